"""The device entry points inside CUDA graphs: every call is stream-ordered, with no
host synchronisation or allocation in the library once a device has made its
first eager call, so a caller can capture it (a decode loop, a training step) and
replay it. A replay must give the eager result bit for bit, also after new inputs
were copied into the captured buffers."""
import pytest
import torch

from online_softmax_merge_gb300.inputs import Workload, make_dout, make_merge_inputs, make_qkv

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def capture(fn):
    """One eager call on a side stream, then fn captured into a graph."""
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream(DEV).wait_stream(side)
    torch.cuda.synchronize(DEV)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize(DEV)
    return g


def replay(g, outs):
    for t in outs:
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize(DEV)
    assert ra.last_error(DEV) == 0
    return [t.clone() for t in outs]


W = Workload("graph", 2, 4 * (2 * 128 + 40), 4, 2, 128, 4, "striped", True, 700)


def test_forward_graph_replays_bit_exact():
    q, k, v = (t.to(DEV) for t in make_qkv(W))
    o = torch.empty_like(q)
    lse = torch.empty((W.batch, W.heads, W.seqlen), dtype=torch.float32, device=DEV)
    g = capture(lambda: ra.fwd(q, k, v, W.P, W.layout, W.causal, out=o, lse=lse))
    for seed in (None, 701):
        if seed is not None:                      # new inputs into the captured buffers
            q2, k2, v2 = make_qkv(W, seed=seed)
            q.copy_(q2)
            k.copy_(k2)
            v.copy_(v2)
        got = replay(g, [o, lse])
        ref = ra.fwd(q, k, v, W.P, W.layout, W.causal)
        torch.cuda.synchronize(DEV)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


def test_backward_graph_replays_bit_exact():
    q, k, v = (t.to(DEV) for t in make_qkv(W))
    do = make_dout(W).to(DEV)
    o, lse = ra.fwd(q, k, v, W.P, W.layout, W.causal)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = ra.bwd_workspace_bytes(W.batch, W.seqlen, W.heads, W.kv_heads, W.head_dim, W.P,
                                  W.layout, W.causal)
    ws = torch.empty(need // 4 + 4, dtype=torch.float32, device=DEV)
    g = capture(lambda: ra.bwd(q, k, v, o, lse, do, W.P, W.layout, W.causal, dq=dq, dk=dk,
                               dv=dv, workspace=ws))
    got = replay(g, [dq, dk, dv])
    ref = ra.bwd(q, k, v, o, lse, do, W.P, W.layout, W.causal)
    torch.cuda.synchronize(DEV)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


# P = 4: four partials per row group, merged inside a thread-block cluster (one launch);
# P = 16: sixteen partials, through the workspace and the merge kernel (two launches)
@pytest.mark.parametrize("P", [4, 16])
def test_decode_graph_replays_bit_exact(P):
    w = W.with_(P=P)                              # 1184 tokens: 296 per shard at P = 4, 74 at 16
    _, k, v = (t.to(DEV) for t in make_qkv(w))
    n_q = 2
    gen = torch.Generator(device="cpu").manual_seed(702)
    qd = torch.randn((w.batch, n_q, w.heads, w.head_dim), generator=gen).to(torch.bfloat16).to(DEV)
    need = ra.decode_workspace_bytes(w.batch, w.seqlen, w.heads, w.kv_heads, w.head_dim, w.P,
                                     n_q, w.layout, w.causal)
    ws = torch.empty(need // 4 + 4, dtype=torch.float32, device=DEV)
    o = torch.empty_like(qd)
    lse = torch.empty((w.batch, w.heads, n_q), dtype=torch.float32, device=DEV)
    pos = w.seqlen - n_q
    g = capture(lambda: ra.decode(qd, k, v, w.P, pos, w.layout, w.causal, workspace=ws, out=o,
                                  lse=lse))
    for step in range(2):
        if step:                                  # the next token's query
            qd.copy_(torch.randn(qd.shape, generator=gen).to(torch.bfloat16))
        got = replay(g, [o, lse])
        ref = ra.decode(qd, k, v, w.P, pos, w.layout, w.causal)
        torch.cuda.synchronize(DEV)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


def test_fp32_output_forward_graph_replays_bit_exact():
    q, k, v = (t.to(DEV) for t in make_qkv(W))
    o = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    lse = torch.empty((W.batch, W.heads, W.seqlen), dtype=torch.float32, device=DEV)
    g = capture(lambda: ra.fwd(q, k, v, W.P, W.layout, W.causal, out=o, lse=lse,
                               out_dtype=torch.float32))
    got = replay(g, [o, lse])
    ref = ra.fwd(q, k, v, W.P, W.layout, W.causal, out_dtype=torch.float32)
    torch.cuda.synchronize(DEV)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


def test_merge_and_step_path_graphs_replay_bit_exact():
    o_p, l_p = make_merge_inputs(4, 1, 1000, 8, 128, device=DEV, seed=703)
    mo = torch.empty((1, 1000, 8, 128), dtype=torch.bfloat16, device=DEV)
    ml = torch.empty((1, 8, 1000), dtype=torch.float32, device=DEV)
    g = capture(lambda: ra.merge(o_p, l_p, out=mo, lse=ml))
    got = replay(g, [mo, ml])
    ref = ra.merge(o_p, l_p)
    torch.cuda.synchronize(DEV)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])

    q, k, v = (t.to(DEV) for t in make_qkv(W))
    state = ra.empty_state(q)
    so = torch.empty_like(q)
    sl = torch.empty((W.batch, W.heads, W.seqlen), dtype=torch.float32, device=DEV)

    def composed():
        for s in range(W.P):
            ra.step(q, k, v, W.P, s, state, s == 0, W.layout, W.causal)
        ra.finalize(state, W.P, W.layout, W.causal, out=so, lse=sl)

    g = capture(composed)
    got = replay(g, [so, sl])
    state2 = ra.empty_state(q)
    for s in range(W.P):
        ra.step(q, k, v, W.P, s, state2, s == 0, W.layout, W.causal)
    ref = ra.finalize(state2, W.P, W.layout, W.causal)
    torch.cuda.synchronize(DEV)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
