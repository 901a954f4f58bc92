"""GPU parity of the step API (tensor-core and SIMT), finalize and merge.

The step state (m, z, y) is compared with the oracle's ring recurrence after
every step; visiting the steps in any order gives the oracle's dense result;
per-shard partials merged by ring_attn_merge equal the fused forward."""
import itertools

import numpy as np
import pytest
import torch

from gpu_helpers import TOL_LSE, TOL_O, compare_full, host32
from online_softmax_merge_gb300.inputs import Workload, make_merge_inputs, make_qkv
from oracle import merge as OM
from oracle import ring as OR

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def _inputs(w):
    q, k, v = make_qkv(w)
    return q.to(DEV), k.to(DEV), v.to(DEV)


STEP_CASES = [
    Workload("st-contig", 1, 4 * (2 * 128 + 24), 4, 2, 128, 4, "contiguous", True, 21),
    Workload("st-striped", 1, 4 * (2 * 128 + 24), 4, 2, 128, 4, "striped", True, 22),
    Workload("st-full-d64", 1, 3 * 200, 2, 1, 64, 3, "contiguous", False, 23),
    Workload("st-mha", 2, 2 * 300, 3, 3, 128, 2, "striped", True, 24),
    Workload("st-zigzag", 1, 6 * 200, 4, 2, 128, 3, "zigzag", True, 30),
]


@pytest.mark.parametrize("impl", ["tc", "simt"])
@pytest.mark.parametrize("w", STEP_CASES, ids=[w.name for w in STEP_CASES])
def test_step_state_follows_oracle_recurrence(w, impl):
    q, k, v = _inputs(w)
    fn = ra.step if impl == "tc" else ra.step_simt
    state = ra.empty_state(q)
    # oracle states after each step, per (batch, head, shard)
    want = {}

    def trace(b, h, u, s, shard, st):
        want[(b, h, u, s)] = (st.m.copy(), st.z.copy(), st.y.copy())

    OR.ring_attention(host32(q).astype(np.float64), host32(k).astype(np.float64),
                      host32(v).astype(np.float64), w.P, w.layout, w.causal, trace=trace)
    from oracle.shardmap import shard_tokens
    for s in range(w.P):
        fn(q, k, v, w.P, s, state, first=(s == 0), layout=w.layout, causal=w.causal)
        torch.cuda.synchronize()
        m, z, y = (host32(t).astype(np.float64) for t in state)
        for b in range(w.batch):
            for h in range(w.heads):
                for u in range(w.P):
                    tq = shard_tokens(w.layout, w.seqlen, w.P, u)
                    mw, zw, yw = want[(b, h, u, s)]
                    seen = np.isfinite(mw)
                    assert np.array_equal(np.isfinite(m[b, h, tq]), seen)
                    assert np.abs(m[b, h, tq][seen] - mw[seen]).max(initial=0) <= 1e-4
                    assert np.all(z[b, h, tq][~seen] == 0)
                    zr = np.abs(z[b, h, tq][seen] / zw[seen] - 1).max(initial=0)
                    assert zr <= 1e-3, zr
                    on = y[b, tq, h][seen] / z[b, h, tq][seen][:, None]
                    ow = yw[seen] / zw[seen][:, None]
                    assert np.abs(on - ow).max(initial=0) <= TOL_O
    o, lse = ra.finalize(state, w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    eo, el = compare_full(o, lse, q, k, v, w.causal)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_steps_in_any_order_give_dense_result(layout):
    w = Workload("order", 1, 5 * 160, 4, 2, 128, 5, layout, True, 25)
    q, k, v = _inputs(w)
    rng = np.random.default_rng(3)
    outs = []
    for perm in ([0, 1, 2, 3, 4], [4, 3, 2, 1, 0], list(rng.permutation(5))):
        state = ra.empty_state(q)
        for i, s in enumerate(perm):
            ra.step(q, k, v, w.P, int(s), state, first=(i == 0), layout=layout, causal=True)
        o, lse = ra.finalize(state, w.P, layout, True)
        torch.cuda.synchronize()
        eo, el = compare_full(o, lse, q, k, v, True)
        assert eo <= TOL_O and el <= TOL_LSE, (perm, eo, el)
        outs.append((o, lse))
    of, lf = ra.fwd(q, k, v, w.P, layout, True)
    torch.cuda.synchronize()
    for o, lse in outs:
        assert float((o.float() - of.float()).abs().max()) <= 2 * TOL_O
        assert float((lse - lf).abs().max()) <= 2 * TOL_LSE


def test_tc_step_matches_simt_step():
    w = Workload("tcsimt", 1, 2 * 384, 8, 2, 128, 2, "striped", True, 26)
    q, k, v = _inputs(w)
    a, b = ra.empty_state(q), ra.empty_state(q)
    for s in range(w.P):
        ra.step(q, k, v, w.P, s, a, first=(s == 0), layout=w.layout, causal=True)
        ra.step_simt(q, k, v, w.P, s, b, first=(s == 0), layout=w.layout, causal=True)
    oa, la = ra.finalize(a, w.P, w.layout)
    ob, lb = ra.finalize(b, w.P, w.layout)
    torch.cuda.synchronize()
    assert float((oa.float() - ob.float()).abs().max()) <= 2 * TOL_O
    assert float((la - lb).abs().max()) <= 2 * TOL_LSE


def test_finalize_matches_oracle():
    g = torch.Generator().manual_seed(27)
    B, N, H, d = 2, 100, 3, 128
    m = torch.randn((B, H, N), generator=g)
    z = torch.rand((B, H, N), generator=g) * 5 + 0.5
    z[0, 1, :7] = 0.0
    m[0, 1, :7] = -float("inf")
    y = torch.randn((B, N, H, d), generator=g) * 3
    o, lse = ra.finalize((m.to(DEV), z.to(DEV), y.to(DEV)))
    torch.cuda.synchronize()
    Ow, Lw = OM.finalize(m.double().numpy(), z.double().numpy(), y.double().numpy())
    # |O| reaches ~20 here: the bound is bf16 rounding of the output (half an ulp)
    assert np.all(np.abs(host32(o) - Ow) <= 2.0 ** -8 * np.abs(Ow) + 1e-6)
    fin = np.isfinite(Lw)
    got = host32(lse)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - Lw[fin]).max() <= 1e-5


@pytest.mark.parametrize("n,B,N,H,d", [(8, 1, 1000, 4, 128), (16, 2, 257, 3, 64), (1, 1, 64, 2, 128),
                                       (5, 1, 33, 1, 128), (64, 1, 128, 2, 128)])
def test_merge_matches_oracle(n, B, N, H, d):
    o_p, l_p = make_merge_inputs(n, B, N, H, d, seed=n + N)
    l_p[:, 0, 0, :3] = -float("inf")            # a row with every part empty
    o, lse = ra.merge(o_p.to(DEV), l_p.to(DEV))
    torch.cuda.synchronize()
    Ow, Lw = OM.merge(o_p.double().numpy(), l_p.double().numpy())
    assert np.abs(host32(o) - Ow).max() <= TOL_O
    got = host32(lse)
    fin = np.isfinite(Lw)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - Lw[fin]).max() <= 1e-5
    assert np.all(host32(o)[0, :3, 0] == 0)


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_merge_of_oracle_shard_partials_equals_dense(layout):
    w = Workload("mp", 1, 4 * 96, 4, 2, 128, 4, layout, True, 28)
    q, k, v = make_qkv(w)
    Op, Lp = OR.shard_partials(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                               w.P, layout, True)
    o, lse = ra.merge(torch.from_numpy(Op).float().to(DEV), torch.from_numpy(Lp).float().to(DEV))
    torch.cuda.synchronize()
    eo, el = compare_full(o, lse, q.to(DEV), k.to(DEV), v.to(DEV), True)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


def test_gpu_shard_partials_merge_to_fused_forward():
    """Each shard's partial from one GPU step (per virtual device), merged by
    the merge kernel, equals the fused forward."""
    w = Workload("pm", 1, 4 * 160, 4, 2, 128, 4, "contiguous", False, 29)
    q, k, v = _inputs(w)
    parts_o, parts_l = [], []
    for s in range(w.P):
        st = ra.empty_state(q)
        ra.step(q, k, v, w.P, s, st, first=True, layout=w.layout, causal=False)
        o_s, l_s = ra.finalize(st, w.P, w.layout, False)
        parts_o.append(o_s.float())
        parts_l.append(l_s)
    o, lse = ra.merge(torch.stack(parts_o).contiguous(), torch.stack(parts_l).contiguous())
    of, lf = ra.fwd(q, k, v, w.P, w.layout, False)
    torch.cuda.synchronize()
    assert float((o.float() - of.float()).abs().max()) <= 2 * TOL_O
    assert float((lse - lf).abs().max()) <= 2 * TOL_LSE


def test_finalize_fp32_output_matches_oracle():
    g = torch.Generator().manual_seed(31)
    B, N, H, d = 1, 70, 2, 64
    m = torch.randn((B, H, N), generator=g)
    z = torch.rand((B, H, N), generator=g) * 5 + 0.5
    z[0, 0, :3] = 0.0
    m[0, 0, :3] = -float("inf")
    y = torch.randn((B, N, H, d), generator=g) * 3
    st = (m.to(DEV), z.to(DEV), y.to(DEV))
    o32, l32 = ra.finalize(st, out_dtype=torch.float32)
    o16, l16 = ra.finalize(st)
    torch.cuda.synchronize()
    Ow, _ = OM.finalize(m.double().numpy(), z.double().numpy(), y.double().numpy())
    # y * (1/z) in fp32: two roundings of 2^-24 each
    assert np.all(np.abs(host32(o32) - Ow) <= 2.0 ** -22 * np.abs(Ow) + 1e-30)
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)


def test_step_path_fp32_finalize_equals_fused_fp32_forward():
    w = Workload("sf32", 1, 4 * 200, 4, 2, 128, 4, "striped", True, 32)
    q, k, v = _inputs(w)
    st = ra.empty_state(q)
    for s in range(w.P):
        ra.step(q, k, v, w.P, s, st, first=(s == 0), layout=w.layout, causal=True)
    o, lse = ra.finalize(st, w.P, w.layout, out_dtype=torch.float32)
    of, lf = ra.fwd(q, k, v, w.P, w.layout, True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    eo, el = compare_full(o, lse, q, k, v, True)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)
    # same fp32 recurrence, different summation order
    assert float((o - of).abs().max()) <= 1e-3
