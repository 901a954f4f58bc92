"""Seeded random problem shapes: the forward, the backward, pass-Q decode and the
composed step path against the fp64 oracle over every layout, both head sizes,
GQA/MHA/MQA head groupings, shard lengths that are not multiples of the 128-row
tile, P = 1 and one-token shards. Each shape is drawn from a fixed seed, so a
failure names a reproducible case."""
import numpy as np
import pytest
import torch

from gpu_helpers import TOL_LSE, TOL_O, compare_full, host32
from oracle import backward as OB
from oracle.attention import attention_at
from online_softmax_merge_gb300.inputs import Workload, make_dout, make_qkv

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

N_CASES = 24
TOL_GRAD_MAX = 2.0 ** -6      # the backward's bars (derived in test_gpu_bwd.py)
TOL_GRAD_FRO = 2.0 ** -7


def draw(i: int) -> Workload:
    """Shape i: layout, causal, d, heads/kv heads, P and a shard length up to 400."""
    rng = np.random.default_rng(5000 + i)
    layout = ("contiguous", "striped", "zigzag")[i % 3]
    causal = bool(rng.integers(0, 4))                     # 3 in 4 causal
    d = int(rng.choice([64, 128]))
    G, hpg = [(1, 1), (1, 2), (2, 2), (1, 3), (2, 3), (3, 1), (1, 4), (2, 4)][rng.integers(0, 8)]
    P = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 16]))
    S = int(rng.integers(1, 401))
    if layout == "zigzag":
        S += S % 2                                        # two equal chunks per shard
    B = int(rng.integers(1, 3))
    return Workload(f"fuzz{i}", B, P * S, G * hpg, G, d, P, layout, causal, 6000 + i)


CASES = [draw(i) for i in range(N_CASES)] + [
    # wide head groupings: 64 query heads on one kv head (32 head pairs per CTA group,
    # 64 decode rows per kv head), 48 heads MHA, 64 over 4
    Workload("wide-mqa", 1, 2 * 300, 64, 1, 64, 2, "striped", True, 6100),
    Workload("wide-mha", 1, 3 * 160, 48, 48, 128, 3, "contiguous", True, 6101),
    Workload("wide-gqa16", 2, 4 * 96, 64, 4, 128, 4, "zigzag", True, 6102),
]
IDS = [f"{w.name}-{w.layout}-{'c' if w.causal else 'n'}-d{w.head_dim}-H{w.heads}G{w.kv_heads}"
       f"-P{w.P}-S{w.shard_len}-B{w.batch}" for w in CASES]
WIDE = CASES[N_CASES:]


def test_draws_cover_the_edge_shapes():
    """The fixed draws include each layout, both d, P = 1, a shard shorter than one
    tile, one longer than two tiles with a ragged tail, and MQA."""
    assert {w.layout for w in CASES} == {"contiguous", "striped", "zigzag"}
    assert {w.head_dim for w in CASES} == {64, 128}
    assert any(w.P == 1 for w in CASES)
    assert any(w.shard_len < 128 for w in CASES)
    assert any(w.shard_len > 256 and w.shard_len % 128 for w in CASES)
    assert any(w.kv_heads == 1 and w.heads > 1 for w in CASES)
    assert any(not w.causal for w in CASES)


@pytest.mark.parametrize("w", CASES, ids=IDS)
def test_fuzz_forward_and_backward(w):
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    o, lse = ra.fwd(q, k, v, w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    eo, el = compare_full(o, lse, q, k, v, w.causal)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)

    do = make_dout(w).to(DEV)
    grads = ra.bwd(q, k, v, o, lse, do, w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    hq, hk, hv, hdo = (host32(t).astype(np.float64) for t in (q, k, v, do))
    ref = OB.attention_grads(hq, hk, hv, hdo, w.causal)
    for name, got, r in zip(("dq", "dk", "dv"), grads, ref):
        dlt = host32(got).astype(np.float64) - r
        em = float(np.abs(dlt).max() / max(np.abs(r).max(), 1e-30))
        ef = float(np.linalg.norm(dlt) / max(np.linalg.norm(r), 1e-30))
        assert em <= TOL_GRAD_MAX and ef <= TOL_GRAD_FRO, (name, em, ef)


@pytest.mark.parametrize("w", CASES[:N_CASES:3] + WIDE, ids=IDS[:N_CASES:3] + IDS[N_CASES:])
def test_fuzz_decode(w):
    """The last two tokens (or one, for one-token sequences) as decode queries."""
    _, k, v = make_qkv(w)
    n_q = min(2, w.seqlen)
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn((w.batch, n_q, w.heads, w.head_dim), generator=g).to(torch.bfloat16)
    q_pos0 = w.seqlen - n_q
    o, lse = ra.decode(q.to(DEV), k.to(DEV), v.to(DEV), w.P, q_pos0, w.layout, w.causal)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    rows = np.arange(q_pos0, w.seqlen)
    O_ref, L_ref = attention_at(host32(q), rows, list(range(w.heads)), w.heads, host32(k),
                                host32(v), w.causal)
    assert float(np.abs(host32(o) - O_ref).max()) <= TOL_O
    assert float(np.abs(host32(lse) - L_ref).max()) <= TOL_LSE


@pytest.mark.parametrize("w", CASES[1::4], ids=IDS[1::4])
def test_fuzz_step_path(w):
    """P ring_attn_step calls (state in HBM) and ring_attn_finalize: the same O and
    LSE as the oracle."""
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    state = ra.empty_state(q)
    for s in range(w.P):
        ra.step(q, k, v, w.P, s, state, s == 0, w.layout, w.causal)
    o, lse = ra.finalize(state, w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    eo, el = compare_full(o, lse, q, k, v, w.causal)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)
