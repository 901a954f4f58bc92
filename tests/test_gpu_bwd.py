"""Parity of the backward ring (ring_attn_bwd) with the gradient oracle.

Tolerance, per gradient tensor, derived from the arithmetic: the kernels round
the probabilities A and the products dS to bf16 before the tensor-core
contractions, accumulate in fp32 and write bf16 results -- each a relative
rounding of at most u = 2^-9. Replaying exactly those roundings on the CPU gives
at most 2.8u of max|ref| (elementwise) and of ||ref||_F on the stress inputs
(1.2u on plain ones). The bar: max|d| <= 2^-6 max|ref| (8u) and
||d||_F <= 2^-7 ||ref||_F (4u). Comparisons of two GPU results (different
layouts, i.e. different summation orders) allow twice that.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import host32
from oracle import attention as OA
from oracle import backward as OB
from online_softmax_merge_gb300.inputs import WORKLOADS, Workload, make_dout, make_qkv

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

TOL_MAX = 2.0 ** -6
TOL_FRO = 2.0 ** -7

CASES = [
    Workload("gqa-contig-causal-tail", 1, 4 * (3 * 128 + 40), 4, 2, 128, 4, "contiguous", True, 200),
    Workload("gqa-striped-causal-tail", 1, 4 * (3 * 128 + 40), 4, 2, 128, 4, "striped", True, 201),
    Workload("zigzag-causal", 1, 8 * (2 * 128 + 40), 2, 1, 128, 4, "zigzag", True, 202),
    Workload("zigzag-noncausal-d64", 1, 4 * (128 + 20), 2, 2, 64, 2, "zigzag", False, 203),
    Workload("mha-noncausal-d64-b2", 2, 2 * (2 * 128 + 7), 2, 2, 64, 2, "contiguous", False, 204),
    Workload("gqa3-striped", 1, 2 * (3 * 128 + 1), 6, 2, 128, 2, "striped", True, 205),
    Workload("p1-causal", 1, 300, 2, 1, 128, 1, "contiguous", True, 206),
    Workload("tiny", 1, 8, 2, 1, 64, 2, "contiguous", True, 207),
    Workload("stress", 1, 4 * 256, 4, 2, 128, 4, "contiguous", True, 9,
             stress_frac=0.05, stress_factor=8.0),
    # degenerate shapes: every token its own shard, a single partial tile, odd tile
    # counts with MHA, one-token zigzag chunks
    Workload("s1-every-token-a-shard", 1, 64, 2, 1, 128, 64, "striped", True, 212),
    Workload("tiny-noncausal", 1, 5, 2, 2, 128, 1, "contiguous", False, 213),
    Workload("mha-odd-tiles", 1, 3 * (5 * 128 + 8), 3, 3, 128, 3, "contiguous", True, 214),
    Workload("zigzag-s2", 1, 64, 4, 2, 128, 32, "zigzag", True, 215),
    Workload("d64-striped-causal", 1, 4 * 300, 2, 2, 64, 4, "striped", True, 216),
]


def grad_errors(got: np.ndarray, ref: np.ndarray):
    """(max|got - ref| / max|ref|, ||got - ref||_F / ||ref||_F)."""
    d = got.astype(np.float64) - ref
    return (float(np.abs(d).max() / max(np.abs(ref).max(), 1e-30)),
            float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)))


def assert_close(got, ref, name, scale=1.0):
    em, ef = grad_errors(got, ref)
    assert em <= scale * TOL_MAX and ef <= scale * TOL_FRO, (name, em, ef)


def _inputs(w):
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    do = make_dout(w).to(DEV)
    return q, k, v, do


def _bwd(w, q, k, v, o, lse, do, layout=None):
    dq, dk, dv = ra.bwd(q, k, v, o, lse, do, w.P, layout or w.layout, w.causal)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    return dq, dk, dv


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_bwd_from_oracle_statistics(w):
    """The backward alone: O (rounded to bf16) and LSE come from the oracle."""
    q, k, v, do = _inputs(w)
    hq, hk, hv, hdo = (host32(t).astype(np.float64) for t in (q, k, v, do))
    O, LSE = OA.dense_attention(hq, hk, hv, w.causal)
    o = torch.from_numpy(O).to(torch.bfloat16).to(DEV)
    lse = torch.from_numpy(LSE).to(torch.float32).to(DEV)
    dq, dk, dv = _bwd(w, q, k, v, o, lse, do)
    ref = OB.attention_grads(hq, hk, hv, hdo, w.causal)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(host32(got), r, name)


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_bwd_after_gpu_forward(w):
    """The training path: the GPU forward's O and LSE feed the GPU backward."""
    q, k, v, do = _inputs(w)
    o, lse = ra.fwd(q, k, v, w.P, w.layout, w.causal)
    dq, dk, dv = _bwd(w, q, k, v, o, lse, do)
    hq, hk, hv, hdo = (host32(t).astype(np.float64) for t in (q, k, v, do))
    ref = OB.attention_grads(hq, hk, hv, hdo, w.causal)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(host32(got), r, name)


@pytest.mark.parametrize("w", [CASES[1], CASES[3], CASES[8]], ids=["striped", "zigzag-d64", "stress"])
def test_bwd_from_fp32_forward_output(w):
    """The saved O may be the forward's fp32 output (RA_DTYPE_F32): the statistics
    pass reads it as fp32."""
    q, k, v, do = _inputs(w)
    o, lse = ra.fwd(q, k, v, w.P, w.layout, w.causal, out_dtype=torch.float32)
    dq, dk, dv = _bwd(w, q, k, v, o, lse, do)
    hq, hk, hv, hdo = (host32(t).astype(np.float64) for t in (q, k, v, do))
    ref = OB.attention_grads(hq, hk, hv, hdo, w.causal)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(host32(got), r, name)


def test_bwd_layouts_agree_and_runs_are_deterministic():
    w = Workload("gqa", 1, 8 * (128 + 84), 4, 2, 128, 4, "contiguous", True, 210)
    q, k, v, do = _inputs(w)
    outs = {}
    for layout in ("contiguous", "striped", "zigzag"):
        o, lse = ra.fwd(q, k, v, w.P, layout, True)
        outs[layout] = _bwd(w, q, k, v, o, lse, do, layout)
        again = _bwd(w, q, k, v, o, lse, do, layout)
        for a, b in zip(outs[layout], again):
            assert torch.equal(a, b), layout          # no atomics: bit-identical reruns
    for layout in ("striped", "zigzag"):
        for name, a, b in zip(("dq", "dk", "dv"), outs["contiguous"], outs[layout]):
            assert_close(host32(b), host32(a).astype(np.float64), name + "/" + layout, scale=2.0)


def test_bwd_rows_without_keys_and_outputs_fully_written():
    """A row whose saved LSE is -inf contributes nothing, and every output
    element is overwritten (buffers start as NaN)."""
    w = Workload("t", 1, 2 * 200, 2, 1, 128, 2, "striped", True, 211)
    q, k, v, do = _inputs(w)
    o, lse = ra.fwd(q, k, v, w.P, w.layout, True)
    lse2 = lse.clone()
    lse2[:, :, 17] = -float("inf")
    nan = float("nan")
    dq = torch.full_like(q, nan)
    dk = torch.full_like(k, nan)
    dv = torch.full_like(v, nan)
    ra.bwd(q, k, v, o, lse2, do, w.P, w.layout, True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    for t in (dq, dk, dv):
        assert not torch.isnan(t).any()
    assert float(dq[:, 17].float().abs().max()) == 0.0
    # the same gradients as dropping row 17's upstream gradient, up to rounding
    do0 = do.clone()
    do0[:, 17] = 0
    dq0, dk0, dv0 = ra.bwd(q, k, v, o, lse, do0, w.P, w.layout, True)
    torch.cuda.synchronize()
    for a, b in ((dk, dk0), (dv, dv0)):
        assert_close(host32(a), host32(b).astype(np.float64), "no-key row", scale=2.0)


def _sampled(w, rows, keys, groups):
    """Full-size run; for batch 0 and the listed kv heads, dQ is checked on
    sampled query rows of every query head of the group and dK/dV on sampled
    keys (the oracle sums over every query row that sees them). One group is an
    exact sub-problem: its query heads, its kv head."""
    q, k, v = make_qkv(w, device=DEV)
    do = make_dout(w, device=DEV)
    o, lse = ra.fwd(q, k, v, w.P, w.layout, w.causal)
    dq, dk, dv = _bwd(w, q, k, v, o, lse, do)
    hpg = w.heads // w.kv_heads
    for g in groups:
        hs = slice(g * hpg, (g + 1) * hpg)
        hq = host32(q[:1, :, hs]).astype(np.float64)
        hk = host32(k[:1, :, g:g + 1]).astype(np.float64)
        hv = host32(v[:1, :, g:g + 1]).astype(np.float64)
        hdo = host32(do[:1, :, hs]).astype(np.float64)
        ref_q = OB.query_grads_at(rows, range(hpg), hq, hk, hv, hdo, w.causal)
        assert_close(host32(dq[:1, rows, hs]), ref_q, f"dq g={g}")
        ref_k, ref_v = OB.key_grads_at(keys, hq, hk, hv, hdo, w.causal)
        assert_close(host32(dk[:1, keys, g:g + 1]), ref_k, f"dk g={g}")
        assert_close(host32(dv[:1, keys, g:g + 1]), ref_v, f"dv g={g}")


def test_bwd_c2_sampled():
    w = WORKLOADS["c2"]
    N = w.seqlen
    rng = np.random.default_rng(12)
    rows = sorted({0, 1, 127, 128, N // 2, N - 1} | set(rng.integers(0, N, 6).tolist()))
    keys = [N - 1, N - 2, N - 129, N - 400]
    _sampled(w, rows, keys, groups=[0, w.kv_heads - 1])


def test_bwd_c4_sampled():
    w = WORKLOADS["c4"]
    N = w.seqlen
    rng = np.random.default_rng(14)
    rows = sorted({0, 8191, 8192, N - 1} | set(rng.integers(0, N, 4).tolist()))
    keys = [N - 1, N - 128, N - 300]
    _sampled(w, rows, keys, groups=[3])


def test_bwd_c4_shape_at_head_size_64_sampled():
    """d = 64 on the c4 shape: both backward kernels keep a second score buffer there
    (and dK/dV a third Q/dO stage)."""
    w = WORKLOADS["c4"].with_(head_dim=64)
    N = w.seqlen
    rng = np.random.default_rng(16)
    rows = sorted({0, 8191, 8192, N - 1} | set(rng.integers(0, N, 4).tolist()))
    keys = [N - 1, N - 128, N - 300]
    _sampled(w, rows, keys, groups=[0, 6])


def test_bwd_c4_zigzag_sampled():
    """The c4 workload with the zigzag layout: every shard holds two chunks, so each
    key tile meets the queries of both of its shard's segments."""
    w = WORKLOADS["c4"].with_(layout="zigzag")
    N = w.seqlen
    rng = np.random.default_rng(17)
    chunk = N // (2 * w.P)
    rows = sorted({0, chunk - 1, chunk, N - chunk, N - 1} | set(rng.integers(0, N, 4).tolist()))
    # late keys (the oracle's cost grows with the queries that see a key) in the last two
    # chunks, which belong to different shards: chunk 2P-1 to shard 0, chunk 2P-2 to shard 1
    keys = [N - 1, N - 100, N - chunk - 1]
    _sampled(w, rows, keys, groups=[2])


def test_bwd_c3_striped_sampled():
    w = WORKLOADS["c3"]
    N = w.seqlen
    rng = np.random.default_rng(13)
    # first and last tokens of a few shards, plus random rows
    rows = sorted({0, w.P - 1, w.P, N - 1, N - w.P} | set(rng.integers(0, N, 5).tolist()))
    keys = [N - 1, N - 2, N - 17, N - 300]
    _sampled(w, rows, keys, groups=[5])


def test_bwd_c5_one_million_tokens_sampled():
    """The largest workload (1,048,576 tokens, striped over 64 shards): the backward
    from the GPU forward, checked on sampled query rows and on the last keys."""
    w = WORKLOADS["c5"]
    N = w.seqlen
    rng = np.random.default_rng(15)
    rows = sorted({0, w.P, N - 1} | set(rng.integers(0, N, 3).tolist()))
    keys = [N - 1, N - 65, N - 200]
    _sampled(w, rows, keys, groups=[7])


@pytest.mark.parametrize("scale,layout,d", [(0.05, "contiguous", 128), (0.3, "striped", 128),
                                            (0.5, "zigzag", 64)])
def test_fwd_and_bwd_with_explicit_scale(scale, layout, d):
    """A score scale other than 1/sqrt(d): the forward's O and LSE and all three
    gradients follow the oracle run with the same scale (the backward folds
    -LSE/scale into its products, so a wrong scale anywhere shows here)."""
    w = Workload("scale", 1, 4 * (2 * 128 + 40), 4, 2, d, 4, layout, True, 217)
    q, k, v, do = _inputs(w)
    o, lse = ra.fwd(q, k, v, w.P, w.layout, w.causal, scale)
    dq, dk, dv = ra.bwd(q, k, v, o, lse, do, w.P, w.layout, w.causal, scale)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    hq, hk, hv, hdo = (host32(t).astype(np.float64) for t in (q, k, v, do))
    O, LSE = OA.dense_attention(hq, hk, hv, w.causal, scale=scale)
    assert np.abs(host32(o) - O).max() <= 1e-2
    assert np.abs(host32(lse) - LSE).max() <= 1e-3
    ref = OB.attention_grads(hq, hk, hv, hdo, w.causal, scale=scale)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(host32(got), r, name)
