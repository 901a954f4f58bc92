"""GPU parity of the fused ring forward (ring_attn_fwd) against the fp64 oracle,
at sizes the oracle computes in full: several 128-row tiles, ragged shard tails,
both layouts, causal and not, GQA and MHA, d in {64, 128}, and the degenerate
cases of the method."""
import json
import math
import os

import numpy as np
import pytest
import torch

from gpu_helpers import TOL_LSE, TOL_O, compare_full, host32
from online_softmax_merge_gb300.inputs import Workload, make_qkv
from oracle import attention as OA

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


def _run(w: Workload, scale=0.0):
    q, k, v = make_qkv(w)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = ra.fwd(q, k, v, w.P, w.layout, w.causal, scale)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    return q, k, v, o, lse


CASES = [
    # name, B, N, H, G, d, P, layout, causal
    ("gqa-contig-causal-tail", 1, 4 * (3 * 128 + 40), 4, 2, 128, 4, "contiguous", True),
    ("gqa-striped-causal-tail", 1, 4 * (3 * 128 + 40), 4, 2, 128, 4, "striped", True),
    ("gqa-contig-full-tail", 1, 2 * (2 * 128 + 72), 4, 2, 128, 2, "contiguous", False),
    ("gqa-striped-full", 2, 8 * 64, 8, 2, 128, 8, "striped", False),
    ("mha-odd-tiles", 1, 3 * (5 * 128 + 8), 3, 3, 128, 3, "contiguous", True),
    ("gqa3-striped", 1, 2 * (3 * 128 + 1), 6, 2, 128, 2, "striped", True),
    ("d64-contig-causal", 2, 4 * 200, 4, 1, 64, 4, "contiguous", True),
    ("d64-striped-causal", 1, 4 * 300, 2, 2, 64, 4, "striped", True),
    ("p1-plain", 1, 700, 2, 1, 128, 1, "contiguous", True),
    ("s1-every-token-a-shard", 1, 64, 2, 1, 128, 64, "striped", True),
    ("s1-contig", 1, 48, 2, 2, 64, 48, "contiguous", True),
    ("tiny", 1, 5, 2, 2, 128, 1, "contiguous", False),
    ("zigzag-causal-tail", 1, 8 * (128 + 40), 4, 2, 128, 4, "zigzag", True),
    ("zigzag-full-aligned", 1, 4 * 256, 4, 2, 128, 2, "zigzag", False),
    ("zigzag-mha-d64", 2, 6 * 100, 3, 3, 64, 3, "zigzag", True),
    ("zigzag-p1", 1, 2 * 300, 2, 1, 128, 1, "zigzag", True),
    ("zigzag-s2", 1, 64, 4, 2, 128, 32, "zigzag", True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fwd_matches_oracle(case):
    name, B, N, H, G, d, P, layout, causal = case
    w = Workload(name, B, N, H, G, d, P, layout, causal, seed=100 + CASES.index(case))
    q, k, v, o, lse = _run(w)
    eo, el = compare_full(o, lse, q, k, v, causal)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


# Two GPU results are each within TOL of the exact value, so within 2 TOL of
# each other (two bf16 roundings of nearly equal values can differ by an ulp).
def test_contiguous_equals_striped_and_zigzag_on_same_tensors():
    w = Workload("cs", 1, 8 * 192, 4, 2, 128, 8, "contiguous", True, seed=5)
    q, k, v, o1, l1 = _run(w)
    for layout in ("striped", "zigzag"):
        o2, l2 = ra.fwd(q, k, v, w.P, layout, True)
        torch.cuda.synchronize()
        assert float((o1.float() - o2.float()).abs().max()) <= 2 * TOL_O
        assert float((l1 - l2).abs().max()) <= 2 * TOL_LSE


def test_p_invariance_and_p1_is_plain_attention():
    w = Workload("pinv", 1, 1024, 4, 2, 128, 1, "contiguous", True, seed=6)
    q, k, v, o1, l1 = _run(w)
    for P in (2, 4, 8):
        for layout in ("contiguous", "striped"):
            o2, l2 = ra.fwd(q, k, v, P, layout, True)
            torch.cuda.synchronize()
            assert float((o1.float() - o2.float()).abs().max()) <= 2 * TOL_O
            assert float((l1 - l2).abs().max()) <= 2 * TOL_LSE


def test_worked_example_zero_padded():
    """The chapter's printed example (d = 1, raw products as scores), padded to
    d = 64 with zeros and run with scale 1."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))
    q = torch.zeros((1, 4, 1, 64), dtype=torch.bfloat16)
    k = torch.zeros_like(q)
    v = torch.zeros_like(q)
    q[0, :, 0, 0] = torch.tensor(g["Q"], dtype=torch.bfloat16)
    k[0, :, 0, 0] = torch.tensor(g["K"], dtype=torch.bfloat16)
    v[0, :, 0, 0] = torch.tensor(g["V"], dtype=torch.bfloat16)
    o, lse = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), g["P"], "contiguous", False, scale=1.0)
    torch.cuda.synchronize()
    got = host32(o)[0, :, 0, 0]
    want = np.array(g["outputs"]["values"])
    # bf16 rounding of P (2^-9 relative) weighted by |V| <= 40, plus bf16 output rounding
    tol = 2.0 ** -8 * 40 + 2.0 ** -8 * np.abs(want)
    assert np.all(np.abs(got - want) <= tol), (got, want)
    lse_want = [math.log(sum(math.exp(qq * kk) for kk in g["K"])) for qq in g["Q"]]
    assert np.abs(host32(lse)[0, 0] - np.array(lse_want)).max() <= TOL_LSE
    assert np.all(host32(o)[0, :, 0, 1:] == 0)


def test_zero_queries_give_mean_of_visible_values():
    w = Workload("q0", 1, 4 * 160, 2, 1, 128, 4, "striped", True, seed=7)
    q, k, v = make_qkv(w)
    q = torch.zeros_like(q)
    o, lse = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, True)
    torch.cuda.synchronize()
    vv = v[0, :, 0].double()
    mean = torch.cumsum(vv, 0) / torch.arange(1, w.seqlen + 1, dtype=torch.float64)[:, None]
    assert float((o[0, :, 0].cpu().double() - mean).abs().max()) <= TOL_O
    want_lse = torch.log(torch.arange(1, w.seqlen + 1, dtype=torch.float64))
    assert float((lse[0, 0].cpu().double() - want_lse).abs().max()) <= TOL_LSE


def test_constant_values_and_first_token():
    w = Workload("v1", 1, 2 * 256, 4, 2, 128, 2, "contiguous", True, seed=8)
    q, k, v = make_qkv(w)
    ones = torch.ones_like(v)
    o, lse = ra.fwd(q.to(DEV), k.to(DEV), ones.to(DEV), w.P, w.layout, True)
    torch.cuda.synchronize()
    # rows sum to 1 (P is rounded to bf16 for the MMA, the denominator is not)
    assert float((o.float() - 1.0).abs().max()) <= TOL_O
    o, lse = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, True)
    torch.cuda.synchronize()
    assert torch.equal(o[:, 0].cpu(), v[:, 0].repeat_interleave(2, dim=1))   # token 0 sees itself
    s00 = (q[0, 0].double() * k[0, 0].repeat_interleave(2, dim=0).double()).sum(-1) / math.sqrt(128)
    assert float((lse[0, :, 0].cpu().double() - s00).abs().max()) <= TOL_LSE


def test_large_logits_stress():
    # keys scaled x8 on 1% of rows (like the 131072-token stress configuration)
    w = Workload("stress", 1, 4 * 256, 4, 2, 128, 4, "contiguous", True, seed=9,
                 stress_frac=0.05, stress_factor=8.0)
    q, k, v, o, lse = _run(w)
    eo, el = compare_full(o, lse, q, k, v, True)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


def test_repeated_calls_are_deterministic():
    w = Workload("det", 1, 2 * 384, 4, 2, 128, 2, "striped", True, seed=10)
    q, k, v, o1, l1 = _run(w)
    o2, l2 = ra.fwd(q, k, v, w.P, w.layout, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("factor", [4, 16, 64])
def test_large_logits_stay_within_the_arithmetic_bounds(factor):
    """Q and K scaled by `factor` (score spread ~ factor^2), past the configurations'
    inputs. The errors follow the arithmetic, not the N(0, 1) bars:
      * LSE: each score is an fp32 sum of d products, so its rounding error is of the
        order 2^-24 sum_k |q_k k_k| scale; the bound allows 2^-21 of it (8x).
      * O: P is rounded to bf16 for the tensor core (relative 2^-9, at most 2^-9 max|V|
        in O) and O itself to bf16 (half an ulp, at most 2^-8 |O|)."""
    w = Workload("big", 1, 4 * 300, 4, 2, 128, 4, "contiguous", True, 950)
    q, k, v = make_qkv(w)
    q = (q.float() * factor).to(torch.bfloat16)
    k = (k.float() * factor).to(torch.bfloat16)
    o, lse = ra.fwd(q.to(DEV), k.to(DEV), v.to(DEV), w.P, w.layout, w.causal)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    hq, hk, hv = (t.double().numpy() for t in (q, k, v))
    O, L = OA.dense_attention(hq, hk, hv, True)
    scale = 1.0 / np.sqrt(w.head_dim)
    dot_mag = 0.0
    for h in range(w.heads):
        g = h * w.kv_heads // w.heads
        dot_mag = max(dot_mag, float((np.abs(hq[0, :, h]) @ np.abs(hk[0, :, g]).T).max()) * scale)
    el = float(np.abs(host32(lse) - L).max())
    eo = float(np.abs(host32(o) - O).max())
    assert el <= 2.0 ** -21 * dot_mag + 1e-6, (el, dot_mag)
    assert eo <= 2.0 ** -9 * float(np.abs(hv).max()) + 2.0 ** -8 * float(np.abs(O).max()) + 1e-4, eo


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fwd_fp32_output(case):
    """O written as fp32 (RA_DTYPE_F32): within the bar of the oracle, and the bf16
    output of the same call is exactly its rounding to nearest even (one
    computation, two stores)."""
    name, B, N, H, G, d, P, layout, causal = case
    w = Workload(name, B, N, H, G, d, P, layout, causal, seed=100 + CASES.index(case))
    q, k, v, o16, l16 = _run(w)
    o32, l32 = ra.fwd(q, k, v, P, layout, causal, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    assert o32.dtype == torch.float32
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)
    eo, el = compare_full(o32, l32, q, k, v, causal)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)
