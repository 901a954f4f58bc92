"""Parity at the five measured configurations, in the launch configuration the
bench times (one ring_attn_fwd call on the full-size inputs).

Every call runs twice, once writing O as fp32 and once as bf16. The two are one
computation with two stores, so the bf16 output must be exactly the fp32 output
rounded to nearest even, over the whole tensor; the fp32 output is then held to the
stated bars against the fp64 oracle (O max-abs 1e-2, LSE max-abs 1e-3), and the
bf16 output to the same bar plus the half unit in the last place that its own
rounding adds at each |O|.

The 1024-token configuration is checked on every row, the 32768-token one on every
row of three heads (one in each of three kv groups) and, like the larger ones, on
sampled rows, each computed exactly by the oracle, per (sequence, query head) for
every head: the first and last local row of every shard, 256 seeded random rows,
and the 16 rows with the largest |O| in the output; the configuration with 1% of its
keys scaled by 8 adds the 16 rows with the largest LSE (their largest score sits on a
scaled key, which the test confirms) and 16 of the scaled positions themselves --
the large-logit rows where the running max is rescaled hardest ("Ring Attention:
what the near-infinite context paper actually says", "Failure modes in practice").
The GPU output only chooses rows; the oracle computes every checked value.
"""
import json
import os

import numpy as np
import pytest
import torch

from gpu_helpers import TOL_LSE, TOL_O, compare_full, edge_rows
from online_softmax_merge_gb300.inputs import WORKLOADS, make_qkv, stress_positions
from oracle.attention import kv_head_of
from oracle_pool import bf16_half_ulp, errors, gather_rows, oracle_rows, row_sets

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

N_RANDOM = 256
N_TOP = 16
FULL_HEADS_C2 = (0, 13, 31)


def _report(name, **kw):
    """Appends the measured maxima to the file RA_PARITY_REPORT names, if set."""
    path = os.environ.get("RA_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"config": name, **kw}) + "\n")


def _fwd_both(w, q, k, v, layout):
    o32, l32 = ra.fwd(q, k, v, w.P, layout, w.causal, out_dtype=torch.float32)
    o16, l16 = ra.fwd(q, k, v, w.P, layout, w.causal)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    # one computation, two stores: bf16 = the fp32 result rounded to nearest even
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(l16, l32)
    return o32, o16, l32


def _select(w, layout, o32, lse, seed, stress=None):
    """Rows to check for every (b, h): shard edges, seeded random rows, the largest
    |O| rows and, with stress positions, the largest-LSE rows and stressed positions."""
    B, N, H = w.batch, w.seqlen, w.heads
    edges = sorted(edge_rows(layout, N, w.P))
    amax = torch.maximum(o32.amax(3), -o32.amin(3))                   # [B, N, H]
    top_o = amax.permute(0, 2, 1).topk(N_TOP, dim=2).indices.cpu().numpy()
    top_l = lse.topk(N_TOP, dim=2).indices.cpu().numpy() if stress is not None else None
    sel, picked = {}, {}
    for b in range(B):
        for h in range(H):
            rng = np.random.default_rng(seed * 100003 + b * H + h)
            r = set(edges)
            r.update(int(x) for x in rng.integers(0, N, N_RANDOM))
            r.update(int(x) for x in top_o[b, h])
            if stress is not None:
                r.update(int(x) for x in top_l[b, h])
                sp = stress[b].numpy()
                r.update(int(x) for x in rng.choice(sp, size=min(N_TOP, len(sp)), replace=False))
                picked[(b, h)] = top_l[b, h]
            sel[(b, h)] = np.array(sorted(r), dtype=np.int64)
    return sel, picked


def _check_sampled(name, w, layout, q, k, v, o32, o16, lse, sel):
    k_host = k.float().cpu().numpy()
    v_host = v.float().cpu().numpy()
    ref = oracle_rows(k_host, v_host, w.heads, row_sets(q, sel), w.causal)
    o32r = gather_rows(o32, sel, "bnhd")
    o16r = gather_rows(o16, sel, "bnhd")
    lr = gather_rows(lse, sel, "bhn")
    eo, el = errors(o32r, lr, ref)
    eo16, _ = errors(o16r, lr, ref)
    # bf16: the bar plus the half ulp its rounding adds at the exact value's size
    # (at the size of the rounded fp32 value, which is within 1e-2 of the exact one)
    excess = max(float((np.abs(o16r[x] - ref[x][0]) -
                        bf16_half_ulp(np.abs(ref[x][0]) + TOL_O)).max()) for x in ref)
    over = sum(int((np.abs(o16r[x] - ref[x][0]) > TOL_O).sum()) for x in ref)
    omax = max(float(np.abs(ref[x][0]).max()) for x in ref)
    n_rows = sum(len(s) for s in sel.values())
    _report(name, layout=layout, rows=n_rows, max_abs_o_fp32=eo, max_abs_lse=el,
            max_abs_o_bf16=eo16, bf16_elements_over_1e2=over, max_abs_o_ref=omax,
            bf16_excess_over_half_ulp=excess)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)
    assert excess <= TOL_O, excess
    return ref


def test_c1_full():
    w = WORKLOADS["c1"]
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    o32, o16, lse = _fwd_both(w, q, k, v, w.layout)
    eo, el = compare_full(o32, lse, q, k, v, w.causal)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)
    eo16, _ = compare_full(o16, lse, q, k, v, w.causal)
    _report("c1", layout=w.layout, rows="all", max_abs_o_fp32=eo, max_abs_lse=el,
            max_abs_o_bf16=eo16)
    assert eo16 <= TOL_O


def test_c2_sampled_and_three_heads_in_full():
    w = WORKLOADS["c2"]
    q, k, v = make_qkv(w, device=DEV)
    o32, o16, lse = _fwd_both(w, q, k, v, w.layout)
    sel, _ = _select(w, w.layout, o32, lse, seed=20)
    for h in FULL_HEADS_C2:                 # every row of three heads (three kv groups)
        sel[(0, h)] = np.arange(w.seqlen)
    _check_sampled("c2", w, w.layout, q, k, v, o32, o16, lse, sel)


def test_c3_three_layouts_on_same_tensors():
    w = WORKLOADS["c3"]
    q, k, v = make_qkv(w, device=DEV)
    out = {}
    for i, layout in enumerate(("striped", "contiguous", "zigzag")):
        o32, o16, lse = _fwd_both(w, q, k, v, layout)
        sel, _ = _select(w, layout, o32, lse, seed=30 + i)
        _check_sampled("c3", w, layout, q, k, v, o32, o16, lse, sel)
        out[layout] = (o32, lse)
        del o16
    # the layout is an index map: every order of the same ring reaches the same result
    for layout in ("contiguous", "zigzag"):
        assert float((out["striped"][0] - out[layout][0]).abs().max()) <= 2 * TOL_O
        assert float((out["striped"][1] - out[layout][1]).abs().max()) <= 2 * TOL_LSE


def _argmax_keys(q, k, w, b, h, rows):
    """Key position of each row's largest score (fp32 on the GPU, causal): used only
    to confirm what kind of rows the selection picked."""
    g = kv_head_of(h, w.heads, w.kv_heads)
    rows_t = torch.as_tensor(rows, device=q.device)
    s = q[b, rows_t, h].float() @ k[b, :, g].float().T                  # [R, N]
    keys = torch.arange(w.seqlen, device=q.device)
    s = s.masked_fill(keys[None, :] > rows_t[:, None], float("-inf"))
    return s.argmax(dim=1).cpu().numpy()


def test_c4_sampled_with_stress_rows():
    w = WORKLOADS["c4"]
    q, k, v = make_qkv(w, device=DEV)
    o32, o16, lse = _fwd_both(w, q, k, v, w.layout)
    stress = stress_positions(w)
    sel, picked = _select(w, w.layout, o32, lse, seed=40, stress=stress)
    # the largest-LSE rows are rows whose largest score sits on a x8 key
    on_stress, total = 0, 0
    for (b, h), rows in picked.items():
        am = _argmax_keys(q, k, w, b, h, rows)
        on_stress += int(np.isin(am, stress[b].numpy()).sum())
        total += len(rows)
    assert on_stress >= 0.9 * total, (on_stress, total)
    _check_sampled("c4", w, w.layout, q, k, v, o32, o16, lse, sel)


def test_c4_shape_at_head_size_64():
    """The c4 workload at d = 64, where the kernel keeps a third score buffer in the
    TMEM columns O leaves free: the same sample, stress rows included."""
    w = WORKLOADS["c4"].with_(head_dim=64)
    q, k, v = make_qkv(w, device=DEV)
    o32, o16, lse = _fwd_both(w, q, k, v, w.layout)
    sel, _ = _select(w, w.layout, o32, lse, seed=44, stress=stress_positions(w))
    _check_sampled("c4-d64", w, w.layout, q, k, v, o32, o16, lse, sel)


def test_c5_sampled():
    w = WORKLOADS["c5"]
    q, k, v = make_qkv(w, device=DEV)
    o32, o16, lse = _fwd_both(w, q, k, v, w.layout)
    sel, _ = _select(w, w.layout, o32, lse, seed=50)
    _check_sampled("c5", w, w.layout, q, k, v, o32, o16, lse, sel)
