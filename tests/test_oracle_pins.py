"""Pins for the oracle: each check ties it to something other than itself.

Printed values from the pages (tests/golden), a library routine for the special
case of plain attention (torch scaled_dot_product_attention / logsumexp in fp64),
closed forms, brute force in pure Python on tiny inputs, and the invariants the
pages state (ring = dense, any visit order, any shard count, rows sum to 1).
"""
import itertools
import json
import math
import os
import random

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import merge as OM
from oracle import ring as OR
from oracle import shardmap as OS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_qkv(rng, B, N, H, G, d):
    """bf16-exact random inputs as fp64 arrays."""
    def bf(shape):
        x = torch.from_numpy(rng.standard_normal(shape)).to(torch.bfloat16)
        return x.double().numpy()
    return bf((B, N, H, d)), bf((B, N, G, d)), bf((B, N, G, d))


# --------------------------------------------------------------------------- #
# Printed worked example ("Ring Attention: Distributed Attention Across
# Devices", "Worked example: tracing the ring by hand").
# --------------------------------------------------------------------------- #

def _worked():
    g = _load("worked_example.json")
    q = np.array(g["Q"], dtype=np.float64).reshape(1, 4, 1, 1)
    k = np.array(g["K"], dtype=np.float64).reshape(1, 4, 1, 1)
    v = np.array(g["V"], dtype=np.float64).reshape(1, 4, 1, 1)
    return g, q, k, v


def test_worked_example_dense_outputs():
    g, q, k, v = _worked()
    O, _ = OA.dense_attention(q, k, v, causal=False, scale=g["scale"])
    tol = 0.5 * 10 ** -g["outputs"]["decimals"]
    assert np.abs(O[0, :, 0, 0] - np.array(g["outputs"]["values"])).max() <= tol


def test_worked_example_dense_intermediates():
    g, q, k, v = _worked()
    A = OA.attention_weights(q, k, causal=False, scale=g["scale"])
    inter = g["q1_dense_intermediates"]
    tol = 0.5 * 10 ** -inter["decimals"]
    # exp(score - max) / Z are the weights; their ratio to the max entry is exp_shifted.
    w = A[0, 0, 0]
    assert np.abs(w / w.max() - np.array(inter["exp_shifted"])).max() <= tol
    assert abs(1.0 / w.max() - inter["Z"]) <= tol


def test_worked_example_ring_outputs_both_orders():
    g, q, k, v = _worked()
    want = np.array(g["outputs"]["values"])
    tol = 0.5 * 10 ** -g["outputs"]["decimals"]
    for order in (None, lambda u: list(reversed(OR.ring_order(u, g["P"])))):
        O, _ = OR.ring_attention(q, k, v, g["P"], "contiguous", causal=False,
                                 scale=g["scale"], order=order)
        assert np.abs(O[0, :, 0, 0] - want).max() <= tol


def test_worked_example_q1_trace():
    g, q, k, v = _worked()
    tr = g["q1_trace"]
    tol = 0.5 * 10 ** -tr["decimals"]
    seen = {}

    def trace(b, h, u, s, shard, st):
        if u == 0:
            seen[s] = (shard, float(st.m[0]), float(st.z[0]), float(st.y[0, 0]))

    O, _ = OR.ring_attention(q, k, v, g["P"], "contiguous", causal=False,
                             scale=g["scale"], trace=trace)
    assert seen[0][0] == 0 and seen[1][0] == 1        # own block first, then the neighbour's
    for s, key in ((0, "after_step0"), (1, "after_step1")):
        _, m, z, y = seen[s]
        assert abs(m - tr[key]["m"]) <= tol
        assert abs(z - tr[key]["l"]) <= tol
        assert abs(y - tr[key]["acc"]) <= tol
    assert abs(O[0, 0, 0, 0] - tr["output"]) <= tol


def test_worked_example_lse_closed_form():
    # q2 = 0: every score is 0, so LSE = ln 4 and O = mean(V) = 25 exactly.
    g, q, k, v = _worked()
    O, L = OA.dense_attention(q, k, v, causal=False, scale=g["scale"])
    assert L[0, 0, 1] == pytest.approx(math.log(4.0), abs=1e-15)
    assert O[0, 1, 0, 0] == pytest.approx(25.0, abs=1e-12)
    # every row: LSE = ln sum_j exp(q_t k_j) by hand
    for t in range(4):
        want = math.log(math.fsum(math.exp(g["Q"][t] * kj) for kj in g["K"]))
        assert L[0, 0, t] == pytest.approx(want, abs=1e-13)


# --------------------------------------------------------------------------- #
# Special case reducing to a library routine: torch SDPA in fp64 on the CPU.
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("B,N,H,G,d,causal,scale", [
    (1, 37, 1, 1, 8, False, None),
    (2, 64, 4, 2, 16, True, None),
    (1, 50, 8, 2, 32, True, 0.3),
    (1, 33, 6, 3, 4, False, None),
    (2, 19, 4, 4, 8, True, 1.0),
    (1, 40, 8, 1, 16, True, None),
])
def test_dense_matches_sdpa_fp64(B, N, H, G, d, causal, scale):
    rng = np.random.default_rng(N * 7 + H)
    q, k, v = _rand_qkv(rng, B, N, H, G, d)
    O, L = OA.dense_attention(q, k, v, causal=causal, scale=scale)
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)                 # [B, H, N, d]
    tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(H // G, dim=1)
    tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(H // G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                           scale=scale)
    assert np.abs(O - ref.permute(0, 2, 1, 3).numpy()).max() < 1e-12
    sc = (1.0 / math.sqrt(d)) if scale is None else scale
    s = torch.matmul(tq, tk.transpose(-1, -2)) * sc
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    lse_ref = torch.logsumexp(s, dim=-1).numpy()
    assert np.abs(L - lse_ref).max() < 1e-12


def test_gqa_mapping_is_grouped_not_strided():
    # kv head = floor(h * G / H): heads 0..3 -> 0, 4..7 -> 1 for H=8, G=2.
    assert [OA.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [OA.kv_head_of(h, 32, 8) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    # GQA equals MHA with kv heads repeated in groups
    rng = np.random.default_rng(3)
    q, k, v = _rand_qkv(rng, 1, 24, 8, 2, 8)
    O, L = OA.dense_attention(q, k, v, causal=True)
    O2, L2 = OA.dense_attention(q, np.repeat(k, 4, axis=2), np.repeat(v, 4, axis=2), causal=True)
    assert np.abs(O - O2).max() == 0.0 and np.abs(L - L2).max() == 0.0


# --------------------------------------------------------------------------- #
# Closed forms.
# --------------------------------------------------------------------------- #

def test_zero_queries_give_mean_of_visible_values():
    rng = np.random.default_rng(5)
    _, k, v = _rand_qkv(rng, 1, 30, 2, 1, 8)
    q = np.zeros((1, 30, 2, 8))
    for causal in (False, True):
        O, L = OA.dense_attention(q, k, v, causal=causal)
        for t in range(30):
            J = t + 1 if causal else 30
            assert np.abs(O[0, t, :, :] - v[0, :J, 0, :].mean(axis=0)).max() < 1e-13
            assert np.abs(L[0, :, t] - math.log(J)).max() < 1e-13


def test_causal_first_token_sees_only_itself():
    rng = np.random.default_rng(6)
    q, k, v = _rand_qkv(rng, 2, 17, 4, 2, 16)
    O, L = OA.dense_attention(q, k, v, causal=True)
    for b in range(2):
        for h in range(4):
            g = OA.kv_head_of(h, 4, 2)
            assert np.abs(O[b, 0, h] - v[b, 0, g]).max() == 0.0
            s00 = float(q[b, 0, h] @ k[b, 0, g]) / 4.0
            assert L[b, h, 0] == pytest.approx(s00, abs=1e-14)


def test_constant_values_give_constant_output():
    rng = np.random.default_rng(7)
    q, k, _ = _rand_qkv(rng, 1, 21, 2, 2, 8)
    v = np.ones((1, 21, 2, 8))
    for causal in (False, True):
        O, _ = OA.dense_attention(q, k, v, causal=causal)
        assert np.abs(O - 1.0).max() < 1e-14


def test_one_hot_values_give_attention_rows_summing_to_one():
    rng = np.random.default_rng(8)
    N = d = 16
    q, k, _ = _rand_qkv(rng, 1, N, 1, 1, d)
    v = np.eye(N).reshape(1, N, 1, d)
    for causal in (False, True):
        O, _ = OA.dense_attention(q, k, v, causal=causal)
        rows = O[0, :, 0, :]
        assert np.abs(rows.sum(axis=1) - 1.0).max() < 1e-12
        if causal:
            assert np.abs(np.triu(rows, 1)).max() == 0.0
        A = OA.attention_weights(q, k, causal=causal)
        assert np.abs(rows - A[0, 0]).max() < 1e-15


def test_shift_invariance():
    # Add c to every score of a row via an extra dimension: q' = [q, 1], k' = [k, c/scale].
    rng = np.random.default_rng(9)
    q, k, v = _rand_qkv(rng, 1, 25, 2, 1, 8)
    scale = 0.25
    c = 3.75
    q2 = np.concatenate([q, np.ones((1, 25, 2, 1))], axis=3)
    k2 = np.concatenate([k, np.full((1, 25, 1, 1), c / scale)], axis=3)
    v2 = v
    for causal in (False, True):
        O, L = OA.dense_attention(q, k, v, causal=causal, scale=scale)
        # pad v to the new width is not needed: v keeps d columns, q/k gain one
        Oa, La = OA.dense_attention(q2, k2, np.concatenate([v2, np.zeros((1, 25, 1, 1))], 3),
                                    causal=causal, scale=scale)
        assert np.abs(Oa[..., :8] - O).max() < 1e-12
        assert np.abs(La - (L + c)).max() < 1e-12
        Or_, Lr = OR.ring_attention(q2, k2, np.concatenate([v2, np.zeros((1, 25, 1, 1))], 3),
                                    5, "striped", causal, scale=scale)
        assert np.abs(Or_[..., :8] - O).max() < 1e-12
        assert np.abs(Lr - (L + c)).max() < 1e-12


# --------------------------------------------------------------------------- #
# Brute force in pure Python (math.fsum) on tiny inputs.
# --------------------------------------------------------------------------- #

def _brute(q, k, v, causal, scale):
    B, N, H, d = q.shape
    G = k.shape[2]
    O = np.zeros_like(q)
    L = np.zeros((B, H, N))
    for b, h, t in itertools.product(range(B), range(H), range(N)):
        g = (h * G) // H
        J = range(t + 1) if causal else range(N)
        s = [scale * math.fsum(float(q[b, t, h, c]) * float(k[b, j, g, c]) for c in range(d))
             for j in J]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        z = math.fsum(e)
        for c in range(d):
            O[b, t, h, c] = math.fsum(ei * float(v[b, j, g, c]) for ei, j in zip(e, J)) / z
        L[b, h, t] = mx + math.log(z)
    return O, L


@pytest.mark.parametrize("N,H,G,d,causal", [(5, 1, 1, 3, False), (9, 2, 1, 4, True),
                                            (12, 4, 2, 2, True), (16, 3, 3, 4, False)])
def test_dense_matches_brute_force(N, H, G, d, causal):
    rng = np.random.default_rng(N + 100 * H)
    q, k, v = _rand_qkv(rng, 1, N, H, G, d)
    scale = 1.0 / math.sqrt(d)
    O, L = OA.dense_attention(q, k, v, causal=causal)
    Ob, Lb = _brute(q, k, v, causal, scale)
    assert np.abs(O - Ob).max() < 1e-12
    assert np.abs(L - Lb).max() < 1e-12


# --------------------------------------------------------------------------- #
# Invariants the pages state: ring = dense, any visit order, any P.
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_ring_equals_dense(layout, causal, P):
    rng = np.random.default_rng(P + 10 * causal)
    q, k, v = _rand_qkv(rng, 2, 48, 4, 2, 8)
    O, L = OA.dense_attention(q, k, v, causal=causal)
    Or_, Lr = OR.ring_attention(q, k, v, P, layout, causal)
    assert np.abs(Or_ - O).max() < 1e-12
    assert np.abs(Lr - L).max() < 1e-12


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_ring_any_visit_order(layout):
    rng = np.random.default_rng(11)
    q, k, v = _rand_qkv(rng, 1, 40, 2, 1, 8)
    P = 5
    O, L = OA.dense_attention(q, k, v, causal=True)
    pr = random.Random(4)
    perms = {u: pr.sample(range(P), P) for u in range(P)}
    Or_, Lr = OR.ring_attention(q, k, v, P, layout, True, order=lambda u: perms[u])
    assert np.abs(Or_ - O).max() < 1e-12
    assert np.abs(Lr - L).max() < 1e-12


def test_ring_fold_order_and_state_scale():
    # The running max after all folds is the row max of the admitted scores.
    rng = np.random.default_rng(12)
    q, k, v = _rand_qkv(rng, 1, 32, 1, 1, 4)
    P = 4
    final = {}

    def trace(b, h, u, s, shard, st):
        if s == P - 1:
            final[u] = st.copy()

    OR.ring_attention(q, k, v, P, "contiguous", True, trace=trace)
    for u in range(P):
        tq = OS.shard_tokens("contiguous", 32, P, u)
        S = (q[0, :, 0, :] @ k[0, :, 0, :].T) * 0.5
        S = np.where(np.arange(32)[None, :] <= np.arange(32)[:, None], S, -np.inf)
        assert np.abs(final[u].m - S[tq].max(axis=1)).max() == 0.0


def test_fold_leaves_unseen_rows_unchanged():
    st = OR.RowState(2, 3)
    S = np.array([[-np.inf, -np.inf], [0.5, -np.inf]])
    V = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    OR.fold(st, S, V)
    assert st.m[0] == -np.inf and st.z[0] == 0.0 and not st.y[0].any()
    assert st.m[1] == 0.5 and st.z[1] == 1.0 and list(st.y[1]) == [1.0, 2.0, 3.0]
    O, L = OR.finalize(st)
    assert not O[0].any() and L[0] == -np.inf
    assert list(O[1]) == [1.0, 2.0, 3.0] and L[1] == 0.5


# --------------------------------------------------------------------------- #
# Merge of partials and finalize.
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("causal", [False, True])
def test_merge_of_shard_partials_equals_dense(layout, causal):
    rng = np.random.default_rng(13)
    q, k, v = _rand_qkv(rng, 1, 36, 4, 2, 8)
    P = 6
    Op, Lp = OR.shard_partials(q, k, v, P, layout, causal)
    if causal:
        assert np.isinf(Lp).any()          # some rows see nothing in a later shard
    O, L = OM.merge(Op, Lp)
    Od, Ld = OA.dense_attention(q, k, v, causal=causal)
    assert np.abs(O - Od).max() < 1e-12
    assert np.abs(L - Ld).max() < 1e-12


def test_merge_closed_forms():
    o = np.random.default_rng(14).standard_normal((2, 1, 3, 1, 4))
    # two parts with equal LSE a: LSE = a + ln 2, O = mean
    lse = np.full((2, 1, 1, 3), 1.25)
    O, L = OM.merge(o, lse)
    assert np.abs(L - (1.25 + math.log(2))).max() < 1e-15
    assert np.abs(O - o.mean(axis=0)).max() < 1e-15
    # weights e^{l1} / (e^{l1} + e^{l2})
    lse = np.stack([np.full((1, 1, 3), 0.0), np.full((1, 1, 3), math.log(3.0))])
    O, L = OM.merge(o, lse)
    assert np.abs(O - (0.25 * o[0] + 0.75 * o[1])).max() < 1e-15
    assert np.abs(L - math.log(4.0)).max() < 1e-15
    # a -inf part contributes nothing; all -inf gives O = 0, LSE = -inf
    lse = np.stack([np.full((1, 1, 3), -np.inf), np.full((1, 1, 3), 2.0)])
    O, L = OM.merge(o, lse)
    assert np.abs(O - o[1]).max() == 0.0 and np.abs(L - 2.0).max() == 0.0
    O, L = OM.merge(o, np.full((2, 1, 1, 3), -np.inf))
    assert not O.any() and np.all(L == -np.inf)
    # a single part is returned unchanged
    O, L = OM.merge(o[:1], lse[1:])
    assert np.abs(O - o[0]).max() == 0.0 and np.abs(L - 2.0).max() == 0.0


def test_finalize_closed_form():
    m = np.array([[[0.5, -np.inf]]])
    z = np.array([[[2.0, 0.0]]])
    y = np.array([[[[4.0, 6.0]], [[1.0, 1.0]]]])      # [B=1, N=2, H=1, d=2]
    O, L = OM.finalize(m, z, y)
    assert list(O[0, 0, 0]) == [2.0, 3.0] and not O[0, 1, 0].any()
    assert L[0, 0, 0] == pytest.approx(0.5 + math.log(2.0), abs=1e-15)
    assert L[0, 0, 1] == -np.inf
