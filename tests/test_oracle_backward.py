"""Pins for the backward oracle (oracle/backward.py).

The gradient has a plain definition -- the derivative of the forward -- so the
dense chain rule is pinned to (i) central finite differences of the already
pinned forward oracle, (ii) torch autograd through a plain fp64 softmax
attention built from library ops, and (iii) closed forms and invariants that a
dropped term, a wrong sign or a transposed operand would break.  The backward
ring (the pages' second ring, reverse direction) is then pinned to the dense
gradient for every layout and shard count, and the sampled-row / sampled-key
helpers to the full gradient.
"""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import backward as OB
from oracle import shardmap as OS


def _bf(rng, shape):
    x = torch.from_numpy(rng.standard_normal(shape)).to(torch.bfloat16)
    return x.double().numpy()


def _inputs(seed, B, N, H, G, d):
    rng = np.random.default_rng(seed)
    return (_bf(rng, (B, N, H, d)), _bf(rng, (B, N, G, d)), _bf(rng, (B, N, G, d)),
            _bf(rng, (B, N, H, d)))


# --------------------------------------------------------------------------- #
# (i) finite differences of the forward oracle
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("B,N,H,G,d,causal", [
    (1, 5, 2, 1, 3, True), (1, 5, 2, 1, 3, False), (1, 4, 4, 2, 2, True),
    (2, 3, 2, 2, 4, False)])
def test_grads_match_central_differences(B, N, H, G, d, causal):
    q, k, v, do = _inputs(11, B, N, H, G, d)
    scale = 0.7
    dq, dk, dv = OB.attention_grads(q, k, v, do, causal, scale)

    def loss(q_, k_, v_):
        O, _ = OA.dense_attention(q_, k_, v_, causal, scale)
        return float((O * do).sum())

    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        args = [q.copy(), k.copy(), v.copy()]
        fd = np.zeros_like(args[which])
        for idx in np.ndindex(args[which].shape):
            x0 = args[which][idx]
            args[which][idx] = x0 + eps
            lp = loss(*args)
            args[which][idx] = x0 - eps
            lm = loss(*args)
            args[which][idx] = x0
            fd[idx] = (lp - lm) / (2 * eps)
        assert np.abs(fd - grad).max() <= 1e-7 * max(1.0, np.abs(grad).max()), which


# --------------------------------------------------------------------------- #
# (ii) torch autograd through library softmax, fp64
# --------------------------------------------------------------------------- #

def _torch_attention(q, k, v, causal, scale):
    H, G = q.shape[2], k.shape[2]
    idx = torch.tensor([(h * G) // H for h in range(H)])
    kk, vv = k[:, :, idx], v[:, :, idx]
    S = torch.einsum("bihd,bjhd->bhij", q, kk) * scale
    if causal:
        N = q.shape[1]
        keep = torch.ones(N, N, dtype=torch.bool).tril()
        S = S.masked_fill(~keep, float("-inf"))
    A = torch.softmax(S, dim=-1)
    return torch.einsum("bhij,bjhd->bihd", A, vv)


@pytest.mark.parametrize("B,N,H,G,d,causal", [
    (2, 37, 4, 2, 8, True), (1, 29, 6, 3, 16, False), (1, 40, 8, 1, 4, True)])
def test_grads_match_torch_autograd(B, N, H, G, d, causal):
    q, k, v, do = _inputs(12, B, N, H, G, d)
    scale = 1.0 / np.sqrt(d)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    O = _torch_attention(tq, tk, tv, causal, scale)
    O.backward(torch.from_numpy(do))
    dq, dk, dv = OB.attention_grads(q, k, v, do, causal, scale)
    for ours, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        ref = ref.numpy()
        assert np.abs(ours - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


# --------------------------------------------------------------------------- #
# (iii) closed forms and invariants
# --------------------------------------------------------------------------- #

def test_causal_first_query_has_zero_dq_and_last_key_closed_form():
    """Under the causal mask query 0 sees only key 0, so its softmax weight is
    exactly 1 and dS = 0: dQ_0 = 0.  Key N-1 is seen only by query N-1, with
    weight A[N-1, N-1]: dV_{N-1} = sum over the group's heads of A dO_{N-1}."""
    B, N, H, G, d = 1, 9, 4, 2, 5
    q, k, v, do = _inputs(13, B, N, H, G, d)
    dq, dk, dv = OB.attention_grads(q, k, v, do, True)
    assert np.all(dq[:, 0] == 0.0)
    A = OA.attention_weights(q, k, True)
    for g in range(G):
        want = sum(A[0, h, N - 1, N - 1] * do[0, N - 1, h] for h in range(H) if (h * G) // H == g)
        assert np.abs(dv[0, N - 1, g] - want).max() <= 1e-14


@pytest.mark.parametrize("causal", [True, False])
def test_column_sums(causal):
    """Rows of A sum to 1, so summing dV over keys gives the sum of dO over the
    group's query rows; rows of dS sum to 0, so dK sums to 0 over keys."""
    B, N, H, G, d = 2, 23, 4, 2, 6
    q, k, v, do = _inputs(14, B, N, H, G, d)
    _, dk, dv = OB.attention_grads(q, k, v, do, causal)
    for b in range(B):
        for g in range(G):
            hs = [h for h in range(H) if (h * G) // H == g]
            assert np.abs(dv[b, :, g].sum(0) - do[b][:, hs].sum((0, 1))).max() <= 1e-12
            assert np.abs(dk[b, :, g].sum(0)).max() <= 1e-12


def test_key_shift_invariance():
    """Adding one vector c to every key adds q_i . c to a whole row of scores,
    which the softmax ignores: all three gradients are unchanged (dQ because
    each row of dS sums to 0)."""
    B, N, H, G, d = 1, 17, 2, 1, 4
    q, k, v, do = _inputs(15, B, N, H, G, d)
    c = np.random.default_rng(16).standard_normal(d)
    a = OB.attention_grads(q, k, v, do, True)
    b_ = OB.attention_grads(q, k + c, v, do, True)
    for x, y in zip(a, b_):
        assert np.abs(x - y).max() <= 1e-11


def test_identical_keys_give_zero_dq():
    """With every key equal, each row's weights are uniform over its visible
    keys, independent of q: dQ = 0."""
    B, N, H, G, d = 1, 8, 2, 1, 3
    q, _, v, do = _inputs(17, B, N, H, G, d)
    k = np.broadcast_to(np.arange(1.0, d + 1), (B, N, G, d)).copy()
    dq, _, _ = OB.attention_grads(q, k, v, do, True)
    assert np.abs(dq).max() <= 1e-14


def test_value_gradient_is_linear_in_do():
    B, N, H, G, d = 1, 11, 2, 2, 3
    q, k, v, do = _inputs(18, B, N, H, G, d)
    do2 = np.random.default_rng(19).standard_normal(do.shape)
    g1 = OB.attention_grads(q, k, v, do, True)
    g2 = OB.attention_grads(q, k, v, do2, True)
    g3 = OB.attention_grads(q, k, v, 2.0 * do - do2, True)
    for a, b, c in zip(g1, g2, g3):
        assert np.abs(2.0 * a - b - c).max() <= 1e-12


# --------------------------------------------------------------------------- #
# the backward ring
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("layout", OS.LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_ring_backward_equals_dense(layout, causal, P):
    B, N, H, G, d = 2, 24, 4, 2, 8
    q, k, v, do = _inputs(20 + P, B, N, H, G, d)
    o, lse = OA.dense_attention(q, k, v, causal)
    ring = OB.ring_backward(q, k, v, o, lse, do, P, layout, causal)
    dense = OB.attention_grads(q, k, v, do, causal)
    for a, b in zip(ring, dense):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max())


def test_ring_backward_visits_reverse_ring():
    P = 4
    seen = []
    q, k, v, do = _inputs(30, 1, 8, 1, 1, 2)
    o, lse = OA.dense_attention(q, k, v, True)
    OB.ring_backward(q, k, v, o, lse, do, P, "contiguous", True,
                     trace=lambda bi, h, b, s, u: seen.append((b, s, u)))
    assert len(seen) == P * P
    for b, s, u in seen:
        assert u == (b - s) % P
        assert (u + s) % P == b          # device u holds block (u + s) mod P at step s


def test_ring_backward_any_visit_order():
    """The visit order changes only the summation order."""
    B, N, H, G, d, P = 1, 16, 2, 1, 4, 4
    q, k, v, do = _inputs(31, B, N, H, G, d)
    o, lse = OA.dense_attention(q, k, v, True)
    a = OB.ring_backward(q, k, v, o, lse, do, P, "striped", True)
    b_ = OB.ring_backward(q, k, v, o, lse, do, P, "striped", True,
                          order=lambda b: [(b + s) % P for s in range(P)])
    for x, y in zip(a, b_):
        assert np.abs(x - y).max() <= 1e-13


def test_ring_backward_uses_saved_statistics():
    """The ring takes A from the saved LSE and D from the saved output: a
    wrong LSE or output changes the result (so it does read them)."""
    B, N, H, G, d, P = 1, 8, 1, 1, 4, 2
    q, k, v, do = _inputs(32, B, N, H, G, d)
    o, lse = OA.dense_attention(q, k, v, True)
    ref = OB.ring_backward(q, k, v, o, lse, do, P, "contiguous", True)
    off = OB.ring_backward(q, k, v, o, lse + 0.5, do, P, "contiguous", True)
    assert np.abs(off[2] - np.exp(-0.5) * ref[2]).max() <= 1e-12   # dV scales by e^{-0.5}
    bad_o = OB.ring_backward(q, k, v, 0.0 * o, lse, do, P, "contiguous", True)
    assert np.abs(bad_o[0] - ref[0]).max() > 1e-3


# --------------------------------------------------------------------------- #
# sampled helpers
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("causal", [True, False])
def test_sampled_rows_and_keys_match_full(causal):
    B, N, H, G, d = 2, 40, 4, 2, 8
    q, k, v, do = _inputs(40, B, N, H, G, d)
    dq, dk, dv = OB.attention_grads(q, k, v, do, causal)
    rows, heads = [0, 7, 39], [1, 3]
    got = OB.query_grads_at(rows, heads, q, k, v, do, causal)
    assert np.abs(got - dq[:, rows][:, :, heads]).max() <= 1e-13
    keys = [3, 21, 38, 39]
    gk, gv = OB.key_grads_at(keys, q, k, v, do, causal, rows_per_chunk=7)
    assert np.abs(gk - dk[:, keys]).max() <= 1e-13
    assert np.abs(gv - dv[:, keys]).max() <= 1e-13
