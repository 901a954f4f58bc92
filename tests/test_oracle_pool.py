"""The worker-pool runner of the oracle (tests/oracle_pool.py), on the CPU: on
sampled rows of a small causal GQA problem it returns what the oracle returns
when called once on the whole problem, so the parity tests that use it at full
size check against the oracle itself."""
import numpy as np
import pytest
import torch

from online_softmax_merge_gb300.inputs import Workload, make_qkv
from oracle.attention import dense_attention
from oracle_pool import bf16_half_ulp, gather_rows, oracle_rows, row_sets


@pytest.mark.parametrize("workers", [3, 8])
def test_pool_rows_equal_the_oracle_on_the_whole_problem(workers):
    w = Workload("pool", 2, 1536, 4, 2, 64, 4, "contiguous", True, seed=77,
                 stress_frac=0.02, stress_factor=8.0)
    q, k, v = make_qkv(w)
    rng = np.random.default_rng(0)
    sel = {(b, h): np.unique(np.concatenate([rng.integers(0, w.seqlen, 700), [0, w.seqlen - 1]]))
           for b in range(w.batch) for h in range(w.heads)}
    got = oracle_rows(k.float().numpy(), v.float().numpy(), w.heads, row_sets(q, sel), True,
                      workers=workers)
    O, L = dense_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), True)
    for (b, h), rows in sel.items():
        o, lse = got[(b, h)]
        assert np.abs(o - O[b, rows, h]).max() <= 1e-12
        assert np.abs(lse - L[b, h, rows]).max() <= 1e-12


def test_pool_non_causal_and_gather():
    w = Workload("pool2", 1, 300, 3, 1, 64, 3, "striped", False, seed=78)
    q, k, v = make_qkv(w)
    sel = {(0, h): np.array([5, 0, 299, 17]) for h in range(3)}
    got = oracle_rows(k.float().numpy(), v.float().numpy(), 3, row_sets(q, sel), False, workers=1)
    O, L = dense_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(), False)
    qs = gather_rows(q, sel, "bnhd")
    for h in range(3):
        assert np.abs(got[(0, h)][0] - O[0, [5, 0, 299, 17], h]).max() <= 1e-12
        assert np.array_equal(qs[(0, h)], q[0, [5, 0, 299, 17], h].double().numpy())


def test_bf16_half_ulp():
    x = np.array([1.0, 1.5, 2.0, 3.99, 4.0, 7.9, -5.0, 0.3])
    got = bf16_half_ulp(x)
    want = np.array([2 ** -8, 2 ** -8, 2 ** -7, 2 ** -7, 2 ** -6, 2 ** -6, 2 ** -6, 2 ** -10])
    assert np.array_equal(got, want)
    # and it is what rounding to bf16 can move a value by
    t = torch.from_numpy(rng_vals := np.random.default_rng(1).uniform(-8, 8, 10000))
    r = t.to(torch.bfloat16).double().numpy()
    assert np.all(np.abs(r - rng_vals) <= bf16_half_ulp(rng_vals))
