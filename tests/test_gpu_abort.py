"""The kernels' abort path on the GPU, made to run by a short wait limit (no broken
kernel, no fault, no hang).

ring_attn_selftest_wait_limit lowers the time limit of every device-side wait of
the kernels launched afterwards. In the debug build (libringattn_debug.so, loaded
with RA_DEBUG=1) each wait tests its barrier without blocking and looks at the
limit on every poll, so with a limit of 1 ns the real waits of the forward, step,
backward and decode kernels run out on an ordinary small problem: the role that
gives up records RA_ERR_TIMEOUT and raises its CTA's abort flag, the others stop at
their next wait, the copies and products in flight are let finish (with the
drain's own fixed limit), the tensor memory is freed and the kernel returns. Limits
of a few microseconds let some waits finish and others run out part way through
the pipeline, so those calls end either way (RA_OK or RA_ERR_TIMEOUT). After each,
the default limit is restored and the next call must be correct against the oracle
with a clean status word: the context is still usable.

These tests run in a child process on the debug build. In the release build the
hook is only checked to be harmless (its waits first block in hardware for a short
time, so a tiny limit need not make them run out)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from gpu_helpers import TOL_LSE, TOL_O, compare_full, host32
from online_softmax_merge_gb300 import _lib
from online_softmax_merge_gb300.inputs import Workload, make_dout, make_qkv
from oracle import backward as OB
from oracle.attention import attention_at

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
IN_DEBUG = os.environ.get("RA_DEBUG") == "1"
debug_only = pytest.mark.skipif(not IN_DEBUG, reason="runs in the debug-build child process")

LIMITS = (1, 1, 1000, 4000)      # nanoseconds: the first ones run out at once


def _under_limit(limit_ns, call):
    """Runs call() with the wait limit lowered; returns the status word after it."""
    ra.last_error(DEV)
    ra.selftest_wait_limit(limit_ns)
    try:
        call()
        torch.cuda.synchronize()
    finally:
        ra.selftest_wait_limit(0)
    return ra.last_error(DEV)


def _assert_codes(codes):
    assert codes[0] == _lib.RA_ERR_TIMEOUT and codes[1] == _lib.RA_ERR_TIMEOUT, codes
    assert all(c in (_lib.RA_OK, _lib.RA_ERR_TIMEOUT) for c in codes), codes


def test_wait_limit_argument():
    lib = ra.load()
    assert lib.ring_attn_selftest_wait_limit(3_000_000_000) == _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_selftest_wait_limit(0) == _lib.RA_OK


def test_short_limit_leaves_the_context_usable():
    """In either build: a call under a 1 ns limit ends (cleanly or timed out) and the
    next call under the default limit is correct."""
    w = Workload("abort-any", 1, 4 * 640, 4, 2, 128, 4, "striped", True, seed=599)
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    code = _under_limit(1, lambda: ra.fwd(q, k, v, w.P, w.layout, True))
    assert code in (_lib.RA_OK, _lib.RA_ERR_TIMEOUT)
    o, lse = ra.fwd(q, k, v, w.P, w.layout, True)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    eo, el = compare_full(o, lse, q, k, v, True)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


@debug_only
@pytest.mark.parametrize("d,layout", [(128, "contiguous"), (64, "striped"), (128, "zigzag")])
def test_forward_abort_path(d, layout):
    w = Workload("abort-fwd", 1, 4 * 640, 4, 2, d, 4, layout, True, seed=600 + d)
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    _assert_codes([_under_limit(lim, lambda: ra.fwd(q, k, v, w.P, layout, True))
                   for lim in LIMITS])
    # the step path (the same kernel reading and writing the state in HBM)
    st = ra.empty_state(q)
    assert _under_limit(1, lambda: ra.step(q, k, v, w.P, 0, st, True, layout, True)) == \
        _lib.RA_ERR_TIMEOUT
    # the context is intact: the next call is correct and clean
    o, lse = ra.fwd(q, k, v, w.P, layout, True)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    eo, el = compare_full(o, lse, q, k, v, True)
    assert eo <= TOL_O and el <= TOL_LSE, (eo, el)


@debug_only
@pytest.mark.parametrize("d,layout", [(128, "striped"), (64, "zigzag")])
def test_backward_abort_path(d, layout):
    w = Workload("abort-bwd", 1, 4 * 384, 4, 2, d, 4, layout, True, seed=610 + d)
    q, k, v = (t.to(DEV) for t in make_qkv(w))
    do = make_dout(w).to(DEV)
    o, lse = ra.fwd(q, k, v, w.P, layout, True)
    torch.cuda.synchronize()
    _assert_codes([_under_limit(lim, lambda: ra.bwd(q, k, v, o, lse, do, w.P, layout, True))
                   for lim in LIMITS])
    dq, dk, dv = ra.bwd(q, k, v, o, lse, do, w.P, layout, True)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    hq, hk, hv, hdo = (host32(t).astype(np.float64) for t in (q, k, v, do))
    ref = OB.attention_grads(hq, hk, hv, hdo, True)
    for got, r in zip((dq, dk, dv), ref):
        d_ = host32(got).astype(np.float64) - r
        assert np.abs(d_).max() <= 2.0 ** -6 * np.abs(r).max()


@debug_only
def test_decode_abort_path():
    """The two-launch decode (64 shards: partials, then the merge kernel)."""
    w = Workload("abort-dec", 2, 16384, 8, 2, 128, 64, "contiguous", True, seed=620)
    _, k, v = (t.to(DEV) for t in make_qkv(w))
    g = torch.Generator().manual_seed(21)
    q = torch.randn((w.batch, 2, w.heads, w.head_dim), generator=g).to(torch.bfloat16).to(DEV)
    pos = w.seqlen - 2
    _assert_codes([_under_limit(lim, lambda: ra.decode(q, k, v, w.P, pos, w.layout, True))
                   for lim in LIMITS])
    _check_decode(w, q, k, v, pos)


@debug_only
def test_decode_in_a_cluster_under_a_short_limit():
    """The one-launch decode (8 shards, partials merged inside a thread-block cluster):
    its K/V loads often land before the first poll, so a 1 ns limit need not make a
    wait run out; every call must end, cleanly or timed out, and leave the context
    usable."""
    w = Workload("abort-decc", 1, 2048, 8, 2, 128, 8, "contiguous", True, seed=621)
    _, k, v = (t.to(DEV) for t in make_qkv(w))
    g = torch.Generator().manual_seed(22)
    q = torch.randn((1, 1, w.heads, w.head_dim), generator=g).to(torch.bfloat16).to(DEV)
    pos = w.seqlen - 1
    codes = [_under_limit(1, lambda: ra.decode(q, k, v, w.P, pos, w.layout, True))
             for _ in range(6)]
    assert all(c in (_lib.RA_OK, _lib.RA_ERR_TIMEOUT) for c in codes), codes
    _check_decode(w, q, k, v, pos)


def _check_decode(w, q, k, v, pos):
    n_q = q.shape[1]
    o, lse = ra.decode(q, k, v, w.P, pos, w.layout, True)
    torch.cuda.synchronize()
    assert ra.last_error(DEV) == 0
    rows = np.arange(pos, pos + n_q)
    O, L = attention_at(host32(q), rows, list(range(w.heads)), w.heads, host32(k), host32(v), True)
    assert float(np.abs(host32(o) - O).max()) <= TOL_O
    assert float(np.abs(host32(lse) - L).max()) <= TOL_LSE


@pytest.mark.skipif(IN_DEBUG, reason="this process already runs the debug build")
def test_abort_paths_on_the_debug_build():
    env = dict(os.environ, RA_DEBUG="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_abort.py", "-m", "gpu",
                        "-q", "-x", "-p", "no:cacheprovider", "-k", "not on_the_debug_build"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert "skipped" not in r.stdout.splitlines()[-1], r.stdout[-2000:]
