"""Pointer residency at the C boundary: host memory given where the ABI wants device
memory is refused with RA_ERR_INVALID_ARG before anything is launched, while device
memory from every PyTorch allocator (the caching allocator, its expandable
virtual-memory segments, the cudaMallocAsync backend) is accepted and gives the same
results bit for bit."""
import ctypes
import hashlib
import os
import subprocess
import sys

import pytest
import torch

from online_softmax_merge_gb300 import _lib
from online_softmax_merge_gb300.inputs import Workload, make_dout, make_qkv

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")
DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W = Workload("res", 1, 4 * 200, 4, 2, 128, 4, "striped", True, 800)


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("pinned", [False, True])
def test_host_memory_is_refused_before_any_launch(pinned):
    lib = ra.load()
    q, k, v = (t.to(DEV) for t in make_qkv(W))
    o = torch.empty_like(q)
    lse = torch.empty((W.batch, W.heads, W.seqlen), dtype=torch.float32, device=DEV)
    host_q = q.cpu().pin_memory() if pinned else q.cpu()
    pr = ra.problem(W.batch, W.seqlen, W.heads, W.kv_heads, W.head_dim, W.P, True, W.layout)
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    o.fill_(7)
    code = lib.ring_attn_fwd(ctypes.byref(pr), _p(host_q), _p(k), _p(v), _p(o), _p(lse), stream)
    assert code == _lib.RA_ERR_INVALID_ARG
    host_lse = torch.empty(lse.shape, dtype=torch.float32, pin_memory=pinned)
    code = lib.ring_attn_fwd(ctypes.byref(pr), _p(q), _p(k), _p(v), _p(o), _p(host_lse), stream)
    assert code == _lib.RA_ERR_INVALID_ARG
    torch.cuda.synchronize(DEV)
    assert ra.last_error(DEV) == 0
    assert bool((o == 7).all())                       # nothing was written
    # the same call on device memory still works afterwards
    ra.fwd(q, k, v, W.P, W.layout, True, out=o, lse=lse)
    torch.cuda.synchronize(DEV)
    assert ra.last_error(DEV) == 0


CHILD = r"""
import hashlib, sys, torch
sys.path.insert(0, sys.argv[1])
import online_softmax_merge_gb300 as ra
from online_softmax_merge_gb300.inputs import Workload, make_dout, make_qkv
dev = torch.device("cuda:0")
w = Workload("res", 1, 4 * 200, 4, 2, 128, 4, "striped", True, 800)
q, k, v = (t.to(dev) for t in make_qkv(w))
o, lse = ra.fwd(q, k, v, w.P, w.layout, True)
dq, dk, dv = ra.bwd(q, k, v, o, lse, make_dout(w).to(dev), w.P, w.layout, True)
od, ld = ra.decode(q[:, -2:].contiguous(), k, v, w.P, w.seqlen - 2, w.layout, True)
torch.cuda.synchronize(dev)
assert ra.last_error(dev) == 0
h = hashlib.sha256()
for t in (o, lse, dq, dk, dv, od, ld):
    h.update(t.cpu().view(torch.uint8).numpy().tobytes())
print(h.hexdigest())
"""


def test_every_pytorch_allocator_is_accepted_with_identical_results():
    digests = {}
    for conf in ("", "expandable_segments:True", "backend:cudaMallocAsync"):
        env = dict(os.environ, PYTORCH_ALLOC_CONF=conf)
        r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, cwd=ROOT,
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, (conf, r.stderr[-3000:])
        digests[conf] = r.stdout.strip().splitlines()[-1]
    assert len(set(digests.values())) == 1, digests


def test_outputs_overlapping_inputs_are_refused_and_nothing_is_written():
    """There is no in-place form: o over q, z over m, dq over dout and a
    merge output over its partials are refused before any launch (the binding surfaces
    RA_ERR_INVALID_ARG), and the aliased buffers keep their contents."""
    q, k, v = (t.to(DEV) for t in make_qkv(W))
    q0 = q.clone()
    with pytest.raises(ra.RingAttnError) as e:
        ra.fwd(q, k, v, W.P, W.layout, W.causal, out=q)
    assert e.value.code == _lib.RA_ERR_INVALID_ARG
    o, lse = ra.fwd(q, k, k, W.P, W.layout, W.causal)              # inputs may alias
    torch.cuda.synchronize()
    m, z, y = ra.empty_state(q)
    with pytest.raises(ra.RingAttnError):
        ra.step(q, k, v, W.P, 0, (m, m, y), True, W.layout, W.causal)   # z over m
    dout = make_dout(W).to(DEV)
    d0 = dout.clone()
    o, lse = ra.fwd(q, k, v, W.P, W.layout, W.causal)
    with pytest.raises(ra.RingAttnError):
        ra.bwd(q, k, v, o, lse, dout, W.P, W.layout, W.causal, dq=dout)
    parts = torch.randn((3,) + tuple(o.shape), device=DEV)
    lparts = torch.randn((3,) + tuple(lse.shape), device=DEV)
    p0 = parts.clone()
    with pytest.raises(ra.RingAttnError):
        ra.merge(parts, lparts, lse=lparts[0])
    torch.cuda.synchronize()
    assert torch.equal(q, q0) and torch.equal(dout, d0) and torch.equal(parts, p0)
    assert ra.last_error(DEV) == 0
