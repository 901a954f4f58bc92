"""ring_attn_decode_noalloc, the decode entry point for callers that cannot
allocate device memory when they decode (a serving loop that must not stall on an
allocator, a plugin whose host owns the device memory): its per-shard partials
live in a fixed scratch array inside the library instead of a caller workspace.

Called through the C ABI. It runs the same kernels as ring_attn_decode on the same
inputs, so its outputs must equal that entry point's bit for bit. The calls come in
the order large, small, large: a small call after a larger one would show a stale
partial left in the shared scratch by the earlier call (the small call is also
checked against the oracle directly)."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import TOL_LSE, TOL_O, host32
from online_softmax_merge_gb300 import _lib
from online_softmax_merge_gb300.inputs import Workload, make_qkv
from oracle.attention import attention_at

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_decode_equals_decode_on_calls_in_a_row():
    lib = ra.load()
    dev = torch.device("cuda:0")
    # 32 shards: more partials per row group than one thread-block cluster merges, so
    # the partials go through the scratch and the merge kernel
    w = Workload("noalloc", 2, 64 * 1024, 8, 2, 128, 32, "contiguous", True, seed=41)
    _, k, v = (t.to(dev) for t in make_qkv(w))
    pr = ra.problem(w.batch, w.seqlen, w.heads, w.kv_heads, w.head_dim, w.P, True, w.layout)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    big = lib.ring_attn_decode_workspace_bytes(ctypes.byref(pr), 16)
    small = lib.ring_attn_decode_workspace_bytes(ctypes.byref(pr), 1)
    assert small < big <= _lib.RA_DECODE_SCRATCH_BYTES
    # (n_q, first query position, seed): large, then small, then large again
    calls = ((16, 40000, 1), (1, w.seqlen - 1, 2), (16, w.seqlen - 16, 3))
    for n_q, q_pos0, seed in calls:
        g = torch.Generator(device=dev).manual_seed(seed)
        q = torch.randn((w.batch, n_q, w.heads, w.head_dim), generator=g,
                        device=dev).to(torch.bfloat16)
        o_ref, l_ref = ra.decode(q, k, v, w.P, q_pos0, w.layout, True)
        o = torch.empty_like(o_ref)
        lse = torch.empty_like(l_ref)
        st = lib.ring_attn_decode_noalloc(ctypes.byref(pr), n_q, q_pos0, _p(q), _p(k), _p(v),
                                          _p(o), _p(lse), stream)
        assert st == _lib.RA_OK
        torch.cuda.synchronize(dev)
        assert ra.last_error(dev) == 0
        assert torch.equal(o, o_ref), (n_q, q_pos0)
        assert torch.equal(lse, l_ref), (n_q, q_pos0)
        if n_q == 1:
            rows = np.arange(q_pos0, q_pos0 + n_q)
            O, L = attention_at(host32(q), rows, list(range(w.heads)), w.heads, host32(k),
                                host32(v), True)
            assert float(np.abs(host32(o) - O).max()) <= TOL_O
            assert float(np.abs(host32(lse) - L).max()) <= TOL_LSE


def test_noalloc_decode_rejects_problems_beyond_the_scratch():
    lib = ra.load()
    big = ra.problem(8, 1 << 20, 64, 8, 128, 64, True, "contiguous")
    need = lib.ring_attn_decode_workspace_bytes(ctypes.byref(big), 16)
    assert need > _lib.RA_DECODE_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)
    assert lib.ring_attn_decode_noalloc(ctypes.byref(big), 16, 0, fake, fake, fake, fake, fake,
                                        None) == _lib.RA_ERR_INVALID_ARG
