"""ring_attn_decode_noalloc, the decode entry point for callers that cannot
allocate device memory when they decode (its partials live in a fixed scratch
array inside the library). Called through the C ABI and checked against
ring_attn_decode on two calls in a row, which also shows that a call does not
depend on what the previous call left in the shared scratch."""
import ctypes

import pytest
import torch

from gpu_helpers import TOL_LSE, TOL_O
from online_softmax_merge_gb300 import _lib
from online_softmax_merge_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu

ra = pytest.importorskip("online_softmax_merge_gb300")


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_noalloc_decode_matches_decode_on_two_calls_in_a_row():
    lib = ra.load()
    dev = torch.device("cuda:0")
    w = Workload("noalloc", 2, 4 * 1024, 8, 2, 128, 4, "contiguous", True, seed=41)
    _, k, v = (t.to(dev) for t in make_qkv(w))
    pr = ra.problem(w.batch, w.seqlen, w.heads, w.kv_heads, w.head_dim, w.P, True, w.layout)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for n_q, q_pos0, seed in ((3, 1500, 1), (1, w.seqlen - 1, 2)):
        g = torch.Generator(device=dev).manual_seed(seed)
        q = torch.randn((w.batch, n_q, w.heads, w.head_dim), generator=g, device=dev).to(torch.bfloat16)
        o_ref, l_ref = ra.decode(q, k, v, w.P, q_pos0, w.layout, True)
        o = torch.empty_like(o_ref)
        lse = torch.empty_like(l_ref)
        st = lib.ring_attn_decode_noalloc(ctypes.byref(pr), n_q, q_pos0, _p(q), _p(k), _p(v),
                                          _p(o), _p(lse), stream)
        assert st == _lib.RA_OK
        torch.cuda.synchronize(dev)
        assert ra.last_error(dev) == 0
        assert float((o.float() - o_ref.float()).abs().max()) <= TOL_O
        assert float((lse - l_ref).abs().max()) <= TOL_LSE


def test_noalloc_decode_rejects_problems_beyond_the_scratch():
    lib = ra.load()
    big = ra.problem(8, 1 << 20, 64, 8, 128, 64, True, "contiguous")
    need = lib.ring_attn_decode_workspace_bytes(ctypes.byref(big), 16)
    assert need > (16 << 20)
    fake = ctypes.c_void_p(0x10000)
    assert lib.ring_attn_decode_noalloc(ctypes.byref(big), 16, 0, fake, fake, fake, fake, fake,
                                        None) == _lib.RA_ERR_INVALID_ARG
