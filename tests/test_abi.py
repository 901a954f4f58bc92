"""The C ABI on the CPU: the library builds, loads, exports every symbol the
header declares, checks its arguments before touching the GPU, and its host
shard map is bit-exact against the oracle's."""
import ctypes
import os
import re

import pytest
import torch

from online_softmax_merge_gb300 import _lib
from online_softmax_merge_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ringattn.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|ra_status|int32_t|size_t)\s+(\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declarations_match_binding():
    assert _declared() == sorted(_lib.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert lib.ring_attn_version() == 102


def test_debug_build_exports_the_same_symbols_and_reports_its_checks(lib):
    """libringattn_debug.so (the kernels with index checks) has the same ABI; only
    ring_attn_debug_checks tells the two apart."""
    dbg = ctypes.CDLL(B.build(debug=True))
    for name in _declared():
        assert hasattr(dbg, name), name
    dbg.ring_attn_debug_checks.restype = ctypes.c_int32
    assert dbg.ring_attn_debug_checks() == 1
    if os.environ.get("RA_DEBUG") != "1":
        assert lib.ring_attn_debug_checks() == 0


def test_binding_constants_match_the_header():
    text = open(HEADER).read()
    m = re.search(r"#define RA_DECODE_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m is not None
    assert _lib.RA_DECODE_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
    assert re.search(r"#define RA_TILE %d\b" % _lib.TILE, text)


def test_status_strings(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert lib.ra_status_str(code).decode() == name


def test_cuda_error_behind_ra_err_cuda_is_reported(lib):
    assert lib.ring_attn_cuda_error_name(0).decode() == "cudaSuccess"
    assert lib.ring_attn_cuda_error_name(2).decode() == "cudaErrorMemoryAllocation"
    if torch.cuda.is_available():
        pytest.skip("needs a process without a usable GPU")
    code = ctypes.c_int32(-1)
    # without a GPU the call cannot find a device: RA_ERR_CUDA, and the CUDA error it got
    assert lib.ring_attn_last_error(ctypes.byref(code)) == _lib.RA_ERR_CUDA
    err = lib.ring_attn_last_cuda_error()
    assert err != 0 and lib.ring_attn_cuda_error_name(err).decode().startswith("cudaError")
    with pytest.raises(_lib.RingAttnError, match=r"RA_ERR_CUDA \(cudaError"):
        _lib.check("ring_attn_last_error", lib.ring_attn_last_error(ctypes.byref(code)))


def _pr(**kw):
    base = dict(batch=1, seqlen=256, heads=4, kv_heads=2, head_dim=128, P=2, causal=1, layout=0,
                scale=0.0)
    base.update(kw)
    return _lib.RaProblem(**base)


FAKE = ctypes.c_void_p(0x10000)      # aligned, never dereferenced: checks fail first


@pytest.mark.parametrize("bad,code", [
    (dict(seqlen=255), _lib.RA_ERR_INVALID_ARG),          # N % P != 0
    (dict(heads=3), _lib.RA_ERR_INVALID_ARG),             # H % G != 0
    (dict(batch=0), _lib.RA_ERR_INVALID_ARG),
    (dict(P=0), _lib.RA_ERR_INVALID_ARG),
    (dict(P=512), _lib.RA_ERR_INVALID_ARG),               # P > N
    (dict(layout=3), _lib.RA_ERR_INVALID_ARG),
    (dict(layout=2, seqlen=258, P=2), _lib.RA_ERR_INVALID_ARG),   # zigzag: 258 % 4 != 0
    (dict(causal=2), _lib.RA_ERR_INVALID_ARG),
    (dict(scale=-1.0), _lib.RA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _lib.RA_ERR_INVALID_ARG),
    (dict(head_dim=96), _lib.RA_ERR_UNSUPPORTED),
    # 2^31 forward CTAs (batch x heads x shards x query tiles): past the 1-D grid
    (dict(batch=1024, seqlen=1 << 20, heads=256, kv_heads=256, head_dim=64, P=8),
     _lib.RA_ERR_UNSUPPORTED),
])
def test_fwd_rejects_bad_problems_before_any_launch(lib, bad, code):
    pr = _pr(**bad)
    assert lib.ring_attn_fwd(ctypes.byref(pr), FAKE, FAKE, FAKE, FAKE, FAKE, None) == code


def test_null_and_misaligned_pointers_rejected(lib):
    pr = _pr()
    assert lib.ring_attn_fwd(None, FAKE, FAKE, FAKE, FAKE, FAKE, None) == _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_fwd(ctypes.byref(pr), None, FAKE, FAKE, FAKE, FAKE, None) == \
        _lib.RA_ERR_INVALID_ARG
    odd = ctypes.c_void_p(0x10008)
    assert lib.ring_attn_fwd(ctypes.byref(pr), FAKE, odd, FAKE, FAKE, FAKE, None) == \
        _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_step(ctypes.byref(pr), 2, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                              None) == _lib.RA_ERR_INVALID_ARG        # s >= P
    assert lib.ring_attn_merge(0, 1, 8, 1, 128, FAKE, FAKE, FAKE, FAKE, None) == \
        _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_merge(2, 1, 8, 1, 80, FAKE, FAKE, FAKE, FAKE, None) == \
        _lib.RA_ERR_UNSUPPORTED
    assert lib.ring_attn_tile_classes(ctypes.byref(pr), 2, 0, FAKE, None) == \
        _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_selftest_timeout(0, None) == _lib.RA_ERR_INVALID_ARG


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("N,P", [(8, 4), (12, 3), (1024, 16), (96, 96), (7, 1), (10, 1)])
def test_host_shard_map_bit_exact_vs_oracle(lib, layout, N, P):
    if layout == "zigzag" and N % (2 * P):
        pytest.skip("zigzag needs N divisible by 2P")
    from oracle import shardmap as OS
    import online_softmax_merge_gb300 as ra
    got = ra.shard_map(layout, N, P)
    want = OS.shard_map(layout, N, P)
    assert got == tuple(want) or list(got) == list(want)


def test_host_shard_map_rejects_bad_sizes(lib):
    arr = (ctypes.c_int32 * 10)()
    assert lib.ring_attn_shard_map(0, 10, 3, arr, arr, arr) == _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_shard_map(5, 10, 2, arr, arr, arr) == _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_shard_map(2, 10, 2, arr, arr, arr) == _lib.RA_ERR_INVALID_ARG  # 10 % 4
    assert lib.ring_attn_shard_map(0, 10, 2, None, arr, arr) == _lib.RA_ERR_INVALID_ARG


def test_decode_workspace_and_argument_checks(lib):
    pr = _pr(seqlen=8192, P=4)                       # S = 2048: one key chunk per shard
    need = lib.ring_attn_decode_workspace_bytes(ctypes.byref(pr), 3)
    assert need == 4 * 1 * 4 * 3 * (128 + 1) * 4     # parts * B * H * n_q * (d + 1) floats
    assert lib.ring_attn_decode_workspace_bytes(ctypes.byref(_pr(heads=3)), 3) == 0
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE]
    assert lib.ring_attn_decode(ctypes.byref(pr), 3, 8189, *args, need - 4, None) == \
        _lib.RA_ERR_INVALID_ARG                      # workspace too small
    assert lib.ring_attn_decode(ctypes.byref(pr), 3, 8190, *args, need, None) == \
        _lib.RA_ERR_INVALID_ARG                      # query positions past the cache
    assert lib.ring_attn_decode(ctypes.byref(pr), 0, 0, *args, need, None) == \
        _lib.RA_ERR_INVALID_ARG


@pytest.mark.parametrize("layout,N,P,tiles_per_bh", [
    (0, 1000, 4, 4 * 2),        # 4 shards of 250 rows: 2 tiles each
    (1, 1000, 4, 4 * 2),        # striped: the same per shard
    (2, 1040, 4, 8 * 2),        # zigzag: 8 chunks of 130 rows: 2 tiles each
    (0, 256, 1, 2),
])
@pytest.mark.parametrize("d", [64, 128])
def test_bwd_workspace_bytes(lib, layout, N, P, tiles_per_bh, d):
    pr = _pr(seqlen=N, P=P, layout=layout, heads=6, kv_heads=3, batch=2, head_dim=d)
    # per query tile: 1 KiB of statistics and two 4 KiB extension tiles; one 4 KiB key-side tile
    assert lib.ring_attn_bwd_workspace_bytes(ctypes.byref(pr)) == \
        2 * 6 * tiles_per_bh * (1024 + 2 * 4096) + 4096
    assert lib.ring_attn_bwd_workspace_bytes(ctypes.byref(_pr(heads=3))) == 0
    assert lib.ring_attn_bwd_workspace_bytes(None) == 0


def test_bwd_argument_checks(lib):
    pr = _pr()
    need = lib.ring_attn_bwd_workspace_bytes(ctypes.byref(pr))
    good = [FAKE] * 9
    assert lib.ring_attn_bwd(ctypes.byref(pr), *good, FAKE, need - 16, None) == \
        _lib.RA_ERR_INVALID_ARG                      # workspace too small
    for i in range(10):
        ptrs = [FAKE] * 10
        ptrs[i] = None
        assert lib.ring_attn_bwd(ctypes.byref(pr), *ptrs, need, None) == _lib.RA_ERR_INVALID_ARG
        ptrs[i] = ctypes.c_void_p(0x10004)
        assert lib.ring_attn_bwd(ctypes.byref(pr), *ptrs, need, None) == _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_bwd(ctypes.byref(_pr(head_dim=96)), *[FAKE] * 10, need, None) == \
        _lib.RA_ERR_UNSUPPORTED
    assert lib.ring_attn_bwd(None, *[FAKE] * 10, need, None) == _lib.RA_ERR_INVALID_ARG


def test_fwd_host_workspace_and_argument_checks(lib):
    pr = _pr(batch=3, seqlen=1000, heads=4, kv_heads=2, head_dim=128, P=4)
    r = lambda x: (x + 255) // 256 * 256
    # a piece: 2 query heads (one kv group) and 1 kv head of one sequence
    slot = r(1000 * 2 * 128 * 2) * 2 + r(1000 * 1 * 128 * 2) * 2 + r(2 * 1000 * 4)
    # recommended: one slot per piece up to sixteen (here 3 x 2 = 6 pieces); two suffice
    assert lib.ring_attn_fwd_host_workspace_bytes(ctypes.byref(pr)) == 6 * slot
    many = _pr(batch=12, seqlen=1000, heads=4, kv_heads=2, head_dim=128, P=4)
    assert lib.ring_attn_fwd_host_workspace_bytes(ctypes.byref(many)) == 16 * slot
    one = _pr(batch=1, seqlen=1000, heads=4, kv_heads=1, head_dim=128, P=4)
    slot1 = r(1000 * 4 * 128 * 2) * 2 + r(1000 * 1 * 128 * 2) * 2 + r(4 * 1000 * 4)
    assert lib.ring_attn_fwd_host_workspace_bytes(ctypes.byref(one)) == slot1
    assert lib.ring_attn_fwd_host_workspace_bytes(ctypes.byref(_pr(heads=3))) == 0
    ptrs = [FAKE] * 5
    assert lib.ring_attn_fwd_host(ctypes.byref(pr), *ptrs, FAKE, 2 * slot - 1, None, None) == \
        _lib.RA_ERR_INVALID_ARG                     # workspace too small
    assert lib.ring_attn_fwd_host(ctypes.byref(pr), *ptrs, ctypes.c_void_p(0x10008), 2 * slot,
                                  None, None) == _lib.RA_ERR_INVALID_ARG   # misaligned workspace
    for i in range(5):
        bad = list(ptrs)
        bad[i] = None
        assert lib.ring_attn_fwd_host(ctypes.byref(pr), *bad, FAKE, 2 * slot, None, None) == \
            _lib.RA_ERR_INVALID_ARG


def test_host_mapped_refuses_pageable_null_and_empty_ranges(lib):
    """Pageable memory, a null pointer and an empty range read 0, with or without a
    device (without one every range reads 0); the query launches nothing."""
    buf = ctypes.create_string_buffer(4096)
    assert lib.ring_attn_host_mapped(ctypes.addressof(buf), 4096) == 0
    assert lib.ring_attn_host_mapped(None, 4096) == 0
    assert lib.ring_attn_host_mapped(ctypes.addressof(buf), 0) == 0


# Far-apart fake addresses (aligned, never dereferenced): every range of the small
# problems below fits between two of them.
def _at(i, off=0):
    return ctypes.c_void_p(0x1000_0000_0000 + i * 0x1_0000_0000 + off)


def _no_device_reached(code):
    """A call whose arguments passed every host-side check stops at the device lookup
    (RA_ERR_CUDA or RA_ERR_UNSUPPORTED here); on a machine with a GPU the fake
    addresses fail the residency check instead, so only the overlap cases are decided."""
    if torch.cuda.is_available():
        return True
    return code in (_lib.RA_ERR_CUDA, _lib.RA_ERR_UNSUPPORTED)


def test_written_ranges_may_not_overlap_other_arguments(lib):
    pr = _pr()                                      # B=1 N=256 H=4 G=2 d=128
    bq, bkv, brows, by = 256 * 4 * 128 * 2, 256 * 2 * 128 * 2, 4 * 256 * 4, 256 * 4 * 128 * 4
    q, k, v, o, lse = (_at(i) for i in range(5))
    fwd = lambda *a: lib.ring_attn_fwd(ctypes.byref(pr), *a, None)
    assert _no_device_reached(fwd(q, k, v, o, lse))
    assert _no_device_reached(fwd(q, k, k, o, lse))                 # inputs may alias
    assert fwd(q, k, v, q, lse) == _lib.RA_ERR_INVALID_ARG           # o over q: no in-place form
    assert fwd(q, k, v, _at(0, bq - 16), lse) == _lib.RA_ERR_INVALID_ARG   # o over q's tail
    assert _no_device_reached(fwd(q, k, v, _at(0, bq), lse))        # o right after q
    assert fwd(q, k, v, o, _at(3, bq - 16)) == _lib.RA_ERR_INVALID_ARG     # lse inside o
    assert fwd(q, k, v, o, _at(2, bkv - 16)) == _lib.RA_ERR_INVALID_ARG    # lse over v's tail
    m, z, y = _at(5), _at(6), _at(7)
    step = lambda *a: lib.ring_attn_step(ctypes.byref(pr), 0, 1, *a, None)
    assert _no_device_reached(step(q, k, v, m, z, y))
    assert step(q, k, v, m, z, _at(1, 16)) == _lib.RA_ERR_INVALID_ARG      # y over k
    assert step(q, k, v, m, _at(5, brows - 16), y) == _lib.RA_ERR_INVALID_ARG   # z over m
    fin = lambda *a: lib.ring_attn_finalize(ctypes.byref(pr), *a, None)
    assert _no_device_reached(fin(m, z, y, o, lse))
    assert fin(m, z, y, o, _at(7, by - 16)) == _lib.RA_ERR_INVALID_ARG      # lse over y
    n = 3
    merge = lambda *a: lib.ring_attn_merge(n, 1, 256, 4, 128, *a, None)
    assert _no_device_reached(merge(_at(8), _at(9), o, lse))
    assert merge(_at(8), _at(9), _at(8, n * 256 * 4 * 128 * 4 - 16), lse) == \
        _lib.RA_ERR_INVALID_ARG                                        # o over o_parts' tail
    ws = _at(10)
    need = lib.ring_attn_bwd_workspace_bytes(ctypes.byref(pr))
    bwd = lambda *a: lib.ring_attn_bwd(ctypes.byref(pr), *a, need, None)
    dout, dq, dk, dv = _at(11), _at(12), _at(13), _at(14)
    assert _no_device_reached(bwd(q, k, v, o, lse, dout, dq, dk, dv, ws))
    assert bwd(q, k, v, o, lse, dout, dout, dk, dv, ws) == _lib.RA_ERR_INVALID_ARG   # dq = dout
    assert bwd(q, k, v, o, lse, dout, dq, dk, dv, _at(14, bkv - 16)) == \
        _lib.RA_ERR_INVALID_ARG                                        # workspace over dv
    assert bwd(q, k, v, o, lse, dout, dq, dk, dk, ws) == _lib.RA_ERR_INVALID_ARG     # dk = dv
    dpr = _pr(seqlen=8192, P=4)
    dneed = lib.ring_attn_decode_workspace_bytes(ctypes.byref(dpr), 1)
    dec = lambda *a: lib.ring_attn_decode(ctypes.byref(dpr), 1, 8191, *a, dneed, None)
    assert _no_device_reached(dec(q, k, v, o, lse, ws))
    assert dec(q, k, v, o, lse, _at(1, 64)) == _lib.RA_ERR_INVALID_ARG      # workspace over k
    hneed = lib.ring_attn_fwd_host_workspace_bytes(ctypes.byref(pr))
    host = lambda *a: lib.ring_attn_fwd_host(ctypes.byref(pr), *a, hneed, None, None)
    assert _no_device_reached(host(q, k, v, o, lse, ws))
    assert host(q, k, v, o, lse, _at(3, 256)) == _lib.RA_ERR_INVALID_ARG    # workspace over o
    assert host(q, k, v, o, _at(2), ws) == _lib.RA_ERR_INVALID_ARG          # lse = v


def test_fp32_output_ranges_and_bad_dtype(lib):
    """With o_dtype = RA_DTYPE_F32 the written range of o is 4 bytes per element, so
    a range that clears a bf16 o may overlap as fp32; any other o_dtype is refused."""
    pr = _pr(o_dtype=_lib.RA_DTYPE_F32)             # B=1 N=256 H=4 G=2 d=128
    bq = 256 * 4 * 128 * 2
    q, k, v, o = (_at(i) for i in range(4))
    fwd = lambda p, *a: lib.ring_attn_fwd(ctypes.byref(p), *a, None)
    assert _no_device_reached(fwd(pr, q, k, v, o, _at(3, 2 * bq)))       # lse right after o
    assert fwd(pr, q, k, v, o, _at(3, bq)) == _lib.RA_ERR_INVALID_ARG    # lse inside fp32 o
    assert _no_device_reached(fwd(_pr(), q, k, v, o, _at(3, bq)))       # ... but after bf16 o
    bad = _pr(o_dtype=2)
    assert fwd(bad, q, k, v, o, _at(4)) == _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_finalize(ctypes.byref(bad), q, k, v, o, _at(4), None) == \
        _lib.RA_ERR_INVALID_ARG


def test_selftest_wait_limit_is_host_only_and_checked(lib):
    """The abort-path test hook only sets the limit later launches get."""
    assert lib.ring_attn_selftest_wait_limit(ctypes.c_uint64(3_000_000_000)) == \
        _lib.RA_ERR_INVALID_ARG
    assert lib.ring_attn_selftest_wait_limit(ctypes.c_uint64(5)) == _lib.RA_OK
    assert lib.ring_attn_selftest_wait_limit(ctypes.c_uint64(0)) == _lib.RA_OK
