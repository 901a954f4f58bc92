"""ctypes loader for libringattn.so (the C ABI in include/ringattn.h).

Loading fails loudly when the library has not been built: there is no fallback.
With RA_DEBUG=1 in the environment the debug build libringattn_debug.so (the same
kernels with index checks) is loaded instead.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libringattn_debug.so" if os.environ.get("RA_DEBUG") == "1"
                        else "libringattn.so")

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_TIMEOUT, RA_ERR_BOUNDS = range(6)
STATUS_NAMES = {0: "RA_OK", 1: "RA_ERR_INVALID_ARG", 2: "RA_ERR_UNSUPPORTED", 3: "RA_ERR_CUDA",
                4: "RA_ERR_TIMEOUT", 5: "RA_ERR_BOUNDS"}
LAYOUTS = {"contiguous": 0, "striped": 1, "zigzag": 2}
RA_DTYPE_BF16, RA_DTYPE_F32 = 0, 1
TILE = 128
# bytes of the fixed scratch array of ring_attn_decode_noalloc (RA_DECODE_SCRATCH_BYTES)
RA_DECODE_SCRATCH_BYTES = 16 << 20

# Every exported function of include/ringattn.h, with (restype, argtypes).
_i32, _u64, _vp, _fp = ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_void_p


class RaProblem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seqlen", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("P", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("layout", ctypes.c_int32), ("scale", ctypes.c_float),
                ("o_dtype", ctypes.c_int32)]


_PP = ctypes.POINTER(RaProblem)
SIGNATURES = {
    "ring_attn_fwd": (_i32, [_PP, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_fwd_host": (_i32, [_PP, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp, _vp]),
    "ring_attn_fwd_host_workspace_bytes": (ctypes.c_size_t, [_PP]),
    "ring_attn_host_mapped": (_i32, [_vp, ctypes.c_size_t]),
    "ring_attn_step": (_i32, [_PP, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_step_simt": (_i32, [_PP, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_finalize": (_i32, [_PP, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_merge": (_i32, [_i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_decode": (_i32, [_PP, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "ring_attn_decode_workspace_bytes": (ctypes.c_size_t, [_PP, _i32]),
    "ring_attn_decode_noalloc": (_i32, [_PP, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "ring_attn_bwd": (_i32, [_PP, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]),
    "ring_attn_bwd_workspace_bytes": (ctypes.c_size_t, [_PP]),
    "ring_attn_shard_map": (_i32, [_i32, _i32, _i32, _vp, _vp, _vp]),
    "ring_attn_shard_map_device": (_i32, [_i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "ring_attn_tile_classes": (_i32, [_PP, _i32, _i32, _vp, _vp]),
    "ring_attn_mask": (_i32, [_PP, _i32, _i32, _vp, _vp]),
    "ring_attn_last_error": (_i32, [ctypes.POINTER(ctypes.c_int32)]),
    "ring_attn_selftest_timeout": (_i32, [_u64, _vp]),
    "ring_attn_selftest_wait_limit": (_i32, [_u64]),
    "ring_attn_selftest_bounds": (_i32, [_vp]),
    "ring_attn_debug_checks": (_i32, []),
    "ra_status_str": (ctypes.c_char_p, [_i32]),
    "ring_attn_last_cuda_error": (_i32, []),
    "ring_attn_cuda_error_name": (ctypes.c_char_p, [_i32]),
    "ring_attn_version": (_i32, []),
}

_LIB = None


class RingAttnError(RuntimeError):
    def __init__(self, fn: str, code: int, cuda_error: int = 0, cuda_name: str = ""):
        what = f"{fn} returned {STATUS_NAMES.get(code, code)}"
        if cuda_error:
            what += f" ({cuda_name or 'cudaError'} = {cuda_error})"
        super().__init__(what)
        self.fn = fn
        self.code = code
        self.cuda_error = cuda_error


def load() -> ctypes.CDLL:
    """Load (once) and return the library; raises if it is not built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(or python online_softmax_merge_gb300/build.py [--debug]) first")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def check(fn: str, code: int) -> None:
    if code != RA_OK:
        cuda_error, name = 0, ""
        if code == RA_ERR_CUDA and _LIB is not None:
            cuda_error = int(_LIB.ring_attn_last_cuda_error())
            name = (_LIB.ring_attn_cuda_error_name(cuda_error) or b"").decode()
        raise RingAttnError(fn, code, cuda_error, name)
