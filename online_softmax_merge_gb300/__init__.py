"""Ring Attention's online-softmax merge on one GB300: Python binding.

Thin wrappers over the C ABI of libringattn.so (include/ringattn.h). They check
shapes, dtypes and devices, allocate outputs with PyTorch when none are given,
and pass raw pointers plus the current CUDA stream. Every step of the path runs
in the library's CUDA kernels; nothing here computes attention.

Tensor layouts (original token order, whatever the shard layout):
  q [B, N, H, d] bf16;  o [B, N, H, d] bf16, or fp32 where a call takes
  out_dtype=torch.float32 (O kept at fp32, not rounded to bf16);
  k, v [B, N, G, d] bf16;  lse, m, z [B, H, N] fp32;
  y [B, N, H, d] fp32;  o_parts [n, B, N, H, d] fp32;  lse_parts [n, B, H, N] fp32.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import (LAYOUTS, RA_ERR_BOUNDS, RA_ERR_CUDA, RA_ERR_INVALID_ARG,  # noqa: F401
                   RA_ERR_TIMEOUT, RA_ERR_UNSUPPORTED, RA_OK, TILE, RingAttnError, check, load)

__all__ = ["fwd", "fwd_host", "fwd_host_workspace_bytes", "host_mapped", "bwd", "bwd_workspace_bytes", "decode", "decode_workspace_bytes", "step", "step_simt", "finalize", "merge", "shard_map", "shard_map_device",
           "tile_classes", "mask", "last_error", "selftest_timeout", "selftest_bounds",
           "selftest_wait_limit",
           "debug_checks", "problem", "RingAttnError",
           "empty_state", "LAYOUTS", "TILE"]


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _same_device(ref: torch.Tensor, **tensors):
    """Every tensor passed by name lives on ref's GPU (the kernels are launched there)."""
    for name, t in tensors.items():
        if t.device != ref.device:
            raise ValueError(f"{name} is on {t.device}, the call runs on {ref.device}")


_O_DTYPES = {torch.bfloat16: _lib.RA_DTYPE_BF16, torch.float32: _lib.RA_DTYPE_F32}


def _o_dtype_code(out_dtype) -> int:
    if out_dtype not in _O_DTYPES:
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    return _O_DTYPES[out_dtype]


def problem(batch: int, seqlen: int, heads: int, kv_heads: int, head_dim: int, P: int,
            causal: bool, layout: str = "contiguous", scale: float = 0.0,
            out_dtype=torch.bfloat16) -> _lib.RaProblem:
    """The ra_problem struct (scale 0 means 1/sqrt(head_dim); out_dtype is the
    element type of o)."""
    if layout not in LAYOUTS:
        raise ValueError(f"layout must be one of {tuple(LAYOUTS)}")
    return _lib.RaProblem(batch, seqlen, heads, kv_heads, head_dim, P, int(bool(causal)),
                          LAYOUTS[layout], float(scale), _o_dtype_code(out_dtype))


def _qkv_problem(q, k, v, P, layout, causal, scale, out_dtype=torch.bfloat16):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, N, H, d] and k, v [B, N, G, d]")
    B, N, H, d = q.shape
    G = k.shape[2]
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, (B, N, G, d))
    _need(v, "v", torch.bfloat16, (B, N, G, d))
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k, v must be on one device")
    return problem(B, N, H, G, d, P, causal, layout, scale, out_dtype), (B, N, H, G, d)


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, layout: str = "contiguous",
        causal: bool = True, scale: float = 0.0, out: Optional[torch.Tensor] = None,
        lse: Optional[torch.Tensor] = None,
        out_dtype=torch.bfloat16) -> Tuple[torch.Tensor, torch.Tensor]:
    """Full ring forward over P virtual shards (ring_attn_fwd). Returns (O, LSE);
    O is bf16, or fp32 with out_dtype=torch.float32."""
    lib = load()
    pr, (B, N, H, G, d) = _qkv_problem(q, k, v, P, layout, causal, scale, out_dtype)
    if out is None:
        out = torch.empty((B, N, H, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _need(out, "out", out_dtype, (B, N, H, d))
    _need(lse, "lse", torch.float32, (B, H, N))
    _same_device(q, out=out, lse=lse)
    with torch.cuda.device(q.device):
        check("ring_attn_fwd", lib.ring_attn_fwd(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v),
                                                 _ptr(out), _ptr(lse), _stream(q.device)))
    return out, lse


def _need_host(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


_COPY_STREAMS = {}


def fwd_host_workspace_bytes(batch: int, seqlen: int, heads: int, kv_heads: int, head_dim: int,
                             P: int, layout: str = "contiguous", causal: bool = True,
                             out_dtype=torch.bfloat16) -> int:
    """Device workspace bytes ring_attn_fwd_host needs."""
    lib = load()
    pr = problem(batch, seqlen, heads, kv_heads, head_dim, P, causal, layout, 0.0, out_dtype)
    return int(lib.ring_attn_fwd_host_workspace_bytes(ctypes.byref(pr)))


def fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int,
             layout: str = "contiguous", causal: bool = True, scale: float = 0.0,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, device=None,
             copy_stream: Optional[torch.cuda.Stream] = None, out_dtype=torch.bfloat16):
    """Ring forward for host tensors (ring_attn_fwd_host): q [B, N, H, d], k, v
    [B, N, G, d] bf16 on the CPU (pinned for overlap); returns host (O, LSE), O in
    out_dtype (bf16 or fp32). Runs
    on `device` (default: the current CUDA device) and its current stream; copies
    go on copy_stream (default: one cached side stream per device)."""
    lib = load()
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, N, H, d] and k, v [B, N, G, d]")
    B, N, H, d = q.shape
    G = k.shape[2]
    _need_host(q, "q", torch.bfloat16, (B, N, H, d))
    _need_host(k, "k", torch.bfloat16, (B, N, G, d))
    _need_host(v, "v", torch.bfloat16, (B, N, G, d))
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    pr = problem(B, N, H, G, d, P, causal, layout, scale, out_dtype)
    need = int(lib.ring_attn_fwd_host_workspace_bytes(ctypes.byref(pr)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    # any workspace of at least two slots works (the library checks the size); the
    # recommended one, `need` bytes, holds sixteen (or one per piece)
    if workspace.device != dev:
        raise ValueError(f"workspace is on {workspace.device}, the call runs on {dev}")
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, N, H, d), dtype=out_dtype, pin_memory=pin)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    _need_host(out, "out", out_dtype, (B, N, H, d))
    _need_host(lse, "lse", torch.float32, (B, H, N))
    if copy_stream is None:
        copy_stream = _COPY_STREAMS.get(dev.index)
        if copy_stream is None:
            copy_stream = torch.cuda.Stream(device=dev)
            _COPY_STREAMS[dev.index] = copy_stream
    with torch.cuda.device(dev):
        check("ring_attn_fwd_host", lib.ring_attn_fwd_host(
            ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(workspace),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(dev),
            ctypes.c_void_p(copy_stream.cuda_stream)))
    return out, lse


def host_mapped(t: torch.Tensor, device=None) -> bool:
    """Whether ring_attn_fwd_host moves host tensor `t` (its whole storage extent
    from its first element) with copy kernels rather than the copy engines
    (ring_attn_host_mapped): page-locked memory that `device` (default: the current
    CUDA device) maps at the same address, inside one allocation."""
    lib = load()
    if t.device.type != "cpu":
        raise ValueError("host_mapped takes a CPU tensor")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return bool(lib.ring_attn_host_mapped(_ptr(t), ctypes.c_size_t(t.numel() * t.element_size())))


def bwd_workspace_bytes(batch: int, seqlen: int, heads: int, kv_heads: int, head_dim: int,
                        P: int, layout: str = "contiguous", causal: bool = True) -> int:
    """Workspace bytes ring_attn_bwd needs (ring_attn_bwd_workspace_bytes)."""
    lib = load()
    pr = problem(batch, seqlen, heads, kv_heads, head_dim, P, causal, layout)
    return int(lib.ring_attn_bwd_workspace_bytes(ctypes.byref(pr)))


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
        dout: torch.Tensor, P: int, layout: str = "contiguous", causal: bool = True,
        scale: float = 0.0, dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
        dv: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """Backward ring (ring_attn_bwd): gradients of the forward for upstream gradient
    dout, from the forward's saved o (bf16 or fp32) and lse. Returns (dq, dk, dv)."""
    lib = load()
    pr, (B, N, H, G, d) = _qkv_problem(q, k, v, P, layout, causal, scale,
                                       o.dtype if o.dtype == torch.float32 else torch.bfloat16)
    _need(o, "o", torch.bfloat16 if o.dtype != torch.float32 else torch.float32, (B, N, H, d))
    _need(lse, "lse", torch.float32, (B, H, N))
    _need(dout, "dout", torch.bfloat16, (B, N, H, d))
    need = int(lib.ring_attn_bwd_workspace_bytes(ctypes.byref(pr)))
    if workspace is None:
        workspace = torch.empty(max(need, 16) // 4, dtype=torch.float32, device=q.device)
    _need(workspace, "workspace", torch.float32)
    if dq is None:
        dq = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=q.device)
    if dk is None:
        dk = torch.empty((B, N, G, d), dtype=torch.bfloat16, device=q.device)
    if dv is None:
        dv = torch.empty((B, N, G, d), dtype=torch.bfloat16, device=q.device)
    _need(dq, "dq", torch.bfloat16, (B, N, H, d))
    _need(dk, "dk", torch.bfloat16, (B, N, G, d))
    _need(dv, "dv", torch.bfloat16, (B, N, G, d))
    _same_device(q, o=o, lse=lse, dout=dout, workspace=workspace, dq=dq, dk=dk, dv=dv)
    with torch.cuda.device(q.device):
        check("ring_attn_bwd", lib.ring_attn_bwd(
            ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
            ctypes.c_size_t(workspace.numel() * 4), _stream(q.device)))
    return dq, dk, dv


def decode_workspace_bytes(batch: int, seqlen: int, heads: int, kv_heads: int, head_dim: int,
                           P: int, n_q: int, layout: str = "contiguous", causal: bool = True) -> int:
    """Workspace bytes ring_attn_decode needs (ring_attn_decode_workspace_bytes)."""
    lib = load()
    pr = problem(batch, seqlen, heads, kv_heads, head_dim, P, causal, layout)
    return int(lib.ring_attn_decode_workspace_bytes(ctypes.byref(pr), int(n_q)))


def decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, q_pos0: int,
           layout: str = "contiguous", causal: bool = True, scale: float = 0.0,
           workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
           lse: Optional[torch.Tensor] = None, out_dtype=torch.bfloat16):
    """Pass-Q decode (ring_attn_decode): q [B, n_q, H, d] at positions q_pos0.. against the
    KV cache k, v [B, N, G, d] in P stationary virtual shards. Returns (O, LSE), O in
    out_dtype (bf16 or fp32)."""
    lib = load()
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, n_q, H, d] and k, v [B, N, G, d]")
    B, n_q, H, d = q.shape
    N, G = k.shape[1], k.shape[2]
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, (B, N, G, d))
    _need(v, "v", torch.bfloat16, (B, N, G, d))
    pr = problem(B, N, H, G, d, P, causal, layout, scale, out_dtype)
    need = int(lib.ring_attn_decode_workspace_bytes(ctypes.byref(pr), n_q))
    if workspace is None:
        workspace = torch.empty(max(need, 16) // 4 + 4, dtype=torch.float32, device=q.device)
    _need(workspace, "workspace", torch.float32)
    if out is None:
        out = torch.empty((B, n_q, H, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q.device)
    _need(out, "out", out_dtype, (B, n_q, H, d))
    _need(lse, "lse", torch.float32, (B, H, n_q))
    _same_device(q, k=k, v=v, workspace=workspace, out=out, lse=lse)
    with torch.cuda.device(q.device):
        check("ring_attn_decode", lib.ring_attn_decode(
            ctypes.byref(pr), int(n_q), int(q_pos0), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
            _ptr(lse), _ptr(workspace), ctypes.c_size_t(workspace.numel() * 4),
            _stream(q.device)))
    return out, lse


def empty_state(q: torch.Tensor):
    """Uninitialised (m, z, y) buffers for the step API (start with first=True)."""
    B, N, H, d = q.shape
    m = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    z = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    y = torch.empty((B, N, H, d), dtype=torch.float32, device=q.device)
    return m, z, y


def _step(fn_name, q, k, v, P, s, state, first, layout, causal, scale):
    lib = load()
    pr, (B, N, H, G, d) = _qkv_problem(q, k, v, P, layout, causal, scale)
    m, z, y = state
    _need(m, "m", torch.float32, (B, H, N))
    _need(z, "z", torch.float32, (B, H, N))
    _need(y, "y", torch.float32, (B, N, H, d))
    _same_device(q, m=m, z=z, y=y)
    with torch.cuda.device(q.device):
        check(fn_name, getattr(lib, fn_name)(ctypes.byref(pr), int(s), int(bool(first)), _ptr(q),
                                             _ptr(k), _ptr(v), _ptr(m), _ptr(z), _ptr(y),
                                             _stream(q.device)))
    return state


def step(q, k, v, P: int, s: int, state, first: bool, layout: str = "contiguous",
         causal: bool = True, scale: float = 0.0):
    """One ring step s for every virtual device (ring_attn_step); updates state in place."""
    return _step("ring_attn_step", q, k, v, P, s, state, first, layout, causal, scale)


def step_simt(q, k, v, P: int, s: int, state, first: bool, layout: str = "contiguous",
              causal: bool = True, scale: float = 0.0):
    """ring_attn_step_simt: the fp32 SIMT cross-check of step()."""
    return _step("ring_attn_step_simt", q, k, v, P, s, state, first, layout, causal, scale)


def finalize(state, P: int = 1, layout: str = "contiguous", causal: bool = True,
             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             out_dtype=torch.bfloat16):
    """(m, z, y) -> (O, LSE) (ring_attn_finalize); O in out_dtype (bf16 or fp32)."""
    lib = load()
    m, z, y = state
    B, N, H, d = y.shape
    _need(y, "y", torch.float32)
    _need(m, "m", torch.float32, (B, H, N))
    _need(z, "z", torch.float32, (B, H, N))
    if out is None:
        out = torch.empty((B, N, H, d), dtype=out_dtype, device=y.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=y.device)
    _need(out, "out", out_dtype, (B, N, H, d))
    _need(lse, "lse", torch.float32, (B, H, N))
    _same_device(y, m=m, z=z, out=out, lse=lse)
    pr = problem(B, N, H, H, d, P, causal, layout, 0.0, out_dtype)
    with torch.cuda.device(y.device):
        check("ring_attn_finalize", lib.ring_attn_finalize(ctypes.byref(pr), _ptr(m), _ptr(z),
                                                           _ptr(y), _ptr(out), _ptr(lse),
                                                           _stream(y.device)))
    return out, lse


def merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out: Optional[torch.Tensor] = None,
          lse: Optional[torch.Tensor] = None):
    """Merge n normalised partials (ring_attn_merge). Returns (O bf16, LSE fp32)."""
    lib = load()
    if o_parts.dim() != 5:
        raise ValueError("o_parts must be [n, B, N, H, d]")
    n, B, N, H, d = o_parts.shape
    _need(o_parts, "o_parts", torch.float32)
    _need(lse_parts, "lse_parts", torch.float32, (n, B, H, N))
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=o_parts.device)
    _need(out, "out", torch.bfloat16, (B, N, H, d))
    _need(lse, "lse", torch.float32, (B, H, N))
    _same_device(o_parts, lse_parts=lse_parts, out=out, lse=lse)
    with torch.cuda.device(o_parts.device):
        check("ring_attn_merge", lib.ring_attn_merge(n, B, N, H, d, _ptr(o_parts), _ptr(lse_parts),
                                                     _ptr(out), _ptr(lse),
                                                     _stream(o_parts.device)))
    return out, lse


def shard_map(layout: str, seqlen: int, P: int):
    """Host shard maps (ring_attn_shard_map): owner[N], local[N], token_of[N] lists."""
    lib = load()
    arr = ctypes.c_int32 * seqlen
    own, loc, tok = arr(), arr(), arr()
    check("ring_attn_shard_map", lib.ring_attn_shard_map(LAYOUTS[layout], seqlen, P, own, loc,
                                                         tok))
    return list(own), list(loc), list(tok)


def shard_map_device(layout: str, seqlen: int, P: int, device="cuda"):
    """The same maps computed on the GPU (ring_attn_shard_map_device), as int32 tensors."""
    lib = load()
    device = torch.device(device)
    own = torch.empty(seqlen, dtype=torch.int32, device=device)
    loc = torch.empty_like(own)
    tok = torch.empty_like(own)
    with torch.cuda.device(device):
        check("ring_attn_shard_map_device",
              lib.ring_attn_shard_map_device(LAYOUTS[layout], seqlen, P, _ptr(own), _ptr(loc),
                                             _ptr(tok), _stream(device)))
    return own, loc, tok


def tile_classes(pr: _lib.RaProblem, u: int, b: int, device="cuda") -> torch.Tensor:
    """Tile classes of shard pair (u, b) as the kernels see them (int8 [nt, nt])."""
    lib = load()
    device = torch.device(device)
    S = pr.seqlen // pr.P
    nt = (S + TILE - 1) // TILE
    out = torch.empty((nt, nt), dtype=torch.int8, device=device)
    with torch.cuda.device(device):
        check("ring_attn_tile_classes",
              lib.ring_attn_tile_classes(ctypes.byref(pr), u, b, _ptr(out), _stream(device)))
    return out


def mask(pr: _lib.RaProblem, u: int, b: int, device="cuda") -> torch.Tensor:
    """Element mask of shard pair (u, b) from the kernels' visibility rule (uint8 [S, S])."""
    lib = load()
    device = torch.device(device)
    S = pr.seqlen // pr.P
    out = torch.empty((S, S), dtype=torch.uint8, device=device)
    with torch.cuda.device(device):
        check("ring_attn_mask", lib.ring_attn_mask(ctypes.byref(pr), u, b, _ptr(out),
                                                   _stream(device)))
    return out


def last_error(device="cuda") -> int:
    """Read and clear the GPU's status word (call after synchronising)."""
    lib = load()
    code = ctypes.c_int32(0)
    with torch.cuda.device(torch.device(device)):
        check("ring_attn_last_error", lib.ring_attn_last_error(ctypes.byref(code)))
    return int(code.value)


def debug_checks() -> bool:
    """True if the loaded library is the debug build (kernels check their indices)."""
    return bool(load().ring_attn_debug_checks())


def selftest_bounds(device="cuda") -> None:
    """Launch the index-check self test: a debug build records RA_ERR_BOUNDS, a
    release build nothing (no memory is accessed either way)."""
    lib = load()
    device = torch.device(device)
    with torch.cuda.device(device):
        check("ring_attn_selftest_bounds", lib.ring_attn_selftest_bounds(_stream(device)))


def selftest_timeout(limit_ns: int, device="cuda") -> None:
    """Launch the bounded-wait self test (it records RA_ERR_TIMEOUT after limit_ns)."""
    lib = load()
    device = torch.device(device)
    with torch.cuda.device(device):
        check("ring_attn_selftest_timeout",
              lib.ring_attn_selftest_timeout(int(limit_ns), _stream(device)))


def selftest_wait_limit(limit_ns: int) -> None:
    """Test hook (ring_attn_selftest_wait_limit): the time limit of every device-side
    wait in the kernels of later calls; 0 restores the default (2 s). A few
    nanoseconds make the kernels' real waits run out, exercising their abort path."""
    check("ring_attn_selftest_wait_limit", load().ring_attn_selftest_wait_limit(int(limit_ns)))
