"""The fp64 oracle on many sampled query rows of a large problem, spread over
worker processes.

Test infrastructure. The workers run `oracle.attention.attention_at` as it stands
on exact copies of the bf16 inputs (every bf16 value is exact in fp32 and fp64);
nothing from the GPU result enters them. A task is a run of position-sorted rows of
one (sequence, kv head). The workers are started with the `spawn` method, so they
are safe to create after CUDA was initialised in the parent; the key and value rows
reach them as fp64 .npy files that every worker maps (RAM-backed when there is room),
not through pipes.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os
import tempfile
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

RowSet = Tuple[np.ndarray, np.ndarray]          # (token positions [R], q rows fp32 [R, d])


def _available_bytes() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 16 << 30


_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _task(args):
    kpath, vpath, causal, scale, rows, qr, block = args
    from oracle.attention import attention_at
    K = np.load(kpath, mmap_mode="r")[None, :, None, :]     # [1, N, 1, d] fp64
    V = np.load(vpath, mmap_mode="r")[None, :, None, :]
    N, d = K.shape[1], K.shape[3]
    O = np.empty((len(rows), d))
    L = np.empty(len(rows))
    # The rows come in position order. Under the causal mask a block's rows see no key
    # past its last row, so the oracle is given only the keys up to there: the keys
    # left out would each add exactly zero to its sums (and nothing to its max).
    for i in range(0, len(rows), block):
        rr = rows[i:i + block]
        n_keys = int(rr.max()) + 1 if causal else N
        o, lse = attention_at(qr[i:i + block][None, :, None, :], rr, [0], 1, K[:, :n_keys],
                              V[:, :n_keys], causal, scale, max_chunk_elems=len(rr) * n_keys)
        O[i:i + len(rr)] = o[0, :, 0, :]
        L[i:i + len(rr)] = lse[0, 0, :]
    return O, L


def _scratch_dir(need: int) -> Optional[str]:
    """A RAM-backed directory with room for `need` bytes, else None (the default)."""
    import shutil
    try:
        if os.path.isdir("/dev/shm") and shutil.disk_usage("/dev/shm").free > 2 * need:
            return "/dev/shm"
    except OSError:
        pass
    return None


def oracle_rows(k_host: np.ndarray, v_host: np.ndarray, H: int,
                sel: Dict[Tuple[int, int], RowSet], causal: bool,
                scale: Optional[float] = None, workers: Optional[int] = None,
                timeout_s: float = 1200.0) -> Dict[Tuple[int, int], Tuple[np.ndarray, np.ndarray]]:
    """O [R, d] and LSE [R] (fp64) of the oracle for every (batch, query head) in
    `sel`, whose value holds the query rows' token positions and their q vectors.
    k_host, v_host: [B, N, G, d] fp32 host arrays with the exact input values.

    Rows of the query heads of one kv head are pooled (a row's attention depends
    only on its q vector, its position and that kv head), sorted by position and
    cut into blocks whose key prefix the oracle sees; the blocks of one kv head are
    split over tasks of about equal work."""
    from oracle.attention import kv_head_of
    B, N, G, d = k_host.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    pooled: Dict[Tuple[int, int], List] = {}
    for (b, h), (rows, qr) in sel.items():
        pooled.setdefault((b, kv_head_of(h, H, G)), []).append(
            (h, np.asarray(rows, dtype=np.int64), np.asarray(qr, dtype=np.float32)))
    results: Dict[Tuple[int, int], Tuple[np.ndarray, np.ndarray]] = {}
    if not pooled:
        return results
    # rows per block: about 2^26 scores of fp64 (a few such matrices live at once)
    block = int(max(8, min(512, (1 << 26) // max(N, 1))))
    per_worker = 4 * block * N * 8 + (1 << 28)
    cap = max(1, int(_available_bytes() // 2 // per_worker))
    target = max(1, min(workers or os.cpu_count() or 1, cap))
    kv_bytes = len(pooled) * 2 * N * d * 8
    with tempfile.TemporaryDirectory(prefix="oracle_rows_", dir=_scratch_dir(kv_bytes)) as tmp:
        tasks = []     # (key, order slice, args)
        parts = max(1, -(-target // len(pooled)))
        for (b, g), heads in sorted(pooled.items()):
            kp = os.path.join(tmp, f"k_{b}_{g}.npy")
            vp = os.path.join(tmp, f"v_{b}_{g}.npy")
            # fp64 files: every worker maps them (no per-task conversion copies)
            np.save(kp, np.ascontiguousarray(k_host[b, :, g, :], dtype=np.float64))
            np.save(vp, np.ascontiguousarray(v_host[b, :, g, :], dtype=np.float64))
            pos = np.concatenate([r for _, r, _ in heads])
            qs = np.concatenate([q for _, _, q in heads])
            tag = np.concatenate([np.full(len(r), i) for i, (_, r, _) in enumerate(heads)])
            idx = np.concatenate([np.arange(len(r)) for _, r, _ in heads])
            order = np.argsort(pos, kind="stable")
            # split into parts of about equal work (rows x visible keys)
            work = np.cumsum(pos[order] + 1 if causal else np.full(len(order), N))
            cuts = np.searchsorted(work, work[-1] * np.arange(1, parts) / parts)
            for sl in np.split(order, cuts):
                if len(sl):
                    tasks.append(((b, g, heads, tag[sl], idx[sl]),
                                  (kp, vp, causal, scale, pos[sl], qs[sl], block)))
        n = min(target, len(tasks))
        if n == 1:
            outs = [_task(a) for _, a in tasks]
        else:
            # One BLAS thread per worker (the pool supplies the parallelism): the workers
            # inherit these variables before their numpy loads. A worker that dies makes
            # the pool raise (BrokenProcessPool) instead of waiting.
            saved = {v: os.environ.get(v) for v in _BLAS_VARS}
            os.environ.update({v: "1" for v in _BLAS_VARS})
            try:
                with cf.ProcessPoolExecutor(n, mp_context=mp.get_context("spawn")) as ex:
                    outs = list(ex.map(_task, [a for _, a in tasks], timeout=timeout_s))
            finally:
                for v, val in saved.items():
                    if val is None:
                        os.environ.pop(v, None)
                    else:
                        os.environ[v] = val
        for ((b, g, heads, tg, ix), _), (O, L) in zip(tasks, outs):
            for i, (h, rows, _) in enumerate(heads):
                if (b, h) not in results:
                    results[(b, h)] = (np.empty((len(rows), d)), np.empty(len(rows)))
                m = tg == i
                results[(b, h)][0][ix[m]] = O[m]
                results[(b, h)][1][ix[m]] = L[m]
    return results


def gather_rows(t, sel_rows: Dict[Tuple[int, int], np.ndarray], layout: str):
    """Host fp64 copies of the selected rows of a GPU tensor: layout "bnhd" for q and o
    ([B, N, H, d]) gives {(b, h): [R, d]}, "bhn" for lse ([B, H, N]) gives {(b, h): [R]}."""
    import torch
    keys = sorted(sel_rows)
    bi = np.concatenate([np.full(len(sel_rows[k]), k[0]) for k in keys]).astype(np.int64)
    hi = np.concatenate([np.full(len(sel_rows[k]), k[1]) for k in keys]).astype(np.int64)
    ri = np.concatenate([np.asarray(sel_rows[k], dtype=np.int64) for k in keys])
    dev = t.device
    B_, H_, R_ = (torch.as_tensor(x, device=dev) for x in (bi, hi, ri))
    if layout == "bnhd":
        g = t[B_, R_, H_].float().cpu().numpy().astype(np.float64)
    else:
        g = t[B_, H_, R_].float().cpu().numpy().astype(np.float64)
    out, i = {}, 0
    for k in keys:
        r = len(sel_rows[k])
        out[k] = g[i:i + r]
        i += r
    return out


def row_sets(q, sel_rows: Dict[Tuple[int, int], np.ndarray]) -> Dict[Tuple[int, int], RowSet]:
    """(positions, exact fp32 q rows) for every selected (b, h)."""
    qs = gather_rows(q, sel_rows, "bnhd")
    return {k: (np.asarray(sel_rows[k], dtype=np.int64), qs[k].astype(np.float32))
            for k in sel_rows}


def errors(o_rows, lse_rows, ref) -> Tuple[float, float]:
    """Max |O - O_ref| and |LSE - LSE_ref| over every selected (b, h)."""
    eo = max(float(np.abs(o_rows[k] - ref[k][0]).max()) for k in ref)
    el = max(float(np.abs(lse_rows[k] - ref[k][1]).max()) for k in ref)
    return eo, el


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |x| (8 significant bits): the most that
    rounding a value of that size to bf16 can change it."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 8)
