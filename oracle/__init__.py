"""Plain CPU fp64 oracle for the chunk-forward kkt_solve step of Gated DeltaNet.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's
CPU-baseline / reference leg may import this module; the product path never
does.  It shares no code with the CUDA path.  The arithmetic lives in
``kkt_solve_oracle.c`` (dense explicit loops in double precision); this file
compiles it with gcc, loads it with ctypes and converts inputs to float64
(bf16 -> float64 is exact).  See the header of ``kkt_solve_oracle.c`` for the
definition and the passages it follows.
"""
from __future__ import annotations

import concurrent.futures as _cf
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kkt_solve_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_kkt_solve.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build (plain gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d, i64, vp = ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p
            lib.oracle_kkt_solve_chunk.argtypes = [i64, i64, i64, d, i64, d, i64, d, i64, d, i64]
            lib.oracle_kkt_solve_chunk.restype = ctypes.c_int
            lib.oracle_kkt_solve.argtypes = [d, d, d, vp, i64, i64, i64, i64, i64, d, i64, i64]
            lib.oracle_kkt_solve.restype = ctypes.c_int
            lib.oracle_chunk_A_chunk.argtypes = [i64, i64, i64, d, i64, d, i64, d, i64, d, i64]
            lib.oracle_chunk_A_chunk.restype = ctypes.c_int
            lib.oracle_solve_tril_chunk.argtypes = [i64, i64, d, i64, d, i64]
            lib.oracle_solve_tril_chunk.restype = ctypes.c_int
            lib.oracle_chunk_A.argtypes = [d, d, d, vp, i64, i64, i64, i64, i64, d, i64, i64]
            lib.oracle_chunk_A.restype = ctypes.c_int
            lib.oracle_solve_tril.argtypes = [d, vp, i64, i64, i64, i64, d, i64, i64]
            lib.oracle_solve_tril.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):              # torch tensor (any float dtype, CPU)
        import torch
        return np.ascontiguousarray(x.detach().cpu().to(torch.float64).numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def kkt_solve_ref(k, g=None, beta=None, cu_seqlens=None, chunk_size: int = 64,
                  threads: int | None = None) -> np.ndarray:
    """(I + A)^{-1} for every chunk and head, in float64.

    k: [B, T, H, K] (or [1, T, H, K] with cu_seqlens [N+1]); g, beta: [B, T, H]
    or None.  Returns [B, T, H, chunk_size]; rows outside every sequence are 0.
    Heads are split over ``threads`` host threads (each runs the same plain loop
    on its own heads)."""
    lib = _load()
    kd = _f64(k)
    lead = kd.shape[:2]
    H, K = kd.shape[2], kd.shape[3]
    ntok = lead[0] * lead[1]
    kd = kd.reshape(ntok, H, K)
    gd = None if g is None else _f64(g).reshape(ntok, H)
    bd = None if beta is None else _f64(beta).reshape(ntok, H)
    out = np.zeros((ntok, H, chunk_size), dtype=np.float64)
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int32))
        nseq, T = len(cu) - 1, lead[1]
    else:
        cu, nseq, T = None, lead[0], lead[1]
    threads = max(1, min(threads or os.cpu_count() or 1, H))
    bounds = [(H * t // threads, H * (t + 1) // threads) for t in range(threads)]

    def run(hb, he):
        return lib.oracle_kkt_solve(_ptr(kd), _ptr(gd), _ptr(bd), _ptr(cu), nseq, T, H, K,
                                    chunk_size, _ptr(out), hb, he)

    if threads == 1:
        rcs = [run(0, H)]
    else:
        with _cf.ThreadPoolExecutor(threads) as ex:
            rcs = list(ex.map(lambda b: run(*b), bounds))
    if any(rcs):
        raise RuntimeError(f"oracle failed: {rcs}")
    return out.reshape(*lead, H, chunk_size)


def kkt_solve_ref_tiles(k, g, beta, tiles, chunk_size: int = 64, threads: int | None = None):
    """The oracle on selected tiles only.  ``tiles`` holds (n, c, h, row0, L)
    tuples (row0 = first token row of the chunk in the flattened token axis).
    Returns a list of float64 arrays of shape [L, chunk_size]."""
    lib = _load()
    H = k.shape[2]
    K = k.shape[3]
    kf = k.reshape(-1, H, K)
    gf = None if g is None else g.reshape(-1, H)
    bf = None if beta is None else beta.reshape(-1, H)

    def one(t):
        _, _, h, r0, L = t
        kc = _f64(kf[r0:r0 + L, h, :])
        gc = None if gf is None else _f64(gf[r0:r0 + L, h])
        bc = None if bf is None else _f64(bf[r0:r0 + L, h])
        o = np.zeros((L, chunk_size), dtype=np.float64)
        rc = lib.oracle_kkt_solve_chunk(L, chunk_size, K, _ptr(kc), K, _ptr(gc), 1, _ptr(bc), 1,
                                        _ptr(o), chunk_size)
        if rc:
            raise RuntimeError("oracle chunk failed")
        return o

    threads = max(1, threads or os.cpu_count() or 1)
    if threads == 1 or len(tiles) < 8:
        return [one(t) for t in tiles]
    with _cf.ThreadPoolExecutor(threads) as ex:
        return list(ex.map(one, tiles))


def kkt_solve_ref_chunk(kc, gc=None, bc=None, chunk_size: int = 64) -> np.ndarray:
    """One chunk given directly: kc [L, K], gc/bc [L] or None -> [L, chunk_size]."""
    lib = _load()
    kd = _f64(kc)
    L, K = kd.shape
    gd = None if gc is None else _f64(gc).reshape(L)
    bd = None if bc is None else _f64(bc).reshape(L)
    o = np.zeros((L, chunk_size), dtype=np.float64)
    rc = lib.oracle_kkt_solve_chunk(L, chunk_size, K, _ptr(kd), K, _ptr(gd), 1, _ptr(bd), 1,
                                    _ptr(o), chunk_size)
    if rc:
        raise RuntimeError("oracle chunk failed")
    return o


def _layout(lead, cu_seqlens):
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int32))
        return cu, len(cu) - 1, lead[1]
    return None, lead[0], lead[1]


def _over_heads(H, threads, run):
    threads = max(1, min(threads or os.cpu_count() or 1, H))
    bounds = [(H * t // threads, H * (t + 1) // threads) for t in range(threads)]
    if threads == 1:
        rcs = [run(0, H)]
    else:
        with _cf.ThreadPoolExecutor(threads) as ex:
            rcs = list(ex.map(lambda b: run(*b), bounds))
    if any(rcs):
        raise RuntimeError(f"oracle failed: {rcs}")


def chunk_A_ref(k, g=None, beta=None, cu_seqlens=None, chunk_size: int = 64,
                threads: int | None = None) -> np.ndarray:
    """A of every chunk and head in float64, in the page's layout [B, T, H, chunk]:
    A[i][j] = beta_i (k_i . k_j) exp(g_i - g_j) for j < i, zero elsewhere; rows
    outside every sequence are 0."""
    lib = _load()
    kd = _f64(k)
    lead = kd.shape[:2]
    H, K = kd.shape[2], kd.shape[3]
    ntok = lead[0] * lead[1]
    kd = kd.reshape(ntok, H, K)
    gd = None if g is None else _f64(g).reshape(ntok, H)
    bd = None if beta is None else _f64(beta).reshape(ntok, H)
    A = np.zeros((ntok, H, chunk_size), dtype=np.float64)
    cu, nseq, T = _layout(lead, cu_seqlens)
    _over_heads(H, threads, lambda hb, he: lib.oracle_chunk_A(
        _ptr(kd), _ptr(gd), _ptr(bd), _ptr(cu), nseq, T, H, K, chunk_size, _ptr(A), hb, he))
    return A.reshape(*lead, H, chunk_size)


def solve_tril_ref(A, cu_seqlens=None, chunk_size: int = 64, threads: int | None = None) -> np.ndarray:
    """(I + A)^{-1} of every chunk and head from a given A [B, T, H, chunk]
    (only its strictly lower part inside each chunk is read), in float64."""
    lib = _load()
    Ad = _f64(A)
    lead = Ad.shape[:2]
    H = Ad.shape[2]
    ntok = lead[0] * lead[1]
    Ad = np.ascontiguousarray(Ad.reshape(ntok, H, chunk_size))
    out = np.zeros((ntok, H, chunk_size), dtype=np.float64)
    cu, nseq, T = _layout(lead, cu_seqlens)
    _over_heads(H, threads, lambda hb, he: lib.oracle_solve_tril(
        _ptr(Ad), _ptr(cu), nseq, T, H, chunk_size, _ptr(out), hb, he))
    return out.reshape(*lead, H, chunk_size)
