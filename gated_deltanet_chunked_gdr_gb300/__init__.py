"""GB300 (sm_103a) chunk-forward kkt_solve of Gated DeltaNet.

Thin Python binding over the C ABI declared in include/gdr_kkt_solve.h.  This
module only marshals arguments (pointers, sizes, the current CUDA stream);
every step of the computation runs in the CUDA library.  There is no CPU
fallback: if the library is missing or no sm_103 GPU is present, calls raise.

Python signature mirrors the API of the MindSpeed-Ops PR #135 page ("feat(triton):
add chunk_gated_delta_rule_fwd_kkt_solve", API block):
    kkt_solve(k, g=None, beta=None, cu_seqlens=None, chunk_size=64, output_dtype=None)
    -> (I + A)^{-1} as [B, T, H, 64]
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

GDR_OK = 0
GDR_ERR_NULL = -1
GDR_ERR_SHAPE = -2
GDR_ERR_CHUNK = -3
GDR_ERR_DTYPE = -4
GDR_ERR_ALIGN = -5
GDR_ERR_DEVICE = -6
GDR_ERR_CUDA = -7
GDR_ERR_TIMEOUT = -8
GDR_ERR_SCRATCH = -9
GDR_ERR_CU_SEQLENS = -10
GDR_F32 = 0
GDR_BF16 = 1
GDR_F16 = 2

EXPORTED_SYMBOLS = ("gdr_kkt_solve", "gdr_kkt_solve_ex", "gdr_chunk_scaled_dot_kkt",
                    "gdr_solve_tril", "gdr_kkt_solve_unfused_noalloc", "gdr_kkt_solve_host",
                    "gdr_kkt_solve_host_workspace_bytes", "gdr_status_string",
                    "gdr_kkt_solve_device_status", "gdr_kkt_solve_num_sms", "gdr_selftest_bounded_wait",
                    "gdr_check_cu_seqlens")

_lib = None
_lock = threading.Lock()


class GdrError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load the compiled library (building it first if the sources are newer)."""
    global _lib
    with _lock:
        if _lib is None:
            if _build.needs_build():
                _build.build()
            lib = ctypes.CDLL(_build.LIB_PATH)
            vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.gdr_kkt_solve.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ci, ci, vp, vp]
            lib.gdr_kkt_solve.restype = ci
            lib.gdr_kkt_solve_ex.argtypes = [vp, ci, vp, vp, ci, vp, i64, i64, i64, i64, ci, ci, vp, vp]
            lib.gdr_kkt_solve_ex.restype = ci
            lib.gdr_chunk_scaled_dot_kkt.argtypes = [vp, ci, vp, vp, ci, vp, i64, i64, i64, i64, ci, vp, vp]
            lib.gdr_chunk_scaled_dot_kkt.restype = ci
            lib.gdr_solve_tril.argtypes = [vp, vp, i64, i64, i64, ci, ci, vp, vp]
            lib.gdr_solve_tril.restype = ci
            lib.gdr_kkt_solve_unfused_noalloc.argtypes = [vp, ci, vp, vp, ci, vp, i64, i64, i64, i64, ci, ci,
                                                          vp, vp]
            lib.gdr_kkt_solve_unfused_noalloc.restype = ci
            lib.gdr_kkt_solve_host.argtypes = [vp, ci, vp, vp, ci, vp, i64, i64, i64, i64, ci, ci, vp, vp, i64,
                                               vp]
            lib.gdr_kkt_solve_host.restype = ci
            lib.gdr_kkt_solve_host_workspace_bytes.argtypes = [ci, i64, i64, i64, i64, ci, ci]
            lib.gdr_kkt_solve_host_workspace_bytes.restype = i64
            lib.gdr_status_string.argtypes = [ci]
            lib.gdr_status_string.restype = ctypes.c_char_p
            lib.gdr_kkt_solve_device_status.argtypes = [ctypes.POINTER(ci)]
            lib.gdr_kkt_solve_device_status.restype = ci
            lib.gdr_selftest_bounded_wait.argtypes = [vp]
            lib.gdr_selftest_bounded_wait.restype = ci
            lib.gdr_check_cu_seqlens.argtypes = [vp, i64, i64, vp]
            lib.gdr_check_cu_seqlens.restype = ci
            lib.gdr_kkt_solve_num_sms.argtypes = []
            lib.gdr_kkt_solve_num_sms.restype = ci
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().gdr_status_string(int(status)).decode()


def kkt_solve_raw(k_ptr: int, g_ptr: int, beta_ptr: int, cu_ptr: int, B: int, T: int, H: int,
                  K: int, chunk_size: int, out_dtype: int, out_ptr: int, stream: int) -> int:
    """Direct C-ABI call with integer pointers; returns the gdr_status code."""
    return load_library().gdr_kkt_solve(k_ptr or None, g_ptr or None, beta_ptr or None,
                                        cu_ptr or None, B, T, H, K, chunk_size, out_dtype,
                                        out_ptr or None, stream or None)


def kkt_solve_ex_raw(k_ptr: int, k_dtype: int, g_ptr: int, beta_ptr: int, beta_dtype: int,
                     cu_ptr: int, B: int, T: int, H: int, K: int, chunk_size: int,
                     out_dtype: int, out_ptr: int, stream: int) -> int:
    """Direct call of gdr_kkt_solve_ex with integer pointers; returns the gdr_status code."""
    return load_library().gdr_kkt_solve_ex(k_ptr or None, k_dtype, g_ptr or None, beta_ptr or None,
                                           beta_dtype, cu_ptr or None, B, T, H, K, chunk_size,
                                           out_dtype, out_ptr or None, stream or None)


def chunk_scaled_dot_kkt_raw(k_ptr: int, k_dtype: int, g_ptr: int, beta_ptr: int, beta_dtype: int,
                             cu_ptr: int, B: int, T: int, H: int, K: int, chunk_size: int,
                             A_ptr: int, stream: int) -> int:
    """Direct call of gdr_chunk_scaled_dot_kkt with integer pointers; returns the status."""
    return load_library().gdr_chunk_scaled_dot_kkt(k_ptr or None, k_dtype, g_ptr or None,
                                                   beta_ptr or None, beta_dtype, cu_ptr or None,
                                                   B, T, H, K, chunk_size, A_ptr or None,
                                                   stream or None)


def solve_tril_raw(A_ptr: int, cu_ptr: int, B: int, T: int, H: int, chunk_size: int,
                   out_dtype: int, out_ptr: int, stream: int) -> int:
    """Direct call of gdr_solve_tril with integer pointers; returns the status."""
    return load_library().gdr_solve_tril(A_ptr or None, cu_ptr or None, B, T, H, chunk_size,
                                         out_dtype, out_ptr or None, stream or None)


def kkt_solve_unfused_noalloc_raw(k_ptr: int, k_dtype: int, g_ptr: int, beta_ptr: int,
                                  beta_dtype: int, cu_ptr: int, B: int, T: int, H: int, K: int,
                                  chunk_size: int, out_dtype: int, out_ptr: int, stream: int) -> int:
    """Direct call of gdr_kkt_solve_unfused_noalloc (the allocation-free chain, for
    callers that may not allocate device memory while running; at most 262144
    token-heads per call); returns the gdr_status code."""
    return load_library().gdr_kkt_solve_unfused_noalloc(k_ptr or None, k_dtype, g_ptr or None,
                                                        beta_ptr or None, beta_dtype, cu_ptr or None,
                                                        B, T, H, K, chunk_size, out_dtype,
                                                        out_ptr or None, stream or None)


def kkt_solve_host_raw(k_ptr: int, k_dtype: int, g_ptr: int, beta_ptr: int, beta_dtype: int, cu_ptr: int,
                       B: int, T: int, H: int, K: int, chunk_size: int, out_dtype: int, out_ptr: int,
                       ws_ptr: int, ws_bytes: int, stream: int) -> int:
    """Direct call of gdr_kkt_solve_host (host input and output pointers, a device
    workspace); returns the gdr_status code."""
    return load_library().gdr_kkt_solve_host(k_ptr or None, k_dtype, g_ptr or None, beta_ptr or None,
                                             beta_dtype, cu_ptr or None, B, T, H, K, chunk_size, out_dtype,
                                             out_ptr or None, ws_ptr or None, ws_bytes, stream or None)


def kkt_solve_host_workspace_bytes(k_dtype: int, B: int, T: int, H: int, K: int, chunk_size: int,
                                   out_dtype: int) -> int:
    """Device workspace bytes gdr_kkt_solve_host needs (raises on invalid arguments)."""
    n = load_library().gdr_kkt_solve_host_workspace_bytes(k_dtype, B, T, H, K, chunk_size, out_dtype)
    if n < 0:
        raise GdrError(int(n), "gdr_kkt_solve_host_workspace_bytes")
    return int(n)


def check_cu_seqlens_raw(cu_ptr: int, B: int, T: int, stream: int) -> int:
    """Direct call of gdr_check_cu_seqlens (enqueues the device-side check of the
    packed-sequence contract); returns the gdr_status code of the enqueue."""
    return load_library().gdr_check_cu_seqlens(cu_ptr or None, B, T, stream or None)


def check_cu_seqlens(cu_seqlens, T: int, stream=None) -> None:
    """Enqueues the device-side check that cu_seqlens (int32 [B + 1] CUDA tensor)
    starts at 0, never decreases and ends at most at T.  A broken array is
    reported as GDR_ERR_CU_SEQLENS by the next device_status()."""
    import torch

    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_cuda:
        raise TypeError("cu_seqlens must be a 1-D int32 CUDA tensor")
    cu_seqlens = cu_seqlens.contiguous()
    if stream is None:
        stream = torch.cuda.current_stream(cu_seqlens.device).cuda_stream
    with torch.cuda.device(cu_seqlens.device):
        rc = check_cu_seqlens_raw(cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, int(T), int(stream))
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_check_cu_seqlens")


def _gdr_dtype(dt, what: str) -> int:
    import torch

    table = {torch.float32: GDR_F32, torch.bfloat16: GDR_BF16, torch.float16: GDR_F16}
    if dt not in table:
        raise TypeError(f"{what} must be torch.float32, torch.bfloat16 or torch.float16")
    return table[dt]


def device_status() -> int:
    """Reads and clears the device-side status word (synchronises the device)."""
    v = ctypes.c_int(0)
    rc = load_library().gdr_kkt_solve_device_status(ctypes.byref(v))
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_kkt_solve_device_status")
    return v.value


def selftest_bounded_wait(stream: int = 0) -> int:
    """Enqueues the bounded-wait self-test kernel (see the C header); returns the status."""
    return load_library().gdr_selftest_bounded_wait(stream or None)


def num_sms() -> int:
    rc = load_library().gdr_kkt_solve_num_sms()
    if rc < 0:
        raise GdrError(rc, "gdr_kkt_solve_num_sms")
    return rc


def kkt_solve(k, g=None, beta=None, cu_seqlens=None, chunk_size: int = 64, output_dtype=None,
              out=None, stream=None, validate_cu_seqlens: bool = False):
    """(I + A)^{-1} of every 64-token chunk and head, on the GPU.

    k: bf16 or fp16 [B, T, H, K] CUDA tensor, K in {64, 128, 192, 256}
    (K in {64, 128} for chunk_size 128), or fp32 with K in {64, 128} and
    chunk_size 64
    ([1, T, H, K] with cu_seqlens); g: fp32 [B, T, H] or None; beta: fp32,
    bf16 or fp16 [B, T, H] or None; cu_seqlens: int32 [N + 1] CUDA tensor or
    None; output_dtype: torch.float32 (default), torch.bfloat16 or
    torch.float16; chunk_size: 64 or 128.  validate_cu_seqlens=True first
    enqueues the device-side check of the cu_seqlens contract (see
    check_cu_seqlens).  Returns out [B, T, H, chunk_size]."""
    import torch

    if chunk_size not in (64, 128):
        raise ValueError("chunk_size must be 64 or 128")
    if output_dtype is None:
        output_dtype = torch.float32
    out_code = _gdr_dtype(output_dtype, "output_dtype")
    if k.dtype not in (torch.bfloat16, torch.float16, torch.float32) or k.dim() != 4 or not k.is_cuda:
        raise TypeError("k must be a 4-D bf16, fp16 or fp32 CUDA tensor")
    k_code = _gdr_dtype(k.dtype, "k")
    beta_code = GDR_F32 if beta is None else _gdr_dtype(beta.dtype, "beta")
    for name, t, dt in (("g", g, torch.float32), ("cu_seqlens", cu_seqlens, torch.int32)):
        if t is not None and (t.dtype != dt or t.device != k.device):
            raise TypeError(f"{name} must be a {dt} tensor on {k.device}")
    if beta is not None and beta.device != k.device:
        raise TypeError(f"beta must be on {k.device}")
    Bk, T, H, K = k.shape
    if cu_seqlens is not None:
        if Bk != 1 or cu_seqlens.dim() != 1:
            raise ValueError("with cu_seqlens, k must be [1, T, H, K] and cu_seqlens 1-D")
        B = cu_seqlens.numel() - 1
    else:
        B = Bk
    for name, t in (("g", g), ("beta", beta)):
        if t is not None and tuple(t.shape) != (Bk, T, H):
            raise ValueError(f"{name} must have shape {(Bk, T, H)}")
    k = k.contiguous()
    g = None if g is None else g.contiguous()
    beta = None if beta is None else beta.contiguous()
    cu_seqlens = None if cu_seqlens is None else cu_seqlens.contiguous()
    if out is None:
        out = torch.empty((Bk, T, H, chunk_size), dtype=output_dtype, device=k.device)
    elif out.dtype != output_dtype or tuple(out.shape) != (Bk, T, H, chunk_size) or not out.is_contiguous():
        raise ValueError("out has the wrong dtype, shape or layout")
    if stream is None:
        stream = torch.cuda.current_stream(k.device).cuda_stream
    if validate_cu_seqlens and cu_seqlens is not None:
        check_cu_seqlens(cu_seqlens, T, stream)
    with torch.cuda.device(k.device):
        rc = kkt_solve_ex_raw(k.data_ptr(), k_code, 0 if g is None else g.data_ptr(),
                              0 if beta is None else beta.data_ptr(), beta_code,
                              0 if cu_seqlens is None else cu_seqlens.data_ptr(),
                              B, T, H, K, chunk_size, out_code, out.data_ptr(), int(stream))
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_kkt_solve_ex")
    return out


def kkt_solve_host(k, g=None, beta=None, cu_seqlens=None, chunk_size: int = 64, output_dtype=None,
                   out=None, workspace=None, stream=None, device=None):
    """kkt_solve on HOST tensors (gdr_kkt_solve_host): k, g, beta, cu_seqlens are
    CPU tensors (page-locked for overlapped copies), out a CPU tensor or None
    (then a page-locked one is allocated).  `workspace` is a uint8 CUDA tensor of
    at least kkt_solve_host_workspace_bytes(...) bytes, or None (then one is
    allocated on `device`, default the current CUDA device, and kept from reuse
    until `stream` has passed the call); a workspace passed in must not be used
    for anything else until then.  The call is asynchronous on `stream` (default
    the device's current stream): synchronise it before reading out.  Returns
    out [B, T, H, chunk_size]."""
    import torch

    if output_dtype is None:
        output_dtype = torch.float32
    out_code = _gdr_dtype(output_dtype, "output_dtype")
    if k.dim() != 4 or k.is_cuda:
        raise TypeError("k must be a 4-D CPU tensor")
    for name, t in (("g", g), ("beta", beta), ("cu_seqlens", cu_seqlens)):
        if t is not None and t.is_cuda:
            raise TypeError(f"{name} must be a CPU tensor")
    if g is not None and g.dtype != torch.float32:
        raise TypeError("g must be float32")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    k_code = _gdr_dtype(k.dtype, "k")
    beta_code = GDR_F32 if beta is None else _gdr_dtype(beta.dtype, "beta")
    Bk, T, H, K = k.shape
    B = Bk if cu_seqlens is None else cu_seqlens.numel() - 1
    k = k.contiguous()
    g = None if g is None else g.contiguous()
    beta = None if beta is None else beta.contiguous()
    cu_seqlens = None if cu_seqlens is None else cu_seqlens.contiguous()
    if out is not None and (out.is_cuda or out.dtype != output_dtype or tuple(out.shape) != (Bk, T, H, chunk_size)
                            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous CPU tensor of the output's dtype and shape")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty((Bk, T, H, chunk_size), dtype=output_dtype, pin_memory=True)
    need = kkt_solve_host_workspace_bytes(k_code, B, T, H, K, chunk_size, out_code)
    own_workspace = workspace is None
    if own_workspace:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        rc = kkt_solve_host_raw(k.data_ptr(), k_code, 0 if g is None else g.data_ptr(),
                                0 if beta is None else beta.data_ptr(), beta_code,
                                0 if cu_seqlens is None else cu_seqlens.data_ptr(), B, T, H, K, chunk_size,
                                out_code, out.data_ptr(), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), int(stream))
    if own_workspace:
        # The call's internal streams use the workspace; the caller's stream waits
        # for them, so the allocator may reuse it once that stream passes here.
        workspace.record_stream(torch.cuda.ExternalStream(int(stream), device=dev))
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_kkt_solve_host")
    return out


def _check_inputs(k, g, beta, cu_seqlens, chunk_size):
    import torch

    if chunk_size != 64:
        raise ValueError("chunk_size must be 64")
    if k.dtype not in (torch.bfloat16, torch.float16) or k.dim() != 4 or not k.is_cuda:
        raise TypeError("k must be a 4-D bf16 or fp16 CUDA tensor")
    for name, t, dt in (("g", g, torch.float32), ("cu_seqlens", cu_seqlens, torch.int32)):
        if t is not None and (t.dtype != dt or t.device != k.device):
            raise TypeError(f"{name} must be a {dt} tensor on {k.device}")
    if beta is not None and beta.device != k.device:
        raise TypeError(f"beta must be on {k.device}")
    Bk, T, H, _ = k.shape
    for name, t in (("g", g), ("beta", beta)):
        if t is not None and tuple(t.shape) != (Bk, T, H):
            raise ValueError(f"{name} must have shape {(Bk, T, H)}")
    if cu_seqlens is not None and (Bk != 1 or cu_seqlens.dim() != 1):
        raise ValueError("with cu_seqlens, k must be [1, T, H, K] and cu_seqlens 1-D")
    return cu_seqlens.numel() - 1 if cu_seqlens is not None else Bk


def chunk_scaled_dot_kkt(k, g=None, beta=None, cu_seqlens=None, chunk_size: int = 64, A=None,
                         stream=None):
    """The unfused chain's first half: A [B, T, H, 64] fp32 with
    A[i][j] = beta_i (k_i . k_j) exp(g_i - g_j) for j < i, zero elsewhere."""
    import torch

    B = _check_inputs(k, g, beta, cu_seqlens, chunk_size)
    Bk, T, H, K = k.shape
    k = k.contiguous()
    g = None if g is None else g.contiguous()
    beta = None if beta is None else beta.contiguous()
    if A is None:
        A = torch.empty((Bk, T, H, 64), dtype=torch.float32, device=k.device)
    elif A.dtype != torch.float32 or tuple(A.shape) != (Bk, T, H, 64) or not A.is_contiguous():
        raise ValueError("A has the wrong dtype, shape or layout")
    if stream is None:
        stream = torch.cuda.current_stream(k.device).cuda_stream
    with torch.cuda.device(k.device):
        rc = chunk_scaled_dot_kkt_raw(k.data_ptr(), _gdr_dtype(k.dtype, "k"),
                                      0 if g is None else g.data_ptr(),
                                      0 if beta is None else beta.data_ptr(),
                                      GDR_F32 if beta is None else _gdr_dtype(beta.dtype, "beta"),
                                      0 if cu_seqlens is None else cu_seqlens.contiguous().data_ptr(),
                                      B, T, H, K, chunk_size, A.data_ptr(), int(stream))
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_chunk_scaled_dot_kkt")
    return A


def solve_tril(A, cu_seqlens=None, chunk_size: int = 64, output_dtype=None, out=None, stream=None):
    """The unfused chain's second half: (I + A)^{-1} of every chunk from A
    [B, T, H, 64] fp32 (only each chunk's strictly lower part is read)."""
    import torch

    if chunk_size != 64:
        raise ValueError("chunk_size must be 64")
    if A.dtype != torch.float32 or A.dim() != 4 or A.shape[3] != 64 or not A.is_cuda:
        raise TypeError("A must be a [B, T, H, 64] fp32 CUDA tensor")
    if output_dtype is None:
        output_dtype = torch.float32
    out_code = _gdr_dtype(output_dtype, "output_dtype")
    Bk, T, H, _ = A.shape
    if cu_seqlens is not None:
        if Bk != 1 or cu_seqlens.dim() != 1 or cu_seqlens.dtype != torch.int32:
            raise ValueError("with cu_seqlens, A must be [1, T, H, 64] and cu_seqlens 1-D int32")
        B = cu_seqlens.numel() - 1
    else:
        B = Bk
    A = A.contiguous()
    if out is None:
        out = torch.empty((Bk, T, H, 64), dtype=output_dtype, device=A.device)
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    with torch.cuda.device(A.device):
        rc = solve_tril_raw(A.data_ptr(), 0 if cu_seqlens is None else cu_seqlens.contiguous().data_ptr(),
                            B, T, H, chunk_size, out_code, out.data_ptr(), int(stream))
    if rc != GDR_OK:
        raise GdrError(rc, "gdr_solve_tril")
    return out


__all__ = ["kkt_solve", "chunk_scaled_dot_kkt", "solve_tril", "kkt_solve_raw", "kkt_solve_ex_raw",
           "chunk_scaled_dot_kkt_raw", "solve_tril_raw", "kkt_solve_unfused_noalloc_raw", "check_cu_seqlens",
           "check_cu_seqlens_raw", "device_status", "num_sms", "build", "load_library",
           "status_string", "GdrError", "EXPORTED_SYMBOLS"]
