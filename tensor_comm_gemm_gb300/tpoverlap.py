"""Python binding of libtpoverlap (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: torch tensors are turned into device pointers, the
current torch stream into a cudaStream_t, and status codes into exceptions.
The CUDA library is required: if ``libtpoverlap.so`` is missing or fails to
load, importing this module's functions raises; there is no fallback path.
"""

from __future__ import annotations

import array
import ctypes
import os
from typing import Optional, Sequence

from . import build as _build

TPO_BF16, TPO_FP8_E4M3 = 0, 1
TPO_ERR_INVALID_ARG, TPO_ERR_UNSUPPORTED = 1, 2
STATUS = {0: "TPO_OK", 1: "TPO_ERR_INVALID_ARG", 2: "TPO_ERR_UNSUPPORTED", 3: "TPO_ERR_CUDA",
          4: "TPO_ERR_TIMEOUT", 5: "TPO_ERR_OOM"}
TPO_TRACE_START, TPO_TRACE_END, TPO_TRACE_PUBLISH, TPO_TRACE_ACQUIRE = 0, 1, 2, 18
TPO_TRACE_WAIT_NS, TPO_TRACE_CHUNK_DONE, TPO_TRACE_WORDS = 34, 35, 128
TPO_TRACE_CYC_TMA_EMPTY, TPO_TRACE_CYC_MMA_FULL, TPO_TRACE_CYC_MMA_TEMPTY = 100, 101, 102
TPO_TRACE_CYC_EPI_TFULL, TPO_TRACE_CYC_GEMM, TPO_TRACE_KBLOCKS = 103, 104, 105
TPO_MAX_TP, TPO_MAX_ROW_CHUNKS = 16, 64

# Every symbol the public header declares.
EXPORTS = ["tpo_ctx_create", "tpo_ctx_destroy", "tpo_ag_gemm", "tpo_gemm_rs", "tpo_gemm_ar", "tpo_set_opt",
           "tpo_get_opt", "tpo_sync_status", "tpo_last_device_error", "tpo_last_error", "tpo_staging_ptr",
           "tpo_done_counters", "tpo_read_trace", "tpo_version", "tpo_ag_gemm_noalloc", "tpo_set_fp8_scales"]
TPO_NOALLOC_MAX_STAGING_BYTES = 32 << 20


class TpoError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s: %s" % (STATUS.get(status, str(status)), msg))
        self.status = status


_lib = None


def lib(path: Optional[str] = None):
    """Load libtpoverlap.so (raises if it is not built).  The environment
    variable TPO_LIBRARY names another build of the library to load instead."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("TPO_LIBRARY") or _build.LIB
    if not os.path.exists(path):
        raise ImportError("libtpoverlap.so not built (run tensor_comm_gemm_gb300.build.build()): " + path)
    L = ctypes.CDLL(path)
    p, i64, i32, u32p = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_uint32)
    L.tpo_ctx_create.argtypes = [i32, i64, i64, i64, i32]
    L.tpo_ctx_create.restype = p
    L.tpo_ctx_destroy.argtypes = [p]
    L.tpo_ag_gemm.argtypes = [p, p, p, p, p, p, p]
    L.tpo_gemm_rs.argtypes = [p, p, p, p, p]
    L.tpo_gemm_ar.argtypes = [p, p, p, p, i32, p]
    L.tpo_set_opt.argtypes = [p, ctypes.c_char_p, i64]
    L.tpo_get_opt.argtypes = [p, ctypes.c_char_p, ctypes.POINTER(i64)]
    L.tpo_sync_status.argtypes = [p]
    L.tpo_last_device_error.argtypes = [p, u32p]
    L.tpo_last_error.restype = ctypes.c_char_p
    L.tpo_staging_ptr.argtypes = [p]
    L.tpo_staging_ptr.restype = p
    L.tpo_done_counters.argtypes = [p, u32p]
    L.tpo_done_counters.restype = p
    L.tpo_read_trace.argtypes = [p, ctypes.POINTER(ctypes.c_uint64), i32]
    L.tpo_version.restype = ctypes.c_char_p
    L.tpo_ag_gemm_noalloc.argtypes = [i32, i64, i64, i64, i32, p, p, p, p, p, p]
    L.tpo_set_fp8_scales.argtypes = [p, p, p]
    L.tpo_set_fp8_scales.restype = ctypes.c_int
    L.tpo_ag_gemm_noalloc.restype = ctypes.c_int
    for name in ("tpo_ctx_destroy", "tpo_ag_gemm", "tpo_gemm_rs", "tpo_gemm_ar", "tpo_set_opt", "tpo_get_opt",
                 "tpo_sync_status", "tpo_last_device_error", "tpo_read_trace"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def tpo_last_error() -> str:
    return lib().tpo_last_error().decode()


def _check(st: int):
    if st != 0:
        raise TpoError(st, tpo_last_error())


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _ptr_array(ts: Sequence) -> array.array:
    """The pointers as a C array of 64-bit words (pass _addr of it; keep the
    array referenced until the call returns)."""
    return array.array("Q", [_ptr(t) for t in ts])


def _addr(a: array.array) -> int:
    return a.buffer_info()[0]


def _check_tensor(name, t, shape, elem_bytes):
    """Torch tensors handed to the C ABI must be dense CUDA tensors of the shape
    and element size the context expects: a strided view would be read as if it
    were row-major.  Raw integer pointers pass unchecked to the library's own
    argument checks.  A mismatch raises TpoError with TPO_ERR_INVALID_ARG."""
    if t is None or isinstance(t, int):
        return
    if t.is_cuda and t.element_size() == elem_bytes and t.numel() == shape[0] * shape[1] and t.is_contiguous():
        return
    why = None
    if not t.is_cuda:
        why = "must be a CUDA tensor"
    elif not t.is_contiguous():
        why = "must be contiguous (row-major)"
    elif t.element_size() != elem_bytes:
        why = "has %d-byte elements, expected %d" % (t.element_size(), elem_bytes)
    elif t.numel() != shape[0] * shape[1]:
        why = "has %d elements, expected %d x %d" % (t.numel(), shape[0], shape[1])
    if why:
        raise TpoError(TPO_ERR_INVALID_ARG, "%s %s" % (name, why))


_SIZES = {}      # context handle -> (tp, n, k, m, dtype), filled on first use


def _sizes(ctx):
    sz = _SIZES.get(ctx)
    if sz is None:
        sz = _SIZES[ctx] = tuple(tpo_get_opt(ctx, k) for k in ("tp", "n", "k", "m", "dtype"))
    return sz


def _stream(stream) -> int:
    if stream is None:
        import torch
        if _RAW_STREAM is not None:  # the current stream of the current device, as a raw handle
            return _RAW_STREAM(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _raw_stream_getter():
    try:
        import torch
        return getattr(torch._C, "_cuda_getCurrentRawStream", None)
    except Exception:
        return None


_RAW_STREAM = _raw_stream_getter()


def tpo_version() -> str:
    return lib().tpo_version().decode()


def tpo_ctx_create(tp: int, n: int, k: int, m: int, dtype: int) -> int:
    h = lib().tpo_ctx_create(tp, n, k, m, dtype)
    if not h:
        raise TpoError(-1, tpo_last_error())
    _SIZES.pop(h, None)
    return h


def tpo_ctx_destroy(ctx: int) -> None:
    _SIZES.pop(ctx, None)
    _check(lib().tpo_ctx_destroy(ctx))


def tpo_ag_gemm(ctx: int, x: Sequence, w, y, scale_inv_x=None, scale_inv_w=None, stream=None) -> None:
    tp, n, k, m, dt = _sizes(ctx)
    eb = 1 if dt == TPO_FP8_E4M3 else 2
    if len(x) != tp:
        raise TpoError(TPO_ERR_INVALID_ARG, "x must hold tp=%d chunks" % tp)
    for r, xr in enumerate(x):
        _check_tensor("x[%d]" % r, xr, (n // tp, k), eb)
    _check_tensor("w", w, (m, k), eb)
    _check_tensor("y", y, (n, m), 2)
    xa = _ptr_array(x)
    _check(lib().tpo_ag_gemm(ctx, _addr(xa), _ptr(w), _ptr(y), _ptr(scale_inv_x), _ptr(scale_inv_w),
                             _stream(stream)))


def _check_ksplit(ctx, x, w):
    tp, n, k, m, dt = _sizes(ctx)
    eb = 1 if dt == TPO_FP8_E4M3 else 2
    if len(x) != tp or len(w) != tp:
        raise TpoError(TPO_ERR_INVALID_ARG, "x and w must hold tp=%d slices each" % tp)
    for r in range(tp):
        _check_tensor("x[%d]" % r, x[r], (n, k // tp), eb)
        _check_tensor("w[%d]" % r, w[r], (m, k // tp), eb)
    return tp, n, m


def tpo_gemm_rs(ctx: int, x: Sequence, w: Sequence, y: Sequence, stream=None) -> None:
    tp, n, m = _check_ksplit(ctx, x, w)
    if len(y) != tp:
        raise TpoError(TPO_ERR_INVALID_ARG, "y must hold tp=%d row blocks" % tp)
    for b, yb in enumerate(y):
        _check_tensor("y[%d]" % b, yb, (n // tp, m), 2)
    xa, wa, ya = _ptr_array(x), _ptr_array(w), _ptr_array(y)
    _check(lib().tpo_gemm_rs(ctx, _addr(xa), _addr(wa), _addr(ya), _stream(stream)))


def tpo_gemm_ar(ctx: int, x: Sequence, w: Sequence, y, n_row_chunks: int, stream=None) -> None:
    tp, n, m = _check_ksplit(ctx, x, w)
    _check_tensor("y", y, (n, m), 2)
    xa, wa = _ptr_array(x), _ptr_array(w)
    _check(lib().tpo_gemm_ar(ctx, _addr(xa), _addr(wa), _ptr(y), n_row_chunks, _stream(stream)))


def tpo_set_fp8_scales(ctx: int, scale_inv_x, scale_inv_w) -> None:
    _check(lib().tpo_set_fp8_scales(ctx, _ptr(scale_inv_x), _ptr(scale_inv_w)))


def tpo_set_opt(ctx: int, key: str, value: int) -> None:
    _check(lib().tpo_set_opt(ctx, key.encode(), int(value)))


def tpo_get_opt(ctx: int, key: str) -> int:
    v = ctypes.c_int64()
    _check(lib().tpo_get_opt(ctx, key.encode(), ctypes.byref(v)))
    return v.value


def tpo_sync_status(ctx: int) -> int:
    """Returns the status code (0 = TPO_OK) instead of raising, since a device
    timeout is an expected outcome of the fault-injection options."""
    return lib().tpo_sync_status(ctx)


def tpo_last_device_error(ctx: int):
    out = (ctypes.c_uint32 * 4)()
    _check(lib().tpo_last_device_error(ctx, out))
    return list(out)


def tpo_staging_ptr(ctx: int) -> int:
    return lib().tpo_staging_ptr(ctx) or 0


def tpo_done_counters(ctx: int):
    t = ctypes.c_uint32()
    p = lib().tpo_done_counters(ctx, ctypes.byref(t))
    return (p or 0), t.value


def tpo_read_trace(ctx: int):
    out = (ctypes.c_uint64 * TPO_TRACE_WORDS)()
    _check(lib().tpo_read_trace(ctx, out, TPO_TRACE_WORDS))
    return list(out)


def tpo_ag_gemm_noalloc(tp: int, n: int, k: int, m: int, dtype: int, x: Sequence, w, y, scale_inv_x=None,
                        scale_inv_w=None, stream=None) -> None:
    """AG+GEMM with no device allocation (scratch in the library's static
    array); blocks until the call's work on the stream has finished."""
    xa = _ptr_array(x)
    _check(lib().tpo_ag_gemm_noalloc(tp, n, k, m, dtype, _addr(xa), _ptr(w), _ptr(y), _ptr(scale_inv_x),
                                     _ptr(scale_inv_w), _stream(stream)))
