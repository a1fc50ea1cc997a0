"""dense_packed_bit_gb300 -- fp32 dense GEMM, packed 2-bit GEMV / skinny GEMM and packed
4-bit GEMV on GB300.

Thin ctypes binding over libmm.so (the C ABI declared in include/mm.h).  The
functions keep the C names and argument order; tensors are torch CUDA tensors
(only their device pointers are passed) and `stream` defaults to torch's
current stream.  Every step of the computation runs in libmm's CUDA kernels:
there is no CPU or PyTorch fallback, and a missing or unloadable libmm.so is
an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "MMError", "load_library", "library_path", "mm_version", "mm_last_error",
    "mm_gemm_f32", "mm_gemm_f32_ex", "mm_gemv_packed2", "mm_gemv_packed2_ex",
    "mm_gemm_packed2", "mm_gemm_packed2_ex", "mm_gemv_packed4", "mm_gemv_packed4_ex",
    "mm_check_device_error", "mm_gemm_f32_splitk", "mm_gemm_f32_splitk_workspace", "mm_gemm_f32_splitk_noalloc",
    "MM_SPLITK_NOALLOC_MAX_FLOATS", "mm_gemm_f32_bias_act", "MM_ACT_NONE", "MM_ACT_GELU_TANH",
    "mm_gemv_packed2_strided_batched", "mm_gemv_packed2_strided_batched_ex", "mm_gemm_f32_bias_act_splitk",
    "mm_gemm_f32_split_plan", "mm_gemm_f32_splitk_ex", "mm_gemm_f32_splitk_workspace_ex", "mm_gemm_f32_split_plan_ex",
    "mm_probe_bounded_wait", "mm_attention_fwd", "mm_attention_bwd",
    "MM_OK", "MM_ERR_INVALID_ARG", "MM_ERR_UNSUPPORTED", "MM_ERR_CUDA", "MM_ERR_TIMEOUT",
    "MM_GEMM_AUTO", "MM_GEMM_FFMA", "MM_GEMM_TF32X3",
    "MM_DEQ_AUTO", "MM_DEQ_SELECT", "MM_DEQ_AFFINE", "MM_DEQ_MMA", "MM_DEQ_FP8", "MM_DEQ_TC", "MM_DEQ_MXF4",
]

MM_OK, MM_ERR_INVALID_ARG, MM_ERR_UNSUPPORTED, MM_ERR_CUDA, MM_ERR_TIMEOUT = 0, 1, 2, 3, 4
MM_GEMM_AUTO, MM_GEMM_FFMA, MM_GEMM_TF32X3 = 0, 1, 2
MM_DEQ_AUTO, MM_DEQ_SELECT, MM_DEQ_AFFINE, MM_DEQ_MMA, MM_DEQ_FP8, MM_DEQ_TC, MM_DEQ_MXF4 = 0, 1, 2, 3, 4, 5, 6
MM_SPLITK_NOALLOC_MAX_FLOATS = 4194304  # floats of the static split-K scratch (16 MiB), as in mm.h
MM_ACT_NONE, MM_ACT_GELU_TANH = 0, 1

_PKG = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None

# symbol -> (argtypes, restype); mirrors include/mm.h
_P, _I64, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int


class GemmOpts(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("tile", ctypes.c_int), ("splitk", ctypes.c_int), ("reserved", ctypes.c_int * 5)]


class GemvOpts(ctypes.Structure):
    _fields_ = [("split", ctypes.c_int), ("rows_per_lane", ctypes.c_int), ("warps", ctypes.c_int),
                ("dequant", ctypes.c_int), ("pdl", ctypes.c_int), ("weights_static", ctypes.c_int),
                ("independent", ctypes.c_int), ("staging", ctypes.c_int), ("reserved", ctypes.c_int * 4)]


class GemmPacked2Opts(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int), ("splitk", ctypes.c_int), ("pdl", ctypes.c_int),
                ("weights_static", ctypes.c_int), ("ntok", ctypes.c_int), ("reserved", ctypes.c_int * 3)]


class Gemv4Opts(ctypes.Structure):
    _fields_ = [("blocks", ctypes.c_int), ("pdl", ctypes.c_int), ("weights_static", ctypes.c_int),
                ("independent", ctypes.c_int), ("staging", ctypes.c_int), ("reserved", ctypes.c_int * 3)]


SIGNATURES = {
    "mm_version": ([], ctypes.c_int),
    "mm_last_error": ([], ctypes.c_char_p),
    "mm_gemm_f32": ([_I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P], ctypes.c_int),
    "mm_gemm_f32_ex": ([_I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _P,
                        ctypes.POINTER(GemmOpts)], ctypes.c_int),
    "mm_gemv_packed2": ([_P, _P, _P, _P, _I64, _I64, _P, _P], ctypes.c_int),
    "mm_gemv_packed2_ex": ([_P, _P, _P, _P, _I64, _I64, _P, _P, ctypes.POINTER(GemvOpts)], ctypes.c_int),
    "mm_gemm_packed2": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _P], ctypes.c_int),
    "mm_gemv_packed4": ([_P, _P, _P, _P, _I64, _I64, _P, _P], ctypes.c_int),
    "mm_gemv_packed4_ex": ([_P, _P, _P, _P, _I64, _I64, _P, _P, ctypes.POINTER(Gemv4Opts)], ctypes.c_int),
    "mm_gemm_packed2_ex": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _P, ctypes.POINTER(GemmPacked2Opts)],
                           ctypes.c_int),
    "mm_check_device_error": ([_P], ctypes.c_int),
    "mm_gemm_f32_splitk_workspace": ([_I64, _I64, _I64, _I, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "mm_gemm_f32_splitk": ([_I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I, _P, _I64, _P],
                           ctypes.c_int),
    "mm_gemm_f32_splitk_noalloc": ([_I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I, _P],
                                   ctypes.c_int),
    "mm_gemm_f32_bias_act": ([_I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I, _P, _I64, _P], ctypes.c_int),
    "mm_gemm_f32_split_plan": ([_I64, _I64, _I64, _I, _P, _P], ctypes.c_int),
    "mm_gemm_f32_splitk_ex": ([_I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I64, _I, _P, _I64, _P,
                               ctypes.POINTER(GemmOpts)], ctypes.c_int),
    "mm_gemm_f32_splitk_workspace_ex": ([_I64, _I64, _I64, _I, ctypes.POINTER(GemmOpts),
                                         ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "mm_gemm_f32_split_plan_ex": ([_I64, _I64, _I64, _I, ctypes.POINTER(GemmOpts), _P, _P], ctypes.c_int),
    "mm_gemm_f32_bias_act_splitk": ([_I, _I, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _I, _P, _I64, _I, _P, _I64,
                                     _P], ctypes.c_int),
    "mm_gemv_packed2_strided_batched": ([_P, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P],
                                        ctypes.c_int),
    "mm_gemv_packed2_strided_batched_ex": ([_P, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I64, _P, _P,
                                            ctypes.POINTER(GemvOpts)], ctypes.c_int),
    "mm_probe_bounded_wait": ([_I, ctypes.c_uint64, _P, _P], ctypes.c_int),
    "mm_attention_fwd": ([_P, _P, _P, _P, _P, _I64, _I64, _I64, _I, ctypes.c_float, _P], ctypes.c_int),
    "mm_attention_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I, ctypes.c_float, _P],
                         ctypes.c_int),
}


class MMError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libmm status {status}: {message}")
        self.status = status


def library_path() -> str:
    return os.environ.get("MM_LIBRARY", os.path.join(_PKG, "libmm.so"))


def load_library():
    """Load libmm.so (built by dense_packed_bit_gb300.build); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise MMError(MM_ERR_UNSUPPORTED,
                              f"{path} not found: build it with `python -m dense_packed_bit_gb300.build`")
            lib = ctypes.CDLL(path)
            for name, (argt, rest) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = argt
                fn.restype = rest
            _lib = lib
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _codebook(cb, n=4):
    if cb is None:
        return None
    vals = [float(v) for v in (cb.tolist() if hasattr(cb, "tolist") else cb)]
    if len(vals) != n:
        raise ValueError(f"codebook needs {n} entries")
    return (ctypes.c_float * n)(*vals)


def _check(status: int):
    if status != MM_OK:
        msg = load_library().mm_last_error()
        raise MMError(status, msg.decode() if msg else "")


def mm_version() -> int:
    return load_library().mm_version()


def mm_last_error() -> str:
    return load_library().mm_last_error().decode()


def mm_gemm_f32(transA, transB, M, N, K, A, lda, B, ldb, C, ldc, stream=None):
    _check(load_library().mm_gemm_f32(int(transA), int(transB), M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                      _ptr(C), ldc, _stream(stream)))


def mm_gemm_f32_ex(transA, transB, M, N, K, A, lda, B, ldb, C, ldc, stream=None, *, path=0, tile=0, splitk=0):
    o = GemmOpts(path, tile, splitk)
    _check(load_library().mm_gemm_f32_ex(int(transA), int(transB), M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                         _ptr(C), ldc, _stream(stream), ctypes.byref(o)))


def mm_gemm_f32_splitk_workspace(M, N, K, splitk=0) -> int:
    """Floats of workspace mm_gemm_f32_splitk needs for these sizes and split (0 = automatic)."""
    out = ctypes.c_int64(0)
    _check(load_library().mm_gemm_f32_splitk_workspace(M, N, K, splitk, ctypes.byref(out)))
    return out.value


def mm_gemm_f32_splitk(transA, transB, M, N, K, A, lda, B, ldb, C, ldc, splitk, workspace, workspace_floats,
                       stream=None):
    _check(load_library().mm_gemm_f32_splitk(int(transA), int(transB), M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                             _ptr(C), ldc, int(splitk), _ptr(workspace), int(workspace_floats),
                                             _stream(stream)))


def mm_gemm_f32_split_plan(M, N, K, sms):
    """(splitk, workspace_floats) of the automatic split on a GPU with `sms` SMs; no device needed."""
    sk = ctypes.c_int(0)
    fl = ctypes.c_int64(0)
    _check(load_library().mm_gemm_f32_split_plan(M, N, K, int(sms), ctypes.byref(sk), ctypes.byref(fl)))
    return sk.value, fl.value


def mm_gemm_f32_splitk_ex(transA, transB, M, N, K, A, lda, B, ldb, C, ldc, splitk, workspace, workspace_floats,
                          stream=None, *, path=0, tile=0, opt_splitk=0):
    """mm_gemm_f32_splitk with a kernel choice (path 1: the FFMA kernel and its stream-K tail)."""
    o = GemmOpts(path, tile, opt_splitk)
    _check(load_library().mm_gemm_f32_splitk_ex(int(transA), int(transB), M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                                _ptr(C), ldc, int(splitk), _ptr(workspace), int(workspace_floats),
                                                _stream(stream), ctypes.byref(o)))


def mm_gemm_f32_splitk_workspace_ex(M, N, K, splitk=0, *, path=0, tile=0, opt_splitk=0) -> int:
    """Floats of workspace mm_gemm_f32_splitk_ex needs for these sizes, split and options."""
    o = GemmOpts(path, tile, opt_splitk)
    out = ctypes.c_int64(0)
    _check(load_library().mm_gemm_f32_splitk_workspace_ex(M, N, K, int(splitk), ctypes.byref(o), ctypes.byref(out)))
    return out.value


def mm_gemm_f32_split_plan_ex(M, N, K, sms, *, path=0, tile=0, opt_splitk=0):
    """(splitk, workspace_floats) of mm_gemm_f32_splitk_ex's automatic split for `sms` SMs; no device needed."""
    o = GemmOpts(path, tile, opt_splitk)
    sk = ctypes.c_int(0)
    fl = ctypes.c_int64(0)
    _check(load_library().mm_gemm_f32_split_plan_ex(M, N, K, int(sms), ctypes.byref(o), ctypes.byref(sk),
                                                    ctypes.byref(fl)))
    return sk.value, fl.value


def mm_gemm_f32_bias_act_splitk(transA, transB, M, N, K, A, lda, B, ldb, bias, act, C, ldc, splitk=0,
                                workspace=None, workspace_floats=0, stream=None):
    """mm_gemm_f32_bias_act with the K split of mm_gemm_f32_splitk (0: automatic, -1: stream-K)."""
    _check(load_library().mm_gemm_f32_bias_act_splitk(
        int(transA), int(transB), M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(bias), int(act), _ptr(C), ldc,
        int(splitk), _ptr(workspace), workspace_floats, _stream(stream)))


def mm_gemv_packed2_strided_batched(codes, codes_stride, scales, scales_stride, x, x_stride, y, y_stride, batch,
                                    rows, cols, codebook, stream=None):
    """y_b = W_b x_b for b < batch, matrix b's operands at b times the strides (x_stride 0: shared x)."""
    _check(load_library().mm_gemv_packed2_strided_batched(
        _ptr(codes), codes_stride, _ptr(scales), scales_stride, _ptr(x), x_stride, _ptr(y), y_stride, batch, rows,
        cols, _codebook(codebook), _stream(stream)))


def mm_gemv_packed2_strided_batched_ex(codes, codes_stride, scales, scales_stride, x, x_stride, y, y_stride, batch,
                                       rows, cols, codebook, stream=None, *, dequant=0, rows_per_lane=0, pdl=0,
                                       weights_static=0, independent=0):
    """mm_gemv_packed2_strided_batched with a decode choice (dequant: 0, MM_DEQ_AFFINE or MM_DEQ_MXF4;
    rows_per_lane: 127-row tiles per CTA for MM_DEQ_MXF4, 0 = automatic; pdl / weights_static /
    independent: programmatic dependent launch options of the fp4 decode)."""
    o = GemvOpts(0, rows_per_lane, 0, dequant, pdl, weights_static, independent, -1)
    _check(load_library().mm_gemv_packed2_strided_batched_ex(
        _ptr(codes), codes_stride, _ptr(scales), scales_stride, _ptr(x), x_stride, _ptr(y), y_stride, batch, rows,
        cols, _codebook(codebook), _stream(stream), ctypes.byref(o)))


def mm_gemm_f32_bias_act(transA, transB, M, N, K, A, lda, B, ldb, bias, act, C, ldc, stream=None):
    """C = act(op(A) op(B) + bias): GPT-2's linear layer (bias per column) and GELU (act=1)."""
    _check(load_library().mm_gemm_f32_bias_act(int(transA), int(transB), M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                               _ptr(bias), int(act), _ptr(C), ldc, _stream(stream)))


def mm_gemm_f32_splitk_noalloc(transA, transB, M, N, K, A, lda, B, ldb, C, ldc, splitk=0, stream=None):
    """Split-K GEMM into the library's static scratch: for callers that cannot allocate device
    memory (or hand over a workspace) where they multiply.  Calls that overlap on the GPU race."""
    _check(load_library().mm_gemm_f32_splitk_noalloc(int(transA), int(transB), M, N, K, _ptr(A), lda, _ptr(B), ldb,
                                                     _ptr(C), ldc, int(splitk), _stream(stream)))


def mm_gemv_packed2(codes, scales, x, y, rows, cols, codebook, stream=None):
    _check(load_library().mm_gemv_packed2(_ptr(codes), _ptr(scales), _ptr(x), _ptr(y), rows, cols,
                                          _codebook(codebook), _stream(stream)))


def mm_gemv_packed2_ex(codes, scales, x, y, rows, cols, codebook, stream=None, *, split=0,
                       rows_per_lane=0, warps=0, dequant=0, pdl=0, weights_static=0, independent=0, staging=-1):
    o = GemvOpts(split, rows_per_lane, warps, dequant, pdl, weights_static, independent, staging)
    _check(load_library().mm_gemv_packed2_ex(_ptr(codes), _ptr(scales), _ptr(x), _ptr(y), rows, cols,
                                             _codebook(codebook), _stream(stream), ctypes.byref(o)))


def mm_gemm_packed2(codes, scales, X, Y, M, rows, cols, codebook, stream=None):
    _check(load_library().mm_gemm_packed2(_ptr(codes), _ptr(scales), _ptr(X), _ptr(Y), M, rows, cols,
                                          _codebook(codebook), _stream(stream)))


def mm_gemm_packed2_ex(codes, scales, X, Y, M, rows, cols, codebook, stream=None, *, tile=0, splitk=0, pdl=0,
                       weights_static=0, ntok=0):
    o = GemmPacked2Opts(tile, splitk, pdl, weights_static, ntok)
    _check(load_library().mm_gemm_packed2_ex(_ptr(codes), _ptr(scales), _ptr(X), _ptr(Y), M, rows, cols,
                                             _codebook(codebook), _stream(stream), ctypes.byref(o)))


def mm_check_device_error(stream=None):
    _check(load_library().mm_check_device_error(_stream(stream)))


def mm_probe_bounded_wait(arrive, limit_ns, out=None, stream=None):
    """One bounded device wait that completes (arrive=1) or runs out after limit_ns (arrive=0);
    out: None or a device int64 tensor of 2 receiving (completed, ns waited)."""
    _check(load_library().mm_probe_bounded_wait(int(arrive), int(limit_ns), _ptr(out), _stream(stream)))


def mm_gemv_packed4(codes, scales, x, y, rows, cols, codebook, stream=None):
    _check(load_library().mm_gemv_packed4(_ptr(codes), _ptr(scales), _ptr(x), _ptr(y), rows, cols,
                                          _codebook(codebook, 16), _stream(stream)))


def mm_gemv_packed4_ex(codes, scales, x, y, rows, cols, codebook, stream=None, *, blocks=0, pdl=0,
                       weights_static=0, independent=0, staging=-1):
    o = Gemv4Opts(blocks, pdl, weights_static, independent, staging)
    _check(load_library().mm_gemv_packed4_ex(_ptr(codes), _ptr(scales), _ptr(x), _ptr(y), rows, cols,
                                             _codebook(codebook, 16), _stream(stream), ctypes.byref(o)))


def mm_attention_fwd(Q, K, V, O, L, heads, T, D, causal, scale, stream=None):
    """O = softmax(scale Q K^T (+ causal mask)) V per head, L = the rows' log-sum-exp; [heads][T][D] fp32."""
    _check(load_library().mm_attention_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(L), heads, T, D, int(causal),
                                           float(scale), _stream(stream)))


def mm_attention_bwd(Q, K, V, O, dO, L, dQ, dK, dV, heads, T, D, causal, scale, stream=None):
    """Gradients of sum(O * dO) with respect to Q, K, V, from the forward's O and L."""
    _check(load_library().mm_attention_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L), _ptr(dQ),
                                           _ptr(dK), _ptr(dV), heads, T, D, int(causal), float(scale),
                                           _stream(stream)))
