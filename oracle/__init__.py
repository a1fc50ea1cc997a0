"""CPU oracle for the dense fp32 GEMM, the packed 2-bit GEMV / skinny GEMM and attention.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
baseline leg may import this package.  The product library never loads it and
there is no fallback from the CUDA path to it.

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation, a scalar
bit unpacker); this module only compiles it with gcc and marshals numpy arrays
through ctypes.  Every function returns the value and T = sum_k |term_k|,
the scale of the acceptance bound |y - y_ref| <= 1e-5 * T.

Pins (tests/test_oracle.py): closed forms (all-ones, identity, rank-1),
textbook small products, exact integer products against numpy int64 matmul,
the fp16 decoder against numpy's float16 for all 65,536 patterns, the unpacker
against a hand-written byte table and a pack/unpack round trip, and the packed
GEMM against dense products of explicitly decoded weights; the GELU of the fused
epilogue (gelu_tanh, gemm_bias_act) against the library's fp64 tanh GELU, its
small-z series, its odd-part identity, the library's normal CDF and special
values, and the bias broadcast on a zero product; attention (attention.c)
against the library's fp64 scaled-dot-product attention, log-sum-exp and
autograd gradients, the uniform-weights closed form (Q = 0) and the causal
first row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SRCS = (_SRC, os.path.join(_HERE, "attention.c"))
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c and attention.c into oracle/liboracle.so with gcc (plain -O2, portable)."""
    if force or not os.path.exists(_LIB) or any(os.path.getmtime(_LIB) < os.path.getmtime(f) for f in _SRCS):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, *_SRCS, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_half_to_double.restype = ctypes.c_double
            lib.orc_unpack2.argtypes = [P, I64, I64, P]
            lib.orc_pack2.argtypes = [P, I64, I64, P]
            lib.orc_gemm.argtypes = [I, I, I64, I64, I64, P, I64, P, I64, P, P, I]
            lib.orc_gemm_at.argtypes = [I, I, I64, P, I64, P, I64, I64, P, P, P, P]
            lib.orc_packed_gemm.argtypes = [P, P, P, I64, I64, I64, P, P, P, I]
            lib.orc_packed_gemm_at.argtypes = [P, P, P, I64, P, I64, P, P, P, P]
            lib.orc_unpack4.argtypes = [P, I64, I64, P]
            lib.orc_pack4.argtypes = [P, I64, I64, P]
            lib.orc_packed4_gemm.argtypes = [P, P, P, I64, I64, I64, P, P, P, I]
            lib.orc_packed4_gemm_at.argtypes = [P, P, P, I64, P, I64, P, P, P, P]
            D = ctypes.c_double
            lib.orc_attention_fwd.argtypes = [P, P, P, I64, I64, I64, I, D, P, P, P, I]
            lib.orc_attention_bwd.argtypes = [P, P, P, P, I64, I64, I64, I, D, P, P, P, P, P, P, I]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count())


def half_to_double(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16).reshape(-1)
    return np.array([lib.orc_half_to_double(int(v)) for v in b], dtype=np.float64)


def unpack2(codes: np.ndarray, rows: int, cols: int) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    assert c.size == rows * ((cols + 3) // 4)
    out = np.empty((rows, cols), dtype=np.uint8)
    lib.orc_unpack2(_ptr(c), rows, cols, _ptr(out))
    return out


def pack2(fields: np.ndarray) -> np.ndarray:
    lib = _load()
    f = np.ascontiguousarray(fields, dtype=np.uint8)
    rows, cols = f.shape
    out = np.empty((rows, (cols + 3) // 4), dtype=np.uint8)
    lib.orc_pack2(_ptr(f), rows, cols, _ptr(out))
    return out


def gemm(transA: int, transB: int, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray,
         lda: int | None = None, ldb: int | None = None, threads: int | None = None):
    """(C, T), both (M, N) float64, of C = op(A) op(B) from fp32 A, B (row-major)."""
    lib = _load()
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    if lda is None:
        lda = A.shape[-1]
    if ldb is None:
        ldb = B.shape[-1]
    C = np.empty((M, N), dtype=np.float64)
    T = np.empty((M, N), dtype=np.float64)
    lib.orc_gemm(int(transA), int(transB), M, N, K, _ptr(A), lda, _ptr(B), ldb,
                 _ptr(C), _ptr(T), threads or default_threads())
    return C, T


def gelu_tanh(z) -> np.ndarray:
    """GELU in the tanh form GPT-2 uses, in fp64:
    gelu(z) = z/2 (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))).
    The pages name GPT-2's training step but print no activation; this is the
    published GPT-2 definition, written out plainly."""
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (z + 0.044715 * z * z * z)))


def gemm_bias_act(transA: int, transB: int, M: int, N: int, K: int, A: np.ndarray, B: np.ndarray,
                  bias=None, act: int = 0, lda: int | None = None, ldb: int | None = None):
    """(Y, T, Z) of Y = act(op(A) op(B) + bias) in fp64: bias has N entries (one per output
    column, broadcast over the rows) or is None; act 0 is the identity, 1 is gelu_tanh.
    Z is the pre-activation op(A) op(B) + bias; T = sum_k |a b| + |bias| bounds the
    error the GEMM and the bias add may make."""
    C, T = gemm(transA, transB, M, N, K, A, B, lda, ldb)
    if bias is not None:
        b = np.asarray(bias, dtype=np.float32).astype(np.float64).reshape(1, N)
        C = C + b
        T = T + np.abs(b)
    Y = gelu_tanh(C) if act == 1 else C
    return Y, T, C


def gemm_at(transA: int, transB: int, K: int, A: np.ndarray, B: np.ndarray, ii, jj,
            lda: int | None = None, ldb: int | None = None):
    """(C, T) at the listed output coordinates (ii[n], jj[n])."""
    lib = _load()
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    if lda is None:
        lda = A.shape[-1]
    if ldb is None:
        ldb = B.shape[-1]
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    C = np.empty(len(ii), dtype=np.float64)
    T = np.empty(len(ii), dtype=np.float64)
    lib.orc_gemm_at(int(transA), int(transB), K, _ptr(A), lda, _ptr(B), ldb, len(ii),
                    _ptr(ii), _ptr(jj), _ptr(C), _ptr(T))
    return C, T


def packed_gemm(codes: np.ndarray, scales: np.ndarray, X: np.ndarray, rows: int, cols: int,
                codebook, threads: int | None = None):
    """(Y, T), both (M, rows) float64, Y[m,r] = sum_k scale_r cb[field(r,k)] X[m,k]."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    X = np.ascontiguousarray(X, dtype=np.uint16).reshape(-1, cols)
    cb = np.ascontiguousarray(codebook, dtype=np.float32)
    assert cb.size == 4 and scales.size == rows and codes.size == rows * ((cols + 3) // 4)
    M = X.shape[0]
    Y = np.empty((M, rows), dtype=np.float64)
    T = np.empty((M, rows), dtype=np.float64)
    lib.orc_packed_gemm(_ptr(codes), _ptr(scales), _ptr(X), M, rows, cols, _ptr(cb),
                        _ptr(Y), _ptr(T), threads or default_threads())
    return Y, T


def packed_gemm_at(codes, scales, X, cols: int, codebook, mm, rr):
    """(Y, T) at the listed coordinates (mm[n], rr[n])."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    X = np.ascontiguousarray(X, dtype=np.uint16).reshape(-1, cols)
    cb = np.ascontiguousarray(codebook, dtype=np.float32)
    mm = np.ascontiguousarray(mm, dtype=np.int64)
    rr = np.ascontiguousarray(rr, dtype=np.int64)
    Y = np.empty(len(mm), dtype=np.float64)
    T = np.empty(len(mm), dtype=np.float64)
    lib.orc_packed_gemm_at(_ptr(codes), _ptr(scales), _ptr(X), cols, _ptr(cb), len(mm),
                           _ptr(mm), _ptr(rr), _ptr(Y), _ptr(T))
    return Y, T


def unpack4(codes: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """(rows, cols) uint8 4-bit fields of packed rows of ceil(cols/2) bytes (low nibble first)."""
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    assert c.size == rows * ((cols + 1) // 2)
    out = np.empty((rows, cols), dtype=np.uint8)
    lib.orc_unpack4(_ptr(c), rows, cols, _ptr(out))
    return out


def pack4(fields: np.ndarray) -> np.ndarray:
    lib = _load()
    f = np.ascontiguousarray(fields, dtype=np.uint8)
    rows, cols = f.shape
    out = np.empty((rows, (cols + 1) // 2), dtype=np.uint8)
    lib.orc_pack4(_ptr(f), rows, cols, _ptr(out))
    return out


def packed4_gemm(codes: np.ndarray, scales: np.ndarray, X: np.ndarray, rows: int, cols: int,
                 codebook, threads: int | None = None):
    """(Y, T), both (M, rows) float64, Y[m,r] = sum_k scale_r cb[field4(r,k)] X[m,k] (16-entry cb)."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    X = np.ascontiguousarray(X, dtype=np.uint16).reshape(-1, cols)
    cb = np.ascontiguousarray(codebook, dtype=np.float32)
    assert cb.size == 16 and scales.size == rows and codes.size == rows * ((cols + 1) // 2)
    M = X.shape[0]
    Y = np.empty((M, rows), dtype=np.float64)
    T = np.empty((M, rows), dtype=np.float64)
    lib.orc_packed4_gemm(_ptr(codes), _ptr(scales), _ptr(X), M, rows, cols, _ptr(cb),
                         _ptr(Y), _ptr(T), threads or default_threads())
    return Y, T


def packed4_gemm_at(codes, scales, X, cols: int, codebook, mm, rr):
    """(Y, T) of the 4-bit form at the listed coordinates (mm[n], rr[n])."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    X = np.ascontiguousarray(X, dtype=np.uint16).reshape(-1, cols)
    cb = np.ascontiguousarray(codebook, dtype=np.float32)
    assert cb.size == 16
    mm = np.ascontiguousarray(mm, dtype=np.int64)
    rr = np.ascontiguousarray(rr, dtype=np.int64)
    Y = np.empty(len(mm), dtype=np.float64)
    T = np.empty(len(mm), dtype=np.float64)
    lib.orc_packed4_gemm_at(_ptr(codes), _ptr(scales), _ptr(X), cols, _ptr(cb), len(mm),
                            _ptr(mm), _ptr(rr), _ptr(Y), _ptr(T))
    return Y, T


# ------------------------------------------------------------------ attention (attention.c)

def attention_fwd(Q, K, V, causal: int, scale: float, threads: int | None = None):
    """(O, L, TO) of softmax(scale Q K^T (+ causal mask)) V per head, in fp64.

    Q, K, V: fp32 arrays of shape (heads, T, D).  L[h, i] = log sum_k exp(S[h, i, k]) (the
    log-sum-exp of the row's scaled, unmasked scores); TO = sum_k P |V|, the bound scale.
    scale is taken as given (pass the fp32 value the GPU multiplies by)."""
    lib = _load()
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    BH, T, D = Q.shape
    assert K.shape == Q.shape and V.shape == Q.shape
    O = np.empty((BH, T, D), dtype=np.float64)
    L = np.empty((BH, T), dtype=np.float64)
    TO = np.empty((BH, T, D), dtype=np.float64)
    lib.orc_attention_fwd(_ptr(Q), _ptr(K), _ptr(V), BH, T, D, int(causal), float(scale), _ptr(O), _ptr(L),
                          _ptr(TO), threads or default_threads())
    return O, L, TO


def attention_bwd(Q, K, V, dO, causal: int, scale: float, threads: int | None = None):
    """(dQ, dK, dV, TdQ, TdK, TdV): the gradients of sum(O * dO) with respect to Q, K and V,
    in fp64, with their bound scales (see attention.c)."""
    lib = _load()
    Q = np.ascontiguousarray(Q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    dO = np.ascontiguousarray(dO, dtype=np.float32)
    BH, T, D = Q.shape
    out = [np.empty((BH, T, D), dtype=np.float64) for _ in range(6)]
    lib.orc_attention_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), BH, T, D, int(causal), float(scale),
                          *[_ptr(a) for a in out], threads or default_threads())
    return tuple(out)
