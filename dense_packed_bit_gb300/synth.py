"""Seeded synthetic inputs shared by the CUDA path, the oracle tests and the bench.

This module holds no arithmetic of the method itself (no products, no sums, no
unpacking): it only draws numbers.  Both sides of every parity comparison take
their inputs from here, so neither needs to trust the other's generator.

Generator: SplitMix64 used as a counter-based generator (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014; the finaliser
constants are Vigna's published ones).  Draw i of stream `seed` is
``mix(seed * 2**32 + i + 1)`` where ``mix`` is the SplitMix64 output function
applied to ``state = counter * golden_gamma``.  It is written out here with
numpy uint64 arithmetic (which wraps mod 2**64), so every machine and numpy
version produces the same integer draws, hence the same codes, bytes and
uniform values.  Normals pass through numpy's log and cos, whose last bit may
differ between platforms before the rounding to fp32 / fp16; nothing stored
depends on them, since every comparison recomputes its expected values from
the inputs of the run.

Value recipes (the shapes and distributions of the workloads on the pages):
  * uniform fp32 on [lo, hi): fp64 ``lo + (hi-lo)*u`` rounded to fp32 (RNE),
    with ``u = (z >> 11) * 2**-53``; a value that rounds up to ``hi`` is
    replaced by the next fp32 below ``hi``.
  * normal(0, sigma): Box-Muller in fp64 from two draws, rounded to fp32 or
    to fp16 (RNE).  fp16 values are returned as their uint16 bit patterns.
  * uniform 2-bit codes: uniformly random bytes (four iid uniform 2-bit
    fields per byte, as the Kernel 0112 page's "random bytes" matrices).
  * ternary codes: each 2-bit field iid with P(field=0)=0.25, P(1)=0.5,
    P(2)=0.25 (field value = ternary value + 1), the fields of one byte
    independent, so the byte is a random draw whose meaning does not depend
    on the bit order inside the byte.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


# Draws are made in chunks of this many numbers, so that the temporaries of each
# elementwise step stay in the CPU's caches; every step is elementwise, so the
# chunking changes no value.
_CHUNK = 1 << 18


def _splitmix64_into(seed: int, out: np.ndarray, offset: int = 0) -> None:
    """Fill the 1-D uint64 array `out` with draws offset, offset+1, ... of stream `seed`."""
    base = np.uint64((int(seed) << 32) & 0xFFFFFFFFFFFFFFFF)
    tmp = np.empty(min(len(out), _CHUNK), dtype=np.uint64)
    with np.errstate(over="ignore"):
        for s in range(0, len(out), _CHUNK):
            z = out[s:s + _CHUNK]
            t = tmp[:len(z)]
            np.add(np.arange(offset + s + 1, offset + s + len(z) + 1, dtype=np.uint64), base, out=z)
            np.multiply(z, _GAMMA, out=z)
            np.right_shift(z, np.uint64(30), out=t)
            np.bitwise_xor(z, t, out=z)
            np.multiply(z, _M1, out=z)
            np.right_shift(z, np.uint64(27), out=t)
            np.bitwise_xor(z, t, out=z)
            np.multiply(z, _M2, out=z)
            np.right_shift(z, np.uint64(31), out=t)
            np.bitwise_xor(z, t, out=z)


def _splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n consecutive SplitMix64 outputs of stream `seed`, starting at draw `offset`."""
    out = np.empty(n, dtype=np.uint64)
    _splitmix64_into(seed, out, offset)
    return out


def _unit_open0(z: np.ndarray) -> np.ndarray:
    """uniform on [0, 1) with 53 random bits."""
    return (z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _unit_open1(z: np.ndarray) -> np.ndarray:
    """uniform on (0, 1] with 53 random bits (safe for log)."""
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def uniform_f32(seed: int, shape, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    u = _unit_open0(_splitmix64(seed, n))
    v = (lo + (hi - lo) * u).astype(np.float32)
    top = np.nextafter(np.float32(hi), np.float32(lo))
    v = np.where(v >= np.float32(hi), top, v)
    return v.reshape(shape)


def _normal_into(seed: int, out: np.ndarray, sigma: float) -> None:
    """Box-Muller normals (value i from draws 2i, 2i+1) rounded to out's dtype, chunk by chunk."""
    z = np.empty(min(2 * len(out), 2 * _CHUNK), dtype=np.uint64)
    for s in range(0, len(out), _CHUNK):
        o = out[s:s + _CHUNK]
        zc = z[:2 * len(o)]
        _splitmix64_into(seed, zc, 2 * s)
        u1 = _unit_open1(zc[0::2])
        u2 = _unit_open0(zc[1::2])
        o[:] = sigma * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def normal_f64(seed: int, n: int, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _normal_into(seed, out, sigma)
    return out


def normal_f32(seed: int, shape, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(int(np.prod(shape)), dtype=np.float32)
    _normal_into(seed, out, sigma)
    return out.reshape(shape)


def normal_f16_bits(seed: int, shape, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(int(np.prod(shape)), dtype=np.float16)
    _normal_into(seed, out, sigma)
    return out.view(np.uint16).reshape(shape)


def uniform_f16_bits(seed: int, shape, lo: float, hi: float) -> np.ndarray:
    """fp16 bit patterns of fp64 uniform[lo, hi) values rounded RNE."""
    n = int(np.prod(shape))
    u = _unit_open0(_splitmix64(seed, n))
    v = (lo + (hi - lo) * u).astype(np.float16)
    top = np.nextafter(np.float16(hi), np.float16(lo))
    v = np.where(v >= np.float16(hi), top, v)
    return v.view(np.uint16).reshape(shape)


def random_bytes(seed: int, n: int) -> np.ndarray:
    """n uniformly random bytes (8 per SplitMix64 draw, low byte first)."""
    words = _splitmix64(seed, (n + 7) // 8)
    # the little-endian representation of a word lists its bytes low byte first
    return words.astype("<u8", copy=False).view(np.uint8)[:n].copy()


def ternary_field_bytes(seed: int, n: int) -> np.ndarray:
    """n bytes whose four 2-bit fields are iid: 0 w.p. 1/4, 1 w.p. 1/2, 2 w.p. 1/4.

    Each field uses two fresh random bits r: r=0 -> 0, r in {1,2} -> 1, r=3 -> 2.
    """
    rnd = random_bytes(seed, n)
    out = np.zeros(n, dtype=np.uint8)
    for f in range(4):
        r = (rnd >> np.uint8(2 * f)) & np.uint8(3)
        field = np.where(r == 0, 0, np.where(r == 3, 2, 1)).astype(np.uint8)
        out |= field << np.uint8(2 * f)
    return out


class Digest:
    """SHA-256 over arrays given one at a time: each array's dtype, shape and raw bytes."""

    def __init__(self):
        self._h = hashlib.sha256()

    def update(self, *arrays) -> "Digest":
        for a in arrays:
            a = np.ascontiguousarray(a)
            self._h.update(str(a.dtype).encode())
            self._h.update(str(a.shape).encode())
            self._h.update(memoryview(a.reshape(-1)).cast("B"))  # the bytes, without a copy
        return self

    def hexdigest(self) -> str:
        return self._h.hexdigest()


def digest(*arrays) -> str:
    """SHA-256 over the raw bytes of the given arrays (detects silent input drift)."""
    return Digest().update(*arrays).hexdigest()


# --------------------------------------------------------------------------
# Workloads.  Each is named by what it is, with its sizes.  Seeds are fixed
# per (workload, tensor, index) so a workload is reproducible bit for bit.
# Workload ids: 1 GPT-2 MLP up-projection, 2 / 12 / 22 square 2048^3 NN / NT /
# TN, 3 2-bit GEMV rotation, 4 ternary encoder block, 5 4-bit GEMV rotation,
# 6 transposed 2-bit GEMV rotation, 7 training-shape set, 8 GPT-2 MLP
# up-projection with bias.  `replica` gives every data-parallel replica (one
# per GPU) its own draws of the same workload; replica 0 is the single-GPU
# workload.  Every field of the seed is range-checked, and no stream draws
# 2**32 numbers, so no two tensors of any workloads or replicas share a draw.
# --------------------------------------------------------------------------

MAX_REPLICAS = 40


def _seed(workload_id: int, tensor_id: int, index: int = 0, replica: int = 0) -> int:
    if not (0 < workload_id < 100 and 0 < tensor_id < 1000 and 0 <= index < 1000
            and 0 <= replica < MAX_REPLICAS):
        raise ValueError(f"seed field out of range: workload {workload_id}, tensor {tensor_id}, "
                         f"index {index}, replica {replica}")
    return ((replica * 100 + workload_id) * 1000 + tensor_id) * 1000 + index


@dataclass
class GemmCase:
    name: str
    transA: int
    transB: int
    M: int
    N: int
    K: int
    A: np.ndarray  # stored (M,K) or (K,M) if transA
    B: np.ndarray  # stored (K,N) or (N,K) if transB
    bias: np.ndarray | None = None  # (N,) fp32, one per output column, for a linear layer


def gemm_case(name, transA, transB, M, N, K, dist, seed_base, sigma=0.02, replica=0):
    a_shape = (K, M) if transA else (M, K)
    b_shape = (N, K) if transB else (K, N)
    if dist == "uniform":
        A = uniform_f32(_seed(seed_base, 1, 0, replica), a_shape, -1.0, 1.0)
        B = uniform_f32(_seed(seed_base, 2, 0, replica), b_shape, -1.0, 1.0)
    elif dist == "normal":
        A = normal_f32(_seed(seed_base, 1, 0, replica), a_shape, sigma)
        B = normal_f32(_seed(seed_base, 2, 0, replica), b_shape, sigma)
    else:
        raise ValueError(dist)
    return GemmCase(name, transA, transB, M, N, K, A, B)


def gpt2_mlp_up_64x768x3072(replica: int = 0) -> GemmCase:
    """GPT-2-small MLP up-projection, 64 tokens: C(64x3072) = A(64x768) B(768x3072), U[-1,1)."""
    return gemm_case("gpt2_mlp_up_m64_k768_n3072_nn", 0, 0, 64, 3072, 768, "uniform", 1, replica=replica)


def square_2048(layout: str, replica: int = 0) -> GemmCase:
    """Square 2048^3 fp32 GEMM, N(0,0.02) operands, layout 'nn' | 'nt' | 'tn'."""
    tA, tB = {"nn": (0, 0), "nt": (0, 1), "tn": (1, 0)}[layout]
    return gemm_case(f"square_2048_{layout}", tA, tB, 2048, 2048, 2048, "normal",
                     2 + {"nn": 0, "nt": 10, "tn": 20}[layout], replica=replica)


def gpt2_mlp_bias_gelu_8192x768x3072(replica: int = 0) -> GemmCase:
    """GPT-2-small MLP up-projection of 8 sequences of 1,024 tokens, with its bias.

    X 8192 x 768 N(0, 1) (the layer-normed activations), W 768 x 3072 N(0, 0.02),
    bias 3072 N(0, 0.02); NN.  The GELU that follows has no inputs of its own.
    """
    X = normal_f32(_seed(8, 1, 0, replica), (8192, 768), 1.0)
    W = normal_f32(_seed(8, 2, 0, replica), (768, 3072), 0.02)
    bias = normal_f32(_seed(8, 3, 0, replica), (3072,), 0.02)
    return GemmCase("gpt2_mlp_up_bias_gelu_m8192_k768_n3072_nn", 0, 0, 8192, 3072, 768, X, W, bias)


_TRAINING_PRODUCTS = {
    # which: (name, transA, transB, M, N, K, stored A, stored B)
    "fwd": ("train_fwd_8192x8192x2048_nn", 0, 0, 8192, 8192, 2048, "A", "B"),
    "dA": ("train_dA_8192x2048x8192_nt", 0, 1, 8192, 2048, 8192, "dC", "B"),
    "dB": ("train_dB_2048x8192x8192_tn", 1, 0, 2048, 8192, 8192, "A", "dC"),
}
_TRAINING_TENSORS = {"A": (1, (8192, 2048)), "B": (2, (2048, 8192)), "dC": (3, (8192, 8192))}


def _training_tensor(name: str, replica: int) -> np.ndarray:
    tensor_id, shape = _TRAINING_TENSORS[name]
    return normal_f32(_seed(7, tensor_id, 0, replica), shape, 0.02)


def training_set_8192(which: str, replica: int = 0) -> GemmCase:
    """Training-shape products (batch 16 x seq 512 = 8192 rows, d=2048, d_ff=8192).

    'fwd': C = A(8192x2048) B(2048x8192)            (NN)
    'dA' : dA = dC(8192x8192) B^T, B stored 2048x8192 (NT: M=8192,N=2048,K=8192)
    'dB' : dB = A^T dC, A stored 8192x2048            (TN: M=2048,N=8192,K=8192)
    All operands N(0,0.02); A, B and dC each come from one fixed stream.  Only the
    two tensors the product reads are drawn.
    """
    if which not in _TRAINING_PRODUCTS:
        raise ValueError(which)
    name, tA, tB, M, N, K, a, b = _TRAINING_PRODUCTS[which]
    return GemmCase(name, tA, tB, M, N, K, _training_tensor(a, replica), _training_tensor(b, replica))


def training_set_8192_all(replica: int = 0) -> tuple:
    """The three products (fwd, dA, dB) of training_set_8192, sharing one draw of A, B and dC."""
    t = {name: _training_tensor(name, replica) for name in _TRAINING_TENSORS}
    out = []
    for which in ("fwd", "dA", "dB"):
        name, tA, tB, M, N, K, a, b = _TRAINING_PRODUCTS[which]
        out.append(GemmCase(name, tA, tB, M, N, K, t[a], t[b]))
    return tuple(out)


@dataclass
class AttentionCase:
    name: str
    heads: int
    T: int
    D: int
    causal: int
    Q: np.ndarray  # (heads, T, D) fp32
    K: np.ndarray
    V: np.ndarray
    dO: np.ndarray  # gradient of the loss with respect to O


def gpt2_attention_4x8x512x64(replica: int = 0) -> AttentionCase:
    """Causal self-attention of a GPT-2 training step at the shape of "I built a GPT-2 in the
    browser", section "Flash Attention 2" (B = 4 sequences, H = 8 heads, T = 512), head dimension
    64 (GPT-2's): Q, K, V and the incoming gradient dO N(0, 1) fp32, heads = B H = 32."""
    shape = (32, 512, 64)
    Q, K, V, dO = (normal_f32(_seed(9, t, 0, replica), shape, 1.0) for t in (1, 2, 3, 4))
    return AttentionCase("gpt2_attention_b4_h8_t512_d64_causal", 32, 512, 64, 1, Q, K, V, dO)


@dataclass
class PackedCase:
    name: str
    rows: int
    cols: int
    codes: np.ndarray      # (rows, ceil(cols/4)) uint8
    scales: np.ndarray     # (rows,) uint16 fp16 bits
    codebook: np.ndarray   # (4,) float32
    X: np.ndarray          # (M, cols) uint16 fp16 bits; M=1 for a GEMV


CODEBOOK_2BIT = np.array([-2.0, -1.0, 0.0, 1.0], dtype=np.float32)
# Ternary values v in {-1,0,+1} are stored as field v+1; field 3 never occurs and means 0.
CODEBOOK_TERNARY = np.array([-1.0, 0.0, 1.0, 0.0], dtype=np.float32)


def _normal_ppf(p: float) -> float:
    """Standard normal quantile by bisection on the CDF 0.5 erfc(-x / sqrt 2) (|error| < 1e-15)."""
    lo, hi = -40.0, 40.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if 0.5 * math.erfc(-mid / math.sqrt(2.0)) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def normal_quantile_codebook() -> np.ndarray:
    """16-entry 4-bit codebook of normal-quantile levels with an exact zero (NF4-style).

    Codes 0..6 are negative, code 7 is 0, codes 8..15 are positive: level i of a
    side of n levels is the standard-normal quantile at 0.5 + 0.48 i / n, and each
    side is divided by its largest level, so the table runs from -1 to 1.  None of
    the non-trivial levels is exact in fp16.
    """
    neg = [-_normal_ppf(0.5 + 0.48 * i / 7) for i in range(1, 8)]
    pos = [_normal_ppf(0.5 + 0.48 * i / 8) for i in range(1, 9)]
    neg = [v / -neg[-1] for v in neg]
    pos = [v / pos[-1] for v in pos]
    return np.array(sorted(neg) + [0.0] + pos, dtype=np.float32)


CODEBOOK_NQ4 = normal_quantile_codebook()


def packed_matrix(seed_base, index, rows, cols, kind, replica=0):
    """Codes (rows x packed bytes) and fp16 scales; kind 'uniform4' packs 4-bit fields."""
    rb = (cols + 1) // 2 if kind == "uniform4" else (cols + 3) // 4
    nbytes = rows * rb
    if kind in ("uniform2", "uniform4"):
        codes = random_bytes(_seed(seed_base, 1, index, replica), nbytes)
    elif kind == "ternary":
        codes = ternary_field_bytes(_seed(seed_base, 1, index, replica), nbytes)
    else:
        raise ValueError(kind)
    scales = uniform_f16_bits(_seed(seed_base, 2, index, replica), (rows,), 0.005, 0.05)
    return codes.reshape(rows, rb), scales


def gemv_2bit_12288x1536(index: int, replica: int = 0) -> PackedCase:
    """One of the 64 rotated 2-bit GEMV matrices: 12288 rows x 1536 cols (4.5 MiB of codes)."""
    codes, scales = packed_matrix(3, index, 12288, 1536, "uniform2", replica)
    x = normal_f16_bits(_seed(3, 3, 0, replica), (1, 1536))
    return PackedCase(f"gemv2_12288x1536_m{index}", 12288, 1536, codes, scales,
                      CODEBOOK_2BIT.copy(), x)


def gemv_2bit_1536x12288(index: int, replica: int = 0) -> PackedCase:
    """The transposed shape (the pages' kernel 0113): 1536 rows x 12288 cols of 2-bit codes,
    4.5 MiB per matrix like the 12288 x 1536 one; same value distributions."""
    codes, scales = packed_matrix(6, index, 1536, 12288, "uniform2", replica)
    x = normal_f16_bits(_seed(6, 3, 0, replica), (1, 12288))
    return PackedCase(f"gemv2_1536x12288_m{index}", 1536, 12288, codes, scales,
                      CODEBOOK_2BIT.copy(), x)


def gemv_4bit_12288x1536(index: int, replica: int = 0) -> PackedCase:
    """One of the 64 rotated 4-bit GEMV matrices: 12288 rows x 1536 cols (9 MiB of codes),
    fields uniform in 0..15 (two per byte), normal-quantile codebook."""
    codes, scales = packed_matrix(5, index, 12288, 1536, "uniform4", replica)
    x = normal_f16_bits(_seed(5, 3, 0, replica), (1, 1536))
    return PackedCase(f"gemv4_12288x1536_m{index}", 12288, 1536, codes, scales,
                      CODEBOOK_NQ4.copy(), x)


def ternary_encoder_layer(layer: int, proj: str, replica: int = 0) -> PackedCase:
    """Layer `layer` (0..15) of the ternary 16-layer encoder block, M = 2 x 111 = 222 rows.

    proj 'up'  : W 3072 x 768  (N=3072, K=768)
    proj 'down': W 768 x 3072  (N=768,  K=3072)
    """
    rows, cols, pid = (3072, 768, 0) if proj == "up" else (768, 3072, 1)
    codes, scales = packed_matrix(4, 2 * layer + pid, rows, cols, "ternary", replica)
    X = normal_f16_bits(_seed(4, 3, 2 * layer + pid, replica), (222, cols))
    return PackedCase(f"ternary_enc_l{layer}_{proj}", rows, cols, codes, scales,
                      CODEBOOK_TERNARY.copy(), X)
