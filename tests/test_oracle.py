"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test is chosen so that a plausible slip in oracle.c fails it: a swapped
operand or transpose flag (hand 4x4 case in all layouts, rank-1 closed form), a
dropped or extra term (all-ones = K, identity), a wrong bit order or field
width (hand byte table, one-hot decoding), a wrong fp16 exponent bias
(IEEE table and numpy's float16 on all 65,536 patterns), a misplaced scale
(hand packed case, constant-field rows), and a wrong |term| sum (T checks).
"""
import numpy as np
import pytest

from conftest import read_golden
from dense_packed_bit_gb300 import synth


def _blocks(lines):
    out, cur = {}, None
    for ln in lines:
        if ln.replace("_", "").isalpha() or ln in ("A", "B", "C", "T"):
            cur = ln
            out[cur] = []
        else:
            out[cur].append([float(v) for v in ln.split()])
    return {k: np.array(v) for k, v in out.items()}


# ---------------------------------------------------------------- generator

def test_splitmix64_published_vector():
    # SplitMix64 started from state 0 yields 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
    # 0x06C45D188009454F (the published reference outputs of Vigna's splitmix64.c).
    z = synth._splitmix64(0, 3)
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_generators_deterministic_and_shaped():
    a = synth.uniform_f32(7, (3, 5))
    b = synth.uniform_f32(7, (3, 5))
    assert a.shape == (3, 5) and a.dtype == np.float32 and np.array_equal(a, b)
    assert a.min() >= -1.0 and a.max() < 1.0
    t = synth.ternary_field_bytes(3, 100000)
    fields = np.stack([(t >> (2 * f)) & 3 for f in range(4)])
    frac = np.bincount(fields.reshape(-1), minlength=4) / fields.size
    assert frac[3] == 0 and abs(frac[0] - 0.25) < 0.01 and abs(frac[1] - 0.5) < 0.01
    s = synth.uniform_f16_bits(1, (10000,), 0.005, 0.05).view(np.float16).astype(np.float64)
    assert s.min() >= 0.005 - 1e-6 and s.max() < 0.05


# ---------------------------------------------------------------- fp16 decoder

def test_fp16_decoder_table(oracle):
    for ln in read_golden("fp16_values.txt"):
        bits, val = ln.split()
        got = oracle.half_to_double([int(bits, 16)])[0]
        assert got == float(val) and np.signbit(got) == np.signbit(float(val)), (bits, got)


def test_fp16_decoder_all_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


# ---------------------------------------------------------------- unpack / pack

def test_unpack_hand_table(oracle):
    for ln in read_golden("unpack2_bytes.txt"):
        parts = ln.split()
        byte = int(parts[0], 16)
        want = [int(v) for v in parts[1:5]]
        got = oracle.unpack2(np.array([byte], np.uint8), 1, 4)[0].tolist()
        assert got == want, (hex(byte), got, want)


def test_pack_unpack_roundtrip_all_bytes(oracle):
    allb = np.arange(256, dtype=np.uint8).reshape(64, 4)       # 64 rows x 16 cols
    fields = oracle.unpack2(allb, 64, 16)
    assert fields.max() <= 3
    assert np.array_equal(oracle.pack2(fields), allb)


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (7, 63), (5, 64), (2, 131)])
def test_unpack_pack_roundtrip_ragged(oracle, rows, cols):
    rng = np.random.default_rng(rows * 1000 + cols)
    fields = rng.integers(0, 4, size=(rows, cols), dtype=np.uint8)
    packed = oracle.pack2(fields)
    assert packed.shape == (rows, (cols + 3) // 4)
    assert np.array_equal(oracle.unpack2(packed, rows, cols), fields)
    # bits past the last column are ignored by unpack
    dirty = packed.copy()
    if cols % 4:
        dirty[:, -1] |= np.uint8((0xFF << (2 * (cols % 4))) & 0xFF)
    assert np.array_equal(oracle.unpack2(dirty, rows, cols), fields)


def test_kernel0112_byte_count(oracle):
    g = dict(ln.split() for ln in read_golden("kernel0112_shape.txt"))
    rows, cols, nbytes = int(g["rows"]), int(g["cols"]), int(g["weight_bytes"])
    assert oracle.pack2(np.zeros((4, cols), np.uint8)).shape[1] * rows == nbytes


# ---------------------------------------------------------------- dense GEMM

def _hand():
    return _blocks(read_golden("gemm_4x4_hand.txt"))


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gemm_hand_4x4_all_layouts(oracle, tA, tB):
    h = _hand()
    A, B = h["A"].astype(np.float32), h["B"].astype(np.float32)
    As = np.ascontiguousarray(A.T) if tA else A
    Bs = np.ascontiguousarray(B.T) if tB else B
    C, T = oracle.gemm(tA, tB, 4, 4, 4, As, Bs)
    assert np.array_equal(C, h["C"])
    assert np.array_equal(T, h["T"])


def test_gemm_textbook_2x2(oracle):
    A = np.array([[1, 2], [3, 4]], np.float32)
    B = np.array([[5, 6], [7, 8]], np.float32)
    C, T = oracle.gemm(0, 0, 2, 2, 2, A, B)
    assert C.tolist() == [[19, 22], [43, 50]]
    assert T.tolist() == [[19, 22], [43, 50]]


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(3, 5, 7), (17, 1, 33), (1, 9, 1)])
def test_gemm_all_ones_is_K(oracle, tA, tB, M, N, K):
    A = np.ones((K, M) if tA else (M, K), np.float32)
    B = np.ones((N, K) if tB else (K, N), np.float32)
    C, T = oracle.gemm(tA, tB, M, N, K, A, B)
    assert np.all(C == K) and np.all(T == K)


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0)])
def test_gemm_identity(oracle, tA, tB):
    rng = np.random.default_rng(5)
    n = 13
    X = rng.standard_normal((n, n)).astype(np.float32)
    I = np.eye(n, dtype=np.float32)
    C, _ = oracle.gemm(tA, tB, n, n, n, X.T.copy() if tA else X, I)
    assert np.array_equal(C, X.astype(np.float64))
    C, _ = oracle.gemm(tA, tB, n, n, n, I, X.T.copy() if tB else X)
    assert np.array_equal(C, X.astype(np.float64))


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0)])
def test_gemm_rank1_closed_form(oracle, tA, tB):
    # A = u p^T (M x K), B = q v^T (K x N)  =>  C = (p.q) u v^T exactly
    # (all values small dyadic rationals, so every product and sum is exact).
    M, N, K = 6, 5, 9
    u = np.array([1, -2, 0.5, 3, -0.25, 4])
    v = np.array([2, -1, 0.5, -3, 1.5])
    p = np.arange(1, K + 1) * 0.5
    q = np.array([1, -1, 2, 0, -2, 1, 3, -0.5, 0.25])
    A = np.outer(u, p).astype(np.float32)
    B = np.outer(q, v).astype(np.float32)
    C, T = oracle.gemm(tA, tB, M, N, K, A.T.copy() if tA else A, B.T.copy() if tB else B)
    assert np.array_equal(C, float(p @ q) * np.outer(u, v))
    assert np.array_equal(T, float(np.abs(p) @ np.abs(q)) * np.outer(np.abs(u), np.abs(v)))


@pytest.mark.parametrize("tA,tB", [(0, 0), (0, 1), (1, 0)])
def test_gemm_small_integers_vs_int64_matmul(oracle, tA, tB):
    rng = np.random.default_rng(11 + 2 * tA + tB)
    M, N, K = 37, 29, 71
    A = rng.integers(-8, 9, size=(M, K))
    B = rng.integers(-8, 9, size=(K, N))
    As = (A.T if tA else A).astype(np.float32)
    Bs = (B.T if tB else B).astype(np.float32)
    C, T = oracle.gemm(tA, tB, M, N, K, As, Bs, threads=3)
    assert np.array_equal(C, (A @ B).astype(np.float64))
    assert np.array_equal(T, (np.abs(A) @ np.abs(B)).astype(np.float64))


def test_gemm_leading_dims_and_sampled(oracle):
    rng = np.random.default_rng(3)
    M, N, K = 10, 7, 12
    A = rng.integers(-5, 6, size=(M, K)).astype(np.float32)
    B = rng.integers(-5, 6, size=(K, N)).astype(np.float32)
    Ap = np.zeros((M, K + 5), np.float32); Ap[:, :K] = A; Ap[:, K:] = 1e6
    Bp = np.zeros((K, N + 3), np.float32); Bp[:, :N] = B; Bp[:, N:] = -1e6
    C, T = oracle.gemm(0, 0, M, N, K, Ap, Bp, lda=K + 5, ldb=N + 3)
    assert np.array_equal(C, A.astype(np.int64) @ B.astype(np.int64))
    ii = np.array([0, 9, 4, 3]); jj = np.array([0, 6, 2, 5])
    Cs, Ts = oracle.gemm_at(0, 0, K, Ap, Bp, ii, jj, lda=K + 5, ldb=N + 3)
    assert np.array_equal(Cs, C[ii, jj]) and np.array_equal(Ts, T[ii, jj])
    # sampled outputs agree with the full product in the transposed layouts too
    for tA, tB in [(0, 1), (1, 0)]:
        As = A.T.copy() if tA else A
        Bs = B.T.copy() if tB else B
        Cs, _ = oracle.gemm_at(tA, tB, K, As, Bs, ii, jj)
        assert np.array_equal(Cs, C[ii, jj])


def test_gemm_fp32_products_exact(oracle):
    # Each fp32*fp32 product is exact in double, so a K=1 product equals the
    # exact product computed with Python fractions.
    from fractions import Fraction
    rng = np.random.default_rng(9)
    a = rng.standard_normal((5, 1)).astype(np.float32)
    b = rng.standard_normal((1, 4)).astype(np.float32)
    C, _ = oracle.gemm(0, 0, 5, 4, 1, a, b)
    for i in range(5):
        for j in range(4):
            assert Fraction(C[i, j]) == Fraction(float(a[i, 0])) * Fraction(float(b[0, j]))


# ---------------------------------------------------------------- packed

def _packed_hand(name="packed_2x6_hand.txt"):
    lines = read_golden(name)
    d, cur = {}, None
    for ln in lines:
        tok = ln.split()
        if tok[0] in ("cols", "codebook"):
            d[tok[0]] = tok[1:]
        elif len(tok) == 1 and tok[0].replace("_", "").isalnum() and not tok[0].startswith("0x") \
                and not tok[0].lstrip("-").replace(".", "").isdigit():
            cur = tok[0]
            d[cur] = []
        else:
            d[cur].append(tok)
    return d


def test_packed_hand_2x6(oracle):
    d = _packed_hand()
    cols = int(d["cols"][0])
    cb = np.array([float(v) for v in d["codebook"]], np.float32)
    codes = np.array([[int(v, 16) for v in row] for row in d["codes"]], np.uint8)
    scales = np.array([int(v, 16) for v in d["scales_fp16"][0]], np.uint16)
    x = np.array([int(v, 16) for v in d["x_fp16"][0]], np.uint16)
    y, T = oracle.packed_gemm(codes, scales, x, 2, cols, cb)
    assert y[0].tolist() == [float(v) for v in d["y"][0]]
    assert T[0].tolist() == [float(v) for v in d["T"][0]]
    ys, Ts = oracle.packed_gemm_at(codes, scales, x, cols, cb, [0, 0], [1, 0])
    assert ys.tolist() == [y[0, 1], y[0, 0]] and Ts.tolist() == [T[0, 1], T[0, 0]]


def _dequant(oracle, codes, scales, rows, cols, cb):
    fields = oracle.unpack2(codes, rows, cols)
    s = scales.view(np.float16).astype(np.float32)
    return (cb[fields] * s[:, None]).astype(np.float32)   # exact: fp16 * small codebook entry


@pytest.mark.parametrize("M,rows,cols", [(1, 37, 64), (1, 9, 1537), (5, 33, 771), (3, 1, 1)])
def test_packed_equals_dense_on_decoded_weights(oracle, M, rows, cols):
    seed = M * 10007 + rows * 31 + cols
    codes = synth.random_bytes(seed, rows * ((cols + 3) // 4)).reshape(rows, -1)
    scales = synth.uniform_f16_bits(seed + 1, (rows,), 0.005, 0.05)
    X = synth.normal_f16_bits(seed + 2, (M, cols))
    cb = synth.CODEBOOK_2BIT
    Y, T = oracle.packed_gemm(codes, scales, X, rows, cols, cb, threads=2)
    W = _dequant(oracle, codes, scales, rows, cols, cb)
    Xf = X.view(np.float16).astype(np.float32)
    C, TC = oracle.gemm(0, 1, M, rows, cols, Xf, W)     # X (M x cols) . W^T
    assert np.array_equal(Y, C)
    assert np.array_equal(T, TC)


def test_packed_constant_field_rows(oracle):
    # a row whose fields are all c gives y = scale * cb[c] * sum_k x_k
    rows, cols = 4, 40
    codes = np.array([[0x00] * 10, [0x55] * 10, [0xAA] * 10, [0xFF] * 10], np.uint8)
    scales = np.array([0x3C00, 0x3800, 0x4000, 0x3400], np.uint16)   # 1, 0.5, 2, 0.25
    x = (np.arange(cols) - 17).astype(np.float16).view(np.uint16)     # exact small ints
    cb = np.array([-2.0, -1.0, 0.0, 1.0], np.float32)
    y, T = oracle.packed_gemm(codes, scales, x, rows, cols, cb)
    sx = float(np.sum(np.arange(cols) - 17))
    sax = float(np.sum(np.abs(np.arange(cols) - 17)))
    s = [1.0, 0.5, 2.0, 0.25]
    assert y[0].tolist() == [s[c] * cb[c] * sx for c in range(4)]
    assert T[0].tolist() == [abs(s[c] * cb[c]) * sax for c in range(4)]


def test_packed_one_hot_reads_single_field(oracle):
    # x = e_k picks scale_r * cb[field(r,k)] for every row: each row's byte
    # decodes per the hand table.
    table = [ln.split() for ln in read_golden("unpack2_bytes.txt")]
    codes = np.array([[int(t[0], 16)] for t in table], np.uint8)
    rows = len(table)
    scales = np.full(rows, 0x3800, np.uint16)   # 0.5
    cb = np.array([-2.0, -1.0, 0.5, 3.0], np.float32)
    for k in range(4):
        x = np.zeros(4, np.uint16); x[k] = 0x3C00
        y, _ = oracle.packed_gemm(codes, scales, x, rows, 4, cb)
        assert y[0].tolist() == [0.5 * float(cb[int(t[1 + k])]) for t in table]


def test_packed_ternary_codebook(oracle):
    # ternary reading: value v stored as field v+1, field 3 decodes to 0
    codes = np.array([[0b00_10_01_00], [0b11_11_11_11]], np.uint8)   # fields 0,1,2,0 and 3,3,3,3
    x = np.array([0x3C00, 0x4000, 0x4200, 0x4400], np.uint16)        # 1,2,3,4
    y, T = oracle.packed_gemm(codes, np.array([0x3C00, 0x3C00], np.uint16), x, 2, 4,
                              synth.CODEBOOK_TERNARY)
    assert y[0].tolist() == [-1 * 1 + 0 * 2 + 1 * 3 + -1 * 4, 0.0]
    assert T[0].tolist() == [1 + 0 + 3 + 4, 0.0]


# ---------------------------------------------------------------- 4-bit form

def test_unpack4_hand_table(oracle):
    for ln in read_golden("unpack4_bytes.txt"):
        parts = ln.split()
        byte = int(parts[0], 16)
        want = [int(v) for v in parts[1:3]]
        got = oracle.unpack4(np.array([byte], np.uint8), 1, 2)[0].tolist()
        assert got == want, (hex(byte), got, want)


def test_pack4_unpack4_roundtrip_all_bytes(oracle):
    allb = np.arange(256, dtype=np.uint8).reshape(32, 8)       # 32 rows x 16 cols
    fields = oracle.unpack4(allb, 32, 16)
    assert fields.max() <= 15
    assert np.array_equal(oracle.pack4(fields), allb)


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (7, 63), (5, 64), (2, 131)])
def test_unpack4_pack4_roundtrip_ragged(oracle, rows, cols):
    rng = np.random.default_rng(rows * 999 + cols)
    fields = rng.integers(0, 16, size=(rows, cols), dtype=np.uint8)
    packed = oracle.pack4(fields)
    assert packed.shape == (rows, (cols + 1) // 2)
    assert np.array_equal(oracle.unpack4(packed, rows, cols), fields)
    dirty = packed.copy()
    if cols % 2:
        dirty[:, -1] |= np.uint8(0xF0)   # the unused high nibble is ignored
    assert np.array_equal(oracle.unpack4(dirty, rows, cols), fields)


def test_packed4_hand_2x5(oracle):
    d = _packed_hand("packed4_2x5_hand.txt")
    cols = int(d["cols"][0])
    cb = np.array([float(v) for v in d["codebook"]], np.float32)
    codes = np.array([[int(v, 16) for v in row] for row in d["codes"]], np.uint8)
    scales = np.array([int(v, 16) for v in d["scales_fp16"][0]], np.uint16)
    x = np.array([int(v, 16) for v in d["x_fp16"][0]], np.uint16)
    y, T = oracle.packed4_gemm(codes, scales, x, 2, cols, cb)
    assert y[0].tolist() == [float(v) for v in d["y"][0]]
    assert T[0].tolist() == [float(v) for v in d["T"][0]]
    ys, Ts = oracle.packed4_gemm_at(codes, scales, x, cols, cb, [0, 0], [1, 0])
    assert ys.tolist() == [y[0, 1], y[0, 0]] and Ts.tolist() == [T[0, 1], T[0, 0]]


@pytest.mark.parametrize("M,rows,cols", [(1, 37, 64), (1, 9, 1537), (4, 33, 771), (3, 1, 1)])
def test_packed4_equals_dense_on_decoded_weights(oracle, M, rows, cols):
    # dyadic codebook (c - 7) / 4: entry x fp16 scale is exact in fp32, so the dense
    # oracle on the decoded weights must give the same sums
    seed = M * 7919 + rows * 13 + cols
    codes = synth.random_bytes(seed, rows * ((cols + 1) // 2)).reshape(rows, -1)
    scales = synth.uniform_f16_bits(seed + 1, (rows,), 0.005, 0.05)
    X = synth.normal_f16_bits(seed + 2, (M, cols))
    cb = ((np.arange(16) - 7) / 4.0).astype(np.float32)
    Y, T = oracle.packed4_gemm(codes, scales, X, rows, cols, cb, threads=2)
    fields = oracle.unpack4(codes, rows, cols)
    W = (cb[fields] * scales.view(np.float16).astype(np.float32)[:, None]).astype(np.float32)
    Xf = X.view(np.float16).astype(np.float32)
    C, TC = oracle.gemm(0, 1, M, rows, cols, Xf, W)
    assert np.array_equal(Y, C)
    assert np.array_equal(T, TC)


def test_packed4_constant_field_rows(oracle):
    # a row whose fields are all c gives y = scale * cb[c] * sum_k x_k
    rows, cols = 16, 30
    codes = np.array([[c * 0x11] * 15 for c in range(16)], np.uint8)
    scales = np.full(rows, 0x3800, np.uint16)                          # 0.5
    x = (np.arange(cols) - 11).astype(np.float16).view(np.uint16)      # exact small ints
    cb = ((np.arange(16) - 7) / 8.0).astype(np.float32)
    y, T = oracle.packed4_gemm(codes, scales, x, rows, cols, cb)
    sx = float(np.sum(np.arange(cols) - 11))
    sax = float(np.sum(np.abs(np.arange(cols) - 11)))
    assert y[0].tolist() == [0.5 * float(cb[c]) * sx for c in range(16)]
    assert T[0].tolist() == [abs(0.5 * float(cb[c])) * sax for c in range(16)]


def test_packed4_one_hot_reads_single_field(oracle):
    table = [ln.split() for ln in read_golden("unpack4_bytes.txt")]
    codes = np.array([[int(t[0], 16)] for t in table], np.uint8)
    rows = len(table)
    scales = np.full(rows, 0x3400, np.uint16)   # 0.25
    cb = synth.CODEBOOK_NQ4
    for k in range(2):
        x = np.zeros(2, np.uint16); x[k] = 0x3C00
        y, _ = oracle.packed4_gemm(codes, scales, x, rows, 2, cb)
        assert y[0].tolist() == [0.25 * float(cb[int(t[1 + k])]) for t in table]


def test_packed4_agrees_with_packed2_on_small_fields(oracle):
    # fields below 4 stored in 4 bits, with the 2-bit codebook in entries 0..3, give the
    # 2-bit sums of the same fields (cross-format check of the nibble and field readings)
    rows, cols = 23, 301
    rng = np.random.default_rng(5)
    fields = rng.integers(0, 4, size=(rows, cols), dtype=np.uint8)
    scales = synth.uniform_f16_bits(6, (rows,), 0.005, 0.05)
    x = synth.normal_f16_bits(7, (cols,))
    cb4 = np.concatenate([synth.CODEBOOK_2BIT, np.full(12, 99.0, np.float32)])
    y4, T4 = oracle.packed4_gemm(oracle.pack4(fields), scales, x, rows, cols, cb4)
    y2, T2 = oracle.packed_gemm(oracle.pack2(fields), scales, x, rows, cols, synth.CODEBOOK_2BIT)
    assert np.array_equal(y4, y2) and np.array_equal(T4, T2)


def test_normal_quantile_codebook():
    # the quantile function against textbook values of the standard normal
    assert synth._normal_ppf(0.5) == pytest.approx(0.0, abs=1e-14)
    assert synth._normal_ppf(0.975) == pytest.approx(1.959963984540054, abs=1e-12)
    assert synth._normal_ppf(0.8413447460685429) == pytest.approx(1.0, abs=1e-12)   # Phi(1)
    assert synth._normal_ppf(0.02) == pytest.approx(-synth._normal_ppf(0.98), abs=1e-12)
    cb = synth.CODEBOOK_NQ4
    assert cb.dtype == np.float32 and cb.size == 16
    assert np.all(np.diff(cb) > 0)
    assert cb[0] == -1.0 and cb[7] == 0.0 and cb[15] == 1.0
    top = synth._normal_ppf(0.98)
    for i in range(1, 9):
        assert cb[7 + i] == np.float32(synth._normal_ppf(0.5 + 0.48 * i / 8) / top)


# ------------------------------------------------------------------ bias + GELU epilogue

def test_gelu_tanh_odd_part_is_identity(oracle):
    # gelu(z) - gelu(-z) = z/2 (1 + t) + z/2 (1 - t) = z for the tanh form, any constants
    z = np.linspace(-9.0, 9.0, 1001)
    assert np.allclose(oracle.gelu_tanh(z) - oracle.gelu_tanh(-z), z, rtol=0, atol=1e-14)


def test_gelu_tanh_matches_erf_form(oracle):
    # the tanh form approximates z Phi(z) (Phi from the library's normal CDF) to within
    # about 5e-4 everywhere; a wrong constant (sqrt(2/pi), 0.044715) or a dropped cubic
    # term misses by far more
    from scipy.special import ndtr
    z = np.linspace(-8.0, 8.0, 4001)
    exact = z * ndtr(z)
    d = np.abs(oracle.gelu_tanh(z) - exact)
    assert d.max() < 1e-3 and d.max() > 1e-5
    wrong_cubic = 0.5 * z * (1 + np.tanh(np.sqrt(2 / np.pi) * z))
    assert np.abs(wrong_cubic - exact).max() > 5e-3


def test_gelu_tanh_matches_the_library_tanh_gelu(oracle):
    # PyTorch's own GELU in its tanh form (an independent implementation of GPT-2's published
    # activation), in fp64 on the CPU: agreement to rounding, so a slip in either constant at any
    # of its printed digits fails -- shown on two planted slips
    import torch
    z = np.linspace(-12.0, 12.0, 24001)
    lib = torch.nn.functional.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    # (where 1 + tanh(u) cancels, below z = -7, the two evaluations differ by rounding, < 1e-15)
    assert np.allclose(oracle.gelu_tanh(z), lib, rtol=1e-13, atol=1e-14)

    def planted(c, a):  # the tanh form with given constants, for the planted slips only
        return 0.5 * z * (1.0 + np.tanh(c * (z + a * z ** 3)))
    c0 = np.sqrt(2.0 / np.pi)
    for c, a in ((c0, 0.04472), (c0 * (1 + 1e-5), 0.044715)):
        assert not np.allclose(planted(c, a), lib, rtol=1e-13, atol=1e-14), (c, a)


def test_gelu_tanh_small_z_series_fixes_the_scale(oracle):
    # z/2 (1 + tanh(c z + ...)) = z/2 + (c/2) z^2 + O(z^4): the z^2 coefficient is 1/sqrt(2 pi), the
    # exact GELU's (z Phi(z) = z/2 + z^2/sqrt(2 pi) + ...), which fixes c = sqrt(2/pi)
    for z in (1e-3, -1e-3, 2e-4):
        coef = (float(oracle.gelu_tanh(z)) - z / 2) / z ** 2
        assert abs(coef * np.sqrt(2 * np.pi) - 1.0) < 1e-5


def test_gelu_tanh_special_values(oracle):
    g = oracle.gelu_tanh(np.array([0.0, 10.0, -10.0, 30.0]))
    assert g[0] == 0.0 and g[1] == 10.0 and g[2] == 0.0 and g[3] == 30.0
    h = 1e-6  # slope 1/2 at the origin
    assert abs((oracle.gelu_tanh(h) - oracle.gelu_tanh(-h)) / (2 * h) - 0.5) < 1e-9


def test_gemm_bias_broadcasts_over_rows(oracle):
    # zero product: every row is the bias vector (one entry per output column)
    M, N, K = 5, 7, 3
    A = np.zeros((M, K), np.float32)
    B = np.ones((K, N), np.float32)
    bias = np.arange(N, dtype=np.float32) - 3.0
    Y, T, Z = oracle.gemm_bias_act(0, 0, M, N, K, A, B, bias, act=0)
    assert np.array_equal(Y, np.tile(bias.astype(np.float64), (M, 1)))
    assert np.array_equal(T, np.tile(np.abs(bias).astype(np.float64), (M, 1)))
    Y1, _, _ = oracle.gemm_bias_act(0, 0, M, N, K, A, B, bias, act=1)
    assert np.array_equal(Y1, oracle.gelu_tanh(np.tile(bias.astype(np.float64), (M, 1))))


def test_gemm_bias_act_without_bias_is_gemm(oracle):
    A = synth.normal_f32(5, (33, 17), 1.0)
    B = synth.normal_f32(6, (17, 21), 1.0)
    C, T = oracle.gemm(0, 0, 33, 21, 17, A, B)
    Y, T2, Z = oracle.gemm_bias_act(0, 0, 33, 21, 17, A, B, None, act=0)
    assert np.array_equal(Y, C) and np.array_equal(T2, T) and np.array_equal(Z, C)


# ------------------------------------------------------------------ attention ("Flash Attention 2")

def _attn_inputs(seed, BH, T, D):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((BH, T, D)).astype(np.float32) for _ in range(4)]


@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("shape", [(2, 37, 16), (1, 64, 64), (3, 5, 8)])
def test_attention_fwd_matches_the_library_attention(oracle, causal, shape):
    # PyTorch's own scaled-dot-product attention and log-sum-exp, in fp64 on the CPU (independent
    # implementations of the definition): agreement to rounding
    import torch
    BH, T, D = shape
    Q, K, V, _ = _attn_inputs(11 + T, BH, T, D)
    scale = np.float32(1.0 / np.sqrt(D))
    O, L, TO = oracle.attention_fwd(Q, K, V, causal, float(scale))
    q, k, v = (torch.from_numpy(a.astype(np.float64)) for a in (Q, K, V))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=bool(causal), scale=float(scale))
    assert np.allclose(O, ref.numpy(), rtol=1e-12, atol=1e-13)
    S = float(scale) * (q @ k.transpose(1, 2))
    if causal:
        S = S.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    assert np.allclose(L, torch.logsumexp(S, dim=-1).numpy(), rtol=1e-13, atol=1e-13)
    assert np.all(TO >= np.abs(O) - 1e-12)


@pytest.mark.parametrize("causal", [0, 1])
def test_attention_bwd_matches_library_autograd(oracle, causal):
    # the gradients of sum(O * dO) by PyTorch autograd through its fp64 attention
    import torch
    BH, T, D = 2, 33, 16
    Q, K, V, dO = _attn_inputs(21 + causal, BH, T, D)
    scale = float(np.float32(0.3))
    dQ, dK, dV, TdQ, TdK, TdV = oracle.attention_bwd(Q, K, V, dO, causal, scale)
    q, k, v = (torch.from_numpy(a.astype(np.float64)).requires_grad_(True) for a in (Q, K, V))
    out = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=bool(causal), scale=scale)
    (out * torch.from_numpy(dO.astype(np.float64))).sum().backward()
    for mine, ref, name in ((dQ, q.grad, "dQ"), (dK, k.grad, "dK"), (dV, v.grad, "dV")):
        assert np.allclose(mine, ref.numpy(), rtol=1e-11, atol=1e-12), name
    for g, t in ((dQ, TdQ), (dK, TdK), (dV, TdV)):
        assert np.all(t >= np.abs(g) - 1e-12)


def test_attention_uniform_closed_form(oracle):
    # Q = 0: every score is 0, so a causal row i weighs keys 0..i equally -- O_i is the mean of
    # V_0..V_i and L_i = log(i + 1); without the mask every row is the mean of all of V, L = log T
    BH, T, D = 2, 12, 8
    _, K, V, _ = _attn_inputs(31, BH, T, D)
    Q = np.zeros_like(K)
    O, L, _ = oracle.attention_fwd(Q, K, V, 1, 0.7)
    means = np.cumsum(V.astype(np.float64), axis=1) / np.arange(1, T + 1).reshape(1, T, 1)
    assert np.allclose(O, means, rtol=0, atol=1e-14)
    assert np.allclose(L, np.log(np.arange(1, T + 1)).reshape(1, T), rtol=0, atol=1e-15)
    O2, L2, _ = oracle.attention_fwd(Q, K, V, 0, 0.7)
    assert np.allclose(O2, np.broadcast_to(V.astype(np.float64).mean(axis=1, keepdims=True), O2.shape), atol=1e-14)
    assert np.allclose(L2, np.log(T), atol=1e-15)


def test_attention_first_causal_row_and_magnitudes(oracle):
    # a causal first row sees only key 0: O_0 = V_0 exactly and L_0 = its one score; with V >= 0
    # the bound scale TO equals O
    BH, T, D = 3, 10, 8
    Q, K, V, _ = _attn_inputs(41, BH, T, D)
    scale = 0.25
    O, L, TO = oracle.attention_fwd(Q, K, V, 1, scale)
    assert np.array_equal(O[:, 0], V[:, 0].astype(np.float64))
    s00 = scale * np.einsum("hd,hd->h", Q[:, 0].astype(np.float64), K[:, 0].astype(np.float64))
    assert np.allclose(L[:, 0], s00, rtol=0, atol=1e-15)
    Vp = np.abs(V)
    O, _, TO = oracle.attention_fwd(Q, K, Vp, 1, scale)
    assert np.allclose(TO, O, rtol=1e-15, atol=0)
