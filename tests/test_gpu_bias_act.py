"""GPU parity of the GEMM with GPT-2's bias + GELU epilogue (C = act(op(A) op(B) + bias)).

Bound per output: |y - y_ref| <= 1.13e-5 T + 2^-20 (1 + |z|), with T = sum_k |a b| + |bias|
and z the exact pre-activation: the GEMM's 1e-5 T bound carried through gelu's
slope (at most 1.13), plus the fp32 evaluation of the activation itself.
"""
import numpy as np
import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import synth
from gpu_util import empty_f32, to_dev, to_host

pytestmark = pytest.mark.gpu

LAYOUTS = {"nn": (0, 0), "nt": (0, 1), "tn": (1, 0), "tt": (1, 1)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_packed_bit_gb300 import build
    build.build()
    mm.load_library()


def operands(tA, tB, M, N, K, seed, lda=None, ldb=None):
    a_shape = (K, lda or M) if tA else (M, lda or K)
    b_shape = (N, ldb or K) if tB else (K, ldb or N)
    return synth.normal_f32(seed, a_shape, 1.0), synth.normal_f32(seed + 1, b_shape, 1.0)


def run(tA, tB, M, N, K, A, B, bias, act, ldc=None):
    ldc = ldc or N
    dA, dB = to_dev(A), to_dev(B)
    dbias = None if bias is None else to_dev(bias)
    dC = empty_f32((M, ldc))
    mm.mm_gemm_f32_bias_act(tA, tB, M, N, K, dA, A.shape[1], dB, B.shape[1], dbias, act, dC, ldc)
    mm.mm_check_device_error()
    return to_host(dC)


def check(got, Y, T, Z, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - Y)
    bound = 1.13e-5 * T + 2.0 ** -20 * (1.0 + np.abs(Z))
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(i), float(got[tuple(i)]), float(Y[tuple(i)]), float(bound[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {int(bad.sum())} outputs outside the bound, e.g. {detail}")


# ragged tiles and K tails; M <= 128 runs single CTAs, larger M CTA pairs (TMA-stored C)
SHAPES = [(1, 1, 4), (5, 7, 3), (65, 129, 33), (128, 256, 16), (200, 300, 96), (257, 130, 1000),
          (64, 3072, 768), (1000, 2900, 72)]


@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("with_bias", [True, False])
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", SHAPES)
def test_bias_act_parity(oracle, shape, layout, with_bias, act):
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = operands(tA, tB, M, N, K, seed=31 * M + 7 * N + K + 1000 * act)
    bias = synth.normal_f32(17 + N, (N,), 2.0) if with_bias else None
    got = run(tA, tB, M, N, K, A, B, bias, act)
    Y, T, Z = oracle.gemm_bias_act(tA, tB, M, N, K, A, B, bias, act)
    check(got, Y, T, Z, f"{layout} {shape} bias={with_bias} act={act}")


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_bias_act_unaligned_leading_dims_general_kernel(oracle, layout):
    # leading dimensions that are not multiples of 4 rule out TMA: the general kernel runs
    tA, tB = LAYOUTS[layout]
    M, N, K = 67, 45, 29
    A2, B = operands(tA, tB, M, N, K, seed=5, lda=(M if tA else K) + 1)
    bias = synth.normal_f32(9, (N,), 1.0)
    dA, dB, db = to_dev(A2), to_dev(B), to_dev(bias)
    dC = empty_f32((M, N + 3))
    mm.mm_gemm_f32_bias_act(tA, tB, M, N, K, dA, A2.shape[1], dB, B.shape[1], db, 1, dC, N + 3)
    mm.mm_check_device_error()
    got = to_host(dC)
    Y, T, Z = oracle.gemm_bias_act(tA, tB, M, N, K, A2, B, bias, 1, lda=A2.shape[1])
    check(got[:, :N], Y, T, Z, f"{layout} unaligned")
    assert np.all(np.isnan(got[:, N:])), "write past N into the padding of C"


def test_bias_act_gpt2_mlp_up_8192x3072x768_sampled(oracle):
    # GPT-2 small's MLP up-projection at 8 sequences of 1024 tokens: every output of
    # sampled rows and columns
    M, N, K = 8192, 3072, 768
    A, B = operands(0, 0, M, N, K, seed=77)
    bias = synth.normal_f32(78, (N,), 1.0)
    got = run(0, 0, M, N, K, A, B, bias, 1)
    rows = np.array([0, 1, 127, 128, 129, 255, 256, 4095, 4096, 8063, 8191])
    cols = np.array([0, 1, 127, 128, 255, 256, 1535, 1536, 3071])
    Yr, Tr, Zr = oracle.gemm_bias_act(0, 0, len(rows), N, K, A[rows], B, bias, 1)
    check(got[rows], Yr, Tr, Zr, "sampled rows")
    Yc, Tc, Zc = oracle.gemm_bias_act(0, 0, M, len(cols), K, A, B[:, cols], bias[cols], 1)
    check(got[:, cols], Yc, Tc, Zc, "sampled columns")


def test_bias_act_identity_is_plain_gemm_and_deterministic():
    # act 0 with no bias is the plain GEMM: same kernel, same bits
    M, N, K = 300, 260, 200
    A, B = operands(0, 0, M, N, K, seed=3)
    dA, dB = to_dev(A), to_dev(B)
    c1, c2 = empty_f32((M, N)), empty_f32((M, N))
    mm.mm_gemm_f32_bias_act(0, 0, M, N, K, dA, K, dB, N, None, 0, c1, N)
    mm.mm_gemm_f32_ex(0, 0, M, N, K, dA, K, dB, N, c2, N, path=mm.MM_GEMM_TF32X3, tile=3)
    mm.mm_check_device_error()
    assert np.array_equal(to_host(c1), to_host(c2))
    b = synth.normal_f32(4, (N,), 1.0)
    db = to_dev(b)
    r = [run(0, 0, M, N, K, A, B, b, 1) for _ in range(2)]
    assert np.array_equal(r[0], r[1])


# ------------------------------------------------------------------ with the K split

def run_split(tA, tB, M, N, K, A, B, bias, act, splitk):
    dA, dB = to_dev(A), to_dev(B)
    dbias = None if bias is None else to_dev(bias)
    dC = empty_f32((M, N))
    need = mm.mm_gemm_f32_splitk_workspace(M, N, K, splitk)
    ws = empty_f32((max(need, 4),), 0.0)
    mm.mm_gemm_f32_bias_act_splitk(tA, tB, M, N, K, dA, A.shape[1], dB, B.shape[1], dbias, act, dC, N, splitk, ws,
                                   need)
    mm.mm_check_device_error()
    return to_host(dC)


@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("splitk", [0, 1, 3, 16, -1])
@pytest.mark.parametrize("layout", ["nn", "nt", "tn"])
@pytest.mark.parametrize("shape", [(64, 3072, 768), (300, 2000, 1000), (129, 257, 33), (2000, 2900, 72)])
def test_bias_act_split_parity(oracle, shape, layout, splitk, act):
    # K slices (bias and act applied by the reduce kernel), stream-K (applied by the segment that
    # completes a tile), the automatic choice, and no split
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = operands(tA, tB, M, N, K, seed=7 * M + N + K + 100 * act)
    bias = synth.normal_f32(5 + N, (N,), 1.0)
    got = run_split(tA, tB, M, N, K, A, B, bias, act, splitk)
    Y, T, Z = oracle.gemm_bias_act(tA, tB, M, N, K, A, B, bias, act)
    check(got, Y, T, Z, f"{layout} {shape} splitk {splitk} act {act}")


def test_bias_act_split_gpt2_mlp_up_sampled(oracle):
    # the 8192 x 3072 x 768 MLP up-projection with its automatic split, sampled rows and columns
    M, N, K = 8192, 3072, 768
    A, B = operands(0, 0, M, N, K, seed=91)
    bias = synth.normal_f32(92, (N,), 1.0)
    got = run_split(0, 0, M, N, K, A, B, bias, 1, 0)
    rows = np.array([0, 127, 128, 255, 256, 4095, 8191])
    cols = np.array([0, 255, 256, 1535, 3071])
    Yr, Tr, Zr = oracle.gemm_bias_act(0, 0, len(rows), N, K, A[rows], B, bias, 1)
    check(got[rows], Yr, Tr, Zr, "sampled rows")
    Yc, Tc, Zc = oracle.gemm_bias_act(0, 0, M, len(cols), K, A, B[:, cols], bias[cols], 1)
    check(got[:, cols], Yc, Tc, Zc, "sampled columns")


@pytest.mark.parametrize("layout", ["nn", "nt", "tn"])
def test_bias_act_padded_leading_dims(oracle, layout):
    # padded lda / ldb (multiples of 4: the tensor-core path) and a padded C whose pad stays untouched
    tA, tB = LAYOUTS[layout]
    M, N, K = 300, 260, 96
    A, B = operands(tA, tB, M, N, K, seed=33, lda=(M if tA else K) + 8, ldb=(K if tB else N) + 4)
    bias = synth.normal_f32(34, (N,), 1.0)
    dA, dB, db = to_dev(A), to_dev(B), to_dev(bias)
    dC = empty_f32((M, N + 12))
    mm.mm_gemm_f32_bias_act(tA, tB, M, N, K, dA, A.shape[1], dB, B.shape[1], db, 1, dC, N + 12)
    mm.mm_check_device_error()
    got = to_host(dC)
    Y, T, Z = oracle.gemm_bias_act(tA, tB, M, N, K, A, B, bias, 1, lda=A.shape[1], ldb=B.shape[1])
    check(got[:, :N], Y, T, Z, f"{layout} padded")
    assert np.all(np.isnan(got[:, N:])), "write into the padding of C"


@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", [(17, 257, 300), (64, 130, 48), (1, 5, 8), (40, 1000, 777), (63, 128, 16)])
def test_bias_act_few_rows_tensor_cores(oracle, shape, layout, act):
    # M <= 64 with leading dimensions a multiple of four: the few-rows 3xTF32 kernel (C computed
    # transposed, K split over a cluster), whose reduction applies bias and GELU to the summed
    # partial tiles; ragged N and K, a padded C whose pad stays untouched
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    lda = (M if tA else K) + 3
    ldb = (K if tB else N) + 3
    lda, ldb = lda + (-lda) % 4, ldb + (-ldb) % 4
    A, B = operands(tA, tB, M, N, K, seed=91 + M + N + K + 7 * act, lda=lda, ldb=ldb)
    bias = synth.normal_f32(35 + N, (N,), 1.0)
    dA, dB, db = to_dev(A), to_dev(B), to_dev(bias)
    dC = empty_f32((M, N + 5))
    mm.mm_gemm_f32_bias_act(tA, tB, M, N, K, dA, A.shape[1], dB, B.shape[1], db, act, dC, N + 5)
    mm.mm_check_device_error()
    got = to_host(dC)
    Y, T, Z = oracle.gemm_bias_act(tA, tB, M, N, K, A, B, bias, act, lda=A.shape[1], ldb=B.shape[1])
    check(got[:, :N], Y, T, Z, f"few rows {layout} {shape} act={act}")
    assert np.all(np.isnan(got[:, N:])), "write into the padding of C"


@pytest.mark.parametrize("M", [48, 1024])
def test_gelu_epilogue_within_the_activation_term_alone(oracle, M):
    # K = 1, A = z_r (row r), B = 1 and bias_j = j 2^-12 make every pre-activation z = z_r + bias_j
    # exact in fp32 (z_r multiples of 2^-6 in [-12, 12]; 3xTF32's hi + lo split of z_r adds back to
    # z_r), so the whole error is the fp32 activation's: it must fit the bound's activation term
    # 2^-20 (1 + |z|) with the GEMM term 1.13e-5 T left out.  M = 48 takes the few-rows kernel,
    # M = 1024 the 3xTF32 one.
    N = 64
    zr = np.round((-12.0 + 24.0 * np.arange(M) / (M - 1)) * 64.0) / 64.0
    A = zr.astype(np.float32).reshape(M, 1)
    B = np.ones((1, N), np.float32)
    bias = (np.arange(N) * 2.0 ** -12).astype(np.float32)
    Y, T, Z = oracle.gemm_bias_act(0, 0, M, N, 1, A, B, bias, act=1)
    assert np.array_equal(Z.astype(np.float32).astype(np.float64), Z), "pre-activations exact in fp32"
    got = run(0, 0, M, N, 1, A, B, bias, 1).astype(np.float64)
    err = np.abs(got - Y)
    bound = 2.0 ** -20 * (1.0 + np.abs(Z))
    assert np.all(err <= bound), f"worst {float(np.max(err / bound)):.3f} of the activation term"
    print(f"M={M}: worst error {float(np.max(err / bound)):.4f} of 2^-20 (1 + |z|)")
