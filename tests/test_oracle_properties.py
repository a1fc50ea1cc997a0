"""Property tests of the CPU oracle over random shapes, codebooks and data.

The fixed-shape pins in test_oracle.py tie the oracle to hand tables and closed
forms; these draw many ragged shapes and check invariants that a transposed
index, a wrong row stride or a misplaced scale would break: packing round
trips, packed = dense on the decoded weights, permuting W's rows permutes Y's
columns, scaling X by a power of two scales Y exactly, and |Y| <= T.
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

SETTINGS = settings(max_examples=40, deadline=None, derandomize=True)


def _case(seed, M, rows, cols, nbits=2):
    rng = np.random.default_rng(seed)
    per = 8 // nbits
    codes = rng.integers(0, 256, size=(rows, -(-cols // per)), dtype=np.uint8)
    scales = rng.uniform(0.005, 0.05, size=rows).astype(np.float16).view(np.uint16)
    X = rng.normal(size=(M, cols)).astype(np.float16).view(np.uint16)
    ncb = 1 << nbits
    cb = rng.uniform(-2.0, 2.0, size=ncb).astype(np.float32)
    return codes, scales, X, cb


def _decoded(oracle, codes, scales, rows, cols, cb, nbits):
    fields = oracle.unpack2(codes, rows, cols) if nbits == 2 else oracle.unpack4(codes, rows, cols)
    # fp16 scale x fp32 entry, kept in fp64 (exact) for the dense comparison
    return cb.astype(np.float64)[fields] * scales.view(np.float16).astype(np.float64)[:, None]


shapes = st.tuples(st.integers(1, 4), st.integers(1, 40), st.integers(1, 70), st.integers(0, 2 ** 31 - 1))


@SETTINGS
@given(shapes, st.sampled_from([2, 4]))
def test_pack_unpack_round_trip(oracle, shape, nbits):
    _, rows, cols, seed = shape
    fields = np.random.default_rng(seed).integers(0, 1 << nbits, size=(rows, cols), dtype=np.uint8)
    if nbits == 2:
        assert np.array_equal(oracle.unpack2(oracle.pack2(fields), rows, cols), fields)
    else:
        assert np.array_equal(oracle.unpack4(oracle.pack4(fields), rows, cols), fields)


@SETTINGS
@given(shapes, st.sampled_from([2, 4]))
def test_packed_matches_dense_and_bounds(oracle, shape, nbits):
    M, rows, cols, seed = shape
    codes, scales, X, cb = _case(seed, M, rows, cols, nbits)
    f = oracle.packed_gemm if nbits == 2 else oracle.packed4_gemm
    Y, T = f(codes, scales, X, rows, cols, cb, threads=1)
    W = _decoded(oracle, codes, scales, rows, cols, cb, nbits)
    Xd = X.view(np.float16).astype(np.float64)
    ref = Xd @ W.T                                   # numpy's fp64 product of the decoded weights
    assert Y.shape == (M, rows) and T.shape == (M, rows)
    assert np.all(np.abs(Y - ref) <= 1e-12 * (np.abs(Xd) @ np.abs(W).T) + 1e-300)
    assert np.all(np.abs(Y) <= T * (1 + 1e-12))
    assert np.allclose(T, np.abs(Xd) @ np.abs(W).T, rtol=1e-12, atol=0)


@SETTINGS
@given(shapes)
def test_row_permutation_and_power_of_two_scaling(oracle, shape):
    M, rows, cols, seed = shape
    codes, scales, X, cb = _case(seed, M, rows, cols)
    Y, T = oracle.packed_gemm(codes, scales, X, rows, cols, cb, threads=1)
    perm = np.random.default_rng(seed + 1).permutation(rows)
    Yp, Tp = oracle.packed_gemm(codes[perm], scales[perm], X, rows, cols, cb, threads=1)
    assert np.array_equal(Yp, Y[:, perm]) and np.array_equal(Tp, T[:, perm])
    X2 = (X.view(np.float16) * np.float16(0.5)).view(np.uint16)   # exact unless it underflows
    if np.array_equal(X2.view(np.float16).astype(np.float64) * 2, X.view(np.float16).astype(np.float64)):
        Y2, _ = oracle.packed_gemm(codes, scales, X2, rows, cols, cb, threads=1)
        assert np.array_equal(Y2 * 2, Y)


@SETTINGS
@given(shapes)
def test_single_active_column_reads_one_field(oracle, shape):
    M, rows, cols, seed = shape
    codes, scales, _, cb = _case(seed, 1, rows, cols)
    k = seed % cols
    x = np.zeros((1, cols), np.float16)
    x[0, k] = np.float16(1.0)
    y, _ = oracle.packed_gemm(codes, scales, x.view(np.uint16), rows, cols, cb, threads=1)
    fields = (codes[:, k // 4] >> (2 * (k % 4))) & 3
    want = cb.astype(np.float64)[fields] * scales.view(np.float16).astype(np.float64)
    assert np.array_equal(y[0], want)


@SETTINGS
@given(st.tuples(st.integers(1, 6), st.integers(1, 9), st.integers(1, 12), st.integers(0, 2 ** 31 - 1)),
       st.sampled_from([(0, 0), (0, 1), (1, 0), (1, 1)]))
def test_dense_matches_numpy_and_bounds(oracle, shape, flags):
    M, N, K, seed = shape
    tA, tB = flags
    rng = np.random.default_rng(seed)
    A = rng.normal(size=(K, M) if tA else (M, K)).astype(np.float32)
    B = rng.normal(size=(N, K) if tB else (K, N)).astype(np.float32)
    C, T = oracle.gemm(tA, tB, M, N, K, A, B, threads=1)
    opA = (A.T if tA else A).astype(np.float64)
    opB = (B.T if tB else B).astype(np.float64)
    assert np.allclose(C, opA @ opB, rtol=0, atol=1e-12 * max(1.0, float(np.max(np.abs(opA) @ np.abs(opB)))))
    assert np.allclose(T, np.abs(opA) @ np.abs(opB), rtol=1e-12, atol=0)
