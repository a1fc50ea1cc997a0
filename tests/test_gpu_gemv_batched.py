"""GPU parity of the strided batch of 2-bit GEMVs (one launch for the whole batch).

Every output of every matrix against the oracle, and bit for bit against one
staged call per matrix (the batched kernel runs the same arithmetic in the same
order); shared and per-matrix x, padded strides, ragged row blocks, CTAs that
span many small matrices, and the per-matrix fallback for shapes the one-launch
kernel does not take.
"""
import numpy as np
import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import synth
from gpu_util import check_bound, empty_f32, to_dev, to_host

pytestmark = pytest.mark.gpu

CB2 = synth.CODEBOOK_2BIT
CB_ODD = np.array([0.3, -1.7, 2.5, 0.01], np.float32)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_packed_bit_gb300 import build
    build.build()
    mm.load_library()


def make_batch(batch, rows, cols, seed, shared_x, pad_rows=0):
    rb = (cols + 3) // 4
    codes = synth.random_bytes(seed, batch * (rows + pad_rows) * rb).reshape(batch, rows + pad_rows, rb)
    scales = synth.uniform_f16_bits(seed + 1, (batch, rows + pad_rows), 0.005, 0.05)
    nx = 1 if shared_x else batch
    x = synth.normal_f16_bits(seed + 2, (nx, cols))
    return codes, scales, x


def run_batched(codes, scales, x, rows, cols, cb, shared_x, dequant=None):
    batch, rtot, rb = codes.shape
    dc, ds, dx = to_dev(codes), to_dev(scales), to_dev(x)
    dy = empty_f32((batch, rtot))
    if dequant is None:
        mm.mm_gemv_packed2_strided_batched(dc, rtot * rb, ds, rtot, dx, 0 if shared_x else cols, dy, rtot, batch,
                                           rows, cols, cb)
    else:
        mm.mm_gemv_packed2_strided_batched_ex(dc, rtot * rb, ds, rtot, dx, 0 if shared_x else cols, dy, rtot, batch,
                                              rows, cols, cb, dequant=dequant)
    mm.mm_check_device_error()
    return to_host(dy)


@pytest.mark.parametrize("shared_x", [True, False])
@pytest.mark.parametrize("batch,rows,cols,pad", [(8, 12288, 1536, 0), (3, 1000, 512, 24), (1, 129, 4096, 0),
                                                 (200, 65, 1024, 0), (37, 300, 2048, 4)])
def test_batched_gemv_parity_and_bitwise_equal_to_single_calls(oracle, batch, rows, cols, pad, shared_x):
    # the staged SIMT affine kernel over the whole batch (the automatic choice takes the fp4
    # tensor-core decode, tested below)
    codes, scales, x = make_batch(batch, rows, cols, seed=batch + rows + cols, shared_x=shared_x, pad_rows=pad)
    y = run_batched(codes, scales, x, rows, cols, CB2, shared_x, dequant=mm.MM_DEQ_AFFINE)
    for b in range(batch):
        xb = x[0 if shared_x else b]
        ref, T = oracle.packed_gemm(codes[b, :rows], scales[b, :rows], xb.reshape(1, cols), rows, cols, CB2)
        check_bound(y[b, :rows], ref[0], T[0], f"matrix {b}")
        assert np.all(np.isnan(y[b, rows:])), "write into the padding rows of y"
    # the same arithmetic as one staged call per matrix
    for b in sorted({0, batch // 2, batch - 1}):
        dc, ds = to_dev(np.ascontiguousarray(codes[b, :rows])), to_dev(np.ascontiguousarray(scales[b, :rows]))
        dx = to_dev(np.ascontiguousarray(x[0 if shared_x else b]))
        dy = empty_f32((rows,))
        mm.mm_gemv_packed2_ex(dc, ds, dx, dy, rows, cols, CB2, dequant=2, staging=1)
        assert np.array_equal(to_host(dy).view(np.uint32), y[b, :rows].view(np.uint32)), f"matrix {b} not bitwise equal"


@pytest.mark.parametrize("cb,cols", [("odd", 1536), ("2bit", 1000), ("2bit", 8192)])
def test_batched_gemv_fallback_shapes(oracle, cb, cols):
    # a non-affine codebook, cols not a multiple of 512, cols above 4096: one call per matrix
    codebook = CB_ODD if cb == "odd" else CB2
    batch, rows = 4, 333
    codes, scales, x = make_batch(batch, rows, cols, seed=cols, shared_x=False)
    y = run_batched(codes, scales, x, rows, cols, codebook, False)
    for b in range(batch):
        ref, T = oracle.packed_gemm(codes[b], scales[b], x[b].reshape(1, cols), rows, cols, codebook)
        check_bound(y[b], ref[0], T[0], f"{cb} {cols} matrix {b}")


def test_batched_gemv_zero_entry_rows_exact(oracle):
    # rows whose fields all hold the zero entry (code 2 of {-2,-1,0,1}) give exactly 0
    batch, rows, cols = 5, 256, 1536
    codes, scales, x = make_batch(batch, rows, cols, seed=3, shared_x=True)
    codes[:, ::7, :] = 0xAA  # every field = 2
    y = run_batched(codes, scales, x, rows, cols, CB2, True)
    assert np.all(y[:, ::7] == 0.0)


def test_batched_gemv_single_matrix_and_unaligned_stride_fallback(oracle):
    # batch 1 runs the one-launch kernel; a codes stride that is not a multiple of 16 bytes
    # (one extra byte per matrix) takes one call per matrix
    rows, cols = 200, 1536
    rb = cols // 4
    codes, scales, x = make_batch(1, rows, cols, seed=61, shared_x=True)
    y = run_batched(codes, scales, x, rows, cols, CB2, True)
    ref, T = oracle.packed_gemm(codes[0], scales[0], x.reshape(1, cols), rows, cols, CB2)
    check_bound(y[0], ref[0], T[0], "batch 1")
    batch = 3
    flat = synth.random_bytes(62, batch * (rows * rb + 1))
    sc = synth.uniform_f16_bits(63, (batch, rows), 0.005, 0.05)
    dflat, dsc, dx = to_dev(flat), to_dev(sc), to_dev(x[0])
    dy = empty_f32((batch, rows))
    mm.mm_gemv_packed2_strided_batched(dflat, rows * rb + 1, dsc, rows, dx, 0, dy, rows, batch, rows, cols, CB2)
    mm.mm_check_device_error()
    yh = to_host(dy)
    for b in range(batch):
        cb_ = flat[b * (rows * rb + 1): b * (rows * rb + 1) + rows * rb].reshape(rows, rb)
        ref, T = oracle.packed_gemm(cb_, sc[b], x[0].reshape(1, cols), rows, cols, CB2)
        check_bound(yh[b], ref[0], T[0], f"unaligned stride, matrix {b}")


def run_batched_mxf4(codes, scales, x, rows, cols, cb, shared_x, tiles=0):
    batch, rtot, rb = codes.shape
    dc, ds, dx = to_dev(codes), to_dev(scales), to_dev(x)
    dy = empty_f32((batch, rtot))
    mm.mm_gemv_packed2_strided_batched_ex(dc, rtot * rb, ds, rtot, dx, 0 if shared_x else cols, dy, rtot, batch,
                                          rows, cols, cb, dequant=mm.MM_DEQ_MXF4, rows_per_lane=tiles)
    mm.mm_check_device_error()
    return to_host(dy)


@pytest.mark.parametrize("tiles", [0, 1, 3, 40])
@pytest.mark.parametrize("shared_x", [True, False])
@pytest.mark.parametrize("batch,rows,cols,pad", [(8, 12288, 1536, 0), (3, 1000, 512, 24), (1, 129, 4096, 0),
                                                 (200, 65, 1024, 0), (37, 300, 2048, 4)])
def test_batched_gemv_mxf4_parity_and_bitwise_equal_to_single_calls(oracle, batch, rows, cols, pad, shared_x, tiles):
    # one launch of the fp4 tensor-core decode over the batch; CTAs whose run of tiles spans
    # several matrices rebuild their x pieces at each matrix when x is not shared
    codes, scales, x = make_batch(batch, rows, cols, seed=batch + rows + cols + 5, shared_x=shared_x, pad_rows=pad)
    y = run_batched_mxf4(codes, scales, x, rows, cols, CB2, shared_x, tiles)
    for b in range(batch):
        xb = x[0 if shared_x else b]
        ref, T = oracle.packed_gemm(codes[b, :rows], scales[b, :rows], xb.reshape(1, cols), rows, cols, CB2)
        check_bound(y[b, :rows], ref[0], T[0], f"matrix {b}")
        assert np.all(np.isnan(y[b, rows:])), "write into the padding rows of y"
    for b in sorted({0, batch // 2, batch - 1}):
        dc, ds = to_dev(np.ascontiguousarray(codes[b, :rows])), to_dev(np.ascontiguousarray(scales[b, :rows]))
        dx = to_dev(np.ascontiguousarray(x[0 if shared_x else b]))
        dy = empty_f32((rows,))
        mm.mm_gemv_packed2_ex(dc, ds, dx, dy, rows, cols, CB2, dequant=mm.MM_DEQ_MXF4)
        assert np.array_equal(to_host(dy).view(np.uint32), y[b, :rows].view(np.uint32)), f"matrix {b} not bitwise equal"


def test_batched_gemv_mxf4_zero_entry_rows_exact():
    batch, rows, cols = 5, 256, 1536
    codes, scales, x = make_batch(batch, rows, cols, seed=4, shared_x=False)
    codes[:, ::7, :] = 0xAA  # every field = 2
    y = run_batched_mxf4(codes, scales, x, rows, cols, CB2, False)
    assert np.all(y[:, ::7] == 0.0)


def test_batched_gemv_mxf4_refusals():
    rows, cols = 100, 1536
    codes, scales, x = make_batch(2, rows, cols, seed=9, shared_x=True)
    with pytest.raises(mm.MMError):  # not affine
        run_batched_mxf4(codes, scales, x, rows, cols, CB_ODD, True)
    with pytest.raises(mm.MMError):  # cols not a multiple of 512
        c2, s2, x2 = make_batch(2, rows, 1000, seed=9, shared_x=True)
        run_batched_mxf4(c2, s2, x2, rows, 1000, CB2, True)
    dc, ds, dx = to_dev(codes), to_dev(scales), to_dev(x)
    dy = empty_f32((2, rows))
    for kw in (dict(dequant=mm.MM_DEQ_FP8), dict(dequant=mm.MM_DEQ_MXF4, rows_per_lane=-1),
               dict(dequant=mm.MM_DEQ_AFFINE, pdl=1), dict(dequant=mm.MM_DEQ_MXF4, pdl=2),
               dict(dequant=mm.MM_DEQ_MXF4, independent=3)):
        with pytest.raises(mm.MMError):
            mm.mm_gemv_packed2_strided_batched_ex(dc, rows * cols // 4, ds, rows, dx, 0, dy, rows, 2, rows, cols,
                                                  CB2, **kw)


def test_batched_gemv_automatic_takes_the_fp4_decode(oracle):
    # without options the batch runs the fp4 tensor-core decode: bit for bit the single calls'
    batch, rows, cols = 6, 1000, 1536
    codes, scales, x = make_batch(batch, rows, cols, seed=17, shared_x=False)
    y = run_batched(codes, scales, x, rows, cols, CB2, False)
    for b in range(batch):
        dc, ds, dx = to_dev(np.ascontiguousarray(codes[b])), to_dev(np.ascontiguousarray(scales[b])), to_dev(x[b])
        dy = empty_f32((rows,))
        mm.mm_gemv_packed2_ex(dc, ds, dx, dy, rows, cols, CB2, dequant=mm.MM_DEQ_MXF4)
        assert np.array_equal(to_host(dy).view(np.uint32), y[b].view(np.uint32)), f"matrix {b}"
        ref, T = oracle.packed_gemm(codes[b], scales[b], x[b].reshape(1, cols), rows, cols, CB2)
        check_bound(y[b], ref[0], T[0], f"matrix {b}")
