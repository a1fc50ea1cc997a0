"""GPU parity of the packed 4-bit GEMV (through the C ABI) against the oracle.

The 12,288 x 1,536 4-bit workload is checked on every output of all 64 rotated
matrices; decoding is checked bit for bit with one-hot activations (normal-
quantile codebook) and with integer codebooks and activations.
"""
import numpy as np
import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import synth
from gpu_util import check_bound, check_exact, empty_f32, to_dev, to_host

pytestmark = pytest.mark.gpu

NQ4 = synth.CODEBOOK_NQ4
CB_INT = (np.arange(16) - 7).astype(np.float32)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_packed_bit_gb300 import build
    build.build()
    mm.load_library()


def gemv4(codes, scales, x, rows, cols, cb, **opts):
    dc, ds, dx = to_dev(codes), to_dev(scales), to_dev(x.reshape(-1))
    dy = empty_f32((rows,))
    if opts:
        mm.mm_gemv_packed4_ex(dc, ds, dx, dy, rows, cols, cb, **opts)
    else:
        mm.mm_gemv_packed4(dc, ds, dx, dy, rows, cols, cb)
    mm.mm_check_device_error()
    return to_host(dy)


def rand_case4(rows, cols, seed=0):
    rb = (cols + 1) // 2
    codes = synth.random_bytes(seed, rows * rb).reshape(rows, rb)
    scales = synth.uniform_f16_bits(seed + 1, (rows,), 0.005, 0.05)
    x = synth.normal_f16_bits(seed + 2, (cols,))
    return codes, scales, x


def test_gemv4_12288x1536_all_64_matrices(oracle):
    worst = 0.0
    for i in range(64):
        c = synth.gemv_4bit_12288x1536(i)
        y = gemv4(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
        ref, T = oracle.packed4_gemm(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
        worst = max(worst, check_bound(y, ref[0], T[0], c.name))
    print(f"64 matrices: worst |err|/T = {worst:.3e}")


MODES = [dict(pdl=0), dict(pdl=1, weights_static=1), dict(pdl=1, independent=1)]


@pytest.mark.parametrize("rows", [1, 63, 64, 65, 1000, 1100])
@pytest.mark.parametrize("cols", [256, 512, 1536, 4096])
@pytest.mark.parametrize("mode", MODES, ids=["serial", "chained", "independent"])
@pytest.mark.parametrize("blocks", [0, 1, 3])
def test_gemv4_staged(oracle, rows, cols, mode, blocks):
    # 64-row blocks through the TMA ring, byte-indexed table decode, ragged last CTAs and blocks
    codes, scales, x = rand_case4(rows, cols, seed=rows * 17 + cols)
    y = gemv4(codes, scales, x, rows, cols, NQ4, staging=1, blocks=blocks, **mode)
    ref, T = oracle.packed4_gemm(codes, scales, x, rows, cols, NQ4)
    check_bound(y, ref[0], T[0], f"{rows}x{cols} {mode} blocks {blocks}")


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (7, 255), (33, 257), (65, 1537), (9, 10000), (130, 2048)])
@pytest.mark.parametrize("staging", [0, -1])
def test_gemv4_generic_shapes(oracle, rows, cols, staging):
    # any shape: the generic kernel (and the automatic choice, which falls back to it)
    codes, scales, x = rand_case4(rows, cols, seed=rows * 3 + cols)
    y = gemv4(codes, scales, x, rows, cols, NQ4, staging=staging)
    ref, T = oracle.packed4_gemm(codes, scales, x, rows, cols, NQ4)
    check_bound(y, ref[0], T[0], f"{rows}x{cols}")


@pytest.mark.parametrize("cols", [5, 257, 1537])
def test_gemv4_ignores_nibble_past_cols(oracle, cols):
    rows = 40
    codes, scales, x = rand_case4(rows, cols, seed=cols)
    clean = codes.copy()
    clean[:, -1] &= np.uint8(0x0F)
    dirty = codes.copy()
    dirty[:, -1] |= np.uint8(0xF0)
    assert np.array_equal(gemv4(clean, scales, x, rows, cols, NQ4), gemv4(dirty, scales, x, rows, cols, NQ4))


@pytest.mark.parametrize("staging", [0, 1])
def test_gemv4_one_hot_decodes_exactly(oracle, staging):
    # x = e_k: y_r must be exactly fp32(scale_r * cb[field(r, k)]) for the normal-quantile codebook
    rows, cols = 257, 1536
    codes, scales, _ = rand_case4(rows, cols, seed=11)
    fields = oracle.unpack4(codes, rows, cols)
    s = scales.view(np.float16).astype(np.float64)
    for k in (0, 1, 2, 31, 32, 255, 256, 511, 777, 1535):
        x = np.zeros(cols, np.uint16)
        x[k] = 0x3C00
        y = gemv4(codes, scales, x, rows, cols, NQ4, staging=staging)
        expect = (s * NQ4[fields[:, k]].astype(np.float64)).astype(np.float32)
        assert np.array_equal(y, expect), k


@pytest.mark.parametrize("staging", [0, 1])
def test_gemv4_integer_bit_exact(oracle, staging):
    rows, cols = 300, 1536
    codes, _, _ = rand_case4(rows, cols, seed=12)
    scales = np.full(rows, 0x3C00, np.uint16)
    rng = np.random.default_rng(13)
    x = rng.integers(-3, 4, size=cols).astype(np.float16).view(np.uint16)
    y = gemv4(codes, scales, x, rows, cols, CB_INT, staging=staging)
    ref, _ = oracle.packed4_gemm(codes, scales, x, rows, cols, CB_INT)
    check_exact(y, ref[0], "integer 4-bit")


@pytest.mark.parametrize("staging", [0, 1])
def test_gemv4_zero_bound_rows_are_zero(oracle, staging):
    rows, cols = 130, 1536
    codes = np.full((rows, cols // 2), 0x77, np.uint8)    # every field 7: the codebook's 0
    scales = synth.uniform_f16_bits(14, (rows,), 0.005, 0.05)
    x = synth.normal_f16_bits(15, (cols,))
    assert np.all(gemv4(codes, scales, x, rows, cols, NQ4, staging=staging) == 0.0)


def test_gemv4_deterministic():
    c = synth.gemv_4bit_12288x1536(7)
    y1 = gemv4(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook, pdl=1, independent=1)
    y2 = gemv4(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook, blocks=3)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
