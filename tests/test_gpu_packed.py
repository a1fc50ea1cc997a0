"""GPU parity of the packed 2-bit GEMV and skinny GEMM (through the C ABI) against the oracle.

The 2-bit 12,288 x 1,536 GEMV is checked on every output of all 64 rotated
matrices; the ternary encoder block on every output of its first and last
layers and sampled outputs of the rest.  Field decoding is checked bit for bit
with one-hot activations and integer-valued activations.
"""
import numpy as np
import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import synth
from gpu_util import check_bound, check_exact, empty_f32, to_dev, to_host

pytestmark = pytest.mark.gpu

CB2 = synth.CODEBOOK_2BIT
CBT = synth.CODEBOOK_TERNARY
CB_ODD = np.array([0.3, -1.7, 2.5, 0.01], np.float32)   # not affine: select decode


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_packed_bit_gb300 import build
    build.build()
    mm.load_library()


def gemv(codes, scales, x, rows, cols, cb, **opts):
    dc, ds, dx = to_dev(codes), to_dev(scales), to_dev(x.reshape(-1))
    dy = empty_f32((rows,))
    if opts:
        mm.mm_gemv_packed2_ex(dc, ds, dx, dy, rows, cols, cb, **opts)
    else:
        mm.mm_gemv_packed2(dc, ds, dx, dy, rows, cols, cb)
    return to_host(dy)


def gemm_packed(codes, scales, X, M, rows, cols, cb, tile=None, splitk=0, **opts):
    dc, ds, dX = to_dev(codes), to_dev(scales), to_dev(X)
    dY = empty_f32((M, rows))
    if tile is None and not splitk and not opts:
        mm.mm_gemm_packed2(dc, ds, dX, dY, M, rows, cols, cb)
    else:
        mm.mm_gemm_packed2_ex(dc, ds, dX, dY, M, rows, cols, cb, tile=tile or 0, splitk=splitk, **opts)
    mm.mm_check_device_error()
    return to_host(dY)


def rand_case(rows, cols, M=1, seed=0, kind="uniform2"):
    rb = (cols + 3) // 4
    codes = (synth.random_bytes(seed, rows * rb) if kind == "uniform2"
             else synth.ternary_field_bytes(seed, rows * rb)).reshape(rows, rb)
    scales = synth.uniform_f16_bits(seed + 1, (rows,), 0.005, 0.05)
    X = synth.normal_f16_bits(seed + 2, (M, cols))
    return codes, scales, X


# ------------------------------------------------------------------ GEMV

def test_gemv_2bit_12288x1536_all_64_matrices(oracle):
    worst = 0.0
    for i in range(64):
        c = synth.gemv_2bit_12288x1536(i)
        y = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
        ref, T = oracle.packed_gemm(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
        worst = max(worst, check_bound(y, ref[0], T[0], c.name))
    print(f"64 matrices: worst |err|/T = {worst:.3e}")


VARIANTS = [dict(split=s, rows_per_lane=r, warps=w, dequant=d, pdl=p, weights_static=ws)
            for s in (4, 8, 16) for r in (1, 2, 4) for w in (2, 4, 8) for d in (1, 2)
            for (p, ws) in ((0, 0), (1, 1))]


MMA_VARIANTS = [dict(split=k, rows_per_lane=r, warps=k * m, dequant=3, pdl=p, weights_static=ws, independent=ind)
                for k in (1, 2, 3, 4, 6) for r in (1, 2, 4) for m in (1, 2) if k * m <= (8 if r >= 2 else 16)
                for (p, ws, ind) in ((0, 0, 0), (1, 1, 0), (1, 0, 1))]


@pytest.mark.parametrize("v", VARIANTS + MMA_VARIANTS,
                         ids=lambda v: "s{split}r{rows_per_lane}w{warps}d{dequant}p{pdl}".format(**v)
                         + ("i" if v.get("independent") else ""))
def test_gemv_variant_matrix(oracle, v):
    # ragged row count; 28 chunks = 7 slabs per row (not a multiple of the split widths)
    rows, cols = 1000, 1536 + 256
    codes, scales, x = rand_case(rows, cols, seed=101)
    y = gemv(codes, scales, x, rows, cols, CB2, **v)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_bound(y, ref[0], T[0], str(v))


@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 64), (7, 3), (33, 63), (129, 64), (65, 65), (300, 100),
                                       (17, 4097), (5, 40000), (2, 192)])
@pytest.mark.parametrize("cb", ["2bit", "odd"])
def test_gemv_edge_shapes(oracle, rows, cols, cb):
    codebook = CB2 if cb == "2bit" else CB_ODD
    codes, scales, x = rand_case(rows, cols, seed=rows * 131 + cols)
    y = gemv(codes, scales, x, rows, cols, codebook)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, codebook)
    check_bound(y, ref[0], T[0], f"{rows}x{cols}")


@pytest.mark.parametrize("cols", [5, 66, 1538])
def test_gemv_ignores_fields_past_cols(oracle, cols):
    rows = 40
    codes, scales, x = rand_case(rows, cols, seed=cols)
    dirty = codes.copy()
    dirty[:, -1] |= np.uint8((0xFF << (2 * (cols % 4))) & 0xFF)
    y_clean = gemv(codes, scales, x, rows, cols, CB2)
    y_dirty = gemv(dirty, scales, x, rows, cols, CB2)
    assert np.array_equal(y_clean, y_dirty)


@pytest.mark.parametrize("dequant", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("cols", [64, 256, 1536, 100])
def test_gemv_one_hot_decodes_exactly(oracle, dequant, cols):
    # x = e_k: every y_r must be exactly fp32(scale_r * cb[field(r, k)])
    rows = 257
    codes, scales, _ = rand_case(rows, cols, seed=5 + cols)
    fields = oracle.unpack2(codes, rows, cols)
    ks = sorted(set([0, 1, 15, 16, 31, cols - 1] + list(range(2, cols, max(1, cols // 37)))))
    for k in ks:
        if k >= cols:
            continue
        x = np.zeros(cols, np.uint16)
        x[k] = 0x3C00
        opts = dict(dequant=dequant) if cols % {3: 256, 4: 512, 5: 512}.get(dequant, 64) == 0 else {}
        y = gemv(codes, scales, x, rows, cols, CB2, **opts)
        ref, _ = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
        check_exact(y, ref[0], f"k={k}")
        s = scales.view(np.float16).astype(np.float64)
        assert np.array_equal(y.astype(np.float64), s * CB2[fields[:, k]].astype(np.float64))


@pytest.mark.parametrize("dequant", [1, 2, 3])
def test_gemv_integer_activations_bit_exact(oracle, dequant):
    rows, cols = 500, 1536
    codes, _, _ = rand_case(rows, cols, seed=77)
    scales = np.full(rows, 0x3C00, np.uint16)
    rng = np.random.default_rng(3)
    x = rng.integers(-3, 4, size=cols).astype(np.float16).view(np.uint16)
    y = gemv(codes, scales, x, rows, cols, CB2, dequant=dequant)
    ref, _ = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_exact(y, ref[0], "integer x")


@pytest.mark.parametrize("dequant", [1, 2, 3])
def test_gemv_tiny_activations_exact(oracle, dequant):
    # one-hot with fp16 subnormal and smallest-normal activations: products far below
    # 1 must still be exact
    rows, cols = 64, 256
    codes, scales, _ = rand_case(rows, cols, seed=91)
    for bits in (0x0001, 0x0003, 0x03FF, 0x0400, 0x8001):
        for k in (0, 9, 130, 255):
            x = np.zeros(cols, np.uint16)
            x[k] = bits
            y = gemv(codes, scales, x, rows, cols, CB2, dequant=dequant)
            ref, _ = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
            check_exact(y, ref[0], f"x[{k}]={bits:#06x}")


def test_gemv_deterministic():
    c = synth.gemv_2bit_12288x1536(3)
    y1 = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
    y2 = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_gemv_zero_bound_rows_are_zero(oracle):
    # rows of field 2 (entry 0) give T = 0, so y must be exactly 0
    rows, cols = 64, 1536
    codes = np.full((rows, cols // 4), 0xAA, np.uint8)
    scales = synth.uniform_f16_bits(9, (rows,), 0.005, 0.05)
    x = synth.normal_f16_bits(10, (cols,))
    for d in (1, 2, 3, 4, 5):
        y = gemv(codes, scales, x, rows, cols, CB2, dequant=d)
        assert np.all(y == 0.0), d
    # zero entry at field 1 or 0 cancels exactly too
    for cb, byte in ((np.array([-1, 0, 1, 2], np.float32), 0x55), (np.array([0, 0.5, 1, 1.5], np.float32), 0x00)):
        codes = np.full((rows, cols // 4), byte, np.uint8)
        for d in (1, 2, 3, 4, 5):
            y = gemv(codes, scales, x, rows, cols, cb, dequant=d)
            assert np.all(y == 0.0), (cb, d)


# ------------------------------------------------------------------ skinny GEMM

@pytest.mark.parametrize("M,rows,cols", [(1, 1, 1), (3, 17, 5), (65, 129, 64), (222, 130, 100),
                                         (7, 64, 768), (130, 33, 1537)])
@pytest.mark.parametrize("cb", ["ternary", "2bit", "odd"])
def test_gemm_packed_edge_shapes(oracle, M, rows, cols, cb):
    codebook = {"ternary": CBT, "2bit": CB2, "odd": CB_ODD}[cb]
    codes, scales, X = rand_case(rows, cols, M=M, seed=M * 1000 + rows + cols,
                                 kind="ternary" if cb == "ternary" else "uniform2")
    Y = gemm_packed(codes, scales, X, M, rows, cols, codebook)
    ref, T = oracle.packed_gemm(codes, scales, X, rows, cols, codebook)
    check_bound(Y, ref, T, f"{M}x{rows}x{cols}")


@pytest.mark.parametrize("layer", [0, 15])
@pytest.mark.parametrize("proj", ["up", "down"])
def test_ternary_encoder_full_layers(oracle, layer, proj):
    c = synth.ternary_encoder_layer(layer, proj)
    M = c.X.shape[0]
    Y = gemm_packed(c.codes, c.scales, c.X, M, c.rows, c.cols, c.codebook)
    ref, T = oracle.packed_gemm(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
    worst = check_bound(Y, ref, T, c.name)
    print(f"{c.name}: worst |err|/T = {worst:.3e}")


@pytest.mark.parametrize("proj", ["up", "down"])
def test_ternary_encoder_other_layers_sampled(oracle, proj):
    rng = np.random.default_rng(11)
    for layer in range(1, 15):
        c = synth.ternary_encoder_layer(layer, proj)
        M = c.X.shape[0]
        Y = gemm_packed(c.codes, c.scales, c.X, M, c.rows, c.cols, c.codebook)
        mm_i = rng.integers(0, M, 3000)
        rr_i = rng.integers(0, c.rows, 3000)
        ref, T = oracle.packed_gemm_at(c.codes, c.scales, c.X, c.cols, c.codebook, mm_i, rr_i)
        check_bound(Y[mm_i, rr_i], ref, T, c.name)


def test_gemm_packed_matches_gemv_rows(oracle):
    # M = 1 skinny GEMM and GEMV compute the same product
    c = synth.gemv_2bit_12288x1536(0)
    y = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
    Y = gemm_packed(c.codes, c.scales, c.X, 1, c.rows, c.cols, c.codebook)
    ref, T = oracle.packed_gemm(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
    check_bound(y, ref[0], T[0], "gemv")
    check_bound(Y[0], ref[0], T[0], "gemm M=1")


@pytest.mark.parametrize("tile", [1, 32, 64, 128])
@pytest.mark.parametrize("M,rows,cols", [(1, 1, 8), (3, 33, 24), (129, 130, 136), (222, 256, 768),
                                         (300, 65, 1536), (17, 3072, 64)])
@pytest.mark.parametrize("cb", ["ternary", "2bit"])
def test_gemm_packed_tile_matrix(oracle, tile, M, rows, cols, cb):
    # tensor-core tiles (32/64/128 W rows per CTA) and the FFMA kernel (tile 1); cols not a
    # multiple of 64 exercise the bytewise code loads and the zero-filled K tail
    codebook = CBT if cb == "ternary" else CB2
    codes, scales, X = rand_case(rows, cols, M=M, seed=7 * M + rows + 3 * cols,
                                 kind="ternary" if cb == "ternary" else "uniform2")
    Y = gemm_packed(codes, scales, X, M, rows, cols, codebook, tile=tile)
    ref, T = oracle.packed_gemm(codes, scales, X, rows, cols, codebook)
    check_bound(Y, ref, T, f"tile {tile} {M}x{rows}x{cols}")


@pytest.mark.parametrize("tile", [32, 128])
def test_gemm_packed_tensor_core_integer_exact(oracle, tile):
    # integer activations and scale 1: every partial sum is a small integer, so exact
    M, rows, cols = 150, 200, 512
    codes, _, _ = rand_case(rows, cols, M=M, seed=5)
    scales = np.full(rows, 0x3C00, np.uint16)
    rng = np.random.default_rng(8)
    X = rng.integers(-4, 5, size=(M, cols)).astype(np.float16).view(np.uint16)
    Y = gemm_packed(codes, scales, X, M, rows, cols, CB2, tile=tile)
    ref, _ = oracle.packed_gemm(codes, scales, X, rows, cols, CB2)
    check_exact(Y, ref, f"tile {tile}")


def test_gemm_packed_tensor_core_deterministic():
    c = synth.ternary_encoder_layer(2, "down")
    M = c.X.shape[0]
    y1 = gemm_packed(c.codes, c.scales, c.X, M, c.rows, c.cols, c.codebook)
    y2 = gemm_packed(c.codes, c.scales, c.X, M, c.rows, c.cols, c.codebook)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("splitk", [1, 2, 4, 8])
@pytest.mark.parametrize("tile", [32, 64, 128])
@pytest.mark.parametrize("M,rows,cols", [(222, 768, 3072), (5, 40, 640), (130, 200, 1000)])
def test_gemm_packed_cluster_splitk(oracle, splitk, tile, M, rows, cols):
    # K split over a cluster, partial tiles summed through distributed shared memory;
    # 1000 columns: 16 k-tiles of 64 with a ragged last one, uneven shares for 8 ranks
    codes, scales, X = rand_case(rows, cols, M=M, seed=splitk * 100 + tile + M, kind="ternary")
    Y = gemm_packed(codes, scales, X, M, rows, cols, CBT, tile=tile, splitk=splitk)
    ref, T = oracle.packed_gemm(codes, scales, X, rows, cols, CBT)
    check_bound(Y, ref, T, f"splitk {splitk} tile {tile}")


# ------------------------------------------------------------------ transposed shape (1,536 x 12,288)

@pytest.mark.parametrize("mode", [dict(), dict(pdl=1, independent=1), dict(pdl=1, weights_static=1),
                                  dict(dequant=2, staging=0, split=16, rows_per_lane=4, warps=8),
                                  dict(dequant=3, split=4, rows_per_lane=2, warps=4),
                                  dict(dequant=1, split=16, rows_per_lane=1, warps=4)])
def test_gemv_transposed_1536x12288(oracle, mode):
    # the pages' transposed kernel shape: few rows, 12,288 fields each; automatic and explicit
    # decodes, every output of two rotated matrices
    for i in (0, 63):
        c = synth.gemv_2bit_1536x12288(i)
        y = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook, **mode)
        ref, T = oracle.packed_gemm(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
        check_bound(y, ref[0], T[0], f"{c.name} {mode}")


# ------------------------------------------------------------------ tile 2: W rows as the MMA's M

TILE2_SHAPES = [(1, 1, 64), (3, 33, 64), (129, 130, 192), (222, 256, 768), (300, 65, 1536), (17, 3072, 64),
                (222, 3072, 768), (222, 768, 3072), (257, 200, 640), (512, 100, 128)]


@pytest.mark.parametrize("M,rows,cols", TILE2_SHAPES)
@pytest.mark.parametrize("cb", ["ternary", "2bit"])
def test_gemm_packed_tile2_auto_split(oracle, M, rows, cols, cb):
    # ragged feature tiles (rows not a multiple of 128), ragged and multiple token tiles
    # (M > 256), the automatic split of K over a cluster
    codebook = CBT if cb == "ternary" else CB2
    codes, scales, X = rand_case(rows, cols, M=M, seed=11 * M + rows + 5 * cols,
                                 kind="ternary" if cb == "ternary" else "uniform2")
    Y = gemm_packed(codes, scales, X, M, rows, cols, codebook, tile=2)
    ref, T = oracle.packed_gemm(codes, scales, X, rows, cols, codebook)
    check_bound(Y, ref, T, f"tile 2 {M}x{rows}x{cols}")


@pytest.mark.parametrize("splitk", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("M,rows,cols", [(222, 300, 512), (40, 128, 1024), (222, 768, 3072), (5, 17, 1600)])
def test_gemm_packed_tile2_cluster_splitk(oracle, splitk, M, rows, cols):
    # every cluster size; 1600 columns: 25 atoms, uneven shares; shares of more than
    # 8 atoms are refused
    atoms = cols // 64
    if splitk > atoms or -(-atoms // splitk) > 8 or (M > 128 and -(-atoms // splitk) > 4):
        pytest.skip("share does not fit one CTA")
    codes, scales, X = rand_case(rows, cols, M=M, seed=splitk * 31 + M + rows, kind="ternary")
    Y = gemm_packed(codes, scales, X, M, rows, cols, CBT, tile=2, splitk=splitk)
    ref, T = oracle.packed_gemm(codes, scales, X, rows, cols, CBT)
    check_bound(Y, ref, T, f"tile 2 splitk {splitk} {M}x{rows}x{cols}")


@pytest.mark.parametrize("splitk", [2, 4])
def test_gemm_packed_tile2_integer_exact(oracle, splitk):
    # integer activations, scale 1, integer codebook: exact in any summation order
    M, rows, cols = 150, 200, 512
    codes, _, _ = rand_case(rows, cols, M=M, seed=5)
    scales = np.full(rows, 0x3C00, np.uint16)
    rng = np.random.default_rng(8)
    X = rng.integers(-4, 5, size=(M, cols)).astype(np.float16).view(np.uint16)
    Y = gemm_packed(codes, scales, X, M, rows, cols, CB2, tile=2, splitk=splitk)
    ref, _ = oracle.packed_gemm(codes, scales, X, rows, cols, CB2)
    check_exact(Y, ref, f"tile 2 splitk {splitk}")


def test_gemm_packed_tile2_deterministic():
    c = synth.ternary_encoder_layer(3, "down")
    M = c.X.shape[0]
    y1 = gemm_packed(c.codes, c.scales, c.X, M, c.rows, c.cols, c.codebook, tile=2)
    y2 = gemm_packed(c.codes, c.scales, c.X, M, c.rows, c.cols, c.codebook, tile=2)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


# ------------------------------------------------------------------ tile 3: decoded weights in TMEM

CB_ODD16 = np.array([0.375, -1.75, 2.5, 0.0078125], np.float32)  # four distinct fp16-exact entries


@pytest.mark.parametrize("M,rows,cols", TILE2_SHAPES)
@pytest.mark.parametrize("cb", ["ternary", "2bit", "odd16"])
def test_gemm_packed_tile3_auto(oracle, M, rows, cols, cb):
    # the automatic token tile and split; every code value decoded through prmt (odd16:
    # four distinct entries, so a swapped field or a wrong byte of an entry shows)
    codebook = {"ternary": CBT, "2bit": CB2, "odd16": CB_ODD16}[cb]
    codes, scales, X = rand_case(rows, cols, M=M, seed=13 * M + rows + 7 * cols,
                                 kind="ternary" if cb == "ternary" else "uniform2")
    Y = gemm_packed(codes, scales, X, M, rows, cols, codebook, tile=3)
    ref, T = oracle.packed_gemm(codes, scales, X, rows, cols, codebook)
    check_bound(Y, ref, T, f"tile 3 {M}x{rows}x{cols} {cb}")


@pytest.mark.parametrize("ntok", [16, 48, 64, 112, 224, 256])
@pytest.mark.parametrize("splitk", [1, 2, 4, 8])
@pytest.mark.parametrize("M,rows,cols", [(222, 300, 1024), (5, 17, 1600), (130, 129, 640)])
def test_gemm_packed_tile3_token_tiles_and_splits(oracle, ntok, splitk, M, rows, cols):
    # explicit token tiles (one, several, a ragged last one) and cluster sizes; 1600
    # columns: 25 atoms, uneven shares; 640: 10 atoms, a ring shallower than 8 for 8 ranks
    if splitk > cols // 64:
        pytest.skip("more ranks than atoms")
    codes, scales, X = rand_case(rows, cols, M=M, seed=ntok + 17 * splitk + M, kind="uniform2")
    Y = gemm_packed(codes, scales, X, M, rows, cols, CB_ODD16, tile=3, splitk=splitk, ntok=ntok)
    ref, T = oracle.packed_gemm(codes, scales, X, rows, cols, CB_ODD16)
    check_bound(Y, ref, T, f"tile 3 ntok {ntok} splitk {splitk} {M}x{rows}x{cols}")


@pytest.mark.parametrize("splitk", [1, 4])
def test_gemm_packed_tile3_integer_exact(oracle, splitk):
    # integer activations, scale 1, integer codebook: exact in any summation order
    M, rows, cols = 150, 200, 512
    codes, _, _ = rand_case(rows, cols, M=M, seed=6)
    scales = np.full(rows, 0x3C00, np.uint16)
    rng = np.random.default_rng(9)
    X = rng.integers(-4, 5, size=(M, cols)).astype(np.float16).view(np.uint16)
    Y = gemm_packed(codes, scales, X, M, rows, cols, CB2, tile=3, splitk=splitk)
    ref, _ = oracle.packed_gemm(codes, scales, X, rows, cols, CB2)
    check_exact(Y, ref, f"tile 3 splitk {splitk}")


def test_gemm_packed_tile3_one_hot_decode_exact(oracle):
    # X one-hot in K: Y[t][r] = scale_r cb[field(r, k_t)] exactly, every field of every
    # row position of the atom, all four codes, through every lane of the tensor memory
    M, rows, cols = 64, 256, 64
    codes, scales, _ = rand_case(rows, cols, M=1, seed=77)
    X = np.zeros((M, cols), np.float16)
    X[np.arange(M), np.arange(M) % cols] = 1.0
    X = X.view(np.uint16)
    Y = gemm_packed(codes, scales, X, M, rows, cols, CB_ODD16, tile=3, ntok=64)
    ref, _ = oracle.packed_gemm(codes, scales, X, rows, cols, CB_ODD16)
    check_exact(Y, ref.astype(np.float32).astype(np.float64), "tile 3 one-hot")


def test_gemm_packed_tile3_deterministic():
    c = synth.ternary_encoder_layer(5, "down")
    M = c.X.shape[0]
    y1 = gemm_packed(c.codes, c.scales, c.X, M, c.rows, c.cols, c.codebook, tile=3)
    y2 = gemm_packed(c.codes, c.scales, c.X, M, c.rows, c.cols, c.codebook, tile=3)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("tile", [2, 3])
@pytest.mark.parametrize("weights_static", [0, 1])
def test_gemm_packed_tile2_pdl_waits_before_writing_and_reading(oracle, weights_static, tile):
    # Back-to-back calls with programmatic dependent launch on one stream.
    # Call 2 writes its Y over the bytes of call 1's X (write after read), and call 3
    # reads as X the bytes call 2 wrote (read after write).  Integer activations, an
    # integer codebook and scale 1 make every Y an integer below 2^11, whose fp32 bits
    # read as two finite fp16 values, so the oracle can follow the chain exactly.
    import torch
    M, rows, cols = 222, 768, 1024
    rng = np.random.default_rng(21)
    cb = CB2
    ones = np.full(rows, 0x3C00, np.uint16)
    codes = [rand_case(rows, cols, M=1, seed=40 + i)[0] for i in range(3)]
    X1 = rng.integers(-2, 3, size=(M, cols)).astype(np.float16).view(np.uint16)
    X2 = rng.integers(-2, 3, size=(M, cols)).astype(np.float16).view(np.uint16)
    dev = torch.device("cuda:0")
    buf = torch.zeros(M * rows * 4, dtype=torch.uint8, device=dev)   # holds X1, then Y2, read as X3
    buf[: X1.nbytes].copy_(torch.from_numpy(X1.view(np.uint8).reshape(-1)))
    dX1 = buf[: X1.nbytes].view(torch.int16).view(M, cols)
    dY2 = buf.view(torch.float32).view(M, rows)
    dX3 = buf.view(torch.int16).view(M, 2 * rows)                     # cols of call 3 = 2 * rows
    codes3 = rand_case(rows, 2 * rows, M=1, seed=43)[0]
    dc = [to_dev(codes[0]), to_dev(codes[1]), to_dev(codes3)]
    ds = to_dev(ones)
    dX2 = to_dev(X2)
    dY1 = empty_f32((M, rows))
    dY3 = empty_f32((M, rows))
    opts = dict(tile=tile, pdl=1, weights_static=weights_static)
    for _ in range(3):
        buf[: X1.nbytes].copy_(torch.from_numpy(X1.view(np.uint8).reshape(-1)))
        mm.mm_gemm_packed2_ex(dc[0], ds, dX1, dY1, M, rows, cols, cb, **opts)
        mm.mm_gemm_packed2_ex(dc[1], ds, dX2, dY2, M, rows, cols, cb, **opts)
        mm.mm_gemm_packed2_ex(dc[2], ds, dX3, dY3, M, rows, 2 * rows, cb, **opts)
        mm.mm_check_device_error()
        ref1, _ = oracle.packed_gemm(codes[0], ones, X1, rows, cols, cb)
        ref2, _ = oracle.packed_gemm(codes[1], ones, X2, rows, cols, cb)
        check_exact(to_host(dY1), ref1, "call 1 read X1 before call 2 overwrote it")
        check_exact(to_host(dY2), ref2, "call 2")
        X3 = ref2.astype(np.float32).view(np.uint16).reshape(M, 2 * rows)
        assert np.all(np.isfinite(X3.view(np.float16)))
        ref3, T3 = oracle.packed_gemm(codes3, ones, X3, rows, 2 * rows, cb)
        check_bound(to_host(dY3), ref3, T3, "call 3 read call 2's Y")


@pytest.mark.parametrize("rows", [1, 63, 64, 65, 1000, 1100])
@pytest.mark.parametrize("cols", [512, 1024, 1536, 4096])
@pytest.mark.parametrize("mode", [dict(pdl=0), dict(pdl=1, weights_static=1), dict(pdl=1, independent=1)],
                         ids=["serial", "chained", "independent"])
@pytest.mark.parametrize("blocks", [0, 1, 3, 8])
@pytest.mark.parametrize("dequant", [2, 3])
def test_gemv_tma_staging(oracle, rows, cols, mode, blocks, dequant):
    # code rows streamed through a TMA ring (blocks per CTA: 0 = automatic): 64-row blocks and one
    # warp per 256-field slab (tensor-core decode), or 128-row blocks and one lane per row (SIMT
    # affine decode); ragged row counts leave partial last CTAs and blocks
    codes, scales, x = rand_case(rows, cols, seed=rows * 7 + cols)
    y = gemv(codes, scales, x, rows, cols, CB2, dequant=dequant, staging=1, rows_per_lane=blocks, **mode)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_bound(y, ref[0], T[0], f"{rows}x{cols} {mode}")


@pytest.mark.parametrize("dequant", [2, 3])
def test_gemv_tma_staging_exactness(oracle, dequant):
    rows, cols = 130, 1536
    codes, scales, _ = rand_case(rows, cols, seed=4)
    fields = oracle.unpack2(codes, rows, cols)
    s = scales.view(np.float16).astype(np.float64)
    for k in (0, 7, 8, 255, 256, 777, 1535):
        for bits in (0x3C00, 0x0001, 0xC400):
            x = np.zeros(cols, np.uint16)
            x[k] = bits
            y = gemv(codes, scales, x, rows, cols, CB2, dequant=dequant, staging=1)
            xv = float(np.array([bits], np.uint16).view(np.float16)[0])
            assert np.array_equal(y.astype(np.float64), s * CB2[fields[:, k]].astype(np.float64) * xv), (k, bits)
    zero = np.full((rows, cols // 4), 0xAA, np.uint8)
    xn = synth.normal_f16_bits(12, (cols,))
    assert np.all(gemv(zero, scales, xn, rows, cols, CB2, dequant=dequant, staging=1) == 0.0)
    for cb, byte in ((np.array([-1, 0, 1, 2], np.float32), 0x55), (np.array([0, 0.5, 1, 1.5], np.float32), 0x00)):
        zr = np.full((rows, cols // 4), byte, np.uint8)
        assert np.all(gemv(zr, scales, xn, rows, cols, cb, dequant=dequant, staging=1) == 0.0)


# ------------------------------------------------------------------ fp8 tensor-core decode

FP8_MODES = [dict(pdl=0), dict(pdl=1, weights_static=1), dict(pdl=1, independent=1)]


@pytest.mark.parametrize("rows", [1, 63, 64, 65, 1000, 1100])
@pytest.mark.parametrize("cols", [512, 1024, 1536, 4096])
@pytest.mark.parametrize("mode", FP8_MODES, ids=["serial", "chained", "independent"])
@pytest.mark.parametrize("blocks", [0, 1, 3, 8])
def test_gemv_fp8(oracle, rows, cols, mode, blocks):
    # codes as e4m3 operands, x as exact e5m2 pieces, mma.sync m16n8k32; 64-row blocks
    # through the TMA ring (0 = automatic count), ragged last CTAs and blocks
    codes, scales, x = rand_case(rows, cols, seed=rows * 11 + cols)
    y = gemv(codes, scales, x, rows, cols, CB2, dequant=4, rows_per_lane=blocks, **mode)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_bound(y, ref[0], T[0], f"{rows}x{cols} {mode} blocks {blocks}")


@pytest.mark.parametrize("rows", [1, 126, 127, 128, 254, 255, 1000, 1100])
@pytest.mark.parametrize("cols", [512, 1024, 1536, 4096, 8192])
@pytest.mark.parametrize("mode", FP8_MODES, ids=["serial", "chained", "independent"])
@pytest.mark.parametrize("tiles", [0, 1, 2, 5])
def test_gemv_tcgen05(oracle, rows, cols, mode, tiles):
    # e4m3 code bytes in tensor memory x e5m2 pieces of x, tcgen05.mma; 127-row tiles
    # (the 128th lane forms sum x), several tiles per CTA, ragged last tiles
    codes, scales, x = rand_case(rows, cols, seed=rows * 13 + cols)
    y = gemv(codes, scales, x, rows, cols, CB2, dequant=5, rows_per_lane=tiles, **mode)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_bound(y, ref[0], T[0], f"{rows}x{cols} {mode} tiles {tiles}")


@pytest.mark.parametrize("rows", [1, 126, 127, 128, 254, 255, 1000, 1100])
@pytest.mark.parametrize("cols", [512, 1024, 1536, 2048, 4096, 8192, 12288, 12800])
@pytest.mark.parametrize("mode", FP8_MODES, ids=["serial", "chained", "independent"])
@pytest.mark.parametrize("tiles", [0, 1, 2, 5])
def test_gemv_mxf4(oracle, rows, cols, mode, tiles):
    # packed e2m1 codes in tensor memory x 14 exact e2m1 digit pieces of x, tcgen05.mma
    # kind::mxf4; 127-row tiles (the 128th lane forms the digit sums), several tiles per CTA,
    # ragged last tiles
    codes, scales, x = rand_case(rows, cols, seed=rows * 17 + cols)
    y = gemv(codes, scales, x, rows, cols, CB2, dequant=6, rows_per_lane=tiles, **mode)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_bound(y, ref[0], T[0], f"{rows}x{cols} {mode} tiles {tiles}")


def test_gemv_mxf4_full_rotation_every_output(oracle):
    # all 64 matrices of the 12,288 x 1,536 rotation, independent calls, every output
    import torch
    dev = torch.device("cuda:0")
    for i in range(64):
        c = synth.gemv_2bit_12288x1536(i)
        y = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook, dequant=6, pdl=1, independent=1)
        ref, T = oracle.packed_gemm(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
        check_bound(y, ref[0], T[0], f"matrix {i}")


def test_gemv_mxf4_transposed_rotation_every_output(oracle):
    # the transposed shape (1,536 rows x 12,288 fields: 13 tiles of 127 rows, 48 stages each) on
    # the fp4 decode, 8 of its 64 matrices as independent calls, every output
    for i in range(0, 64, 8):
        c = synth.gemv_2bit_1536x12288(i)
        y = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook, dequant=6, rows_per_lane=5, pdl=1, independent=1)
        ref, T = oracle.packed_gemm(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook)
        check_bound(y, ref[0], T[0], f"transposed matrix {i}")


def test_gemv_mxf4_refuses_columns_past_the_shared_memory_plan():
    import torch
    rows, cols = 8, 13312
    codes, scales, x = rand_case(rows, cols, seed=3)
    with pytest.raises(mm.MMError, match="cols <= 12800"):
        gemv(codes, scales, x, rows, cols, CB2, dequant=6)


@pytest.mark.parametrize("cb", [CB2, np.array([-1, 0, 1, 2], np.float32), np.array([0, 0.5, 1, 1.5], np.float32),
                                np.array([3, 1, -1, -3], np.float32)])
def test_gemv_mxf4_other_affine_codebooks(oracle, cb):
    rows, cols = 1000, 2048
    codes, scales, x = rand_case(rows, cols, seed=88)
    y = gemv(codes, scales, x, rows, cols, cb, dequant=6)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, cb)
    check_bound(y, ref[0], T[0], f"codebook {cb.tolist()}")


def test_gemv_mxf4_extreme_activations(oracle):
    # the largest finite fp16 and the smallest subnormals in one vector, both signs, every
    # digit position of the split: the result still meets the bound
    rows, cols = 300, 1536
    codes, scales, _ = rand_case(rows, cols, seed=91)
    rng = np.random.default_rng(91)
    pool = np.array([0x7BFF, 0xFBFF, 0x0001, 0x8001, 0x03FF, 0x0400, 0x3C00, 0x7800, 0x5555, 0x2AAA], np.uint16)
    x = pool[rng.integers(0, len(pool), cols)]
    y = gemv(codes, scales, x, rows, cols, CB2, dequant=6)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_bound(y, ref[0], T[0], "extremes")


def test_gemv_mxf4_non_finite_x_gives_nan():
    rows, cols = 300, 1024
    codes, scales, x = rand_case(rows, cols, seed=92)
    for bad in (0x7C00, 0xFC00, 0x7E00):
        xb = x.copy()
        xb[0, 517] = bad
        y = gemv(codes, scales, xb, rows, cols, CB2, dequant=6)
        assert np.all(np.isnan(y)), hex(bad)


def test_gemv_mxf4_options_refused():
    rows, cols = 256, 1024
    codes, scales, x = rand_case(rows, cols, seed=93)
    for opts in (dict(split=4), dict(warps=4), dict(staging=1), dict(rows_per_lane=65)):
        with pytest.raises(mm.MMError):
            gemv(codes, scales, x, rows, cols, CB2, dequant=6, **opts)
    with pytest.raises(mm.MMError):  # cols not a multiple of 512
        c2, s2, x2 = rand_case(rows, 768, seed=94)
        gemv(c2, s2, x2, rows, 768, CB2, dequant=6)
    with pytest.raises(mm.MMError):  # not affine
        gemv(codes, scales, x, rows, cols, CB_ODD, dequant=6)


def _fp16_values(bits):
    return np.array(bits, np.uint16).view(np.float16).astype(np.float64)


@pytest.mark.parametrize("dequant", [4, 5, 6])
def test_gemv_fp8_one_hot_every_window(oracle, dequant):
    # x = v e_k for values on both sides of the 2^-6 window boundary, subnormals, the
    # largest finite fp16 and negative values: y_r must be exactly fp32(scale_r * cb * v)
    rows, cols = 130, 1536
    codes, scales, _ = rand_case(rows, cols, seed=14)
    fields = oracle.unpack2(codes, rows, cols)
    s = scales.view(np.float16).astype(np.float64)
    values = [0x3C00, 0x2400, 0x23FF, 0x0001, 0x0155, 0x03FF, 0x0400, 0x7BFF, 0xFBFF, 0x8001, 0xC4D3, 0x1234]
    for k in (0, 1, 2, 3, 4, 15, 16, 63, 64, 255, 256, 511, 777, 1535):
        for bits in values:
            x = np.zeros(cols, np.uint16)
            x[k] = bits
            y = gemv(codes, scales, x, rows, cols, CB2, dequant=dequant)
            expect = (s * CB2[fields[:, k]].astype(np.float64) * _fp16_values([bits])[0]).astype(np.float32)
            assert np.array_equal(y, expect), (k, hex(bits))


@pytest.mark.parametrize("dequant", [4, 5, 6])
def test_gemv_fp8_integer_activations_bit_exact(oracle, dequant):
    rows, cols = 500, 1536
    codes, _, _ = rand_case(rows, cols, seed=78)
    scales = np.full(rows, 0x3C00, np.uint16)
    rng = np.random.default_rng(4)
    x = rng.integers(-3, 4, size=cols).astype(np.float16).view(np.uint16)
    y = gemv(codes, scales, x, rows, cols, CB2, dequant=dequant)
    ref, _ = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_exact(y, ref[0], "integer x")


@pytest.mark.parametrize("dequant", [4, 5, 6])
def test_gemv_fp8_wide_dynamic_range(oracle, dequant):
    # activations spread over every fp16 binade, subnormals included, both signs
    rows, cols = 257, 2048
    codes, scales, _ = rand_case(rows, cols, seed=21)
    rng = np.random.default_rng(21)
    x = rng.integers(0, 0x7C00, size=cols).astype(np.uint16) | (rng.integers(0, 2, size=cols) << 15).astype(np.uint16)
    y = gemv(codes, scales, x, rows, cols, CB2, dequant=dequant)
    ref, T = oracle.packed_gemm(codes, scales, x, rows, cols, CB2)
    check_bound(y, ref[0], T[0], "wide range")


@pytest.mark.parametrize("cb,zero_code", [(CB2, 2), (np.array([-1, 0, 1, 2], np.float32), 1),
                                          (np.array([0, 0.5, 1, 1.5], np.float32), 0)])
@pytest.mark.parametrize("dequant", [4, 5, 6])
def test_gemv_fp8_zero_rows_at_every_position(oracle, cb, zero_code, dequant):
    # rows whose fields all hold the zero entry sit at every position of the 16-row MMA
    # blocks, between random rows: their outputs must be exactly 0
    rows, cols = 200, 1536
    codes, scales, x = rand_case(rows, cols, seed=30 + zero_code)
    zero_rows = [r for r in range(rows) if r % 3 == 0]
    codes[zero_rows, :] = np.uint8(zero_code * 0x55)
    for x_ in (x, synth.normal_f16_bits(31, (cols,))):
        y = gemv(codes, scales, x_, rows, cols, cb, dequant=dequant)
        assert np.all(y[zero_rows] == 0.0)
        ref, T = oracle.packed_gemm(codes, scales, x_, rows, cols, cb)
        check_bound(y, ref[0], T[0], "zero rows")


@pytest.mark.parametrize("dequant", [4, 5, 6])
def test_gemv_fp8_deterministic(dequant):
    c = synth.gemv_2bit_12288x1536(5)
    y1 = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook, dequant=dequant, pdl=1, independent=1)
    y2 = gemv(c.codes, c.scales, c.X, c.rows, c.cols, c.codebook, dequant=dequant, rows_per_lane=3)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
