"""GPU parity of the dense fp32 GEMM (through the C ABI) against the fp64 oracle.

Sizes span several 128 x 128 tiles with ragged tails in every dimension; the
GPT-2 MLP up-projection (64 x 768 x 3072) and the square 2048^3 layouts are
checked on every output; the training-shape set (8192 / 2048 / 8192) on whole
sampled rows and columns plus random outputs.
"""
import numpy as np
import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import synth
from gpu_util import check_bound, check_exact, empty_f32, to_dev, to_host

pytestmark = pytest.mark.gpu

LAYOUTS = {"nn": (0, 0), "nt": (0, 1), "tn": (1, 0), "tt": (1, 1)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_packed_bit_gb300 import build
    build.build()
    mm.load_library()


def run(tA, tB, M, N, K, A, B, lda=None, ldb=None, ldc=None, path=mm.MM_GEMM_AUTO, tile=0):
    if isinstance(path, tuple):
        path, tile = path
    lda = lda or A.shape[1]
    ldb = ldb or B.shape[1]
    ldc = ldc or N
    dA, dB = to_dev(A), to_dev(B)
    dC = empty_f32((M, ldc))
    mm.mm_gemm_f32_ex(tA, tB, M, N, K, dA, lda, dB, ldb, dC, ldc, path=path, tile=tile)
    mm.mm_check_device_error()
    return to_host(dC)


def stored(tA, tB, M, N, K, seed, kind="normal"):
    a_shape = (K, M) if tA else (M, K)
    b_shape = (N, K) if tB else (K, N)
    if kind == "int":
        rng = np.random.default_rng(seed)
        return (rng.integers(-6, 7, size=a_shape).astype(np.float32),
                rng.integers(-6, 7, size=b_shape).astype(np.float32))
    return synth.normal_f32(seed, a_shape, 1.0), synth.normal_f32(seed + 1, b_shape, 1.0)


SHAPES = [(1, 1, 1), (3, 17, 5), (65, 129, 33), (127, 63, 129), (200, 300, 97), (257, 130, 1000)]


# (path, tile): the 3xTF32 path has two kernels, the persistent warp-specialised one
# (tile 2, the automatic choice) and the two-stage one (tile 1)
PATHS = {"auto": (mm.MM_GEMM_AUTO, 0), "ffma": (mm.MM_GEMM_FFMA, 0), "tf32x3": (mm.MM_GEMM_TF32X3, 2),
         "tf32x3_2stage": (mm.MM_GEMM_TF32X3, 1), "tf32x3_pair": (mm.MM_GEMM_TF32X3, 3)}
TC_PATHS = ("tf32x3", "tf32x3_2stage", "tf32x3_pair")


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", SHAPES)
def test_gemm_ragged_shapes(oracle, layout, shape, path):
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = stored(tA, tB, M, N, K, seed=1000 * list(LAYOUTS).index(layout) + 7 * M + 3 * N + K)
    if path in TC_PATHS and (A.shape[1] % 4 or B.shape[1] % 4):
        pytest.skip("3xTF32 path needs leading dimensions that are multiples of 4")
    C = run(tA, tB, M, N, K, A, B, path=PATHS[path])
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    check_bound(C, ref, T, f"{layout} {shape} {path}")


@pytest.mark.parametrize("tile", [1, 2, 3])
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", [(5, 7, 3), (128, 128, 32), (128, 256, 16), (256, 384, 64), (130, 260, 100),
                                   (384, 128, 1000), (64, 3072, 768), (2000, 2900, 72), (19456, 256, 24)])
def test_gemm_tf32x3_tiles(oracle, layout, shape, tile):
    # 19456 x 256: 76 pair tiles, every pair of the GPU busy at once
    # whole tiles, ragged tiles and K tails on the tensor-core path
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = stored(tA, tB, M, N, K, seed=17 + M + N + K)
    Ap = np.zeros((A.shape[0], (A.shape[1] + 3) // 4 * 4), np.float32); Ap[:, :A.shape[1]] = A
    Bp = np.zeros((B.shape[0], (B.shape[1] + 3) // 4 * 4), np.float32); Bp[:, :B.shape[1]] = B
    C = run(tA, tB, M, N, K, Ap, Bp, lda=Ap.shape[1], ldb=Bp.shape[1], path=mm.MM_GEMM_TF32X3, tile=tile)
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    worst = check_bound(C, ref, T, f"{layout} {shape} tile {tile}")
    print(f"tf32x3 tile {tile} {layout} {shape}: worst |err|/T = {worst:.3e}")


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_gemm_unaligned_leading_dims_use_general_path(oracle, layout):
    # leading dimensions that are not a multiple of 4 floats cannot be described by TMA
    tA, tB = LAYOUTS[layout]
    M, N, K = 70, 45, 83
    A, B = stored(tA, tB, M, N, K, seed=17)
    Ap = np.zeros((A.shape[0], A.shape[1] + 3), np.float32); Ap[:, :A.shape[1]] = A
    Bp = np.zeros((B.shape[0], B.shape[1] + 1), np.float32); Bp[:, :B.shape[1]] = B
    C = run(tA, tB, M, N, K, Ap, Bp, lda=Ap.shape[1], ldb=Bp.shape[1], ldc=N + 5)
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    check_bound(C[:, :N], ref, T, layout)
    assert np.all(np.isnan(C[:, N:])), "columns past N were written"


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_gemm_padded_ld_tma_path_and_canary(oracle, layout):
    tA, tB = LAYOUTS[layout]
    M, N, K = 150, 260, 70
    A, B = stored(tA, tB, M, N, K, seed=23)
    lda = (A.shape[1] + 3) // 4 * 4 + 4   # multiples of 4 floats: the TMA path applies
    ldb = (B.shape[1] + 3) // 4 * 4 + 8
    Ap = np.full((A.shape[0], lda), 7.0, np.float32); Ap[:, :A.shape[1]] = A
    Bp = np.full((B.shape[0], ldb), -5.0, np.float32); Bp[:, :B.shape[1]] = B
    C = run(tA, tB, M, N, K, Ap, Bp, lda=Ap.shape[1], ldb=Bp.shape[1], ldc=N + 12)
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    check_bound(C[:, :N], ref, T, layout)
    assert np.all(np.isnan(C[:, N:])), "columns past N were written"


@pytest.mark.parametrize("layout", ["nn", "nt", "tn"])
def test_gemm_small_integers_bit_exact(oracle, layout):
    # every partial sum is an integer below 2^24, so any summation order is exact
    tA, tB = LAYOUTS[layout]
    M, N, K = 300, 272, 516
    A, B = stored(tA, tB, M, N, K, seed=31, kind="int")
    ref, _ = oracle.gemm(tA, tB, M, N, K, A, B)
    for path in PATHS.values():
        if path[0] == mm.MM_GEMM_TF32X3 and (A.shape[1] % 4 or B.shape[1] % 4):
            continue
        check_exact(run(tA, tB, M, N, K, A, B, path=path), ref, f"{layout} path {path}")


def test_gemm_all_ones_is_K():
    M, N, K = 129, 257, 1000
    C = run(0, 0, M, N, K, np.ones((M, K), np.float32), np.ones((K, N), np.float32))
    assert np.all(C == K)


@pytest.mark.parametrize("path", ["ffma", "tf32x3", "tf32x3_2stage", "tf32x3_pair"])
@pytest.mark.parametrize("layout", ["nn", "nt", "tn"])
def test_gemm_deterministic(layout, path):
    tA, tB = LAYOUTS[layout]
    M, N, K = 332, 444, 556
    A, B = stored(tA, tB, M, N, K, seed=41)
    c1 = run(tA, tB, M, N, K, A, B, path=PATHS[path])
    c2 = run(tA, tB, M, N, K, A, B, path=PATHS[path])
    assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))


@pytest.mark.parametrize("tile", [1, 2, 3])
def test_gemm_tf32x3_all_ones_and_identity(tile):
    M = N = K = 256
    C = run(0, 0, M, N, K, np.ones((M, K), np.float32), np.ones((K, N), np.float32), path=mm.MM_GEMM_TF32X3,
            tile=tile)
    assert np.all(C == K)
    X = synth.normal_f32(3, (M, K), 1.0)
    C = run(0, 0, M, N, K, X, np.eye(K, dtype=np.float32), path=mm.MM_GEMM_TF32X3, tile=tile)
    # x = hi + lo with lo's tf32 rounding dropped: relative error below 2^-21
    assert np.all(np.abs(C - X) <= 2.0 ** -20 * np.abs(X))


def test_gpt2_mlp_up_64x768x3072_all_outputs(oracle):
    c = synth.gpt2_mlp_up_64x768x3072()
    C = run(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B)
    ref, T = oracle.gemm(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B)
    check_bound(C, ref, T, c.name)


@pytest.mark.parametrize("path", ["ffma", "tf32x3", "tf32x3_2stage", "tf32x3_pair"])
@pytest.mark.parametrize("layout", ["nn", "nt", "tn"])
def test_square_2048_all_outputs(oracle, layout, path):
    c = synth.square_2048(layout)
    C = run(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B, path=PATHS[path])
    ref, T = oracle.gemm(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B)
    worst = check_bound(C, ref, T, c.name)
    print(f"{c.name} {path}: worst |err|/T = {worst:.3e}")


@pytest.mark.parametrize("path", ["ffma", "tf32x3", "tf32x3_pair"])
@pytest.mark.parametrize("which", ["fwd", "dA", "dB"])
def test_training_set_sampled(oracle, which, path):
    c = synth.training_set_8192(which)
    C = run(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B, path=PATHS[path])
    rng = np.random.default_rng(7)
    rows = [0, c.M - 1, int(rng.integers(c.M))]
    cols = [0, c.N - 1, int(rng.integers(c.N))]
    ii = np.concatenate([np.repeat(rows, c.N), np.tile(np.arange(c.M), len(cols)), rng.integers(0, c.M, 4000)])
    jj = np.concatenate([np.tile(np.arange(c.N), len(rows)), np.repeat(cols, c.M), rng.integers(0, c.N, 4000)])
    ref, T = oracle.gemm_at(c.transA, c.transB, c.K, c.A, c.B, ii, jj)
    worst = check_bound(C[ii, jj], ref, T, c.name)
    print(f"{c.name}: {len(ii)} outputs, worst |err|/T = {worst:.3e}")


# ------------------------------------------------------------------ split-K with a workspace

def run_splitk(tA, tB, M, N, K, A, B, splitk, lda=None, ldb=None, ldc=None, fill=float("nan")):
    import torch
    lda = lda or A.shape[1]
    ldb = ldb or B.shape[1]
    ldc = ldc or N
    dA, dB = to_dev(A), to_dev(B)
    dC = empty_f32((M, ldc))
    n = mm.mm_gemm_f32_splitk_workspace(M, N, K, splitk)
    ws = torch.full((max(n, 1),), fill, dtype=torch.float32, device=dA.device)  # contents must not matter
    mm.mm_gemm_f32_splitk(tA, tB, M, N, K, dA, lda, dB, ldb, dC, ldc, splitk, ws if n else None, n)
    mm.mm_check_device_error()
    return to_host(dC)


def test_gpt2_mlp_up_splitk_auto_all_outputs(oracle):
    # 64 x 768 x 3072: 12 output tiles, split automatically over the SMs
    c = synth.gpt2_mlp_up_64x768x3072()
    assert mm.mm_gemm_f32_splitk_workspace(c.M, c.N, c.K, 0) > 0
    C = run_splitk(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B, 0)
    ref, T = oracle.gemm(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B)
    check_bound(C, ref, T, c.name + " split-K")


@pytest.mark.parametrize("splitk", [1, 2, 3, 5, 16])
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", [(64, 3072, 768), (100, 300, 500), (300, 260, 1000), (5, 7, 40)])
def test_gemm_splitk_parity(oracle, splitk, layout, shape):
    # single CTAs (M <= 128) and CTA pairs (M > 128), ragged tiles, K tails, uneven slices
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = stored(tA, tB, M, N, K, seed=900 + M + N + K)
    Ap = np.zeros((A.shape[0], (A.shape[1] + 3) // 4 * 4), np.float32); Ap[:, :A.shape[1]] = A
    Bp = np.zeros((B.shape[0], (B.shape[1] + 3) // 4 * 4), np.float32); Bp[:, :B.shape[1]] = B
    C = run_splitk(tA, tB, M, N, K, Ap, Bp, splitk, lda=Ap.shape[1], ldb=Bp.shape[1], ldc=N + 3)
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    check_bound(C[:, :N], ref, T, f"split {splitk} {layout} {shape}")
    assert np.all(np.isnan(C[:, N:])), "columns past N were written"


def test_gemm_splitk_deterministic_and_integer_exact(oracle):
    M, N, K = 96, 520, 1536
    A, B = stored(0, 0, M, N, K, seed=77, kind="int")
    ref, _ = oracle.gemm(0, 0, M, N, K, A, B)
    c1 = run_splitk(0, 0, M, N, K, A, B, 7)
    c2 = run_splitk(0, 0, M, N, K, A, B, 7, fill=123.0)
    check_exact(c1, ref, "split-K integers")
    assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))


def test_gemm_splitk_unaligned_operands_take_general_path(oracle):
    # lda not a multiple of 4: no TMA, no split; the workspace is not needed
    M, N, K = 70, 45, 83
    A, B = stored(0, 0, M, N, K, seed=5)
    Ap = np.zeros((M, K + 3), np.float32); Ap[:, :K] = A
    C = run_splitk(0, 0, M, N, K, Ap, B, 4, lda=K + 3)
    ref, T = oracle.gemm(0, 0, M, N, K, A, B)
    check_bound(C, ref, T, "general path")


@pytest.mark.parametrize("layout", ["nn", "nt", "tn"])
def test_square_2048_stream_k_auto_all_outputs(oracle, layout):
    # 64 pair tiles on 76 pairs: the automatic split is stream-K
    c = synth.square_2048(layout)
    C = run_splitk(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B, 0)
    ref, T = oracle.gemm(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B)
    worst = check_bound(C, ref, T, c.name + " stream-K")
    print(f"{c.name} stream-K: worst |err|/T = {worst:.3e}")


@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", [(300, 2000, 1000), (100, 3000, 2000), (2000, 2900, 72), (129, 257, 33),
                                   (19456, 256, 24), (64, 300, 4096)])
def test_gemm_stream_k_parity(oracle, layout, shape):
    # stream-K forced: tiles fewer and more than the units, one- and multi-segment tiles,
    # short K (a unit spanning several whole tiles), single CTAs and pairs
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = stored(tA, tB, M, N, K, seed=1300 + M + N + K)
    Ap = np.zeros((A.shape[0], (A.shape[1] + 3) // 4 * 4), np.float32); Ap[:, :A.shape[1]] = A
    Bp = np.zeros((B.shape[0], (B.shape[1] + 3) // 4 * 4), np.float32); Bp[:, :B.shape[1]] = B
    C = run_splitk(tA, tB, M, N, K, Ap, Bp, -1, lda=Ap.shape[1], ldb=Bp.shape[1], ldc=N + 2)
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    check_bound(C[:, :N], ref, T, f"stream-K {layout} {shape}")
    assert np.all(np.isnan(C[:, N:])), "columns past N were written"


def test_gemm_stream_k_deterministic_and_integer_exact(oracle):
    M, N, K = 700, 900, 2000
    A, B = stored(0, 1, M, N, K, seed=91, kind="int")
    ref, _ = oracle.gemm(0, 1, M, N, K, A, B)
    c1 = run_splitk(0, 1, M, N, K, A, B, -1)
    c2 = run_splitk(0, 1, M, N, K, A, B, -1, fill=-7.0)
    check_exact(c1, ref, "stream-K integers")
    assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))


def test_training_set_through_the_bench_split_path(oracle):
    # The training-shape set exactly as the bench times it: mm_gemm_f32_splitk with the
    # automatic split (splitk = 0) and one workspace sized for the largest of the three
    # products.  On a 152-SM GB300 that is no split for the forward product and stream-K
    # for dA (8192 x 2048 x 8192) and dB (2048 x 8192 x 8192), whose tiles are each added
    # up from several K segments through the workspace flags.  Checked: whole first, last
    # and random rows and columns, every output of the first, a middle and the last
    # 256 x 256 tile, and random outputs.
    import torch
    cases = synth.training_set_8192_all()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plans = [mm.mm_gemm_f32_split_plan(c.M, c.N, c.K, sms)[0] for c in cases]
    if sms == 152:
        assert plans == [1, -1, -1], plans
    need = max(mm.mm_gemm_f32_splitk_workspace(c.M, c.N, c.K, 0) for c in cases)
    dev = torch.device("cuda:0")
    ws = torch.full((max(need, 4),), float("nan"), dtype=torch.float32, device=dev)
    dA = to_dev(cases[0].A)
    dB = to_dev(cases[0].B)
    ddC = to_dev(cases[1].A)
    rng = np.random.default_rng(11)
    for n, (c, (a, b)) in enumerate(zip(cases, ((dA, dB), (ddC, dB), (dA, ddC)))):
        out = empty_f32((c.M, c.N))
        mm.mm_gemm_f32_splitk(c.transA, c.transB, c.M, c.N, c.K, a, a.shape[1], b, b.shape[1], out, c.N, 0,
                              ws, need)
        mm.mm_check_device_error()
        C = to_host(out)
        rows = [0, c.M - 1, int(rng.integers(c.M))]
        cols = [0, c.N - 1, int(rng.integers(c.N))]
        blocks = []
        for (r0, c0) in ((0, 0), ((c.M // 512) * 256, (c.N // 512) * 256), (c.M - 256, c.N - 256)):
            bi, bj = np.meshgrid(np.arange(r0, r0 + 256), np.arange(c0, c0 + 256), indexing="ij")
            blocks.append((bi.reshape(-1), bj.reshape(-1)))
        ii = np.concatenate([np.repeat(rows, c.N), np.tile(np.arange(c.M), len(cols))] + [b[0] for b in blocks]
                            + [rng.integers(0, c.M, 4000)])
        jj = np.concatenate([np.tile(np.arange(c.N), len(rows)), np.repeat(cols, c.M)] + [b[1] for b in blocks]
                            + [rng.integers(0, c.N, 4000)])
        ref, T = oracle.gemm_at(c.transA, c.transB, c.K, c.A, c.B, ii, jj)
        worst = check_bound(C[ii, jj], ref, T, c.name + " bench split path")
        print(f"{c.name} (split {plans[n]}): {len(ii)} outputs, worst |err|/T = {worst:.3e}")



# ------------------------------------------------------------------ few rows: K split over a cluster

@pytest.mark.parametrize("splitk", [0, 1, 2, 3, 5, 8])
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", [(64, 3072, 768), (1, 1, 1), (7, 130, 45), (64, 200, 1000), (33, 64, 31),
                                   (100, 257, 300)])
@pytest.mark.parametrize("aligned", [False, True])
def test_gemm_skinny_parity(oracle, splitk, layout, shape, aligned):
    # 64 x 64 FFMA tiles, K cut over a thread-block cluster, partial tiles added in rank order
    # through distributed shared memory; ragged M, N and K, rows beyond 64 (a second row of
    # tiles), padded leading dimensions -- a multiple of four floats (16-byte copies) or odd
    # (4-byte copies); columns past N stay untouched
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = stored(tA, tB, M, N, K, seed=2100 + M + N + K)
    lda = (A.shape[1] + 3) // 4 * 4 + 4 if aligned else A.shape[1] + 1 + A.shape[1] % 2
    ldb = (B.shape[1] + 3) // 4 * 4 + 8 if aligned else B.shape[1] + 3 + B.shape[1] % 2
    Ap = np.zeros((A.shape[0], lda), np.float32); Ap[:, :A.shape[1]] = A
    Bp = np.zeros((B.shape[0], ldb), np.float32); Bp[:, :B.shape[1]] = B
    dA, dB = to_dev(Ap), to_dev(Bp)
    dC = empty_f32((M, N + 5))
    mm.mm_gemm_f32_ex(tA, tB, M, N, K, dA, Ap.shape[1], dB, Bp.shape[1], dC, N + 5, path=mm.MM_GEMM_FFMA, tile=4,
                      splitk=splitk)
    mm.mm_check_device_error()
    C = to_host(dC)
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    check_bound(C[:, :N], ref, T, f"skinny split {splitk} {layout} {shape}")
    assert np.all(np.isnan(C[:, N:])), "columns past N were written"


def _few_rows_calls(c, lda, ldb, explicit_path):
    """Automatic, explicit tile 4 on `explicit_path`, automatic again: three C arrays."""
    Ap = np.zeros((c.M, lda), np.float32); Ap[:, :c.K] = c.A
    Bp = np.zeros((c.K, ldb), np.float32); Bp[:, :c.N] = c.B
    dA, dB = to_dev(Ap), to_dev(Bp)
    outs = []
    for explicit in (False, True, False):
        dC = empty_f32((c.M, c.N))
        if explicit:
            mm.mm_gemm_f32_ex(0, 0, c.M, c.N, c.K, dA, lda, dB, ldb, dC, c.N, path=explicit_path, tile=4)
        else:
            mm.mm_gemm_f32(0, 0, c.M, c.N, c.K, dA, lda, dB, ldb, dC, c.N)
        mm.mm_check_device_error()
        outs.append(to_host(dC))
    return outs


@pytest.mark.parametrize("kernel", ["tensor_cores", "ffma"])
def test_gemm_skinny_is_automatic_for_few_rows_and_deterministic(oracle, kernel):
    # the GPT-2 MLP up-projection at 64 tokens through mm_gemm_f32 takes a few-rows kernel: the
    # 3xTF32 one when TMA can describe the operands (leading dimensions multiples of four), the
    # FFMA one otherwise (odd leading dimensions) -- the same bits as the explicit tile-4 call of
    # that path, on every call; small integers are exact
    c = synth.gpt2_mlp_up_64x768x3072()
    tc = kernel == "tensor_cores"
    outs = _few_rows_calls(c, c.K if tc else c.K + 1, c.N if tc else c.N + 3,
                           mm.MM_GEMM_TF32X3 if tc else mm.MM_GEMM_FFMA)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[2].view(np.uint32))
    ref, T = oracle.gemm(0, 0, c.M, c.N, c.K, c.A, c.B)
    check_bound(outs[0], ref, T, f"automatic few-rows path ({kernel})")
    for tA, tB, K in ((1, 1, 777), (0, 1, 776), (1, 0, 300)):
        A, B = stored(tA, tB, 48, 1000, K, seed=5 + K, kind="int")
        C = run(tA, tB, 48, 1000, K, A, B)
        check_exact(C, oracle.gemm(tA, tB, 48, 1000, K, A, B)[0], f"few rows, integers, layout {tA}{tB}, K={K}")


# ------------------------------------------------------------------ few rows on the tensor cores

@pytest.mark.parametrize("splitk", [0, 1, 2, 3, 6, 8])
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", [(64, 3072, 768), (1, 1, 1), (7, 130, 45), (64, 200, 1000), (33, 64, 31),
                                   (17, 257, 300), (64, 128, 16)])
@pytest.mark.parametrize("ldc_pad", [4, 5])
def test_gemm_skinny_tc_parity(oracle, splitk, layout, shape, ldc_pad):
    # 3xTF32 on tcgen05 with C computed transposed (128 columns of C per CTA as the MMA's M, the
    # rows as its N), K cut over a cluster of `splitk` CTAs (a rank without K slabs adds zeros),
    # partial tiles added in rank order through distributed shared memory; ragged M, N and K,
    # padded leading dimensions (multiples of four floats), rows of C a multiple of four floats
    # apart (16-byte stores) or not; columns past N stay untouched
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = stored(tA, tB, M, N, K, seed=3100 + M + N + K)
    lda = (A.shape[1] + 3) // 4 * 4 + 4
    ldb = (B.shape[1] + 3) // 4 * 4 + 8
    Ap = np.zeros((A.shape[0], lda), np.float32); Ap[:, :A.shape[1]] = A
    Bp = np.zeros((B.shape[0], ldb), np.float32); Bp[:, :B.shape[1]] = B
    dA, dB = to_dev(Ap), to_dev(Bp)
    ldc = N + ldc_pad
    dC = empty_f32((M, ldc))
    mm.mm_gemm_f32_ex(tA, tB, M, N, K, dA, lda, dB, ldb, dC, ldc, path=mm.MM_GEMM_TF32X3, tile=4, splitk=splitk)
    mm.mm_check_device_error()
    C = to_host(dC)
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    check_bound(C[:, :N], ref, T, f"tensor-core few rows split {splitk} {layout} {shape} ldc N+{ldc_pad}")
    assert np.all(np.isnan(C[:, N:])), "columns past N were written"


def test_gemm_skinny_tc_k_margin_and_refusals(oracle):
    # K at the 3xTF32 margin runs on the tensor cores within the bound; one slab past it, the
    # automatic call takes the FFMA few-rows kernel, and the explicit tile 4 is refused, as are
    # M > 64 and leading dimensions TMA cannot describe
    M, N = 16, 256
    for K in (16384, 16388):
        A, B = stored(0, 0, M, N, K, seed=K)
        C = run(0, 0, M, N, K, A, B)
        ref, T = oracle.gemm(0, 0, M, N, K, A, B)
        check_bound(C, ref, T, f"few rows, K={K}")
    C = run(0, 0, M, N, 16384, A[:, :16384].copy(), B[:16384].copy(), path=(mm.MM_GEMM_TF32X3, 4))
    ref, T = oracle.gemm(0, 0, M, N, 16384, A[:, :16384], B[:16384])
    check_bound(C, ref, T, "tile 4 at the K margin")
    import torch
    z = torch.zeros(((16388 + 4) * 300,), device="cuda")
    out = torch.empty((65 * 256,), device="cuda")
    for (m, k, lda, ldb) in ((16, 16388, 16388, 256), (65, 64, 64, 256), (16, 64, 65, 256), (16, 64, 64, 258)):
        with pytest.raises(mm.MMError) as e:
            mm.mm_gemm_f32_ex(0, 0, m, 256, k, z, lda, z, ldb, out, 256, path=mm.MM_GEMM_TF32X3, tile=4)
        assert e.value.status == mm.MM_ERR_INVALID_ARG


# ------------------------------------------------------------------ the 3xTF32 accuracy margin on K

def test_tf32x3_k_margin_boundary(oracle):
    # K = 16384 is the longest 3xTF32 accumulation: taken when asked for, and automatically; past it
    # (16388: still a multiple of 4, so that TMA could describe the operands) an explicit 3xTF32
    # request is refused while the automatic path runs the FFMA kernel -- both within the bound.
    # N(0, 0.02) operands, the distribution the margin was measured on.
    M, N = 256, 192
    for K in (16384, 16388):
        A = synth.normal_f32(6100 + K, (M, K), 0.02)
        B = synth.normal_f32(6200 + K, (K, N), 0.02)
        ref, T = oracle.gemm(0, 0, M, N, K, A, B)
        C = run(0, 0, M, N, K, A, B)
        check_bound(C, ref, T, f"automatic path, K={K}")
        if K <= 16384:
            check_bound(run(0, 0, M, N, K, A, B, path=mm.MM_GEMM_TF32X3), ref, T, f"3xTF32, K={K}")
        else:
            with pytest.raises(mm.MMError, match="3xTF32 needs K <= 16384"):
                run(0, 0, M, N, K, A, B, path=mm.MM_GEMM_TF32X3)
            check_bound(run(0, 0, M, N, K, A, B, path=mm.MM_GEMM_FFMA), ref, T, f"FFMA, K={K}")


def test_bias_act_beyond_the_k_margin(oracle):
    # bias + GELU with K past the margin: the TMA-staged FFMA kernel with its fused epilogue
    M, N, K = 160, 130, 16400
    A = synth.normal_f32(6301, (M, K), 0.02)
    B = synth.normal_f32(6302, (K, N), 0.02)
    bias = synth.normal_f32(6303, (N,), 0.02)
    for act in (0, 1):
        Y, T, Z = oracle.gemm_bias_act(0, 0, M, N, K, A, B, bias, act)
        dC = empty_f32((M, N))
        mm.mm_gemm_f32_bias_act(0, 0, M, N, K, to_dev(A), K, to_dev(B), N, to_dev(bias), act, dC, N)
        mm.mm_check_device_error()
        got = to_host(dC).astype(np.float64)
        bound = 1.13e-5 * T + 2.0 ** -20 * (1.0 + np.abs(Z))
        assert np.all(np.abs(got - Y) <= bound), f"act {act}: worst {np.max(np.abs(got - Y) / bound):.3f} of the bound"


def test_splitk_keeps_every_slice_within_the_k_margin(oracle):
    import torch
    # K = 40000 on one output tile: the automatic split takes at least 3 slices of <= 16384; an
    # explicit 2-slice split would leave 20000-long slices, so it runs the FFMA kernel unsplit and
    # needs no workspace; stream-K likewise
    M, N, K = 128, 256, 40000
    A = synth.normal_f32(6401, (M, K), 0.02)
    B = synth.normal_f32(6402, (K, N), 0.02)
    ref, T = oracle.gemm(0, 0, M, N, K, A, B)
    dA, dB = to_dev(A), to_dev(B)
    auto_split, _ = mm.mm_gemm_f32_split_plan(M, N, K, 152)
    assert auto_split >= 3
    for splitk in (0, 2, 3, -1):
        need = mm.mm_gemm_f32_splitk_workspace(M, N, K, splitk)
        if splitk in (2, -1):
            assert need == 0
        ws = torch.full((max(need, 1),), float("nan"), dtype=torch.float32, device=dA.device)
        dC = empty_f32((M, N))
        mm.mm_gemm_f32_splitk(0, 0, M, N, K, dA, K, dB, N, dC, N, splitk, ws if need else None, need)
        mm.mm_check_device_error()
        check_bound(to_host(dC), ref, T, f"split {splitk}, K={K}")


# ------------------------------------------------------------------ FFMA kernel with a stream-K tail

def run_ffma_sk(tA, tB, M, N, K, A, B, splitk=0, lda=None, ldb=None, ldc=None, fill=float("nan")):
    import torch
    lda = lda or A.shape[1]
    ldb = ldb or B.shape[1]
    ldc = ldc or N
    dA, dB = to_dev(A), to_dev(B)
    dC = empty_f32((M, ldc))
    n = mm.mm_gemm_f32_splitk_workspace_ex(M, N, K, splitk, path=mm.MM_GEMM_FFMA)
    ws = torch.full((max(n, 1),), fill, dtype=torch.float32, device=dA.device)  # contents must not matter
    mm.mm_gemm_f32_splitk_ex(tA, tB, M, N, K, dA, lda, dB, ldb, dC, ldc, splitk, ws if n else None, n,
                             path=mm.MM_GEMM_FFMA)
    mm.mm_check_device_error()
    return to_host(dC), n


@pytest.mark.parametrize("splitk", [0, -1, 1])
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", [(500, 700, 3000), (130, 260, 1000), (1700, 1650, 300), (1664, 1664, 300),
                                   (2432, 2176, 200), (129, 129, 257)])
def test_ffma_stream_k_parity(oracle, splitk, layout, shape):
    # fewer tiles than SMs (every tile split), a short last wave after a whole one (the
    # first 152 tiles whole, the rest split), a K too short for a split, ragged tiles and K
    tA, tB = LAYOUTS[layout]
    M, N, K = shape
    A, B = stored(tA, tB, M, N, K, seed=1500 + M + N + K)
    Ap = np.zeros((A.shape[0], (A.shape[1] + 3) // 4 * 4), np.float32); Ap[:, :A.shape[1]] = A
    Bp = np.zeros((B.shape[0], (B.shape[1] + 3) // 4 * 4), np.float32); Bp[:, :B.shape[1]] = B
    C, n = run_ffma_sk(tA, tB, M, N, K, Ap, Bp, splitk, lda=Ap.shape[1], ldb=Bp.shape[1], ldc=N + 2)
    if splitk == 1:
        assert n == 0
    ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
    check_bound(C[:, :N], ref, T, f"FFMA stream-K {splitk} {layout} {shape} (workspace {n})")
    assert np.all(np.isnan(C[:, N:])), "columns past N were written"


@pytest.mark.parametrize("layout", ["nn", "nt", "tn"])
def test_square_2048_ffma_stream_k_all_outputs(oracle, layout):
    # the bench's FFMA phase: 256 tiles on 152 SMs, 152 whole and 104 split over 152 CTAs
    c = synth.square_2048(layout)
    C, n = run_ffma_sk(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B, 0)
    assert n > 0
    ref, T = oracle.gemm(c.transA, c.transB, c.M, c.N, c.K, c.A, c.B)
    worst = check_bound(C, ref, T, c.name + " FFMA stream-K")
    print(f"{c.name} FFMA stream-K: worst |err|/T = {worst:.3e}")


def test_ffma_stream_k_deterministic_and_integer_exact(oracle):
    # integers: every partial sum exact, so the split tiles equal the oracle bit for bit; two
    # runs with different workspace contents give the same bits
    M, N, K = 1700, 1650, 600
    A, B = stored(0, 1, M, N, K, seed=93, kind="int")
    ref, _ = oracle.gemm(0, 1, M, N, K, A, B)
    c1, n = run_ffma_sk(0, 1, M, N, K, A, B, -1)
    c2, _ = run_ffma_sk(0, 1, M, N, K, A, B, -1, fill=-7.0)
    assert n > 0
    check_exact(c1, ref, "FFMA stream-K integers")
    assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))


def test_ffma_stream_k_unaligned_operands_take_general_path(oracle):
    M, N, K = 1700, 1650, 301
    A, B = stored(0, 0, M, N, K, seed=6)
    Ap = np.zeros((M, K + 3), np.float32); Ap[:, :K] = A
    C, _ = run_ffma_sk(0, 0, M, N, K, Ap, B, -1, lda=K + 3)
    ref, T = oracle.gemm(0, 0, M, N, K, A, B)
    check_bound(C, ref, T, "FFMA stream-K request, general path")
