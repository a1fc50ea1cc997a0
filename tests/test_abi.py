"""The C-ABI library builds, loads and exports every symbol include/mm.h declares;
argument checks return their status codes before any CUDA call (no GPU needed).

Every call here is rejected by argument validation, so no pointer passed is
ever dereferenced and no kernel is launched, on any machine.
"""
import ctypes
import os
import re

import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import build as mmbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    mmbuild.build()
    return mm.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "mm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mm_[a-z0-9_]+)\s*\(", src)))


def test_header_lists_the_boundary():
    names = header_functions()
    for n in ["mm_gemm_f32", "mm_gemv_packed2", "mm_gemm_packed2", "mm_last_error", "mm_version",
              "mm_check_device_error", "mm_gemm_f32_ex", "mm_gemv_packed2_ex", "mm_gemm_packed2_ex"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert name in mm.SIGNATURES, f"binding lacks {name}"


def test_library_has_no_oracle_symbols(lib):
    # the product library must not carry the oracle
    for name in ["orc_gemm", "orc_packed_gemm", "orc_unpack2"]:
        with pytest.raises(AttributeError):
            getattr(lib, name)


def test_version(lib):
    assert mm.mm_version() == 100


def _status(fn, *args):
    return fn(*args)


@pytest.mark.parametrize("case", [
    dict(tA=2), dict(M=0), dict(N=-1), dict(K=0), dict(A=None), dict(B=None), dict(C=None),
    dict(lda=3), dict(ldb=4), dict(ldc=5), dict(tA=1, lda=7), dict(tB=1, ldb=7),
])
def test_gemm_argument_errors(lib, case):
    a = dict(tA=0, tB=0, M=8, N=8, K=8, A=FAKE, lda=8, B=FAKE + 4096, ldb=8, C=FAKE + 8192, ldc=8)
    a.update(case)
    st = lib.mm_gemm_f32(a["tA"], a["tB"], a["M"], a["N"], a["K"], a["A"], a["lda"], a["B"], a["ldb"],
                         a["C"], a["ldc"], None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()
    assert lib.mm_last_error()


def test_gemm_overlap_rejected(lib):
    # C overlapping A
    st = lib.mm_gemm_f32(0, 0, 8, 8, 8, FAKE, 8, FAKE + 4096, 8, FAKE + 64, 8, None)
    assert st == mm.MM_ERR_INVALID_ARG and b"overlap" in lib.mm_last_error()


def test_gemm_bad_path_option(lib):
    o = mm.GemmOpts(7, 0)
    st = lib.mm_gemm_f32_ex(0, 0, 8, 8, 8, FAKE, 8, FAKE + 4096, 8, FAKE + 8192, 8, None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG


@pytest.mark.parametrize("path,tile", [(0, 4), (2, -1), (2, 7)])
def test_gemm_bad_tf32x3_tile(lib, path, tile):
    o = mm.GemmOpts(path, tile)
    st = lib.mm_gemm_f32_ex(0, 0, 8, 8, 8, FAKE, 8, FAKE + 4096, 8, FAKE + 8192, 8, None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG and b"tile" in lib.mm_last_error()


@pytest.mark.parametrize("path,tile,splitk", [(1, 3, 0), (1, 5, 0), (1, 4, 9), (1, 4, -1), (1, 0, 2), (0, 0, 2),
                                              (2, 2, 1)])
def test_gemm_bad_ffma_tile_or_split(lib, path, tile, splitk):
    # the few-rows FFMA kernel is tile 4 of the FFMA path; only it takes a cluster split (1..8)
    o = mm.GemmOpts(path, tile, splitk)
    st = lib.mm_gemm_f32_ex(0, 0, 8, 8, 8, FAKE, 8, FAKE + 4096, 8, FAKE + 8192, 8, None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG


def test_gemm_splitk_workspace_size(lib):
    out = ctypes.c_int64(-1)
    assert lib.mm_gemm_f32_splitk_workspace(64, 3072, 768, 4, ctypes.byref(out)) == mm.MM_OK
    assert out.value == 4 * 64 * 3072
    assert lib.mm_gemm_f32_splitk_workspace(64, 3072, 768, 1, ctypes.byref(out)) == mm.MM_OK and out.value == 0
    # a split is capped at one slice per 16-deep slab of K
    assert lib.mm_gemm_f32_splitk_workspace(8, 8, 20, 16, ctypes.byref(out)) == mm.MM_OK and out.value == 2 * 64
    assert lib.mm_gemm_f32_splitk_workspace(64, 3072, 768, 17, ctypes.byref(out)) == mm.MM_ERR_INVALID_ARG
    assert lib.mm_gemm_f32_splitk_workspace(0, 3072, 768, 2, ctypes.byref(out)) == mm.MM_ERR_INVALID_ARG
    assert lib.mm_gemm_f32_splitk_workspace(8, 8, 8, 2, None) == mm.MM_ERR_INVALID_ARG


@pytest.mark.parametrize("case", [dict(splitk=17), dict(splitk=-2), dict(ws=FAKE + 0x100004),
                                  dict(ws_floats=4 * 64 * 64 - 1), dict(ws=None), dict(ws=FAKE + 64),
                                  dict(ws_floats=-5), dict(ldc=10)])
def test_gemm_splitk_argument_errors(lib, case):
    a = dict(M=64, N=64, K=256, A=FAKE, B=FAKE + 0x20000, C=FAKE + 0x40000, ldc=64, splitk=4,
             ws=FAKE + 0x100000, ws_floats=4 * 64 * 64)
    a.update(case)
    st = lib.mm_gemm_f32_splitk(0, 0, a["M"], a["N"], a["K"], a["A"], a["K"], a["B"], a["N"], a["C"], a["ldc"],
                                a["splitk"], a["ws"], a["ws_floats"], None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()


def test_gemm_splitk_noalloc_rejects_oversized_split(lib):
    # 16 slices of 1024 x 1024 need 16 Mi floats, more than the static scratch holds
    assert mm.MM_SPLITK_NOALLOC_MAX_FLOATS == 4194304
    st = lib.mm_gemm_f32_splitk_noalloc(0, 0, 1024, 1024, 4096, FAKE, 4096, FAKE + 0x1000000, 1024,
                                        FAKE + 0x2000000, 1024, 16, None)
    assert st == mm.MM_ERR_INVALID_ARG and b"static scratch" in lib.mm_last_error()
    st = lib.mm_gemm_f32_splitk_noalloc(0, 0, 8, 8, 64, None, 64, FAKE, 8, FAKE + 0x10000, 8, 2, None)
    assert st == mm.MM_ERR_INVALID_ARG


def _cb(*v):
    return (ctypes.c_float * 4)(*v)


@pytest.mark.parametrize("case", [
    dict(codes=None), dict(scales=None), dict(x=None), dict(y=None), dict(rows=0), dict(cols=0),
    dict(cb=None), dict(cb=(0.0, float("nan"), 1.0, 2.0)), dict(cb=(0.0, float("inf"), 1.0, 2.0)),
])
def test_gemv_argument_errors(lib, case):
    a = dict(codes=FAKE, scales=FAKE + 0x100000, x=FAKE + 0x200000, y=FAKE + 0x300000, rows=64, cols=64,
             cb=(-2.0, -1.0, 0.0, 1.0))
    a.update(case)
    cb = None if a["cb"] is None else _cb(*a["cb"])
    st = lib.mm_gemv_packed2(a["codes"], a["scales"], a["x"], a["y"], a["rows"], a["cols"], cb, None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()


def test_gemv_output_overlap_rejected(lib):
    st = lib.mm_gemv_packed2(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 8, 64, 64, _cb(-2, -1, 0, 1), None)
    assert st == mm.MM_ERR_INVALID_ARG and b"overlap" in lib.mm_last_error()


@pytest.mark.parametrize("opt", [dict(split=3), dict(rows_per_lane=3), dict(warps=17), dict(dequant=9),
                                 dict(pdl=2), dict(weights_static=5)])
def test_gemv_bad_options(lib, opt):
    o = mm.GemvOpts(**opt)
    st = lib.mm_gemv_packed2_ex(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 64, 64,
                                _cb(-2, -1, 0, 1), None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG


def test_gemv_affine_decode_needs_affine_codebook(lib):
    o = mm.GemvOpts(dequant=mm.MM_DEQ_AFFINE)
    st = lib.mm_gemv_packed2_ex(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 64, 64,
                                _cb(-1, 0, 1, 0), None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG and b"affine" in lib.mm_last_error()


@pytest.mark.parametrize("case", [dict(M=0), dict(rows=-3), dict(X=None), dict(cb=None)])
def test_gemm_packed_argument_errors(lib, case):
    a = dict(M=4, rows=64, cols=64, X=FAKE + 0x200000, cb=(-1.0, 0.0, 1.0, 0.0))
    a.update(case)
    cb = None if a["cb"] is None else _cb(*a["cb"])
    st = lib.mm_gemm_packed2(FAKE, FAKE + 0x100000, a["X"], FAKE + 0x300000, a["M"], a["rows"], a["cols"],
                             cb, None)
    assert st == mm.MM_ERR_INVALID_ARG


def test_python_binding_raises_with_message(lib):
    with pytest.raises(mm.MMError) as ei:
        mm.mm_gemm_f32(0, 0, 0, 8, 8, FAKE, 8, FAKE, 8, FAKE, 8, stream=0)
    assert ei.value.status == mm.MM_ERR_INVALID_ARG and "M, N, K" in str(ei.value)


def test_missing_library_fails_loudly(monkeypatch):
    # a separate copy of the binding module, so the loaded library stays untouched
    import importlib.util
    spec = importlib.util.spec_from_file_location("mm_binding_copy", mm.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    monkeypatch.setenv("MM_LIBRARY", "/nonexistent/libmm.so")
    with pytest.raises(mod.MMError):
        mod.load_library()


@pytest.mark.parametrize("tile", [-1, 4, 48, 256])
def test_gemm_packed_bad_tile(lib, tile):
    o = mm.GemmPacked2Opts(tile)
    st = lib.mm_gemm_packed2_ex(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 4, 64, 64,
                                _cb(-1, 0, 1, 0), None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG


def test_gemm_packed_tensor_core_tile_needs_fp16_codebook(lib):
    o = mm.GemmPacked2Opts(64)
    st = lib.mm_gemm_packed2_ex(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 4, 64, 64,
                                _cb(0.3, -1.7, 2.5, 0.01), None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG and b"fp16" in lib.mm_last_error()


@pytest.mark.parametrize("opt", [dict(tile=2, cols=100), dict(tile=2, splitk=16, cols=640),
                                 dict(tile=2, splitk=1, cols=1024), dict(pdl=2), dict(pdl=0, weights_static=1),
                                 dict(tile=64, splitk=16), dict(tile=3, cols=100), dict(tile=3, splitk=16),
                                 dict(tile=3, splitk=16, cols=64 * 8), dict(tile=3, ntok=8), dict(tile=3, ntok=272),
                                 dict(tile=3, ntok=40), dict(tile=2, ntok=64), dict(ntok=64),
                                 dict(tile=3, splitk=8, cols=64 * 4)])
def test_gemm_packed_tile2_bad_options(lib, opt):
    # tile 2 needs cols % 64 == 0 and 1 to 8 atoms of 64 per CTA; weights_static needs pdl
    cols = opt.pop("cols", 640)
    o = mm.GemmPacked2Opts(**opt)
    st = lib.mm_gemm_packed2_ex(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 4, 64, cols,
                                _cb(-1, 0, 1, 0), None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()


@pytest.mark.parametrize("splitk", [-1, 3, 16])
def test_gemm_packed_bad_splitk(lib, splitk):
    o = mm.GemmPacked2Opts(0, splitk)
    st = lib.mm_gemm_packed2_ex(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 4, 64, 64,
                                _cb(-1, 0, 1, 0), None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG


@pytest.mark.parametrize("opt", [dict(dequant=3, staging=2), dict(dequant=1, staging=1),
                                 dict(dequant=3, staging=1, split=2), dict(dequant=3, staging=1, rows_per_lane=65),
                                 dict(dequant=2, staging=1, warps=4), dict(dequant=2, staging=1, rows_per_lane=65)])
def test_gemv_bad_staging(lib, opt):
    o = mm.GemvOpts(**opt)
    st = lib.mm_gemv_packed2_ex(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 64, 1536,
                                _cb(-2, -1, 0, 1), None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG


def _cb16(*vals):
    v = list(vals) + [0.0] * (16 - len(vals))
    return (ctypes.c_float * 16)(*v)


def test_header_lists_the_4bit_boundary():
    names = header_functions()
    assert "mm_gemv_packed4" in names and "mm_gemv_packed4_ex" in names


@pytest.mark.parametrize("case", [
    dict(codes=None), dict(scales=None), dict(x=None), dict(y=None), dict(rows=0), dict(cols=-3),
    dict(cb="nan"), dict(cb=None), dict(y="overlap"),
])
def test_gemv4_argument_errors(lib, case):
    a = dict(codes=FAKE, scales=FAKE + 0x100000, x=FAKE + 0x200000, y=FAKE + 0x300000, rows=64, cols=1536,
             cb=_cb16(*range(16)))
    a.update(case)
    if a["cb"] == "nan":
        a["cb"] = _cb16(*([0.0] * 12 + [float("nan")]))
    if a["y"] == "overlap":
        a["y"] = FAKE + 64
    st = lib.mm_gemv_packed4(a["codes"], a["scales"], a["x"], a["y"], a["rows"], a["cols"], a["cb"], None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()
    assert lib.mm_last_error()


@pytest.mark.parametrize("opt", [dict(staging=1, cols=1000), dict(staging=1, cols=8192), dict(staging=2),
                                 dict(blocks=65), dict(blocks=-1), dict(pdl=2), dict(independent=3)])
def test_gemv4_bad_options(lib, opt):
    cols = opt.pop("cols", 1536)
    o = mm.Gemv4Opts(**opt)
    st = lib.mm_gemv_packed4_ex(FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 64, cols,
                                _cb16(*range(16)), None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()


@pytest.mark.parametrize("case", [dict(act=2), dict(act=-1), dict(bias=FAKE + 0x40000 + 4 * 64 * 10),
                                  dict(bias=FAKE + 0x40000 - 8), dict(C=None), dict(K=0), dict(tA=2),
                                  dict(ldc=63)])
def test_gemm_bias_act_argument_errors(lib, case):
    # an unknown activation, a bias overlapping C, and the plain GEMM's own checks
    a = dict(tA=0, M=64, N=64, K=256, A=FAKE, B=FAKE + 0x20000, C=FAKE + 0x40000, ldc=64,
             bias=FAKE + 0x80000, act=1)
    a.update(case)
    st = lib.mm_gemm_f32_bias_act(a["tA"], 0, a["M"], a["N"], a["K"], a["A"], a["K"], a["B"], a["N"],
                                  a["bias"], a["act"], a["C"], a["ldc"], None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()
    assert mm.MM_ACT_NONE == 0 and mm.MM_ACT_GELU_TANH == 1


@pytest.mark.parametrize("case", [dict(batch=0), dict(codes_stride=100), dict(scales_stride=10), dict(y_stride=10),
                                  dict(x_stride=5), dict(x_stride=-64), dict(y=FAKE + 0x400),
                                  dict(y=FAKE + 0x200000 + 16), dict(codes=None)])
def test_gemv_batched_argument_errors(lib, case):
    # batch >= 1; strides cover one matrix (or are 0 for a shared x); no y over any input
    a = dict(codes=FAKE, codes_stride=64 * 16, scales=FAKE + 0x100000, scales_stride=64, x=FAKE + 0x200000,
             x_stride=64, y=FAKE + 0x300000, y_stride=64, batch=3, rows=64, cols=64)
    a.update(case)
    st = lib.mm_gemv_packed2_strided_batched(a["codes"], a["codes_stride"], a["scales"], a["scales_stride"], a["x"],
                                             a["x_stride"], a["y"], a["y_stride"], a["batch"], a["rows"], a["cols"],
                                             _cb(-2, -1, 0, 1), None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()


@pytest.mark.parametrize("case", [dict(act=3), dict(bias=FAKE + 0x40000), dict(splitk=17), dict(splitk=-2),
                                  dict(ws=None, splitk=4), dict(ws_floats=10, splitk=4)])
def test_gemm_bias_act_splitk_argument_errors(lib, case):
    a = dict(M=64, N=64, K=256, A=FAKE, B=FAKE + 0x20000, C=FAKE + 0x40000, bias=FAKE + 0x80000, act=1, splitk=4,
             ws=FAKE + 0x100000, ws_floats=4 * 64 * 64)
    a.update(case)
    st = lib.mm_gemm_f32_bias_act_splitk(0, 0, a["M"], a["N"], a["K"], a["A"], a["K"], a["B"], a["N"], a["bias"],
                                         a["act"], a["C"], a["N"], a["splitk"], a["ws"], a["ws_floats"], None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()


# ------------------------------------------------------------------ the automatic GEMM split (host logic, no GPU)

@pytest.mark.parametrize("shape,split,floats", [
    # GPT-2 MLP up-projection 8192 x 3072 x 768: 384 pair tiles on 76 pairs (a partial 6th wave) but
    # only 48 slabs of 16 per tile, where stream-K measured slower: no split
    ((8192, 3072, 768), 1, 0),
    # training-shape dA / dB and 4096^3: 256 pair tiles = 3.4 waves, 256-512 slabs per tile: stream-K,
    # one 128 x 256 partial tile per CTA of the 76 units (2 x 76 x 32768 floats) + 152 flag words
    ((8192, 2048, 8192), -1, 2 * 76 * 32768 + 152),
    ((2048, 8192, 8192), -1, 2 * 76 * 32768 + 152),
    ((4096, 4096, 4096), -1, 2 * 76 * 32768 + 152),
    # training-shape forward 8192 x 8192 x 2048: 1024 pair tiles, 14 waves of 76 lose < 5%: no split
    ((8192, 8192, 2048), 1, 0),
    # 2048^3: 64 pair tiles, between half a wave and a wave: no split
    ((2048, 2048, 2048), 1, 0),
    # GPT-2 MLP up-projection at 64 tokens: 12 single-CTA tiles on 152 SMs -> 12 K slices of 64
    ((64, 3072, 768), 12, 12 * 64 * 3072),
    # 2 tiles: 76 slices would be too thin, capped at K / 64 = 8 slices
    ((100, 300, 500), 8, 8 * 100 * 300),
    # K past the 3xTF32 margin of 16384: at least ceil(K / 16384) slices, never stream-K nor none
    ((4096, 4096, 16384), -1, 2 * 76 * 32768 + 152),
    ((4096, 4096, 32768), 2, 2 * 4096 * 4096),
    ((8192, 8192, 20000), 2, 2 * 8192 * 8192),
    ((4096, 4096, 40000), 3, 3 * 4096 * 4096),
])
def test_gemm_split_plan(shape, split, floats):
    mm.load_library()
    assert mm.mm_gemm_f32_split_plan(*shape, 152) == (split, floats)


def test_gemm_split_plan_argument_errors(lib):
    sk, fl = ctypes.c_int(0), ctypes.c_int64(0)
    assert lib.mm_gemm_f32_split_plan(0, 8, 8, 152, ctypes.byref(sk), ctypes.byref(fl)) == mm.MM_ERR_INVALID_ARG
    assert lib.mm_gemm_f32_split_plan(8, 8, 8, 1, ctypes.byref(sk), ctypes.byref(fl)) == mm.MM_ERR_INVALID_ARG
    assert lib.mm_gemm_f32_split_plan(8, 8, 8, 152, None, ctypes.byref(fl)) == mm.MM_ERR_INVALID_ARG


@pytest.mark.parametrize("arrive,limit,out", [(2, 10000, None), (-1, 10000, None), (0, 999, None),
                                              (0, 100000001, None), (1, 0, None), (0, 2 ** 63, None),
                                              (0, 10000, FAKE + 4)])
def test_probe_bounded_wait_argument_errors(lib, arrive, limit, out):
    # arrive 0 / 1; limit 1 us .. 0.1 s, so the probe can never hold a GPU long; out 8-byte aligned
    st = lib.mm_probe_bounded_wait(arrive, limit, out, None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()


@pytest.mark.parametrize("K,splitk,floats", [
    (16384, 1, 0), (16384, 2, 2 * 256 * 256),
    # slices longer than 16384 would break the 3xTF32 margin: such a split runs unsplit, no workspace
    (40000, 2, 0), (40000, 3, 3 * 256 * 256), (300000, 16, 0),
])
def test_split_workspace_respects_the_k_margin(K, splitk, floats):
    mm.load_library()
    assert mm.mm_gemm_f32_splitk_workspace(256, 256, K, splitk) == floats


# ------------------------------------------------------------------ attention

_AN = 2 * 16 * 64 * 4  # bytes of one [2][16][64] fp32 tensor


@pytest.mark.parametrize("case,status", [
    (dict(heads=0), mm.MM_ERR_INVALID_ARG), (dict(T=0), mm.MM_ERR_INVALID_ARG), (dict(D=0), mm.MM_ERR_INVALID_ARG),
    (dict(causal=2), mm.MM_ERR_INVALID_ARG), (dict(scale=float("nan")), mm.MM_ERR_INVALID_ARG),
    (dict(scale=float("inf")), mm.MM_ERR_INVALID_ARG), (dict(Q=None), mm.MM_ERR_INVALID_ARG),
    (dict(V=None), mm.MM_ERR_INVALID_ARG), (dict(L=None), mm.MM_ERR_INVALID_ARG), (dict(O=None), mm.MM_ERR_INVALID_ARG),
    (dict(K=FAKE + 5 * _AN + 2), mm.MM_ERR_INVALID_ARG),            # misaligned
    (dict(O=FAKE + 64), mm.MM_ERR_INVALID_ARG),                     # O overlaps Q
    (dict(L=FAKE + 3 * _AN + 16), mm.MM_ERR_INVALID_ARG),           # L overlaps O
    (dict(D=32), mm.MM_ERR_UNSUPPORTED), (dict(D=128), mm.MM_ERR_UNSUPPORTED),
])
def test_attention_fwd_argument_errors(lib, case, status):
    a = dict(Q=FAKE, K=FAKE + _AN, V=FAKE + 2 * _AN, O=FAKE + 3 * _AN, L=FAKE + 4 * _AN, heads=2, T=16, D=64,
             causal=1, scale=0.125)
    a.update(case)
    st = mm.load_library().mm_attention_fwd(a["Q"], a["K"], a["V"], a["O"], a["L"], a["heads"], a["T"], a["D"],
                                            a["causal"], a["scale"], None)
    assert st == status, lib.mm_last_error()
    assert lib.mm_last_error()


@pytest.mark.parametrize("case", [
    dict(dQ=None), dict(dO=None), dict(dK=FAKE + 64), dict(dV=FAKE + 6 * _AN + 64), dict(L=FAKE + 7 * _AN + 4),
])
def test_attention_bwd_argument_errors(lib, case):
    a = dict(Q=FAKE, K=FAKE + _AN, V=FAKE + 2 * _AN, O=FAKE + 3 * _AN, dO=FAKE + 4 * _AN, L=FAKE + 5 * _AN,
             dQ=FAKE + 6 * _AN, dK=FAKE + 7 * _AN, dV=FAKE + 8 * _AN)
    a.update(case)
    st = mm.load_library().mm_attention_bwd(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["L"], a["dQ"], a["dK"],
                                            a["dV"], 2, 16, 64, 1, 0.125, None)
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()


# ------------------------------------------------------------------ FFMA stream-K tail

def _ffma_tail(M, N, K, sms, max_pct=85):
    """The documented rule of the FFMA path's stream-K tail: 128 x 128 tiles, k-steps of 32, one
    CTA per SM; the last wave's tiles (if at most max_pct % of a wave) split over at most `sms`
    shares of >= 8 k-steps, each no longer than one tile's K range.  None = no tail."""
    tn, T, KT = -(-N // 128), -(-M // 128) * -(-N // 128), -(-K // 32)
    rem = T % sms
    if rem == 0 or rem * 100 > sms * max_pct:
        return None
    I = rem * KT
    sk = min(I // 8, sms)
    if sk < rem or sk < 2:
        return None
    return dict(T=T, KT=KT, dp=T - rem, rem=rem, sk=sk, I=I)


def _cover(t):
    """Every k-step of every tail tile in exactly one share, every share in at most two tiles
    (its workspace slots 2j, 2j + 1), and the CTAs the reduce kernel visits for tile u (the
    shares holding its first and last k-step and those between) are exactly those covering u."""
    KT, I, sk = t["KT"], t["I"], t["sk"]
    seen = [[] for _ in range(t["rem"])]
    for j in range(sk):
        s, e = j * I // sk, (j + 1) * I // sk
        assert e - s >= 8
        tiles = list(range(s // KT, (e - 1) // KT + 1))
        assert len(tiles) <= 2
        for q, u in enumerate(tiles):
            lo, hi = max(s, u * KT), min(e, (u + 1) * KT)
            seen[u].append((lo, hi, j, 2 * j + q))
    for u, pieces in enumerate(seen):
        assert pieces[0][0] == u * KT and pieces[-1][1] == (u + 1) * KT
        assert all(a[1] == b[0] for a, b in zip(pieces, pieces[1:]))  # contiguous, in K order
        cta_of = lambda i: ((i + 1) * sk + I - 1) // I - 1
        ja, jb = cta_of(u * KT), cta_of((u + 1) * KT - 1)
        assert [p[2] for p in pieces] == list(range(ja, jb + 1))
        assert [p[3] for p in pieces] == [2 * j + (u - (j * I // sk) // KT) for j in range(ja, jb + 1)]


@pytest.mark.parametrize("shape", [(2048, 2048, 2048), (4096, 4096, 4096), (8192, 8192, 2048), (500, 700, 3000),
                                   (130, 260, 1000), (1700, 1650, 300), (1664, 1664, 300), (1664, 1664, 96),
                                   (2432, 2176, 200), (64, 3072, 768), (1, 1, 1), (129, 129, 257),
                                   (19456, 256, 24), (8192, 2048, 8192)])
@pytest.mark.parametrize("sms", [152, 148, 7])
def test_ffma_stream_k_plan(shape, sms):
    mm.load_library()
    t = _ffma_tail(*shape, sms)
    sk, floats = mm.mm_gemm_f32_split_plan_ex(*shape, sms, path=mm.MM_GEMM_FFMA)
    if t is None:
        assert (sk, floats) == (1, 0)
        return
    assert (sk, floats) == (-1, 2 * t["sk"] * 128 * 128)
    _cover(t)


def test_ffma_stream_k_plan_on_the_bench_shape():
    # 2048^2: 256 tiles on 152 SMs, a last wave of 104 tiles (68%): 152 whole tiles, then
    # 104 x 64 k-steps cut into 152 shares of 43-44 k-steps, two 64 KiB slots per CTA
    t = _ffma_tail(2048, 2048, 2048, 152)
    assert (t["dp"], t["rem"], t["sk"], t["I"]) == (152, 104, 152, 6656)
    mm.load_library()
    assert mm.mm_gemm_f32_split_plan_ex(2048, 2048, 2048, 152, path=mm.MM_GEMM_FFMA) == (-1, 2 * 152 * 16384)
    # the automatic path keeps its own plan (no split on CTA pairs at 2048^3)
    assert mm.mm_gemm_f32_split_plan_ex(2048, 2048, 2048, 152) == mm.mm_gemm_f32_split_plan(2048, 2048, 2048, 152)


@pytest.mark.parametrize("opts,splitk", [((2, 0, 0), 0), ((3, 0, 0), 0), ((1, 4, 0), 0), ((1, 0, 2), 0),
                                         ((0, 1, 0), 0), ((1, 0, 0), 2), ((1, 0, 0), -2), ((1, 0, 0), 16)])
def test_ffma_stream_k_refusals(lib, opts, splitk):
    # split entry points take path 0 or 1 with opts.tile = opts.splitk = 0; the FFMA path takes
    # splitk -1, 0 or 1: every other request is refused before any device call
    o = mm.GemmOpts(*opts)
    st = lib.mm_gemm_f32_splitk_ex(0, 0, 64, 64, 256, FAKE, 256, FAKE + 0x20000, 64, FAKE + 0x40000, 64, splitk,
                                   FAKE + 0x100000, 1 << 20, None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG, lib.mm_last_error()
    out = ctypes.c_int64(-1)
    if opts[0] != 1 or opts[1] or opts[2] or splitk not in (-1, 0, 1):
        assert lib.mm_gemm_f32_splitk_workspace_ex(64, 64, 256, splitk, ctypes.byref(o),
                                                   ctypes.byref(out)) in (mm.MM_ERR_INVALID_ARG,)
    if opts[0] != 1 or opts[1] or opts[2]:
        sk = ctypes.c_int(0)
        assert lib.mm_gemm_f32_split_plan_ex(64, 64, 256, 152, ctypes.byref(o), ctypes.byref(sk),
                                             ctypes.byref(out)) == mm.MM_ERR_INVALID_ARG


def test_ffma_stream_k_workspace_checks(lib):
    # the tail needs 2 x SMs x 128 x 128 floats; without a device the size cannot be known, so a
    # call that asks for no split needs none and a NULL workspace passes validation up to the
    # device check
    o = mm.GemmOpts(1, 0, 0)
    out = ctypes.c_int64(-1)
    assert lib.mm_gemm_f32_splitk_workspace_ex(2048, 2048, 2048, 1, ctypes.byref(o), ctypes.byref(out)) == mm.MM_OK
    assert out.value == 0
    st = lib.mm_gemm_f32_splitk_ex(0, 0, 64, 64, 256, FAKE, 256, FAKE + 0x20000, 64, FAKE + 0x40000, 64, 0,
                                   FAKE + 0x100004, 1 << 20, None, ctypes.byref(o))
    assert st == mm.MM_ERR_INVALID_ARG  # a misaligned workspace
