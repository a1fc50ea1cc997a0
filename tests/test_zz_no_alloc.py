"""The split-K GEMM entry point that allocates nothing, against the one that takes a workspace.

mm_gemm_f32_splitk_noalloc is for callers that cannot call cudaMalloc or hand
over a workspace where they multiply (their device memory belongs to another
allocator, or cudaMalloc's device-wide synchronisation is not acceptable there):
its partial tiles go to a scratch array the library holds in device memory.
Two calls in a row, with different shapes, layouts and splits, so that the
second call also shows that what the first left in the shared scratch does not
leak into its result.  This file sorts last, so a run that stops at the first
failure has run every other test first; it also passes alone in a fresh process,
where its first call sets the scratch up.
"""
import numpy as np
import pytest

import dense_packed_bit_gb300 as mm
from dense_packed_bit_gb300 import synth
from gpu_util import check_bound, empty_f32, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_packed_bit_gb300 import build
    build.build()
    mm.load_library()


def _stored(tA, tB, M, N, K, seed):
    A = synth.normal_f32(seed, (K, M) if tA else (M, K), 1.0)
    B = synth.normal_f32(seed + 1, (N, K) if tB else (K, N), 1.0)
    return A, B


def test_noalloc_splitk_matches_workspace_entry_two_calls(oracle):
    import torch
    calls = [  # (transA, transB, M, N, K, splitk): the GPT-2 MLP up-projection with the automatic
               # split, then a transposed product with an uneven explicit split
        (0, 0, 64, 3072, 768, 0),
        (1, 0, 96, 520, 1536, 7),
    ]
    for i, (tA, tB, M, N, K, splitk) in enumerate(calls):
        A, B = _stored(tA, tB, M, N, K, seed=4100 + 10 * i)
        dA, dB = to_dev(A), to_dev(B)
        need = mm.mm_gemm_f32_splitk_workspace(M, N, K, splitk)
        assert 0 < need <= mm.MM_SPLITK_NOALLOC_MAX_FLOATS

        c_noalloc = empty_f32((M, N))
        mm.mm_gemm_f32_splitk_noalloc(tA, tB, M, N, K, dA, A.shape[1], dB, B.shape[1], c_noalloc, N, splitk)
        mm.mm_check_device_error()

        ws = torch.full((need,), float("nan"), dtype=torch.float32, device=dA.device)
        c_ws = empty_f32((M, N))
        mm.mm_gemm_f32_splitk(tA, tB, M, N, K, dA, A.shape[1], dB, B.shape[1], c_ws, N, splitk, ws, need)
        mm.mm_check_device_error()

        ref, T = oracle.gemm(tA, tB, M, N, K, A, B)
        got, want = to_host(c_noalloc), to_host(c_ws)
        # the tolerance of every GEMM test, between the two entry points and against the oracle
        check_bound(got, want.astype(np.float64), T, f"call {i}: static scratch vs workspace")
        check_bound(got, ref, T, f"call {i}: static scratch vs oracle")


def test_noalloc_automatic_split_falls_back_when_scratch_is_small(oracle):
    # 4096^3: the automatic split (stream-K, 256 pair tiles on 76 pairs) needs more than the
    # static scratch; the entry point then runs the product unsplit instead of refusing it
    M = N = K = 4096
    assert mm.mm_gemm_f32_splitk_workspace(M, N, K, 0) > mm.MM_SPLITK_NOALLOC_MAX_FLOATS
    A = synth.normal_f32(4300, (M, K), 0.02)
    B = synth.normal_f32(4301, (K, N), 0.02)
    dA, dB = to_dev(A), to_dev(B)
    C = empty_f32((M, N))
    mm.mm_gemm_f32_splitk_noalloc(0, 0, M, N, K, dA, K, dB, N, C, N, 0)
    mm.mm_check_device_error()
    got = to_host(C)
    rng = np.random.default_rng(3)
    ii = np.concatenate([np.repeat([0, M - 1], N), rng.integers(0, M, 3000)])
    jj = np.concatenate([np.tile(np.arange(N), 2), rng.integers(0, N, 3000)])
    ref, T = oracle.gemm_at(0, 0, K, A, B, ii, jj)
    check_bound(got[ii, jj], ref, T, "4096^3 through the static-scratch entry point")


def test_noalloc_automatic_split_takes_the_most_slices_that_fit(oracle):
    # 128 x 12288 x 4096: the automatic split is 3 K slices (48 tiles on 152 SMs), 4.7M floats, more
    # than the scratch holds; the entry point then takes the 2 slices that fit (3.1M floats) rather
    # than no split
    M, N, K = 128, 12288, 4096
    assert mm.mm_gemm_f32_split_plan(M, N, K, 152)[0] == 3
    assert 3 * M * N > mm.MM_SPLITK_NOALLOC_MAX_FLOATS >= 2 * M * N
    A = synth.normal_f32(4400, (M, K), 0.02)
    B = synth.normal_f32(4401, (K, N), 0.02)
    dA, dB = to_dev(A), to_dev(B)
    C = empty_f32((M, N))
    mm.mm_gemm_f32_splitk_noalloc(0, 0, M, N, K, dA, K, dB, N, C, N, 0)
    mm.mm_check_device_error()
    got = to_host(C)
    # bit-identical to the workspace entry point's explicit 2-slice split (same kernels, same order)
    import torch
    need = mm.mm_gemm_f32_splitk_workspace(M, N, K, 2)
    ws = torch.empty((need,), dtype=torch.float32, device=dA.device)
    C2 = empty_f32((M, N))
    mm.mm_gemm_f32_splitk(0, 0, M, N, K, dA, K, dB, N, C2, N, 2, ws, need)
    mm.mm_check_device_error()
    assert np.array_equal(got.view(np.uint32), to_host(C2).view(np.uint32))
    rng = np.random.default_rng(4)
    ii = np.concatenate([np.repeat([0, M - 1], N), rng.integers(0, M, 3000)])
    jj = np.concatenate([np.tile(np.arange(N), 2), rng.integers(0, N, 3000)])
    ref, T = oracle.gemm_at(0, 0, K, A, B, ii, jj)
    check_bound(got[ii, jj], ref, T, "128 x 12288 x 4096 through the static-scratch entry point")
