// mm_api.cu -- the extern "C" boundary of libmm (declared in include/mm.h).
//
// Argument checks, variant selection and launches on the caller's stream.
// Every check happens before the first CUDA call, so argument errors are
// reported the same way on machines without a GPU.
#include "mm.h"
#include "mm_internal.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace {

thread_local std::string t_err;

mm_status fail(mm_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_err = buf;
    return s;
}

mm_status ok() {
    t_err.clear();
    return MM_OK;
}

mm_status cuda_fail(cudaError_t e, const char *what) {
    return fail(MM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// bytes spanned by a row-major rows x cols matrix with leading dimension ld
uint64_t span(int64_t rows, int64_t cols, int64_t ld, int64_t elem) {
    return (uint64_t)(((rows - 1) * ld + cols) * elem);
}

bool overlap(const void *a, uint64_t na, const void *b, uint64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// The library holds sm_103a code only; anything else is refused up front.
mm_status check_device() {
    static std::mutex mu;
    static int known[64] = {0};  // 0 unknown, 1 ok, 2 unsupported
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(MM_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(mu);
    if (known[dev] == 0) {
        int major = 0, minor = 0;
        e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        known[dev] = (major == 10 && minor == 3) ? 1 : 2;
        if (known[dev] == 2) return fail(MM_ERR_UNSUPPORTED, "libmm is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
    }
    if (known[dev] == 2) return fail(MM_ERR_UNSUPPORTED, "libmm is built for sm_103a only");
    return MM_OK;
}

mm_status check_codebook(const float *cb, int n = 4) {
    if (!cb) return fail(MM_ERR_INVALID_ARG, "codebook is NULL");
    for (int i = 0; i < n; ++i)
        if (!std::isfinite(cb[i])) return fail(MM_ERR_INVALID_ARG, "codebook[%d] is not finite", i);
    return MM_OK;
}

mm_status check_packed(const uint8_t *codes, const uint16_t *scales, const uint16_t *x, const float *y,
                       int64_t M, int64_t rows, int64_t cols, const float *cb) {
    if (!codes || !scales || !x || !y) return fail(MM_ERR_INVALID_ARG, "NULL pointer argument");
    if (M < 1 || rows < 1 || cols < 1)
        return fail(MM_ERR_INVALID_ARG, "sizes must be >= 1 (M=%lld rows=%lld cols=%lld)", (long long)M,
                    (long long)rows, (long long)cols);
    if (rows > ((int64_t)1 << 40) || cols > ((int64_t)1 << 40) || M > ((int64_t)1 << 31))
        return fail(MM_ERR_INVALID_ARG, "sizes too large");
    mm_status s = check_codebook(cb);
    if (s != MM_OK) return s;
    const uint64_t ybytes = (uint64_t)(M * rows * 4);
    if (overlap(y, ybytes, codes, (uint64_t)(rows * ((cols + 3) / 4))) || overlap(y, ybytes, scales, (uint64_t)rows * 2) ||
        overlap(y, ybytes, x, (uint64_t)(M * cols * 2)))
        return fail(MM_ERR_INVALID_ARG, "output overlaps an input");
    return MM_OK;
}

mm_status check_packed4(const uint8_t *codes, const uint16_t *scales, const uint16_t *x, const float *y,
                        int64_t rows, int64_t cols, const float *cb) {
    if (!codes || !scales || !x || !y) return fail(MM_ERR_INVALID_ARG, "NULL pointer argument");
    if (rows < 1 || cols < 1)
        return fail(MM_ERR_INVALID_ARG, "sizes must be >= 1 (rows=%lld cols=%lld)", (long long)rows, (long long)cols);
    if (rows > ((int64_t)1 << 40) || cols > ((int64_t)1 << 40)) return fail(MM_ERR_INVALID_ARG, "sizes too large");
    mm_status s = check_codebook(cb, 16);
    if (s != MM_OK) return s;
    const uint64_t ybytes = (uint64_t)(rows * 4);
    if (overlap(y, ybytes, codes, (uint64_t)(rows * ((cols + 1) / 2))) || overlap(y, ybytes, scales, (uint64_t)rows * 2) ||
        overlap(y, ybytes, x, (uint64_t)(cols * 2)))
        return fail(MM_ERR_INVALID_ARG, "output overlaps an input");
    return MM_OK;
}

// A product with few rows of C: the 3xTF32 kernel's 128 x 256 tiles would occupy at most a
// quarter of the SMs, so a few-rows kernel whose K range is split over a cluster keeps more of
// the GPU busy (64 x 3072 x 768 on GB300: measured against the 3xTF32 kernel's 12 tiles).
bool skinny_auto(int64_t M, int64_t N) {
    if (M > 64) return false;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return ((N + 255) / 256) * 4 <= sms;
}

}  // namespace

extern "C" {

int mm_version(void) { return 100; }

const char *mm_last_error(void) { return t_err.c_str(); }

mm_status mm_gemm_f32_ex(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                         const float *B, int64_t ldb, float *C, int64_t ldc, mm_stream_t stream,
                         const mm_gemm_opts *opts) {
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1))
        return fail(MM_ERR_INVALID_ARG, "transA/transB must be 0 or 1");
    if (M < 1 || N < 1 || K < 1)
        return fail(MM_ERR_INVALID_ARG, "M, N, K must be >= 1 (got %lld, %lld, %lld)", (long long)M, (long long)N,
                    (long long)K);
    if (!A || !B || !C) return fail(MM_ERR_INVALID_ARG, "NULL matrix pointer");
    const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;
    if (lda < a_cols) return fail(MM_ERR_INVALID_ARG, "lda=%lld < %lld", (long long)lda, (long long)a_cols);
    if (ldb < b_cols) return fail(MM_ERR_INVALID_ARG, "ldb=%lld < %lld", (long long)ldb, (long long)b_cols);
    if (ldc < N) return fail(MM_ERR_INVALID_ARG, "ldc=%lld < N=%lld", (long long)ldc, (long long)N);
    const uint64_t cb = span(M, N, ldc, 4);
    if (overlap(C, cb, A, span(a_rows, a_cols, lda, 4)) || overlap(C, cb, B, span(b_rows, b_cols, ldb, 4)))
        return fail(MM_ERR_INVALID_ARG, "C overlaps A or B");
    int path = MM_GEMM_AUTO;
    if (opts) {
        path = opts->path;
        if (path < MM_GEMM_AUTO || path > MM_GEMM_TF32X3) return fail(MM_ERR_INVALID_ARG, "unknown path %d", path);
    }
    const int tile = opts ? opts->tile : 0;
    const int splitk = opts ? opts->splitk : 0;
    if ((path == MM_GEMM_TF32X3 && (tile < 0 || tile > 4)) || (path == MM_GEMM_AUTO && (tile < 0 || tile > 3)))
        return fail(MM_ERR_INVALID_ARG, "3xTF32 tile must be 0 (automatic), 1 (two-stage), 2 (warp-specialised), "
                                        "3 (CTA pairs) or 4 (few rows, K split in a cluster; 3xTF32 path only)");
    if (path == MM_GEMM_FFMA && tile != 0 && tile != 4)
        return fail(MM_ERR_INVALID_ARG, "FFMA tile must be 0 (TMA-staged 128 x 128) or 4 (few rows, K split in a cluster)");
    if (splitk < 0 || splitk > 8 || (splitk != 0 && !((path == MM_GEMM_FFMA || path == MM_GEMM_TF32X3) && tile == 4)))
        return fail(MM_ERR_INVALID_ARG, "splitk is 0, or 1..8 with tile 4 (FFMA or 3xTF32)");
    mm_status s = check_device();
    if (s != MM_OK) return s;

    mm::GemmArgs g{transA, transB, M, N, K, A, lda, B, ldb, C, ldc};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (path == MM_GEMM_TF32X3 && tile == 4) {
        if (!mm::gemm_skinny_tc_supported(g))
            return fail(MM_ERR_INVALID_ARG, "3xTF32 tile 4 needs M <= 64, K <= %lld, 16-byte aligned A, B and lda, "
                                            "ldb multiples of 4", (long long)mm::kTf32x3MaxK);
        e = mm::launch_gemm_skinny_tc(g, splitk, st);
        if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
        return ok();
    }
    if ((path == MM_GEMM_FFMA && tile == 4) || (path == MM_GEMM_AUTO && tile == 0 && skinny_auto(M, N))) {
        // automatic: the tensor-core few-rows kernel where its operand rules and the 3xTF32 K
        // margin allow, else the FFMA one (any alignment, any K)
        e = path == MM_GEMM_AUTO && mm::gemm_skinny_tc_supported(g) ? mm::launch_gemm_skinny_tc(g, 0, st)
                                                                    : mm::launch_gemm_skinny(g, splitk, st);
        if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
        return ok();
    }
    if (path == MM_GEMM_TF32X3 && !mm::gemm_tf32x3_supported(g))
        return fail(MM_ERR_INVALID_ARG, "3xTF32 path needs 16-byte aligned A, B and lda, ldb multiples of 4");
    // beyond the 3xTF32 accuracy margin: refused when asked for, the FFMA kernels when automatic
    const bool long_k = K > mm::kTf32x3MaxK;
    if (long_k && (path == MM_GEMM_TF32X3 || (path == MM_GEMM_AUTO && tile != 0)))
        return fail(MM_ERR_INVALID_ARG, "3xTF32 needs K <= %lld (its accuracy margin), got K=%lld",
                    (long long)mm::kTf32x3MaxK, (long long)K);
    if ((path == MM_GEMM_TF32X3 || path == MM_GEMM_AUTO) && !long_k && mm::gemm_tf32x3_supported(g))
        // automatic: CTA pairs (256-row tiles) once M fills them, one CTA per 128-row tile below that
        e = tile == 1 ? mm::launch_gemm_tf32x3(g, st)
                      : mm::launch_gemm_tf32x3_ws(g, (tile == 3 || (tile == 0 && M > 128)) ? 1 : 0, st);
    else if (mm::gemm_ffma_supported(g)) e = mm::launch_gemm_ffma(g, 0, st);
    else if (path == MM_GEMM_FFMA || path == MM_GEMM_AUTO) e = mm::launch_gemm_simple(g, st);
    else e = cudaErrorNotSupported;
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return ok();
}

mm_status mm_gemm_f32(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                      const float *B, int64_t ldb, float *C, int64_t ldc, mm_stream_t stream) {
    return mm_gemm_f32_ex(transA, transB, M, N, K, A, lda, B, ldb, C, ldc, stream, nullptr);
}

}  // extern "C"

namespace {

// The split a split-K call uses and the workspace it needs: `splitk` itself when given (1..16
// slices, -1 stream-K), else the automatic choice for the tile shape the call runs (CTA pairs
// when M > 128).  Stream-K sizes depend on the SM count, so they query the device.
// A split whose every accumulation stays within the 3xTF32 accuracy margin (K slices of at most
// kTf32x3MaxK; stream-K segments never exceed K).  Any other split runs the FFMA kernel unsplit,
// needing no workspace.
bool split_within_margin(int64_t K, int sk) {
    return sk == mm::kStreamK ? K <= mm::kTf32x3MaxK : (K + sk - 1) / sk <= mm::kTf32x3MaxK;
}

mm_status resolve_splitk(int64_t M, int64_t N, int64_t K, int splitk, int *out, int64_t *floats) {
    if (splitk < -1 || splitk > 16)
        return fail(MM_ERR_INVALID_ARG, "splitk must be 0 (automatic), 1..16 (slices) or -1 (stream-K)");
    const int pair = M > 128 ? 1 : 0;
    if (splitk > 0) {
        *out = (int)(splitk > (K + 15) / 16 ? (K + 15) / 16 : splitk);
        *floats = split_within_margin(K, *out) ? mm::gemm_splitk_workspace_floats(M, N, K, pair, *out, 0) : 0;
        return MM_OK;
    }
    mm_status s = check_device();
    if (s != MM_OK) return s;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    *out = splitk == mm::kStreamK ? mm::kStreamK : mm::gemm_splitk_auto(M, N, K, pair, sms);
    *floats = split_within_margin(K, *out) ? mm::gemm_splitk_workspace_floats(M, N, K, pair, *out, sms) : 0;
    return MM_OK;
}

// The FFMA path's split: none (splitk 1), or the stream-K tail of the TMA-staged FFMA kernel
// (0: when the last wave is at most kFfmaStreamKAutoTailPct % full; -1: whenever there is one).
mm_status resolve_ffma_split(int64_t M, int64_t N, int64_t K, int splitk, int sms, mm::FfmaStreamKPlan *plan) {
    *plan = mm::FfmaStreamKPlan{};
    if (splitk < -1 || splitk > 1)
        return fail(MM_ERR_INVALID_ARG, "FFMA path: splitk must be 0 (automatic), 1 (no split) or -1 (stream-K tail)");
    if (splitk != 1)
        mm::ffma_streamk_plan(M, N, K, sms, splitk == mm::kStreamK ? 100 : mm::kFfmaStreamKAutoTailPct, plan);
    return MM_OK;
}

// The path of a split call's options: MM_GEMM_AUTO or MM_GEMM_FFMA, tile and splitk fields 0.
mm_status split_path(const mm_gemm_opts *opts, int *path) {
    *path = MM_GEMM_AUTO;
    if (!opts) return MM_OK;
    if (opts->path != MM_GEMM_AUTO && opts->path != MM_GEMM_FFMA)
        return fail(MM_ERR_INVALID_ARG, "split entry points take path 0 (automatic) or 1 (FFMA), got %d", opts->path);
    if (opts->tile != 0 || opts->splitk != 0)
        return fail(MM_ERR_INVALID_ARG, "split entry points take opts.tile = 0 and opts.splitk = 0");
    *path = opts->path;
    return MM_OK;
}

int device_sms(mm_status *st) {
    *st = check_device();
    if (*st != MM_OK) return 0;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) *st = cuda_fail(e, "cudaDeviceGetAttribute");
    return sms;
}

}  // namespace

extern "C" {

mm_status mm_gemm_f32_split_plan_ex(int64_t M, int64_t N, int64_t K, int sms, const mm_gemm_opts *opts,
                                    int *splitk, int64_t *workspace_floats) {
    if (!splitk || !workspace_floats) return fail(MM_ERR_INVALID_ARG, "NULL output");
    if (M < 1 || N < 1 || K < 1) return fail(MM_ERR_INVALID_ARG, "M, N, K must be >= 1");
    if (sms < 2) return fail(MM_ERR_INVALID_ARG, "sms must be >= 2 (got %d)", sms);
    int path = MM_GEMM_AUTO;
    mm_status s = split_path(opts, &path);
    if (s != MM_OK) return s;
    if (path == MM_GEMM_AUTO) return mm_gemm_f32_split_plan(M, N, K, sms, splitk, workspace_floats);
    mm::FfmaStreamKPlan plan;
    s = resolve_ffma_split(M, N, K, 0, sms, &plan);
    if (s != MM_OK) return s;
    *splitk = plan.sk_ctas ? mm::kStreamK : 1;
    *workspace_floats = plan.workspace_floats;
    return ok();
}

mm_status mm_gemm_f32_splitk_workspace_ex(int64_t M, int64_t N, int64_t K, int splitk, const mm_gemm_opts *opts,
                                          int64_t *floats) {
    if (!floats) return fail(MM_ERR_INVALID_ARG, "floats is NULL");
    if (M < 1 || N < 1 || K < 1) return fail(MM_ERR_INVALID_ARG, "M, N, K must be >= 1");
    int path = MM_GEMM_AUTO;
    mm_status s = split_path(opts, &path);
    if (s != MM_OK) return s;
    if (path == MM_GEMM_AUTO) return mm_gemm_f32_splitk_workspace(M, N, K, splitk, floats);
    if (splitk < -1 || splitk > 1)
        return fail(MM_ERR_INVALID_ARG, "FFMA path: splitk must be 0 (automatic), 1 (no split) or -1 (stream-K tail)");
    int sms = 0;
    if (splitk != 1) {
        sms = device_sms(&s);
        if (s != MM_OK) return s;
    }
    mm::FfmaStreamKPlan plan;
    s = resolve_ffma_split(M, N, K, splitk, sms, &plan);
    if (s != MM_OK) return s;
    *floats = plan.workspace_floats;
    return ok();
}

mm_status mm_gemm_f32_split_plan(int64_t M, int64_t N, int64_t K, int sms, int *splitk,
                                 int64_t *workspace_floats) {
    if (!splitk || !workspace_floats) return fail(MM_ERR_INVALID_ARG, "NULL output");
    if (M < 1 || N < 1 || K < 1) return fail(MM_ERR_INVALID_ARG, "M, N, K must be >= 1");
    if (sms < 2) return fail(MM_ERR_INVALID_ARG, "sms must be >= 2 (got %d)", sms);
    const int pair = M > 128 ? 1 : 0;
    *splitk = mm::gemm_splitk_auto(M, N, K, pair, sms);
    *workspace_floats = mm::gemm_splitk_workspace_floats(M, N, K, pair, *splitk, sms);
    return ok();
}

mm_status mm_gemm_f32_splitk_workspace(int64_t M, int64_t N, int64_t K, int splitk, int64_t *floats) {
    if (!floats) return fail(MM_ERR_INVALID_ARG, "floats is NULL");
    if (M < 1 || N < 1 || K < 1) return fail(MM_ERR_INVALID_ARG, "M, N, K must be >= 1");
    int sk = 1;
    mm_status s = resolve_splitk(M, N, K, splitk, &sk, floats);
    if (s != MM_OK) return s;
    return ok();
}

}  // extern "C"

namespace {

// the split GEMM of mm_gemm_f32_splitk, with the linear layer's bias and activation
mm_status gemm_splitk_impl(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                           const float *B, int64_t ldb, const float *bias, int act, float *C, int64_t ldc, int splitk,
                           float *workspace, int64_t workspace_floats, mm_stream_t stream,
                           const mm_gemm_opts *opts = nullptr) {
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1))
        return fail(MM_ERR_INVALID_ARG, "transA/transB must be 0 or 1");
    if (M < 1 || N < 1 || K < 1)
        return fail(MM_ERR_INVALID_ARG, "M, N, K must be >= 1 (got %lld, %lld, %lld)", (long long)M, (long long)N,
                    (long long)K);
    if (!A || !B || !C) return fail(MM_ERR_INVALID_ARG, "NULL matrix pointer");
    const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;
    if (lda < a_cols) return fail(MM_ERR_INVALID_ARG, "lda=%lld < %lld", (long long)lda, (long long)a_cols);
    if (ldb < b_cols) return fail(MM_ERR_INVALID_ARG, "ldb=%lld < %lld", (long long)ldb, (long long)b_cols);
    if (ldc < N) return fail(MM_ERR_INVALID_ARG, "ldc=%lld < N=%lld", (long long)ldc, (long long)N);
    const uint64_t cb = span(M, N, ldc, 4);
    if (overlap(C, cb, A, span(a_rows, a_cols, lda, 4)) || overlap(C, cb, B, span(b_rows, b_cols, ldb, 4)))
        return fail(MM_ERR_INVALID_ARG, "C overlaps A or B");
    if (act != MM_ACT_NONE && act != MM_ACT_GELU_TANH) return fail(MM_ERR_INVALID_ARG, "unknown act %d", act);
    if (bias && overlap(C, cb, bias, (uint64_t)N * 4)) return fail(MM_ERR_INVALID_ARG, "C overlaps bias");
    if (splitk < -1 || splitk > 16)
        return fail(MM_ERR_INVALID_ARG, "splitk must be 0 (automatic), 1..16 (slices) or -1 (stream-K)");
    if (workspace_floats < 0) return fail(MM_ERR_INVALID_ARG, "workspace_floats < 0");
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15))
        return fail(MM_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    if (workspace) {
        const uint64_t wb = (uint64_t)workspace_floats * 4;
        if (overlap(workspace, wb, A, span(a_rows, a_cols, lda, 4)) || overlap(workspace, wb, B, span(b_rows, b_cols, ldb, 4)) ||
            overlap(workspace, wb, C, cb))
            return fail(MM_ERR_INVALID_ARG, "workspace overlaps A, B or C");
    }
    int path = MM_GEMM_AUTO;
    mm_status s = split_path(opts, &path);
    if (s != MM_OK) return s;
    if (path == MM_GEMM_FFMA) {
        // the TMA-staged FFMA kernel, with its stream-K tail when the split asks for one
        if (splitk < -1 || splitk > 1)
            return fail(MM_ERR_INVALID_ARG, "FFMA path: splitk must be 0 (automatic), 1 (no split) or -1 (stream-K tail)");
        int sms = 0;
        if (splitk != 1) {
            sms = device_sms(&s);
            if (s != MM_OK) return s;
        }
        mm::FfmaStreamKPlan plan;
        s = resolve_ffma_split(M, N, K, splitk, sms, &plan);
        if (s != MM_OK) return s;
        if (plan.workspace_floats > 0 && (!workspace || workspace_floats < plan.workspace_floats))
            return fail(MM_ERR_INVALID_ARG, "workspace of %lld floats needed (FFMA stream-K tail)",
                        (long long)plan.workspace_floats);
        s = check_device();
        if (s != MM_OK) return s;
        mm::GemmArgs g{transA, transB, M, N, K, A, lda, B, ldb, C, ldc};
        g.bias = bias;
        g.act = act;
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        const cudaError_t e = !mm::gemm_ffma_supported(g) ? mm::launch_gemm_simple(g, st)
                              : plan.sk_ctas               ? mm::launch_gemm_ffma_streamk(g, plan, workspace, st)
                                                           : mm::launch_gemm_ffma(g, 0, st);
        if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
        return ok();
    }
    int sk = 1;
    int64_t need = 0;
    s = resolve_splitk(M, N, K, splitk, &sk, &need);
    if (s != MM_OK) return s;
    if (need > 0 && (!workspace || workspace_floats < need))
        return fail(MM_ERR_INVALID_ARG, "workspace of %lld floats needed (%s)", (long long)need,
                    sk == mm::kStreamK ? "stream-K" : "K slices");
    s = check_device();
    if (s != MM_OK) return s;
    mm::GemmArgs g{transA, transB, M, N, K, A, lda, B, ldb, C, ldc};
    g.bias = bias;
    g.act = act;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    // operands TMA cannot describe take the unsplit general kernel, and a split whose slices would
    // exceed the 3xTF32 accuracy margin the unsplit FFMA kernel (the workspace is then unused)
    if (mm::gemm_tf32x3_supported(g) && split_within_margin(K, sk))
        e = mm::launch_gemm_tf32x3_ws_splitk(g, M > 128 ? 1 : 0, sk, workspace, st);
    else if (mm::gemm_ffma_supported(g)) e = mm::launch_gemm_ffma(g, 0, st);
    else e = mm::launch_gemm_simple(g, st);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return ok();
}

}  // namespace

extern "C" {

mm_status mm_gemm_f32_splitk(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                             const float *B, int64_t ldb, float *C, int64_t ldc, int splitk, float *workspace,
                             int64_t workspace_floats, mm_stream_t stream) {
    return gemm_splitk_impl(transA, transB, M, N, K, A, lda, B, ldb, nullptr, MM_ACT_NONE, C, ldc, splitk, workspace,
                            workspace_floats, stream);
}

mm_status mm_gemm_f32_splitk_ex(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A,
                                int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc, int splitk,
                                float *workspace, int64_t workspace_floats, mm_stream_t stream,
                                const mm_gemm_opts *opts) {
    return gemm_splitk_impl(transA, transB, M, N, K, A, lda, B, ldb, nullptr, MM_ACT_NONE, C, ldc, splitk, workspace,
                            workspace_floats, stream, opts);
}

mm_status mm_gemm_f32_bias_act_splitk(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A,
                                      int64_t lda, const float *B, int64_t ldb, const float *bias, int act, float *C,
                                      int64_t ldc, int splitk, float *workspace, int64_t workspace_floats,
                                      mm_stream_t stream) {
    return gemm_splitk_impl(transA, transB, M, N, K, A, lda, B, ldb, bias, act, C, ldc, splitk, workspace,
                            workspace_floats, stream);
}

mm_status mm_gemm_f32_bias_act(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                               const float *B, int64_t ldb, const float *bias, int act, float *C, int64_t ldc,
                               mm_stream_t stream) {
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1))
        return fail(MM_ERR_INVALID_ARG, "transA/transB must be 0 or 1");
    if (M < 1 || N < 1 || K < 1)
        return fail(MM_ERR_INVALID_ARG, "M, N, K must be >= 1 (got %lld, %lld, %lld)", (long long)M, (long long)N,
                    (long long)K);
    if (!A || !B || !C) return fail(MM_ERR_INVALID_ARG, "NULL matrix pointer");
    if (act != MM_ACT_NONE && act != MM_ACT_GELU_TANH) return fail(MM_ERR_INVALID_ARG, "unknown act %d", act);
    const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;
    const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;
    if (lda < a_cols) return fail(MM_ERR_INVALID_ARG, "lda=%lld < %lld", (long long)lda, (long long)a_cols);
    if (ldb < b_cols) return fail(MM_ERR_INVALID_ARG, "ldb=%lld < %lld", (long long)ldb, (long long)b_cols);
    if (ldc < N) return fail(MM_ERR_INVALID_ARG, "ldc=%lld < N=%lld", (long long)ldc, (long long)N);
    const uint64_t cb = span(M, N, ldc, 4);
    if (overlap(C, cb, A, span(a_rows, a_cols, lda, 4)) || overlap(C, cb, B, span(b_rows, b_cols, ldb, 4)))
        return fail(MM_ERR_INVALID_ARG, "C overlaps A or B");
    if (bias && overlap(C, cb, bias, (uint64_t)N * 4)) return fail(MM_ERR_INVALID_ARG, "C overlaps bias");
    mm_status s = check_device();
    if (s != MM_OK) return s;
    mm::GemmArgs g{transA, transB, M, N, K, A, lda, B, ldb, C, ldc};
    g.bias = bias;
    g.act = act;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // few rows: the cluster split-K kernels (tensor cores where TMA can describe the operands and K
    // is within the 3xTF32 margin, else FFMA); else the warp-specialised 3xTF32 kernel when TMA can
    // describe the operands, else the plain tiled one
    // (a K beyond the 3xTF32 accuracy margin: the TMA-staged FFMA kernel)
    const bool long_k = K > mm::kTf32x3MaxK;
    cudaError_t e = skinny_auto(M, N) && mm::gemm_skinny_tc_supported(g) ? mm::launch_gemm_skinny_tc(g, 0, st)
                    : skinny_auto(M, N)                           ? mm::launch_gemm_skinny(g, 0, st)
                    : !long_k && mm::gemm_tf32x3_supported(g) ? mm::launch_gemm_tf32x3_ws(g, M > 128 ? 1 : 0, st)
                    : mm::gemm_ffma_supported(g)               ? mm::launch_gemm_ffma(g, 0, st)
                                                               : mm::launch_gemm_simple(g, st);
    if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
    return ok();
}

mm_status mm_gemm_f32_splitk_noalloc(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A,
                                     int64_t lda, const float *B, int64_t ldb, float *C, int64_t ldc, int splitk,
                                     mm_stream_t stream) {
    static_assert(mm::kSplitkStaticFloats == MM_SPLITK_NOALLOC_MAX_FLOATS, "the header states the scratch size");
    // the cheap checks first, so that bad arguments never reach a CUDA call
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1))
        return fail(MM_ERR_INVALID_ARG, "transA/transB must be 0 or 1");
    if (M < 1 || N < 1 || K < 1)
        return fail(MM_ERR_INVALID_ARG, "M, N, K must be >= 1 (got %lld, %lld, %lld)", (long long)M, (long long)N,
                    (long long)K);
    if (!A || !B || !C) return fail(MM_ERR_INVALID_ARG, "NULL matrix pointer");
    if (splitk < 0 || splitk > 16) return fail(MM_ERR_INVALID_ARG, "splitk must be 0 (automatic) or 1..16");
    int64_t need = 0;
    mm_status s = mm_gemm_f32_splitk_workspace(M, N, K, splitk, &need);
    if (s != MM_OK) return s;
    if (!splitk && need > mm::kSplitkStaticFloats) {
        // the automatic split does not fit the scratch: K slices take the most slices that fit (no
        // split below two); stream-K (one partial tile per CTA of a large product) runs unsplit
        int sk = 1;
        int64_t auto_need = 0;
        s = resolve_splitk(M, N, K, 0, &sk, &auto_need);
        if (s != MM_OK) return s;
        const int64_t fit = mm::kSplitkStaticFloats / (M * N);
        splitk = (sk > 1 && fit >= 2) ? (int)(fit < sk ? fit : sk) : 1;
        s = mm_gemm_f32_splitk_workspace(M, N, K, splitk, &need);
        if (s != MM_OK) return s;
    }
    if (need > mm::kSplitkStaticFloats)
        return fail(MM_ERR_INVALID_ARG,
                    "split-K of %lld x %lld needs %lld floats of scratch; the library's static scratch holds %lld "
                    "(pass a smaller splitk, or a workspace to mm_gemm_f32_splitk)",
                    (long long)M, (long long)N, (long long)need, (long long)mm::kSplitkStaticFloats);
    float *scratch = nullptr;
    int64_t cap = 0;
    if (need > 0) {
        s = check_device();
        if (s != MM_OK) return s;
        const cudaError_t e = mm::splitk_static_scratch(&scratch, &cap);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the split-K scratch");
    }
    return mm_gemm_f32_splitk(transA, transB, M, N, K, A, lda, B, ldb, C, ldc, splitk, scratch, cap, stream);
}

mm_status mm_gemv_packed2_ex(const uint8_t *codes, const uint16_t *scales, const uint16_t *x, float *y, int64_t rows,
                             int64_t cols, const float codebook[4], mm_stream_t stream, const mm_gemv_opts *opts) {
    mm_status s = check_packed(codes, scales, x, y, 1, rows, cols, codebook);
    if (s != MM_OK) return s;
    mm::GemvConfig cfg{0, 0, 0, 0, 1, 0, 0, -1, 0};
    bool auto_rl = false, auto_w = false, spread = false;  // register-load kernel: automatic shape
    if (opts) {
        cfg.split = opts->split;
        cfg.rows_per_lane = opts->rows_per_lane;
        cfg.warps = opts->warps;
        cfg.dequant = opts->dequant;
        cfg.pdl = opts->pdl;
        cfg.weights_static = opts->weights_static;
        cfg.independent = opts->independent;
        cfg.staging = opts->staging;
    }
    const bool affine = mm::codebook_is_affine(codebook);
    mm::PackedArgs a{codes, scales, x, y, 1, rows, cols, {codebook[0], codebook[1], codebook[2], codebook[3]}};
    // automatic decode, by measurement on GB300 (12,288 x 1,536): the SIMT affine decode is the
    // fastest both for independent calls (bound by issue throughput) and for chained ones
    if (cfg.dequant == MM_DEQ_AUTO) cfg.dequant = affine ? MM_DEQ_AFFINE : MM_DEQ_SELECT;
    if (cfg.dequant < MM_DEQ_SELECT || cfg.dequant > MM_DEQ_MXF4)
        return fail(MM_ERR_INVALID_ARG, "unknown dequant %d", cfg.dequant);
    if (cfg.dequant != MM_DEQ_SELECT && !affine)
        return fail(MM_ERR_INVALID_ARG, "affine decode needs codebook[c] == codebook[0] + c*(codebook[1]-codebook[0])");
    // automatic staging: the TMA-staged affine kernel is the fastest measured, for independent
    // calls (three 128-row blocks per CTA) and chained ones (one block per CTA, its weights
    // loaded before the wait on the previous kernel when they are promised static); the staged
    // tensor-core decode measured slower than register loads
    if (cfg.staging < 0)
        cfg.staging = (cfg.dequant == MM_DEQ_AFFINE && !cfg.split && !cfg.warps && mm::gemv_rows_supported(a)) ? 1 : 0;
    if (cfg.staging != 0 && cfg.staging != 1) return fail(MM_ERR_INVALID_ARG, "staging must be 0 or 1");
    if (cfg.staging && cfg.dequant < MM_DEQ_FP8 &&
        !(cfg.dequant == MM_DEQ_MMA && mm::gemv_tma_supported(a)) &&
        !(cfg.dequant == MM_DEQ_AFFINE && mm::gemv_rows_supported(a)))
        return fail(MM_ERR_INVALID_ARG, "staging needs the affine or tensor-core decode, cols %% 512 == 0, cols <= 4096 and 16-byte aligned codes and x");
    if (cfg.dequant == MM_DEQ_MXF4) {
        // 127 rows per tile and CTA-wide roles fix split and warps; rows_per_lane counts the
        // tiles a CTA multiplies (automatic: 1)
        if (!mm::gemv_mxf4_supported(a))
            return fail(MM_ERR_INVALID_ARG, "fp4 tensor-core decode needs cols %% 512 == 0, cols <= 12800 and 16-byte aligned codes");
        if (cfg.split || cfg.warps || cfg.staging > 0)
            return fail(MM_ERR_INVALID_ARG, "split, warps and staging are fixed by the fp4 tensor-core decode");
        if (cfg.rows_per_lane < 0 || cfg.rows_per_lane > 64)
            return fail(MM_ERR_INVALID_ARG, "rows_per_lane (127-row tiles per CTA) must be 0..64 with the fp4 tensor-core decode");
        cfg.blocks_per_cta = cfg.rows_per_lane;  // 0: one tile per pipeline (three)
    } else if (cfg.dequant == MM_DEQ_TC) {
        // 127 rows per tile and CTA-wide roles fix split and warps; rows_per_lane counts the
        // tiles a CTA multiplies (automatic: 1)
        if (!mm::gemv_tc_supported(a))
            return fail(MM_ERR_INVALID_ARG, "tcgen05 decode needs cols %% 512 == 0, cols <= 8192 and 16-byte aligned codes and x");
        if (cfg.split || cfg.warps) return fail(MM_ERR_INVALID_ARG, "split and warps are fixed by the tcgen05 decode");
        if (cfg.rows_per_lane < 0 || cfg.rows_per_lane > 64)
            return fail(MM_ERR_INVALID_ARG, "rows_per_lane (127-row tiles per CTA) must be 0..64 with the tcgen05 decode");
        cfg.blocks_per_cta = cfg.rows_per_lane ? cfg.rows_per_lane : 1;
    } else if (cfg.dequant == MM_DEQ_FP8) {
        // one warp per 256-field slab, code rows always staged by TMA; rows_per_lane counts
        // the 64-row blocks a CTA streams (automatic: 2 for independent calls, 1 otherwise)
        if (!mm::gemv_fp8_supported(a))
            return fail(MM_ERR_INVALID_ARG, "fp8 decode needs cols %% 512 == 0, cols <= 4096 and 16-byte aligned codes and x");
        if (cfg.split || cfg.warps) return fail(MM_ERR_INVALID_ARG, "split and warps are fixed by the fp8 decode");
        if (cfg.rows_per_lane < 0 || cfg.rows_per_lane > 64)
            return fail(MM_ERR_INVALID_ARG, "rows_per_lane (64-row blocks per CTA) must be 0..64 with the fp8 decode");
        cfg.blocks_per_cta = cfg.rows_per_lane ? cfg.rows_per_lane : (cfg.independent ? 2 : 1);
    } else if (cfg.dequant == MM_DEQ_AFFINE && cfg.staging) {
        // one lane per row of 128-row TMA blocks, eight warps splitting K; rows_per_lane counts
        // the blocks a CTA streams (automatic: 2 for independent calls, 1 otherwise)
        if (cfg.split || cfg.warps) return fail(MM_ERR_INVALID_ARG, "split and warps are fixed by staging");
        if (cfg.rows_per_lane < 0 || cfg.rows_per_lane > 64)
            return fail(MM_ERR_INVALID_ARG, "rows_per_lane (128-row blocks per CTA) must be 0..64 with staging");
        cfg.blocks_per_cta = cfg.rows_per_lane ? cfg.rows_per_lane : (cfg.independent ? 3 : 1);
    } else if (cfg.dequant == MM_DEQ_MMA && cfg.staging) {
        // one warp per 256-field slab fixes split and warps; rows_per_lane counts the 64-row
        // blocks a CTA streams (automatic: 4 for independent calls, 1 otherwise)
        if (cfg.split || cfg.warps) return fail(MM_ERR_INVALID_ARG, "split and warps are fixed by staging");
        if (cfg.rows_per_lane < 0 || cfg.rows_per_lane > 64)
            return fail(MM_ERR_INVALID_ARG, "rows_per_lane (64-row blocks per CTA) must be 0..64 with staging");
        cfg.blocks_per_cta = cfg.rows_per_lane ? cfg.rows_per_lane : (cfg.independent ? 4 : 1);
    } else if (cfg.dequant == MM_DEQ_MMA) {
        if (!mm::gemv_mma_supported(a))
            return fail(MM_ERR_INVALID_ARG, "tensor-core decode needs cols %% 256 == 0, cols <= 32768, 16-byte aligned codes and x");
        if (!cfg.split) cfg.split = 3;
        if (!cfg.rows_per_lane) cfg.rows_per_lane = 2;
        if (!cfg.warps) cfg.warps = 2 * cfg.split;
        if (cfg.split != 1 && cfg.split != 2 && cfg.split != 3 && cfg.split != 4 && cfg.split != 6)
            return fail(MM_ERR_INVALID_ARG, "split must be 1, 2, 3, 4 or 6 for the tensor-core decode");
        if (cfg.rows_per_lane != 1 && cfg.rows_per_lane != 2 && cfg.rows_per_lane != 4)
            return fail(MM_ERR_INVALID_ARG, "rows_per_lane must be 1, 2 or 4 for the tensor-core decode");
        if (cfg.warps < 1 || cfg.warps > (cfg.rows_per_lane >= 2 ? 8 : 16) || cfg.warps % cfg.split)
            return fail(MM_ERR_INVALID_ARG, "warps must be a multiple of split, at most 16 (8 with rows_per_lane 2 or 4)");
    } else {
        // automatic register-load shape, by measurement on GB300: 16 lanes per row for rows of
        // 8192 fields or more (1,536 x 12,288: 2.0 us per independent call against 2.3 with 8);
        // a call that is not promised independent runs alone, so its rows are spread until the
        // grid covers the SMs (1,536 x 12,288 chained: 9 us per call against 31 with 12 CTAs)
        auto_rl = !cfg.rows_per_lane;
        auto_w = !cfg.warps;
        spread = !cfg.independent && (auto_rl || auto_w);
        if (!cfg.split) cfg.split = a.cols >= 8192 ? 16 : 8;
        if (auto_rl) cfg.rows_per_lane = 4;
        if (auto_w) cfg.warps = 8;
        if (cfg.split != 4 && cfg.split != 8 && cfg.split != 16) return fail(MM_ERR_INVALID_ARG, "split must be 4, 8 or 16");
        if (cfg.rows_per_lane != 1 && cfg.rows_per_lane != 2 && cfg.rows_per_lane != 4)
            return fail(MM_ERR_INVALID_ARG, "rows_per_lane must be 1, 2 or 4");
        if (cfg.warps < 1 || cfg.warps > 16) return fail(MM_ERR_INVALID_ARG, "warps must be 1..16");
    }
    if (cfg.pdl != 0 && cfg.pdl != 1) return fail(MM_ERR_INVALID_ARG, "pdl must be 0 or 1");
    if (cfg.weights_static != 0 && cfg.weights_static != 1) return fail(MM_ERR_INVALID_ARG, "weights_static must be 0 or 1");
    if (cfg.independent != 0 && cfg.independent != 1) return fail(MM_ERR_INVALID_ARG, "independent must be 0 or 1");
    s = check_device();
    if (s != MM_OK) return s;
    if (spread) {
        int dev = 0, sms = 152;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        auto ctas = [&] {
            const int64_t per = (int64_t)cfg.warps * (32 / cfg.split) * cfg.rows_per_lane;
            return (rows + per - 1) / per;
        };
        while (ctas() < sms) {
            if (auto_rl && cfg.rows_per_lane > 2) cfg.rows_per_lane /= 2;
            else if (auto_w && cfg.warps > 4) cfg.warps /= 2;
            else if (auto_rl && cfg.rows_per_lane > 1) cfg.rows_per_lane /= 2;
            else break;
        }
    }
    cudaError_t e = mm::launch_gemv_packed2(a, cfg, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gemv launch");
    return ok();
}

mm_status mm_gemv_packed2(const uint8_t *codes, const uint16_t *scales, const uint16_t *x, float *y, int64_t rows,
                          int64_t cols, const float codebook[4], mm_stream_t stream) {
    return mm_gemv_packed2_ex(codes, scales, x, y, rows, cols, codebook, stream, nullptr);
}

mm_status mm_gemv_packed2_strided_batched(const uint8_t *codes, int64_t codes_stride, const uint16_t *scales,
                                          int64_t scales_stride, const uint16_t *x, int64_t x_stride, float *y,
                                          int64_t y_stride, int64_t batch, int64_t rows, int64_t cols,
                                          const float codebook[4], mm_stream_t stream) {
    return mm_gemv_packed2_strided_batched_ex(codes, codes_stride, scales, scales_stride, x, x_stride, y, y_stride,
                                              batch, rows, cols, codebook, stream, nullptr);
}

mm_status mm_gemv_packed2_strided_batched_ex(const uint8_t *codes, int64_t codes_stride, const uint16_t *scales,
                                             int64_t scales_stride, const uint16_t *x, int64_t x_stride, float *y,
                                             int64_t y_stride, int64_t batch, int64_t rows, int64_t cols,
                                             const float codebook[4], mm_stream_t stream, const mm_gemv_opts *opts) {
    int dequant = opts ? opts->dequant : MM_DEQ_AUTO;
    const int tiles = opts ? opts->rows_per_lane : 0;
    if (opts && (opts->split || opts->warps || opts->staging > 0))
        return fail(MM_ERR_INVALID_ARG,
                    "the batched GEMV takes only dequant, rows_per_lane, pdl, weights_static and independent options");
    mm::GemvConfig cfg{0, 0, 0, 0, 0, 0, 0, -1, 0};  // no programmatic launch unless asked for
    if (opts) {
        cfg.pdl = opts->pdl;
        cfg.weights_static = opts->weights_static;
        cfg.independent = opts->independent;
    }
    if ((cfg.pdl != 0 && cfg.pdl != 1) || (cfg.weights_static != 0 && cfg.weights_static != 1) ||
        (cfg.independent != 0 && cfg.independent != 1))
        return fail(MM_ERR_INVALID_ARG, "pdl, weights_static and independent must be 0 or 1");
    const bool launch_opts = cfg.pdl || cfg.weights_static || cfg.independent;
    if (dequant != MM_DEQ_AUTO && dequant != MM_DEQ_AFFINE && dequant != MM_DEQ_MXF4)
        return fail(MM_ERR_INVALID_ARG, "the batched GEMV decode must be MM_DEQ_AUTO, MM_DEQ_AFFINE or MM_DEQ_MXF4");
    if (tiles < 0 || tiles > 4096) return fail(MM_ERR_INVALID_ARG, "rows_per_lane (tiles per CTA) must be 0..4096");
    if (batch < 1) return fail(MM_ERR_INVALID_ARG, "batch must be >= 1 (got %lld)", (long long)batch);
    mm_status s = check_packed(codes, scales, x, y, 1, rows, cols, codebook);
    if (s != MM_OK) return s;
    const int64_t rowbytes = (cols + 3) / 4;
    if (batch > 1 && (codes_stride < rows * rowbytes || scales_stride < rows || y_stride < rows ||
                      (x_stride != 0 && x_stride < cols)))
        return fail(MM_ERR_INVALID_ARG, "strides must cover one matrix (codes_stride >= rows * ceil(cols/4) bytes, "
                                        "scales_stride >= rows, y_stride >= rows, x_stride 0 or >= cols)");
    if (codes_stride < 0 || scales_stride < 0 || x_stride < 0 || y_stride < 0)
        return fail(MM_ERR_INVALID_ARG, "strides must be >= 0");
    const int64_t nb = batch - 1;
    const uint64_t ybytes = (uint64_t)(nb * y_stride + rows) * 4;
    if (overlap(y, ybytes, codes, (uint64_t)(nb * codes_stride + rows * rowbytes)) ||
        overlap(y, ybytes, scales, (uint64_t)(nb * scales_stride + rows) * 2) ||
        overlap(y, ybytes, x, (uint64_t)(nb * x_stride + cols) * 2))
        return fail(MM_ERR_INVALID_ARG, "an output overlaps an input");
    s = check_device();
    if (s != MM_OK) return s;
    mm::PackedBatch p{codes, codes_stride, scales, scales_stride, x, x_stride, y, y_stride, batch, rows, cols,
                      {codebook[0], codebook[1], codebook[2], codebook[3]}};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dequant == MM_DEQ_MXF4 && !mm::gemv_batched_mxf4_supported(p))
        return fail(MM_ERR_INVALID_ARG, "the fp4 tensor-core decode needs an affine codebook, cols %% 512 == 0, "
                                        "cols <= 12800 and 16-byte aligned codes and codes_stride");
    // automatic: the fp4 tensor-core decode, measured fastest for a batch in one launch on GB300
    // (64 x 12,288 x 1,536: 0.975 us per matrix against 1.42 for the staged SIMT affine kernel)
    if (dequant == MM_DEQ_MXF4 || (dequant == MM_DEQ_AUTO && mm::gemv_batched_mxf4_supported(p))) {
        const cudaError_t e = mm::launch_gemv_batched_mxf4(p, tiles, cfg, st);
        if (e != cudaSuccess) return cuda_fail(e, "batched gemv launch");
        return ok();
    }
    if (launch_opts)
        return fail(MM_ERR_INVALID_ARG, "pdl, weights_static and independent need the fp4 tensor-core batched decode");
    if (mm::gemv_batched_supported(p)) {
        const cudaError_t e = mm::launch_gemv_batched(p, st);
        if (e != cudaSuccess) return cuda_fail(e, "batched gemv launch");
        return ok();
    }
    if (dequant == MM_DEQ_AFFINE && !mm::codebook_is_affine(codebook))
        return fail(MM_ERR_INVALID_ARG, "affine decode needs codebook[c] == codebook[0] + c*(codebook[1]-codebook[0])");
    // shapes the one-launch kernel does not take: one call per matrix
    for (int64_t b = 0; b < batch; ++b) {
        s = mm_gemv_packed2_ex(codes + b * codes_stride, scales + b * scales_stride, x + b * x_stride,
                               y + b * y_stride, rows, cols, codebook, stream, nullptr);
        if (s != MM_OK) return s;
    }
    return ok();
}

mm_status mm_gemm_packed2_ex(const uint8_t *codes, const uint16_t *scales, const uint16_t *X, float *Y, int64_t M,
                             int64_t rows, int64_t cols, const float codebook[4], mm_stream_t stream,
                             const mm_gemm_packed2_opts *opts) {
    mm_status s = check_packed(codes, scales, X, Y, M, rows, cols, codebook);
    if (s != MM_OK) return s;
    const int tile = opts ? opts->tile : 0;
    const int splitk = opts ? opts->splitk : 0;
    const int pdl = opts ? opts->pdl : 0, weights_static = opts ? opts->weights_static : 0;
    const int ntok = opts ? opts->ntok : 0;
    if (tile != 0 && tile != 1 && tile != 2 && tile != 3 && tile != 32 && tile != 64 && tile != 128)
        return fail(MM_ERR_INVALID_ARG, "tile must be 0 (auto), 1 (FFMA), 2, 3, 32, 64 or 128 (tensor cores)");
    if (ntok != 0 && (tile != 3 || ntok < 16 || ntok > 256 || ntok % 16 != 0))
        return fail(MM_ERR_INVALID_ARG, "ntok (tokens per tile) is 0 or, with tile 3, a multiple of 16 in 16..256");
    if (splitk != 0 && splitk != 1 && splitk != 2 && splitk != 4 && splitk != 8 && !(splitk == 16 && tile == 2))
        return fail(MM_ERR_INVALID_ARG, "splitk must be 0 (auto), 1, 2, 4 or 8 (or 16 with tile 2)");
    if ((pdl != 0 && pdl != 1) || (weights_static != 0 && weights_static != 1) || (weights_static && !pdl))
        return fail(MM_ERR_INVALID_ARG, "pdl and weights_static must be 0 or 1, weights_static only with pdl");
    mm::PackedArgs a{codes, scales, X, Y, M, rows, cols, {codebook[0], codebook[1], codebook[2], codebook[3]}};
    const bool tc_ok = mm::gemm_packed2_tc_supported(a);
    const bool tcw_ok = mm::gemm_packed2_tcw_supported(a);
    if (tile >= 32 && !tc_ok)
        return fail(MM_ERR_INVALID_ARG, "tensor-core tile needs fp16-exact codebook entries, cols %% 8 == 0 and 16-byte aligned X");
    if (tile == 2 && !tcw_ok)
        return fail(MM_ERR_INVALID_ARG,
                    "tile 2 needs fp16-exact codebook entries, cols %% 64 == 0 and 16-byte aligned codes and X");
    if (tile == 3 && !mm::gemm_packed2_tcr_supported(a))
        return fail(MM_ERR_INVALID_ARG,
                    "tile 3 needs fp16-exact codebook entries, cols %% 64 == 0 and 16-byte aligned codes and X");
    if (tile == 3 && splitk > cols / 64)
        return fail(MM_ERR_INVALID_ARG, "tile 3: splitk must not exceed the cols / 64 atoms");
    if (tile == 2 && splitk && !mm::gemm_packed2_tcw_fits(M, cols, splitk))
        return fail(MM_ERR_INVALID_ARG,
                    "tile 2: splitk must leave each CTA 1 to 8 of the cols / 64 atoms, within shared memory with X");
    s = check_device();
    if (s != MM_OK) return s;
    cudaError_t e;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // automatic: tile 3 (decoded weights in tensor memory) measured fastest on the ternary
    // encoder shapes (7.9 / 10.4 us per up / down product against 10.4 / 15.3 for the
    // pipelined W-as-N kernel and 13.1 / 16.4 for tile 2); the W-as-N kernel covers the
    // shapes tile 3 does not take (cols % 64 != 0, unaligned codes)
    const bool tcr_auto = tile == 0 && mm::gemm_packed2_tcr_supported(a);
    if (tile == 2) e = mm::launch_gemm_packed2_tcw(a, splitk, pdl, weights_static, st);
    else if (tile == 3 || tcr_auto) e = mm::launch_gemm_packed2_tcr(a, ntok, splitk, pdl, weights_static, st);
    else if (tc_ok && tile != 1) e = mm::launch_gemm_packed2_tc(a, tile, splitk, st);
    else e = mm::launch_gemm_packed2(a, 0, st);
    if (e != cudaSuccess) return cuda_fail(e, "packed gemm launch");
    return ok();
}

mm_status mm_gemm_packed2(const uint8_t *codes, const uint16_t *scales, const uint16_t *X, float *Y, int64_t M,
                          int64_t rows, int64_t cols, const float codebook[4], mm_stream_t stream) {
    return mm_gemm_packed2_ex(codes, scales, X, Y, M, rows, cols, codebook, stream, nullptr);
}

mm_status mm_gemv_packed4_ex(const uint8_t *codes, const uint16_t *scales, const uint16_t *x, float *y, int64_t rows,
                             int64_t cols, const float codebook[16], mm_stream_t stream, const mm_gemv4_opts *opts) {
    mm_status s = check_packed4(codes, scales, x, y, rows, cols, codebook);
    if (s != MM_OK) return s;
    mm::Gemv4Config cfg{1, 0, 0, -1, 0};
    if (opts) {
        cfg.pdl = opts->pdl;
        cfg.weights_static = opts->weights_static;
        cfg.independent = opts->independent;
        cfg.staging = opts->staging;
        cfg.blocks_per_cta = opts->blocks;
    }
    mm::Packed4Args a{codes, scales, x, y, rows, cols, {}};
    for (int i = 0; i < 16; ++i) a.cb[i] = codebook[i];
    if (cfg.staging < 0) cfg.staging = mm::gemv4_lut_supported(a) ? 1 : 0;
    if (cfg.staging != 0 && cfg.staging != 1) return fail(MM_ERR_INVALID_ARG, "staging must be -1, 0 or 1");
    if (cfg.staging && !mm::gemv4_lut_supported(a))
        return fail(MM_ERR_INVALID_ARG, "the staged 4-bit kernel needs cols %% 256 == 0, cols <= 4096 and 16-byte aligned codes and x");
    if (cfg.blocks_per_cta < 0 || cfg.blocks_per_cta > 64)
        return fail(MM_ERR_INVALID_ARG, "blocks (64-row blocks per CTA) must be 0..64");
    if (cfg.staging && !cfg.blocks_per_cta) cfg.blocks_per_cta = cfg.independent ? 2 : 1;
    if (cfg.pdl != 0 && cfg.pdl != 1) return fail(MM_ERR_INVALID_ARG, "pdl must be 0 or 1");
    if (cfg.weights_static != 0 && cfg.weights_static != 1) return fail(MM_ERR_INVALID_ARG, "weights_static must be 0 or 1");
    if (cfg.independent != 0 && cfg.independent != 1) return fail(MM_ERR_INVALID_ARG, "independent must be 0 or 1");
    s = check_device();
    if (s != MM_OK) return s;
    cudaError_t e = mm::launch_gemv_packed4(a, cfg, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gemv4 launch");
    return ok();
}

mm_status mm_gemv_packed4(const uint8_t *codes, const uint16_t *scales, const uint16_t *x, float *y, int64_t rows,
                          int64_t cols, const float codebook[16], mm_stream_t stream) {
    return mm_gemv_packed4_ex(codes, scales, x, y, rows, cols, codebook, stream, nullptr);
}

mm_status mm_check_device_error(mm_stream_t stream) {
    cudaError_t e;
    const unsigned int v = mm::gemm_ffma_take_device_error(reinterpret_cast<cudaStream_t>(stream), &e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (v != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the FFMA GEMM (code %u)", v);
    const unsigned int w = mm::gemm_packed2_tc_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (w != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the tensor-core packed GEMM (code %u)", w);
    const unsigned int z = mm::gemm_tf32x3_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (z != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the 3xTF32 GEMM (code %u)", z);
    const unsigned int zw = mm::gemm_tf32x3_ws_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (zw != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the warp-specialised 3xTF32 GEMM (code %u)", zw);
    const unsigned int sk = mm::gemm_skinny_tc_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (sk != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the few-rows 3xTF32 GEMM (code %u)", sk);
    const unsigned int tw = mm::gemm_packed2_tcw_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (tw != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the tensor-core packed GEMM, tile 2 (code %u)", tw);
    const unsigned int tr = mm::gemm_packed2_tcr_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (tr != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the tensor-core packed GEMM, tile 3 (code %u)", tr);
    const unsigned int q = mm::gemv_tma_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (q != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the staged GEMV (code %u)", q);
    const unsigned int f = mm::gemv_fp8_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (f != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the fp8 GEMV (code %u)", f);
    const unsigned int v2 = mm::gemv_rows_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (v2 != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the staged affine GEMV (code %u)", v2);
    const unsigned int u4 = mm::gemv4_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (u4 != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the 4-bit GEMV (code %u)", u4);
    const unsigned int x4 = mm::gemv_mxf4_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (x4 != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the fp4 tensor-core GEMV (code %u)", x4);
    const unsigned int u = mm::gemv_tc_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (u != 0) return fail(MM_ERR_TIMEOUT, "a bounded device wait ran out in the tcgen05 GEMV (code %u)", u);
    const unsigned int pr = mm::wait_probe_take_device_error(&e);
    if (e != cudaSuccess) return cuda_fail(e, "mm_check_device_error");
    if (pr != 0) return fail(MM_ERR_TIMEOUT, "the failure-detection probe's bounded wait ran out (code %u)", pr);
    return ok();
}

namespace {

// shape, pointers and overlaps of an attention call; nin inputs, nout outputs of `per` floats
// each (L-shaped tensors, heads x T, are listed with their own sizes)
mm_status check_attention(int64_t heads, int64_t T, int64_t D, int causal, float scale, const void *const *in,
                          const uint64_t *in_bytes, int nin, void *const *out, const uint64_t *out_bytes, int nout) {
    if (heads < 1 || T < 1 || D < 1)
        return fail(MM_ERR_INVALID_ARG, "heads, T, D must be >= 1 (got %lld, %lld, %lld)", (long long)heads,
                    (long long)T, (long long)D);
    if (causal != 0 && causal != 1) return fail(MM_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (!std::isfinite(scale)) return fail(MM_ERR_INVALID_ARG, "scale is not finite");
    for (int i = 0; i < nin; ++i)
        if (!in[i] || (reinterpret_cast<uintptr_t>(in[i]) & 3)) return fail(MM_ERR_INVALID_ARG, "NULL or misaligned input %d", i);
    for (int i = 0; i < nout; ++i)
        if (!out[i] || (reinterpret_cast<uintptr_t>(out[i]) & 3))
            return fail(MM_ERR_INVALID_ARG, "NULL or misaligned output %d", i);
    if (!mm::attention_supported(heads, T, D))
        return fail(MM_ERR_UNSUPPORTED, "attention supports D = 64, 1 <= T <= 2^24, heads <= 65535 (got D=%lld)",
                    (long long)D);
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlap(out[i], out_bytes[i], in[j], in_bytes[j])) return fail(MM_ERR_INVALID_ARG, "an output overlaps an input");
        for (int j = 0; j < i; ++j)
            if (overlap(out[i], out_bytes[i], out[j], out_bytes[j])) return fail(MM_ERR_INVALID_ARG, "two outputs overlap");
    }
    return MM_OK;
}

}  // namespace

mm_status mm_attention_fwd(const float *Q, const float *K, const float *V, float *O, float *L, int64_t heads,
                           int64_t T, int64_t D, int causal, float scale, mm_stream_t stream) {
    const uint64_t nb = (uint64_t)heads * (uint64_t)T * (uint64_t)D * 4, lb = (uint64_t)heads * (uint64_t)T * 4;
    const void *in[3] = {Q, K, V};
    const uint64_t inb[3] = {nb, nb, nb};
    void *out[2] = {O, L};
    const uint64_t outb[2] = {nb, lb};
    mm_status s = check_attention(heads, T, D, causal, scale, in, inb, 3, out, outb, 2);
    if (s != MM_OK) return s;
    s = check_device();
    if (s != MM_OK) return s;
    const cudaError_t e =
        mm::launch_attention_fwd(Q, K, V, O, L, heads, T, causal, scale, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attention forward launch");
    return ok();
}

mm_status mm_attention_bwd(const float *Q, const float *K, const float *V, const float *O, const float *dO,
                           const float *L, float *dQ, float *dK, float *dV, int64_t heads, int64_t T, int64_t D,
                           int causal, float scale, mm_stream_t stream) {
    const uint64_t nb = (uint64_t)heads * (uint64_t)T * (uint64_t)D * 4, lb = (uint64_t)heads * (uint64_t)T * 4;
    const void *in[6] = {Q, K, V, O, dO, L};
    const uint64_t inb[6] = {nb, nb, nb, nb, nb, lb};
    void *out[3] = {dQ, dK, dV};
    const uint64_t outb[3] = {nb, nb, nb};
    mm_status s = check_attention(heads, T, D, causal, scale, in, inb, 6, out, outb, 3);
    if (s != MM_OK) return s;
    s = check_device();
    if (s != MM_OK) return s;
    const cudaError_t e = mm::launch_attention_bwd(Q, K, V, O, dO, L, dQ, dK, dV, heads, T, causal, scale,
                                                   reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "attention backward launch");
    return ok();
}

mm_status mm_probe_bounded_wait(int arrive, uint64_t limit_ns, uint64_t *out, mm_stream_t stream) {
    if (arrive != 0 && arrive != 1) return fail(MM_ERR_INVALID_ARG, "arrive must be 0 or 1");
    if (limit_ns < 1000 || limit_ns > 100000000)
        return fail(MM_ERR_INVALID_ARG, "limit_ns must be 1,000 .. 100,000,000 (1 us .. 0.1 s)");
    if (out && (reinterpret_cast<uintptr_t>(out) & 7)) return fail(MM_ERR_INVALID_ARG, "out must be 8-byte aligned");
    mm_status s = check_device();
    if (s != MM_OK) return s;
    cudaError_t e = mm::launch_wait_probe(arrive, (unsigned long long)limit_ns,
                                          reinterpret_cast<unsigned long long *>(out),
                                          reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
    return ok();
}

}  // extern "C"
