// gemm_simple.cu -- C = op(A) . op(B), fp32, for any sizes, strides and
// alignment.  Used where the TMA paths cannot describe the operands (leading
// dimensions that are not a multiple of 4 floats, unaligned base pointers).
//
// "I built a GPT-2 in the browser...", section "The kernel sweep", Step 1
// and Step 2: shared-memory tiles of A and B loaded cooperatively, then each
// thread accumulates a small block of outputs in registers from them (here
// 64 x 64 tiles, 4 x 4 per thread).  Partial tiles are masked at the edges
// ("More Stumbling, This Time in the Browser", section "Four answers per
// worker": the edge masks).  Every output sums k in increasing order.  The
// optional epilogue adds a per-column bias and applies GELU (GPT-2's linear
// layer and MLP activation).
#include "mm_common.cuh"
#include "mm_internal.h"

namespace mm {
namespace {

constexpr int TB = 64, TK = 16;

__global__ void __launch_bounds__(256) gemm_simple_kernel(const GemmArgs g) {
    __shared__ float As[TK][TB + 4];
    __shared__ float Bs[TK][TB + 4];
    const int tid = threadIdx.x;
    const int tm = tid / 16, tn = tid % 16;
    const int64_t m0 = (int64_t)blockIdx.y * TB, n0 = (int64_t)blockIdx.x * TB;
    float acc[4][4] = {};
    for (int64_t k0 = 0; k0 < g.K; k0 += TK) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int idx = tid + 256 * e;
            int mm, kk;
            if (g.transA) { kk = idx / TB; mm = idx % TB; } else { mm = idx / TK; kk = idx % TK; }
            const int64_t m = m0 + mm, k = k0 + kk;
            float v = 0.f;
            if (m < g.M && k < g.K) v = g.transA ? g.A[k * g.lda + m] : g.A[m * g.lda + k];
            As[kk][mm] = v;
            int nn;
            if (g.transB) { nn = idx / TK; kk = idx % TK; } else { kk = idx / TB; nn = idx % TB; }
            const int64_t n = n0 + nn, k2 = k0 + kk;
            float w = 0.f;
            if (n < g.N && k2 < g.K) w = g.transB ? g.B[n * g.ldb + k2] : g.B[k2 * g.ldb + n];
            Bs[kk][nn] = w;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][tm * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tn * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + tm * 4 + i;
        if (m >= g.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tn * 4 + j;
            if (n >= g.N) continue;
            float z = acc[i][j];
            if (g.bias) z += g.bias[n];
            g.C[m * g.ldc + n] = g.act ? gelu_tanh_f(z) : z;
        }
    }
}

}  // namespace

cudaError_t launch_gemm_simple(const GemmArgs &g, cudaStream_t s) {
    const int64_t gx = (g.N + TB - 1) / TB, gy = (g.M + TB - 1) / TB;
    if (gy > 65535) return cudaErrorInvalidConfiguration;
    gemm_simple_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(g);
    return cudaGetLastError();
}

}  // namespace mm
