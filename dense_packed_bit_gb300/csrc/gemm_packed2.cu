// gemm_packed2.cu -- Y = X . (diag(scale) W)^T for 2-bit packed W, short batch X.
//
// "More Stumbling, This Time in the Browser", sections "This time, in a
// browser" and "The attractive ideas that went away": the ternary encoder
// (16 layers, a fixed 111-token input, 2 questions) runs its projections on
// packed ternary weights with their own kernels.  Here a CTA decodes a
// 64-row x 64-field tile of W once into shared memory and reuses it for 64
// rows of X, so the decode cost is spread over the batch; X is converted from
// fp16 once per tile.  4 x 4 outputs per thread, fp32 FMA, the per-row scale
// applied to the finished sum.  Any shape and alignment.
#include "mm_common.cuh"
#include "mm_internal.h"

#include <cuda_fp16.h>

namespace mm {
namespace {

constexpr int TM = 64, TN = 64, TKF = 64;  // tile rows of X, rows of W, fields

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__global__ void __launch_bounds__(256) gemm_packed2_kernel(const PackedArgs a) {
    __shared__ float Xs[TKF][TM + 4];
    __shared__ float Ws[TKF][TN + 4];
    const int tid = threadIdx.x;
    const int tm = tid / 16, tn = tid % 16;
    const int64_t m0 = (int64_t)blockIdx.y * TM, n0 = (int64_t)blockIdx.x * TN;
    const int64_t rowbytes = (a.cols + 3) >> 2;
    float acc[4][4] = {};
    for (int64_t k0 = 0; k0 < a.cols; k0 += TKF) {
        // X tile: 64 x 64 fp16 -> fp32, stored [k][m]
#pragma unroll 4
        for (int e = 0; e < 16; ++e) {
            const int idx = tid + 256 * e;
            const int mm = idx / TKF, kk = idx % TKF;
            const int64_t m = m0 + mm, k = k0 + kk;
            Xs[kk][mm] = (m < a.M && k < a.cols) ? h2f(a.x[m * a.cols + k]) : 0.f;
        }
        // W tile: 64 rows x 16 bytes; each thread decodes 4 bytes = 16 fields
        {
            const int nn = tid / 4, bq = (tid % 4) * 4;
            const int64_t n = n0 + nn;
#pragma unroll
            for (int bi = 0; bi < 4; ++bi) {
                const int64_t byte_idx = k0 / 4 + bq + bi;
                uint32_t byte = 0;
                if (n < a.rows && byte_idx < rowbytes) byte = a.codes[n * rowbytes + byte_idx];
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    const int kk = 4 * (bq + bi) + f;
                    const uint32_t c = (byte >> (2 * f)) & 3u;
                    const float lo = (c & 1u) ? a.cb[1] : a.cb[0];
                    const float hi = (c & 1u) ? a.cb[3] : a.cb[2];
                    const bool valid = n < a.rows && (k0 + kk) < a.cols;
                    Ws[kk][nn] = valid ? ((c & 2u) ? hi : lo) : 0.f;
                }
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < TKF; ++kk) {
            float xa[4], wb[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) xa[i] = Xs[kk][tm * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) wb[j] = Ws[kk][tn * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], wb[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t n = n0 + tn * 4 + j;
        if (n >= a.rows) continue;
        const float scale = h2f(a.scales[n]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = m0 + tm * 4 + i;
            if (m < a.M) a.y[m * a.rows + n] = scale * acc[i][j];
        }
    }
}

}  // namespace

cudaError_t launch_gemm_packed2(const PackedArgs &a, int tile, cudaStream_t s) {
    (void)tile;
    const int64_t gx = (a.rows + TN - 1) / TN, gy = (a.M + TM - 1) / TM;
    if (gy > 65535) return cudaErrorInvalidConfiguration;
    gemm_packed2_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mm
