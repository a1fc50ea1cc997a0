// gemm_ffma.cu -- C = op(A) . op(B), fp32 FFMA, TMA-staged and register-blocked.
//
// "I built a GPT-2 in the browser...", section "The kernel sweep": Step 1
// stages 16 x 16 tiles of A and B in workgroup memory, Step 2 gives each
// thread a 4 x 4 register block so each shared load feeds 4 multiply-adds;
// section "The three things that didn't work": an 8 x 8 block lost on Apple
// hardware through register spills, and 128-bit vector loads won 1.37x.
// "More Stumbling, This Time in the Browser", "Four answers per worker":
// register blocks of outputs, edge masks for partial tiles, one fixed
// accumulation order along k.
//
// GB300 design: a CTA computes a 128 x 128 tile of C with 8 consumer warps
// (8 x 8 outputs per thread, 128-bit shared loads, the multiply-adds as packed
// f32x2 FMAs where an operand read along m or n supplies the pairs -- two
// outputs per instruction, each rounded once as by FFMA: identical bits, at
// 2048^3 NN 13 %, TN 8 % and TT 14 % faster) and one producer warp that
// streams 128 x 32 k-slabs of A and B into a 4-stage shared-memory ring with
// TMA, each stage guarded by a "full" mbarrier (TMA transaction bytes) and an
// "empty" mbarrier (one arrival per consumer thread).  Operands whose
// contiguous dimension is K are loaded with the 128-byte swizzle and read
// along k as float4s; operands contiguous along M/N are loaded unswizzled and
// read along M/N.  The thread-to-row maps are chosen per layout so every
// 128-bit shared load of a warp is bank-conflict free.  Out-of-range parts of
// edge tiles read as zeros (TMA fill) and are masked at the store.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tmap.h"

#include <mutex>

namespace mm {

__device__ unsigned int g_ffma_err;

namespace {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 4;
constexpr int NCONS = 256;
constexpr int NTHREADS = NCONS + 32;
constexpr int TILE_BYTES = BM * BK * 4;  // 16 KiB per operand per stage
constexpr int STAGE_BYTES = 2 * TILE_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

struct FfmaParams {
    int M, N, K;
    float *C;
    int64_t ldc;
    const float *bias;  // C = act(op(A) op(B) + bias): bias per column or null, act 1 = GELU (tanh)
    int act;
};

// A_KC: the A tile sits in shared memory as [m][k] (k contiguous, 128-byte
// swizzled); otherwise as [k][m].  B_KC: B tile as [n][k] swizzled; else [k][n].
template <bool A_KC, bool B_KC>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_ffma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const FfmaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *empty = full + STAGES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int KT = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCONS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCONS / 32) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int issued = 0;
            for (int kt = 0; kt < KT; ++kt) {
                const int s = kt % STAGES;
                const uint32_t round = kt / STAGES;
                if (kt >= STAGES && !mbar_wait(&empty[s], (round - 1) & 1)) {
                    atomicExch(&g_ffma_err, kDevErrWaitEmpty);
                    break;
                }
                uint8_t *st = smem + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                const int k0 = kt * BK;
                if (A_KC) tma_load_2d(st, &tmA, &full[s], k0, m0);
                else tma_load_2d(st, &tmA, &full[s], m0, k0);
                if (B_KC) tma_load_2d(st + TILE_BYTES, &tmB, &full[s], k0, n0);
                else tma_load_2d(st + TILE_BYTES, &tmB, &full[s], n0, k0);
                ++issued;
            }
            // every issued copy must land before this CTA's shared memory is released
            for (int kt = issued > STAGES ? issued - STAGES : 0; kt < issued; ++kt)
                if (!mbar_wait(&full[kt % STAGES], (kt / STAGES) & 1)) {
                    atomicExch(&g_ffma_err, kDevErrDrain);
                    break;
                }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int wm = warp & 3, wn = warp >> 2, tr = lane >> 3, tc = lane & 7;
    int rowA[8], colB[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        rowA[i] = A_KC ? wm * 32 + tr + 4 * i : wm * 32 + (i < 4 ? 4 * tr + i : 16 + 4 * tr + (i - 4));
        colB[i] = B_KC ? wn * 64 + tc + 8 * i : wn * 64 + (i < 4 ? 4 * tc + i : 32 + 4 * tc + (i - 4));
    }

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % STAGES;
        if (!mbar_wait(&full[s], (kt / STAGES) & 1)) {
            atomicExch(&g_ffma_err, kDevErrWaitFull);
            return;
        }
        const float *As = reinterpret_cast<const float *>(smem + s * STAGE_BYTES);
        const float *Bs = reinterpret_cast<const float *>(smem + s * STAGE_BYTES + TILE_BYTES);
#pragma unroll 2
        for (int kg = 0; kg < BK / 4; ++kg) {
            float a[8][4], b[8][4];
            if (A_KC) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int m = rowA[i];
                    const float4 v = reinterpret_cast<const float4 *>(As + m * BK)[kg ^ (m & 7)];
                    a[i][0] = v.x; a[i][1] = v.y; a[i][2] = v.z; a[i][3] = v.w;
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float *row = As + (4 * kg + kk) * BM + wm * 32 + 4 * tr;
                    const float4 v0 = *reinterpret_cast<const float4 *>(row);
                    const float4 v1 = *reinterpret_cast<const float4 *>(row + 16);
                    a[0][kk] = v0.x; a[1][kk] = v0.y; a[2][kk] = v0.z; a[3][kk] = v0.w;
                    a[4][kk] = v1.x; a[5][kk] = v1.y; a[6][kk] = v1.z; a[7][kk] = v1.w;
                }
            }
            if (B_KC) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int n = colB[j];
                    const float4 v = reinterpret_cast<const float4 *>(Bs + n * BK)[kg ^ (n & 7)];
                    b[j][0] = v.x; b[j][1] = v.y; b[j][2] = v.z; b[j][3] = v.w;
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float *row = Bs + (4 * kg + kk) * BN + wn * 64 + 4 * tc;
                    const float4 v0 = *reinterpret_cast<const float4 *>(row);
                    const float4 v1 = *reinterpret_cast<const float4 *>(row + 32);
                    b[0][kk] = v0.x; b[1][kk] = v0.y; b[2][kk] = v0.z; b[3][kk] = v0.w;
                    b[4][kk] = v1.x; b[5][kk] = v1.y; b[6][kk] = v1.z; b[7][kk] = v1.w;
                }
            }
            // Packed f32x2 FMAs pair the outputs along the operand whose values one 16-byte shared
            // load already leaves in adjacent registers: B read along n pairs columns (2 jp, 2 jp + 1),
            // A read along m pairs rows; with both read along k, packing would cost a move per pair
            // and plain FFMAs measured faster.
            if constexpr (!B_KC) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int jp = 0; jp < 4; ++jp)
                            fma2_bcast(acc[i][2 * jp], acc[i][2 * jp + 1], a[i][kk], b[2 * jp][kk], b[2 * jp + 1][kk]);
            } else if constexpr (!A_KC) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int j = 0; j < 8; ++j)
#pragma unroll
                        for (int ip = 0; ip < 4; ++ip)
                            fma2_bcast(acc[2 * ip][j], acc[2 * ip + 1][j], b[j][kk], a[2 * ip][kk], a[2 * ip + 1][kk]);
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i][kk], b[j][kk], acc[i][j]);
            }
        }
        mbar_arrive(&empty[s]);
    }

    // ---------------------------------------------------- epilogue (masked)
    const bool vec_ok = !B_KC && (p.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
    if (p.bias || p.act) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int n = n0 + colB[j];
            const float bj = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float z = acc[i][j] + bj;
                acc[i][j] = p.act ? gelu_tanh_f(z) : z;
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + rowA[i];
        if (m >= p.M) continue;
        float *crow = p.C + (int64_t)m * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + colB[4 * h];
            if (vec_ok && n + 3 < p.N) {
                *reinterpret_cast<float4 *>(crow + n) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
            } else {
#pragma unroll
                for (int j = 4 * h; j < 4 * h + 4; ++j) {
                    const int nj = n0 + colB[j];
                    if (nj < p.N) crow[nj] = acc[i][j];
                }
            }
        }
    }
}

template <bool A_KC, bool B_KC>
cudaError_t launch_ffma(const CUtensorMap &ta, const CUtensorMap &tb, const FfmaParams &p, cudaStream_t s) {
    auto kern = gemm_ffma_kernel<A_KC, B_KC>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    dim3 grid((unsigned)((p.N + BN - 1) / BN), (unsigned)((p.M + BM - 1) / BM));
    kern<<<grid, NTHREADS, SMEM_BYTES, s>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace

bool gemm_ffma_supported(const GemmArgs &g) {
    const int64_t lim = (int64_t)1 << 30;
    return (reinterpret_cast<uintptr_t>(g.A) % 16) == 0 && (reinterpret_cast<uintptr_t>(g.B) % 16) == 0 &&
           g.lda % 4 == 0 && g.ldb % 4 == 0 && g.M < lim && g.N < lim && g.K < lim && (g.N + BN - 1) / BN < 65536 &&
           (g.M + BM - 1) / BM < 65536;
}

cudaError_t launch_gemm_ffma(const GemmArgs &g, int tile, cudaStream_t s) {
    (void)tile;
    if (!gemm_ffma_supported(g)) return cudaErrorNotSupported;
    CUtensorMap ta, tb;
    cudaError_t e;
    if (!g.transA)
        e = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.K, g.M, g.lda * 4, BK, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    else
        e = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.M, g.K, g.lda * 4, BM, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    if (!g.transB)
        e = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.N, g.K, g.ldb * 4, BN, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        e = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.K, g.N, g.ldb * 4, BK, BN,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    FfmaParams p{(int)g.M, (int)g.N, (int)g.K, g.C, g.ldc, g.bias, g.act};
    if (!g.transA && !g.transB) return launch_ffma<true, false>(ta, tb, p, s);
    if (!g.transA && g.transB) return launch_ffma<true, true>(ta, tb, p, s);
    if (g.transA && !g.transB) return launch_ffma<false, false>(ta, tb, p, s);
    return launch_ffma<false, true>(ta, tb, p, s);
}

unsigned int gemm_ffma_take_device_error(cudaStream_t s, cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaStreamSynchronize(s);
    if (*err != cudaSuccess) return 0;
    *err = cudaMemcpyFromSymbol(&v, g_ffma_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_ffma_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
