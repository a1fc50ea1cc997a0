// gemm_tf32x3_ws.cu -- warp-specialised, persistent 3xTF32 GEMM on tcgen05.
//
// The GEMM of "I built a GPT-2 in the browser...", section "The kernel sweep"
// (C = A.B forward, dA = dC.B^T and dB = A^T.dC backward), in fp32 accuracy by
// the three-term split of Ootomo and Yokota (IJHPCA 2022):
//
//     a.b ~= a_hi.b_hi + a_hi.b_lo + a_lo.b_hi,
//     a_hi = a with its 13 low mantissa bits cleared, a_lo = a - a_hi (exact).
//
// The tf32 MMA reads the top 19 bits of each fp32 container, so a raw fp32
// tile that is already in the operand layout *is* the hi operand and only
// its lo tile has to be computed.  Operands are K-major with the 64-byte
// swizzle (rows of 16 fp32 along K; 16-byte chunk c of row r at chunk
// c ^ ((r >> 1) & 3)).  A K-contiguous operand arrives that way from TMA and
// its lo tile is the element-wise map at the same offsets; an M/N-contiguous
// operand arrives as an unswizzled [k][m] tile and the lo pass writes both
// its hi and lo tiles transposed (4 conflict-free column reads, one 16-byte
// conflict-free store per tile).
//
// Roles (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0      one thread issues the TMA loads of each 16-deep k-slab of
//               op(A) (128 x 16) and op(B) (256 x 16) into a ring of 3 or
//               4 stages (as many as fit in shared memory);
//   warp 1      one thread issues 2 x 3 tcgen05.mma kind::tf32 (M = 128,
//               N = 256, K = 8) per slab into one of two TMEM accumulators
//               and commits each slab to the barrier that frees its stage;
//   warps 2-5   compute lo = a - a_hi for each landed slab (and transpose
//               M/N-contiguous operands into the K-major layout);
//   warps 6-9   drain a finished accumulator (tcgen05.ld) into C with edge
//               masks while the MMAs of the next tile run in the other one.
// Every wait is bounded; a wait that runs out records an error, raises a CTA
// flag that the other roles poll, and the CTA drains its copies and MMAs,
// frees its TMEM and returns.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tmap.h"

#include <mutex>

namespace mm {

__device__ unsigned int g_tf32ws_err;

namespace {

constexpr int BM = 128, BN = 256, BK = 16, NACC = 2;
constexpr int A_BYTES = BM * BK * 4;          // 8 KiB: one 128 x 16 fp32 tile
constexpr int B_BYTES = BN * BK * 4;          // 16 KiB: one 256 x 16 fp32 tile
constexpr int RAW_BYTES = A_BYTES + B_BYTES;  // bytes TMA brings per stage
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_CONV0 = 2, NCONV = 128, WARP_EPI0 = 6, NEPI = 128;
constexpr int NTHREADS = 320;
constexpr int TMEM_COLS = NACC * BN;          // 512: the whole tensor memory of the SM
constexpr int SMEM_LIMIT = 227 * 1024;

// Shared-memory plan of one stage.  A K-contiguous operand keeps raw (= hi) and
// lo tiles; an M/N-contiguous one keeps its raw [k][m] tile plus K-major hi and lo.
template <bool A_KC, bool B_KC>
struct Plan {
    static constexpr int A_REGION = (A_KC ? 2 : 3) * A_BYTES;
    static constexpr int B_REGION = (B_KC ? 2 : 3) * B_BYTES;
    static constexpr int STAGE_BYTES = A_REGION + B_REGION;
    static constexpr int RAW_A = 0, HI_A = A_KC ? 0 : A_BYTES, LO_A = A_KC ? A_BYTES : 2 * A_BYTES;
    static constexpr int RAW_B = A_REGION, HI_B = A_REGION + (B_KC ? 0 : B_BYTES),
                         LO_B = A_REGION + (B_KC ? B_BYTES : 2 * B_BYTES);
    static constexpr int NBARS_MAX = 3 * 4 + 2 * NACC + 1;
    static constexpr int FIXED = NBARS_MAX * 8 + 16 + 1024;
    static constexpr int S_FIT = (SMEM_LIMIT - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = S_FIT < 4 ? S_FIT : 4;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + (3 * STAGES + 2 * NACC + 1) * 8 + 16 + 1024;
    static_assert(STAGES >= 3, "at least three stages");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
};

struct WsParams {
    int M, N, K;
    int tiles_m, tiles;
    float *C;
    int64_t ldc;
};

__device__ __forceinline__ float lo_part(float a) {
    return __fsub_rn(a, __uint_as_float(__float_as_uint(a) & 0xFFFFE000u));
}

__device__ __forceinline__ float4 lo_part4(float4 v) {
    return make_float4(lo_part(v.x), lo_part(v.y), lo_part(v.z), lo_part(v.w));
}

// K-contiguous operand: the lo tile at the same (swizzled) offsets as the raw tile.
template <int BYTES>
__device__ __forceinline__ void lo_in_place_layout(const uint8_t *raw, uint8_t *lo, int ct) {
    constexpr int R = BYTES / (16 * NCONV);
    static_assert(BYTES % (16 * NCONV) == 0, "whole float4 rounds");
    float4 v[R];
#pragma unroll
    for (int i = 0; i < R; ++i) v[i] = *reinterpret_cast<const float4 *>(raw + (ct + i * NCONV) * 16);
#pragma unroll
    for (int i = 0; i < R; ++i) *reinterpret_cast<float4 *>(lo + (ct + i * NCONV) * 16) = lo_part4(v[i]);
}

// M/N-contiguous operand: raw [k][r] (BK rows of ROWS fp32, unswizzled) -> K-major
// 64-byte-swizzled hi and lo tiles, row r, 16-byte chunk c at chunk c ^ ((r >> 1) & 3).
// A warp covers 32 consecutive r: each column read is one 128-byte row segment and
// each 8-lane phase of the 16-byte stores hits 8 distinct bank groups.
template <int ROWS>
__device__ __forceinline__ void split_transpose(const uint8_t *raw, uint8_t *hi, uint8_t *lo, int ct) {
    const float *src = reinterpret_cast<const float *>(raw);
    constexpr int TASKS = ROWS * (BK / 4);
    static_assert(TASKS % NCONV == 0, "whole rounds");
#pragma unroll
    for (int i = 0; i < TASKS / NCONV; ++i) {
        const int idx = ct + i * NCONV;
        const int r = idx % ROWS, c = idx / ROWS;
        const float4 v = make_float4(src[(4 * c + 0) * ROWS + r], src[(4 * c + 1) * ROWS + r],
                                     src[(4 * c + 2) * ROWS + r], src[(4 * c + 3) * ROWS + r]);
        const int off = r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
        *reinterpret_cast<float4 *>(hi + off) = v;
        *reinterpret_cast<float4 *>(lo + off) = lo_part4(v);
    }
}

__device__ __forceinline__ void fail(volatile int *abort_flag, unsigned int code) {
    atomicExch(&g_tf32ws_err, code);
    *abort_flag = 1;
}

template <bool A_KC, bool B_KC>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tf32x3_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const WsParams p) {
    using P = Plan<A_KC, B_KC>;
    constexpr int STAGES = P::STAGES, STAGE_BYTES = P::STAGE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);  // TMA -> lo pass
    uint64_t *conv = full + STAGES;                                              // lo pass -> MMA
    uint64_t *empty = conv + STAGES;                                             // MMA -> TMA
    uint64_t *accf = empty + STAGES;                                             // MMA -> epilogue
    uint64_t *acce = accf + NACC;                                                // epilogue -> MMA
    uint64_t *last = acce + NACC;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(last + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = (p.K + BK - 1) / BK;

    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&conv[s], NCONV);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], NEPI);
        }
        mbar_init(last, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == WARP_TMA) {
        if (lane == 0) {
            int it = 0;  // slabs issued so far (ring position)
            bool stop = false;
            for (int t = blockIdx.x; t < p.tiles && !stop; t += gridDim.x) {
                const int m0 = (t % p.tiles_m) * BM, n0 = (t / p.tiles_m) * BN;
                for (int kt = 0; kt < KT; ++kt) {
                    const int s = it % STAGES;
                    const uint32_t use = it / STAGES;
                    if (*abort_flag) { stop = true; break; }
                    if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1)) {
                        fail(abort_flag, kDevErrWaitEmpty);
                        stop = true;
                        break;
                    }
                    uint8_t *st = smem + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s], RAW_BYTES);
                    const int k0 = kt * BK;
                    if (A_KC) tma_load_2d(st + P::RAW_A, &tmA, &full[s], k0, m0);
                    else tma_load_2d(st + P::RAW_A, &tmA, &full[s], m0, k0);
                    if (B_KC) tma_load_2d(st + P::RAW_B, &tmB, &full[s], k0, n0);
                    else tma_load_2d(st + P::RAW_B, &tmB, &full[s], n0, k0);
                    ++it;
                }
            }
            // every copy issued must land before this CTA's shared memory is released
            for (int s = 0; s < STAGES && s < it; ++s) {
                const int lastit = s + ((it - 1 - s) / STAGES) * STAGES;
                if (!mbar_wait(&full[s], (uint32_t)(lastit / STAGES) & 1)) {
                    atomicExch(&g_tf32ws_err, kDevErrDrain);
                    break;
                }
            }
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(kFmtTF32, kFmtTF32, BN, BM);
            int it = 0, tc = 0;
            bool stop = false;
            for (int t = blockIdx.x; t < p.tiles && !stop; t += gridDim.x, ++tc) {
                const int b = tc % NACC;
                const uint32_t ause = tc / NACC;
                if (*abort_flag) break;
                if (ause > 0 && !mbar_wait(&acce[b], (ause - 1) & 1)) {
                    fail(abort_flag, kDevErrWaitEmpty);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * BN);
                for (int kt = 0; kt < KT; ++kt, ++it) {
                    const int s = it % STAGES;
                    const uint32_t use = it / STAGES;
                    if (*abort_flag) { stop = true; break; }
                    if (!mbar_wait(&conv[s], use & 1)) {
                        fail(abort_flag, kDevErrWaitFull);
                        stop = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
#pragma unroll
                    for (int ks = 0; ks < BK / 8; ++ks) {
                        // 8 tf32 of K are 32 bytes along the swizzled 64-byte rows
                        const uint32_t o = 32u * ks;
                        const uint64_t ah = sdesc_make(st + P::HI_A + o, 16, 512, kSdescSw64);
                        const uint64_t al = sdesc_make(st + P::LO_A + o, 16, 512, kSdescSw64);
                        const uint64_t bh = sdesc_make(st + P::HI_B + o, 16, 512, kSdescSw64);
                        const uint64_t bl = sdesc_make(st + P::LO_B + o, 16, 512, kSdescSw64);
                        umma_tf32(d, ah, bh, idesc, (kt > 0 || ks > 0) ? 1u : 0u);
                        umma_tf32(d, ah, bl, idesc, 1u);
                        umma_tf32(d, al, bh, idesc, 1u);
                    }
                    umma_commit(&empty[s]);
                }
                if (!stop) umma_commit(&accf[b]);
            }
            // every MMA issued must be complete before the tensor memory is freed
            umma_commit(last);
            if (!mbar_wait(last, 0)) atomicExch(&g_tf32ws_err, kDevErrWaitMma);
        }
    } else if (warp < WARP_EPI0) {
        // lo pass (and transposes of M/N-contiguous operands)
        const int ct = threadIdx.x - 32 * WARP_CONV0;
        int it = 0;
        bool stop = false;
        for (int t = blockIdx.x; t < p.tiles && !stop; t += gridDim.x) {
            for (int kt = 0; kt < KT; ++kt, ++it) {
                const int s = it % STAGES;
                const uint32_t use = it / STAGES;
                if (*abort_flag) { stop = true; break; }
                if (!mbar_wait(&full[s], use & 1)) {
                    fail(abort_flag, kDevErrWaitFull);
                    stop = true;
                    break;
                }
                uint8_t *st = smem + s * STAGE_BYTES;
                if (A_KC) lo_in_place_layout<A_BYTES>(st + P::RAW_A, st + P::LO_A, ct);
                else split_transpose<BM>(st + P::RAW_A, st + P::HI_A, st + P::LO_A, ct);
                if (B_KC) lo_in_place_layout<B_BYTES>(st + P::RAW_B, st + P::LO_B, ct);
                else split_transpose<BN>(st + P::RAW_B, st + P::HI_B, st + P::LO_B, ct);
                fence_proxy_async_smem();
                mbar_arrive(&conv[s]);
            }
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31
        const int q = warp & 3;
        const bool vec_ok = (p.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
        int tc = 0;
        for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++tc) {
            const int b = tc % NACC;
            const uint32_t ause = tc / NACC;
            if (*abort_flag) break;
            if (!mbar_wait_sleep(&accf[b], ause & 1)) {
                fail(abort_flag, kDevErrWaitMma);
                break;
            }
            tc_fence_after_sync();
            const int m0 = (t % p.tiles_m) * BM, n0 = (t / p.tiles_m) * BN;
            const int row = m0 + 32 * q + lane;
            const uint32_t base = tmem + (uint32_t)(b * BN) + ((uint32_t)(32 * q) << 16);
            float *crow = p.C + (int64_t)row * p.ldc + n0;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                tmem_ld32(base + (uint32_t)c0, v);
                if (row < p.M && n0 + c0 < p.N) {
                    if (vec_ok && n0 + c0 + 32 <= p.N) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(crow + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (n0 + c0 + j < p.N) crow[c0 + j] = v[j];
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&acce[b]);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == WARP_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

template <bool A_KC, bool B_KC>
cudaError_t launch_ws(const CUtensorMap &ta, const CUtensorMap &tb, const WsParams &p, int grid, cudaStream_t s) {
    auto kern = gemm_tf32x3_ws_kernel<A_KC, B_KC>;
    constexpr int smem = Plan<A_KC, B_KC>::SMEM_BYTES;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    kern<<<grid, NTHREADS, smem, s>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_tf32x3_ws(const GemmArgs &g, cudaStream_t s) {
    if (!gemm_tf32x3_supported(g)) return cudaErrorNotSupported;
    CUtensorMap ta, tb;
    cudaError_t e;
    // K-contiguous operands: 16 x rows boxes, 64-byte swizzle (the MMA operand layout);
    // M/N-contiguous: rows x 16 boxes, unswizzled (transposed by the lo pass)
    if (!g.transA)
        e = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.K, g.M, g.lda * 4, BK, BM,
                         CU_TENSOR_MAP_SWIZZLE_64B);
    else
        e = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.M, g.K, g.lda * 4, BM, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    if (g.transB)
        e = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.K, g.N, g.ldb * 4, BK, BN,
                         CU_TENSOR_MAP_SWIZZLE_64B);
    else
        e = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.N, g.K, g.ldb * 4, BN, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int tiles_m = (int)((g.M + BM - 1) / BM), tiles_n = (int)((g.N + BN - 1) / BN);
    WsParams p{(int)g.M, (int)g.N, (int)g.K, tiles_m, tiles_m * tiles_n, g.C, g.ldc};
    const int grid = p.tiles < sms ? p.tiles : sms;
    if (!g.transA && !g.transB) return launch_ws<true, false>(ta, tb, p, grid, s);
    if (!g.transA && g.transB) return launch_ws<true, true>(ta, tb, p, grid, s);
    if (g.transA && !g.transB) return launch_ws<false, false>(ta, tb, p, grid, s);
    return launch_ws<false, true>(ta, tb, p, grid, s);
}

unsigned int gemm_tf32x3_ws_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_tf32ws_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_tf32ws_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
