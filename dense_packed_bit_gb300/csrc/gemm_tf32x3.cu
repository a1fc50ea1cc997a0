// gemm_tf32x3.cu -- C = op(A) . op(B) in fp32 accuracy on the tcgen05 tensor cores.
//
// The GEMM of "I built a GPT-2 in the browser...", section "The kernel sweep"
// (NN forward, NT / TN backward products) is a genuine dense contraction, so
// on GB300 it belongs on the tensor cores.  The tensor cores multiply tf32
// (10 explicit mantissa bits); fp32 accuracy comes from the three-term split
// of Ootomo and Yokota ("Recovering single precision accuracy from Tensor
// Cores while surpassing the FP32 theoretical peak performance", IJHPCA 2022):
//
//     a = a_hi + a_lo,  a_hi = a with its 13 low mantissa bits cleared (exact
//     tf32), a_lo = a - a_hi (exact in fp32, at most 13 significant bits)
//     a.b ~= a_hi.b_hi + a_hi.b_lo + a_lo.b_hi        (a_lo.b_lo dropped)
//
// The dropped term is below 2^-20 |a b| and the tf32 rounding of a_lo, b_lo
// below 2^-21 |a b| each, so every product carries a relative error of about
// 2^-19 at most, far inside 1e-5 of sum |a_ik b_kj|.
//
// Per CTA: a 128 x 128 tile of C in tensor memory (128 lanes x 128 fp32
// columns).  Per 32-deep k-slab: TMA brings the raw fp32 tiles of op(A) and
// op(B) into shared memory (K-contiguous operands with the 128-byte swizzle,
// M/N-contiguous ones unswizzled); the 128 threads write the hi and lo tiles
// as K-major 128-byte-swizzled operands (transposing M/N-contiguous sources
// on the way: 4 scalar loads down a column, one 16-byte store along K, both
// bank-conflict free); one thread issues 3 x 4 tcgen05.mma kind::tf32 (K = 8
// each) and commits them to the stage's mbarrier, which frees the hi/lo
// buffers; two stages overlap the split of slab k+1 with the MMAs of slab k.
// The epilogue reads the accumulator with tcgen05.ld and stores C with edge
// masks; out-of-range parts of edge tiles read as zeros (TMA fill).
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tmap.h"

#include <mutex>

namespace mm {

__device__ unsigned int g_tf32x3_err;

namespace {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 2, NTHREADS = 128;
constexpr int TILE = BM * BK * 4;  // 16 KiB: one operand tile (BN == BM)
// per stage: raw A, raw B, A hi, A lo, B hi, B lo
constexpr int STAGE_BYTES = 6 * TILE;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

struct Tf32x3Params {
    int M, N, K;
    float *C;
    int64_t ldc;
};

__device__ __forceinline__ void split4(const float4 v, float4 &hi, float4 &lo) {
    const float x[4] = {v.x, v.y, v.z, v.w};
    float h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h[i] = __uint_as_float(__float_as_uint(x[i]) & 0xFFFFE000u);
        l[i] = __fsub_rn(x[i], h[i]);
    }
    hi = make_float4(h[0], h[1], h[2], h[3]);
    lo = make_float4(l[0], l[1], l[2], l[3]);
}

// raw K-contiguous tile (already K-major, 128-byte swizzled) -> hi / lo at the same offsets
__device__ __forceinline__ void split_kmajor(const uint8_t *raw, uint8_t *hi, uint8_t *lo, int tid) {
#pragma unroll
    for (int i = 0; i < (TILE / 16) / NTHREADS; ++i) {
        const int off = (tid + i * NTHREADS) * 16;
        float4 h, l;
        split4(*reinterpret_cast<const float4 *>(raw + off), h, l);
        *reinterpret_cast<float4 *>(hi + off) = h;
        *reinterpret_cast<float4 *>(lo + off) = l;
    }
}

// raw M/N-contiguous tile [k][r] (r = 0..127, unswizzled rows of 512 bytes) ->
// K-major 128-byte-swizzled hi / lo: row r, 16-byte chunk kc at chunk kc ^ (r % 8)
__device__ __forceinline__ void split_transpose(const uint8_t *raw, uint8_t *hi, uint8_t *lo, int tid) {
    const float *src = reinterpret_cast<const float *>(raw);
#pragma unroll
    for (int i = 0; i < (TILE / 16) / NTHREADS; ++i) {
        const int idx = tid + i * NTHREADS;
        const int r = idx & 127, kc = idx >> 7;
        const float4 v = make_float4(src[(4 * kc + 0) * 128 + r], src[(4 * kc + 1) * 128 + r],
                                     src[(4 * kc + 2) * 128 + r], src[(4 * kc + 3) * 128 + r]);
        float4 h, l;
        split4(v, h, l);
        const int off = r * 128 + ((kc ^ (r & 7)) << 4);
        *reinterpret_cast<float4 *>(hi + off) = h;
        *reinterpret_cast<float4 *>(lo + off) = l;
    }
}

template <bool A_KC, bool B_KC>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tf32x3_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const Tf32x3Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *done = full + STAGES;
    uint64_t *last = done + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(last + 1);
    int *bad = reinterpret_cast<int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int KT = (p.K + BK - 1) / BK;

    if (warp == 0) {
        tmem_alloc(tmem_slot, BN);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&done[s], 1);
        }
        mbar_init(last, 1);
        *bad = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t idesc = make_idesc(kFmtTF32, kFmtTF32, BN, BM);

    auto issue_tma = [&](int kt) {
        uint8_t *st = smem + (kt % STAGES) * STAGE_BYTES;
        uint64_t *bar = &full[kt % STAGES];
        mbar_arrive_expect_tx(bar, 2 * TILE);
        const int k0 = kt * BK;
        if (A_KC) tma_load_2d(st, &tmA, bar, k0, m0);
        else tma_load_2d(st, &tmA, bar, m0, k0);
        if (B_KC) tma_load_2d(st + TILE, &tmB, bar, k0, n0);
        else tma_load_2d(st + TILE, &tmB, bar, n0, k0);
    };
    int issued = 0;
    if (tid == 0)
        for (int kt = 0; kt < STAGES && kt < KT; ++kt) {
            issue_tma(kt);
            ++issued;
        }

    for (int kt = 0; kt < KT; ++kt) {
        const int s = kt % STAGES;
        const uint32_t use = kt / STAGES;
        // hi/lo buffers of this stage must be free (MMAs of slab kt - STAGES done)
        // and its raw tiles must have landed
        if (kt >= STAGES && !mbar_wait(&done[s], (use - 1) & 1)) {
            atomicExch(&g_tf32x3_err, kDevErrWaitMma);
            *bad = 1;
        }
        if (!mbar_wait(&full[s], use & 1)) {
            atomicExch(&g_tf32x3_err, kDevErrWaitFull);
            *bad = 1;
        }
        __syncthreads();
        if (*bad) break;
        uint8_t *st = smem + s * STAGE_BYTES;
        uint8_t *rawA = st, *rawB = st + TILE, *Ahi = st + 2 * TILE, *Alo = st + 3 * TILE;
        uint8_t *Bhi = st + 4 * TILE, *Blo = st + 5 * TILE;
        if (A_KC) split_kmajor(rawA, Ahi, Alo, tid);
        else split_transpose(rawA, Ahi, Alo, tid);
        if (B_KC) split_kmajor(rawB, Bhi, Blo, tid);
        else split_transpose(rawB, Bhi, Blo, tid);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            // raw tiles of this stage are consumed: refill them with slab kt + STAGES
            if (kt + STAGES < KT) {
                issue_tma(kt + STAGES);
                ++issued;
            }
            tc_fence_after_sync();
            const uint32_t ah = smem_u32(Ahi), al = smem_u32(Alo), bh = smem_u32(Bhi), bl = smem_u32(Blo);
#pragma unroll
            for (int ks = 0; ks < BK / 8; ++ks) {
                const uint32_t o = 32 * ks;
                umma_tf32(tmem, sdesc_kmajor_sw128(ah + o), sdesc_kmajor_sw128(bh + o), idesc,
                          (kt > 0 || ks > 0) ? 1u : 0u);
                umma_tf32(tmem, sdesc_kmajor_sw128(ah + o), sdesc_kmajor_sw128(bl + o), idesc, 1u);
                umma_tf32(tmem, sdesc_kmajor_sw128(al + o), sdesc_kmajor_sw128(bh + o), idesc, 1u);
            }
            umma_commit(&done[s]);
        }
    }

    __syncthreads();
    const bool ok = !*bad;
    if (tid == 0) umma_commit(last);
    if (!mbar_wait(last, 0)) atomicExch(&g_tf32x3_err, kDevErrWaitMma);
    tc_fence_after_sync();
    if (ok) {
        const int row = m0 + 32 * warp + lane;
        const bool vec = (p.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
            if (row < p.M) {
                float *crow = p.C + (int64_t)row * p.ldc + n0 + c0;
                if (vec && n0 + c0 + 32 <= p.N) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(crow + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n0 + c0 + j < p.N) crow[j] = v[j];
                }
            }
        }
    }
    // every TMA copy issued must land before this CTA's shared memory is released
    if (tid == 0)
        for (int kt = issued > STAGES ? issued - STAGES : 0; kt < issued; ++kt)
            if (!mbar_wait(&full[kt % STAGES], (kt / STAGES) & 1)) {
                atomicExch(&g_tf32x3_err, kDevErrDrain);
                break;
            }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, BN);
}

template <bool A_KC, bool B_KC>
cudaError_t launch_x3(const CUtensorMap &ta, const CUtensorMap &tb, const Tf32x3Params &p, cudaStream_t s) {
    auto kern = gemm_tf32x3_kernel<A_KC, B_KC>;
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

bool gemm_tf32x3_supported(const GemmArgs &g) { return gemm_ffma_supported(g); }

cudaError_t launch_gemm_tf32x3(const GemmArgs &g, cudaStream_t s) {
    if (!gemm_tf32x3_supported(g)) return cudaErrorNotSupported;
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
    Tf32x3Params p{(int)g.M, (int)g.N, (int)g.K, g.C, g.ldc};
    if (!g.transA && !g.transB) return launch_x3<true, false>(ta, tb, p, s);
    if (!g.transA && g.transB) return launch_x3<true, true>(ta, tb, p, s);
    if (g.transA && !g.transB) return launch_x3<false, false>(ta, tb, p, s);
    return launch_x3<false, true>(ta, tb, p, s);
}

unsigned int gemm_tf32x3_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_tf32x3_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_tf32x3_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
