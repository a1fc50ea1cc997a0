// gemm_packed2_tc.cu -- Y = X . (diag(scale) W)^T on the tcgen05 tensor cores.
//
// "More Stumbling, This Time in the Browser", sections "This time, in a
// browser" and "The attractive ideas that went away": the 16-layer ternary
// encoder (111-token input, 2 questions) multiplies a short batch of
// activations by packed ternary weights.  That is a dense contraction
// (M = 222 rows, K = 768 or 3072, N = 3072 or 768), so here it runs as one:
//
//  * A = X tile, 128 rows x 64 fp16 along K, loaded by TMA with the 128-byte
//    swizzle (K-major);
//  * B = W tile, BN rows x 64 fields, decoded by the CTA's threads straight
//    into the same swizzled K-major fp16 layout: each code byte (4 fields)
//    indexes a 256-entry table of 4 fp16 codebook entries;
//  * one thread issues tcgen05.mma kind::f16 (fp16 x fp16 products are exact,
//    accumulation in fp32 in tensor memory), 4 MMAs of K = 16 per 64-field
//    stage, and commits each stage to an mbarrier that frees its buffers;
//  * a 3-stage ring overlaps the TMA of stage k+1 and the decode of stage k+1
//    with the MMAs of stage k;
//  * the epilogue reads the 128 x BN fp32 accumulator with tcgen05.ld, applies
//    the per-row fp16 scale of W and stores Y with edge masks.
// The codebook entries must be exact in fp16 (they are for the 2-bit and
// ternary codebooks); others go to the FFMA kernel.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tmap.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {

__device__ unsigned int g_tc_packed_err;

namespace {

constexpr int BM = 128, BK = 64, STAGES = 3, NTHREADS = 128;
constexpr int A_BYTES = BM * BK * 2;  // 16 KiB

struct TcPackedParams {
    const uint8_t *codes;
    const uint16_t *scales;
    float *y;
    int M, rows, cols;
    int64_t rowbytes;
    int ktiles;
    int codes_vec;  // rows 16-byte aligned and cols % 64 == 0
    uint32_t cb16[2];
};

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

template <int BN>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_packed2_tc_kernel(const __grid_constant__ CUtensorMap tmX, const TcPackedParams p) {
    constexpr int B_BYTES = BN * BK * 2;
    constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    constexpr int TPR = NTHREADS / BN;  // threads decoding one W row
    constexpr int BPT = 16 / TPR;       // code bytes per thread per stage
    constexpr int TMEM_COLS = BN < 32 ? 32 : BN;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *done = full + STAGES;
    uint64_t *last = done + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(last + 1);
    int *bad = reinterpret_cast<int *>(tmem_slot + 1);
    uint2 *lut = reinterpret_cast<uint2 *>(tmem_slot + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;

    // byte -> fp16 codebook entries of its 4 fields, in K order
    for (int b = tid; b < 256; b += NTHREADS) {
        uint32_t h[4];
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            const uint32_t c = (b >> (2 * f)) & 3u;
            h[f] = (p.cb16[c >> 1] >> (16 * (c & 1))) & 0xFFFFu;
        }
        lut[b] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, TMEM_COLS);
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
        tma_prefetch_desc(&tmX);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    constexpr uint32_t idesc = make_idesc(kFmtF16, kFmtF16, BN, BM);

    const int r = tid / TPR, part = tid % TPR;  // W row decoded by this thread, and which slice
    const int64_t n = (int64_t)n0 + r;
    const uint8_t *wrow = p.codes + n * p.rowbytes;
    int issued = 0;  // stages whose TMA thread 0 issued

    for (int kt = 0; kt < p.ktiles; ++kt) {
        const int s = kt % STAGES;
        const uint32_t use = kt / STAGES;
        if (kt >= STAGES && !mbar_wait(&done[s], (use - 1) & 1)) {
            atomicExch(&g_tc_packed_err, kDevErrWaitMma);
            *bad = 1;
        }
        __syncthreads();
        if (*bad) break;
        uint8_t *sA = smem + s * STAGE_BYTES;
        uint8_t *sB = sA + A_BYTES;
        if (tid == 0) {
            mbar_arrive_expect_tx(&full[s], A_BYTES);
            tma_load_2d(sA, &tmX, &full[s], kt * BK, m0);
            ++issued;
        }
        // ---- decode BPT code bytes of row r (8 fields -> one 16-byte fp16 chunk per 2 bytes)
        uint8_t bytes[BPT];
        const int64_t b0 = (int64_t)kt * 16 + part * BPT;
        if (n < p.rows) {
            if (p.codes_vec) {
                if (BPT == 16) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(wrow + b0);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < BPT; ++i) bytes[i] = (uint8_t)(w4[i >> 2] >> (8 * (i & 3)));
                } else if (BPT == 8) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(wrow + b0);
                    const uint32_t w2[2] = {v.x, v.y};
#pragma unroll
                    for (int i = 0; i < BPT; ++i) bytes[i] = (uint8_t)(w2[i >> 2] >> (8 * (i & 3)));
                } else {
                    const uint32_t v = *reinterpret_cast<const uint32_t *>(wrow + b0);
#pragma unroll
                    for (int i = 0; i < BPT; ++i) bytes[i] = (uint8_t)(v >> (8 * i));
                }
            } else {
#pragma unroll
                for (int i = 0; i < BPT; ++i) bytes[i] = (b0 + i < p.rowbytes) ? wrow[b0 + i] : (uint8_t)0;
            }
        } else {
#pragma unroll
            for (int i = 0; i < BPT; ++i) bytes[i] = 0;
        }
#pragma unroll
        for (int c = 0; c < BPT / 2; ++c) {
            const uint2 lo = lut[bytes[2 * c]], hi = lut[bytes[2 * c + 1]];
            const int chunk = part * (BPT / 2) + c;  // 16-byte chunk along K (0..7)
            *reinterpret_cast<uint4 *>(sB + r * 128 + ((chunk ^ (r & 7)) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            if (!mbar_wait(&full[s], use & 1)) {
                atomicExch(&g_tc_packed_err, kDevErrWaitFull);
                *bad = 1;
            } else {
                tc_fence_after_sync();
                const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
#pragma unroll
                for (int ks = 0; ks < BK / 16; ++ks)
                    umma_f16(tmem, sdesc_kmajor_sw128(a_base + 32 * ks), sdesc_kmajor_sw128(b_base + 32 * ks), idesc,
                             (kt > 0 || ks > 0) ? 1u : 0u);
            }
            umma_commit(&done[s]);
        }
    }

    // ---- wait for every MMA, then read the accumulator
    __syncthreads();
    const bool ok = !*bad;
    if (tid == 0) umma_commit(last);
    if (!mbar_wait(last, 0)) atomicExch(&g_tc_packed_err, kDevErrWaitMma);
    tc_fence_after_sync();
    if (ok) {
        const int row = m0 + 32 * warp + lane;
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
            if (row < p.M) {
                float *yrow = p.y + (int64_t)row * p.rows;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int nn = n0 + c0 + j;
                    if (nn < p.rows) yrow[nn] = v[j] * h2f(p.scales[nn]);
                }
            }
        }
    }
    // copies still in flight (only after a failed wait) must land before the CTA exits
    if (tid == 0 && !ok)
        for (int kt = issued > STAGES ? issued - STAGES : 0; kt < issued; ++kt)
            if (!mbar_wait(&full[kt % STAGES], (kt / STAGES) & 1)) {
                atomicExch(&g_tc_packed_err, kDevErrDrain);
                break;
            }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

template <int BN>
cudaError_t launch_tc(const CUtensorMap &tm, const TcPackedParams &p, cudaStream_t st) {
    auto kern = gemm_packed2_tc_kernel<BN>;
    constexpr int smem = STAGES * (A_BYTES + BN * BK * 2) + 1024 + 2 * STAGES * 8 + 8 + 8 + 256 * 8 + 64;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
    if (attr_err != cudaSuccess) return attr_err;
    dim3 grid((unsigned)((p.rows + BN - 1) / BN), (unsigned)((p.M + BM - 1) / BM));
    kern<<<grid, NTHREADS, smem, st>>>(tm, p);
    return cudaGetLastError();
}

bool fp16_exact(float v, uint16_t *bits) {
    const __half h = __float2half_rn(v);
    if (__half2float(h) != v) return false;
    *bits = *reinterpret_cast<const uint16_t *>(&h);
    return true;
}

}  // namespace

bool gemm_packed2_tc_supported(const PackedArgs &a) {
    uint16_t b;
    for (int i = 0; i < 4; ++i)
        if (!fp16_exact(a.cb[i], &b)) return false;
    return a.cols % 8 == 0 && (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 && a.M < (1 << 30) &&
           a.rows < (1 << 30) && a.cols < (1 << 30) && (a.M + BM - 1) / BM < 65536;
}

cudaError_t launch_gemm_packed2_tc(const PackedArgs &a, int tile, cudaStream_t st) {
    if (!gemm_packed2_tc_supported(a)) return cudaErrorNotSupported;
    TcPackedParams p{};
    p.codes = a.codes;
    p.scales = a.scales;
    p.y = a.y;
    p.M = (int)a.M;
    p.rows = (int)a.rows;
    p.cols = (int)a.cols;
    p.rowbytes = (a.cols + 3) / 4;
    p.ktiles = (int)((a.cols + BK - 1) / BK);
    p.codes_vec = (a.cols % 64 == 0) && (reinterpret_cast<uintptr_t>(a.codes) % 16 == 0);
    uint16_t h[4];
    for (int i = 0; i < 4; ++i) fp16_exact(a.cb[i], &h[i]);
    p.cb16[0] = h[0] | ((uint32_t)h[1] << 16);
    p.cb16[1] = h[2] | ((uint32_t)h[3] << 16);
    CUtensorMap tm;
    cudaError_t e = make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.x, (uint64_t)a.cols, (uint64_t)a.M,
                                 (uint64_t)a.cols * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    // enough CTAs to cover the SMs: narrower W tiles when there are few rows
    int bn = tile;
    if (bn == 0) {
        const int64_t mt = (a.M + BM - 1) / BM;
        bn = 128;
        while (bn > 32 && ((a.rows + bn - 1) / bn) * mt < 120) bn /= 2;
    }
    switch (bn) {
        case 32: return launch_tc<32>(tm, p, st);
        case 64: return launch_tc<64>(tm, p, st);
        case 128: return launch_tc<128>(tm, p, st);
        default: return cudaErrorInvalidValue;
    }
}

unsigned int gemm_packed2_tc_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_tc_packed_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_tc_packed_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
