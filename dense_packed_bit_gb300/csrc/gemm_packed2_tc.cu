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

constexpr int BM = 128, KATOM = 64;  // 64 fp16 along K = one 128-byte swizzle atom
constexpr int NCONS = 128, NTHREADS = NCONS + 32;  // 4 consumer warps + 1 producer warp
constexpr int ATOM_A = BM * KATOM * 2;             // 16 KiB of X per atom

struct TcPackedParams {
    const uint8_t *codes;
    const uint16_t *scales;
    float *y;
    int M, rows, cols;
    int64_t rowbytes;
    int ktiles;
    uint32_t cb16[2];
};

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// KA atoms (64 fields each) per pipeline stage; STAGES stages in the ring.
template <int BN, bool CODES_TMA, int KA>
struct TcLayout {
    static constexpr int BK = KATOM * KA;
    static constexpr int STAGES = KA == 1 ? 4 : (BN == 128 ? 3 : 2);
    static constexpr int A_BYTES = ATOM_A * KA;                   // X tile
    static constexpr int B_ATOM = BN * 128;                       // decoded W, one atom
    static constexpr int B_BYTES = B_ATOM * KA;
    static constexpr int C_BYTES = CODES_TMA ? BN * 16 * KA : 0;  // raw code bytes
    static constexpr int STAGE_BYTES = (A_BYTES + B_BYTES + C_BYTES + 1023) / 1024 * 1024;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + (2 * STAGES + 1) * 8 + 16 + 256 * 8 + 64;
};

// Output staging: the 128 x BN fp32 tile goes through shared memory (rows padded
// by 4 floats, conflict-free float4 writes from the TMEM-row-per-thread layout)
// so that each warp then stores whole contiguous row segments of Y, scaled by
// the per-row fp16 scale of W.
template <int BN>
__device__ __forceinline__ void stage_row(float *stile, int row_local, int c0, const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4 *>(stile + row_local * (BN + 4) + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
}

template <int BN>
__device__ __forceinline__ void store_staged_rows(const float *stile, int warp, int lane, int m0, int n0,
                                                  const TcPackedParams &p) {
    float sc[BN / 32];
#pragma unroll
    for (int q = 0; q < BN / 32; ++q) {
        const int nn = n0 + lane + 32 * q;
        sc[q] = nn < p.rows ? h2f(p.scales[nn]) : 0.f;
    }
    for (int rr = 0; rr < 32; ++rr) {
        const int rl = 32 * warp + rr, grow = m0 + rl;
        if (grow >= p.M) break;
        float *yrow = p.y + (int64_t)grow * p.rows;
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) {
            const int cc = lane + 32 * q, nn = n0 + cc;
            if (nn < p.rows) yrow[nn] = stile[rl * (BN + 4) + cc] * sc[q];
        }
    }
}

// Warp roles: warp 4 (one thread) streams X tiles -- and, when the code rows
// are 16-byte aligned, the code bytes -- into a STAGES-deep ring with TMA,
// running ahead until a stage's previous MMAs have released it; warps 0-3
// decode the codes of each stage into the swizzled fp16 W tile, thread 0
// issues the MMAs and commits them to the stage's "done" barrier, and after
// the last stage the same 128 threads read the accumulator (TMEM lanes 0-127).
template <int BN, bool CODES_TMA, bool SPLITK, int KA>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_packed2_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                           const TcPackedParams p) {
    using L = TcLayout<BN, CODES_TMA, KA>;
    constexpr int STAGES = L::STAGES;
    constexpr int TPR = NCONS / BN;     // consumer threads decoding one W row
    constexpr int BPT = 16 * KA / TPR;  // code bytes per thread per stage
    constexpr int TMEM_COLS = BN < 32 ? 32 : BN;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * L::STAGE_BYTES);
    uint64_t *done = full + STAGES;
    uint64_t *last = done + STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(last + 1);
    int *cbad = reinterpret_cast<int *>(tmem_slot + 1);
    uint2 *lut = reinterpret_cast<uint2 *>(tmem_slot + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    // split-K: CTA z of the (1, 1, S) cluster owns k-tiles [kt_begin, kt_end)
    const int S = gridDim.z, z = blockIdx.z;
    const int kt_begin = (int)((int64_t)z * p.ktiles / S), kt_end = (int)((int64_t)(z + 1) * p.ktiles / S);

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
        *cbad = 0;
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == NCONS / 32) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            if (CODES_TMA) tma_prefetch_desc(&tmC);
            int issued = 0;
            for (int kt = kt_begin; kt < kt_end; ++kt) {
                const int i = kt - kt_begin;
                const int s = i % STAGES;
                const uint32_t use = i / STAGES;
                if (i >= STAGES && !mbar_wait(&done[s], (use - 1) & 1)) {
                    atomicExch(&g_tc_packed_err, kDevErrWaitEmpty);
                    break;
                }
                uint8_t *st = smem + s * L::STAGE_BYTES;
                mbar_arrive_expect_tx(&full[s], L::A_BYTES + L::C_BYTES);
#pragma unroll
                for (int a = 0; a < KA; ++a) tma_load_2d(st + a * ATOM_A, &tmX, &full[s], kt * L::BK + a * KATOM, m0);
                if (CODES_TMA) tma_load_2d(st + L::A_BYTES + L::B_BYTES, &tmC, &full[s], kt * 16 * KA, n0);
                ++issued;
            }
            for (int kt = issued > STAGES ? issued - STAGES : 0; kt < issued; ++kt)
                if (!mbar_wait(&full[kt % STAGES], (kt / STAGES) & 1)) {
                    atomicExch(&g_tc_packed_err, kDevErrDrain);
                    break;
                }
        }
    } else {
        // ------------------------------------------------------------ consumers
        constexpr uint32_t idesc = make_idesc(kFmtF16, kFmtF16, BN, BM);
        const int r = tid / TPR, part = tid % TPR;  // W row decoded by this thread, and which slice
        const int64_t n = (int64_t)n0 + r;
        const uint8_t *wrow = p.codes + n * p.rowbytes;
        for (int kt = kt_begin; kt < kt_end; ++kt) {
            const int i = kt - kt_begin;
            const int s = i % STAGES;
            const uint32_t use = i / STAGES;
            // the stage's X (and code) tiles have landed; the producer only refilled it after
            // the MMAs of its previous use completed, so the W tile is free as well
            if (!mbar_wait(&full[s], use & 1)) {
                atomicExch(&g_tc_packed_err, kDevErrWaitFull);
                *cbad = 1;
            }
            bar_sync(1, NCONS);
            if (*cbad) break;
            uint8_t *sA = smem + s * L::STAGE_BYTES;
            uint8_t *sB = sA + L::A_BYTES;
            uint8_t bytes[BPT];
            if (CODES_TMA) {
                const uint8_t *src = sB + L::B_BYTES + r * 16 * KA + part * BPT;
                if (BPT == 32) {
                    const uint4 v0 = *reinterpret_cast<const uint4 *>(src);
                    const uint4 v1 = *reinterpret_cast<const uint4 *>(src + 16);
                    const uint32_t w8[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                    for (int i = 0; i < BPT; ++i) bytes[i] = (uint8_t)(w8[i >> 2] >> (8 * (i & 3)));
                } else if (BPT == 16) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(src);
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < BPT; ++i) bytes[i] = (uint8_t)(w4[i >> 2] >> (8 * (i & 3)));
                } else if (BPT == 8) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(src);
                    const uint32_t w2[2] = {v.x, v.y};
#pragma unroll
                    for (int i = 0; i < BPT; ++i) bytes[i] = (uint8_t)(w2[i >> 2] >> (8 * (i & 3)));
                } else {
                    const uint32_t v = *reinterpret_cast<const uint32_t *>(src);
#pragma unroll
                    for (int i = 0; i < BPT; ++i) bytes[i] = (uint8_t)(v >> (8 * i));
                }
            } else {
                const int64_t b0 = (int64_t)kt * 16 * KA + part * BPT;
#pragma unroll
                for (int i = 0; i < BPT; ++i)
                    bytes[i] = (n < p.rows && b0 + i < p.rowbytes) ? wrow[b0 + i] : (uint8_t)0;
            }
#pragma unroll
            for (int c = 0; c < BPT / 2; ++c) {
                const uint2 lo = lut[bytes[2 * c]], hi = lut[bytes[2 * c + 1]];
                const int chunk = part * (BPT / 2) + c;  // 16-byte chunk along K (0 .. 8*KA-1)
                const int atom = chunk >> 3, cc = chunk & 7;
                *reinterpret_cast<uint4 *>(sB + atom * L::B_ATOM + r * 128 + ((cc ^ (r & 7)) << 4)) =
                    make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
            fence_proxy_async_smem();
            bar_sync(1, NCONS);
            if (tid == 0) {
                tc_fence_after_sync();
                const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
#pragma unroll
                for (int ks = 0; ks < L::BK / 16; ++ks) {
                    const uint32_t ao = (ks >> 2) * ATOM_A + 32 * (ks & 3), bo = (ks >> 2) * L::B_ATOM + 32 * (ks & 3);
                    umma_f16(tmem, sdesc_kmajor_sw128(a_base + ao), sdesc_kmajor_sw128(b_base + bo), idesc,
                             (i > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(&done[s]);
            }
        }
        const bool ok = !*cbad && kt_end > kt_begin;
        if (tid == 0) umma_commit(last);
        if (!mbar_wait(last, 0)) atomicExch(&g_tc_packed_err, kDevErrWaitMma);
        tc_fence_after_sync();
        if (!SPLITK && ok) {
            float *stile = reinterpret_cast<float *>(smem);  // the ring is idle: every copy has landed
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
                stage_row<BN>(stile, 32 * warp + lane, c0, v);
            }
            __syncwarp();
            store_staged_rows<BN>(stile, warp, lane, m0, n0, p);
        }
        if (SPLITK && z != 0) {
            // partial tile -> own shared memory (the ring is idle now), row-major 128 x BN fp32
            float *part = reinterpret_cast<float *>(smem);
            const int row = 32 * warp + lane;
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                if (ok) tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
                else
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(part + row * BN + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
        }
    }
    if (SPLITK) {
        // rank 0 adds the partial tiles of ranks 1..S-1 in rank order (deterministic)
        cluster_sync();
        if (z == 0 && warp < NCONS / 32) {
            const int row = 32 * warp + lane;
            const bool ok = !*cbad && kt_end > kt_begin;
            const uint32_t part0 = smem_u32(smem);
#pragma unroll
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                if (ok) tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, v);
                else
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                for (int rk = 1; rk < S; ++rk) {
                    const uint32_t peer = cluster_map(part0, (uint32_t)rk) + (uint32_t)((row * BN + c0) * 4);
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        const float4 q = ld_cluster_v4(peer + 4 * j);
                        v[j] += q.x;
                        v[j + 1] += q.y;
                        v[j + 2] += q.z;
                        v[j + 3] += q.w;
                    }
                }
                // rank 0 never exposes its own ring to the peers: stage the sum there
                stage_row<BN>(reinterpret_cast<float *>(smem), row, c0, v);
            }
            __syncwarp();
            store_staged_rows<BN>(reinterpret_cast<const float *>(smem), warp, lane, m0, n0, p);
        }
        // peers keep their shared memory alive until rank 0 has read it
        cluster_sync();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

template <int BN, bool CODES_TMA, bool SPLITK, int KA>
cudaError_t launch_tc(const CUtensorMap &tx, const CUtensorMap &tc, const TcPackedParams &p, int splitk,
                      cudaStream_t st) {
    using L = TcLayout<BN, CODES_TMA, KA>;
    auto kern = gemm_packed2_tc_kernel<BN, CODES_TMA, SPLITK, KA>;
    constexpr int smem = L::SMEM;
    static_assert(L::STAGES * L::STAGE_BYTES >= BM * (BN + 4) * 4, "tiles must fit the ring");
    static_assert(smem <= 227 * 1024, "shared memory");
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((p.rows + BN - 1) / BN), (unsigned)((p.M + BM - 1) / BM), (unsigned)splitk);
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = smem;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)splitk;
    lc.attrs = attr;
    lc.numAttrs = SPLITK ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kern, tx, tc, p);
}

template <bool CODES_TMA, int KA>
cudaError_t launch_tc_bn(int bn, int splitk, const CUtensorMap &tx, const CUtensorMap &tc, const TcPackedParams &p,
                         cudaStream_t st) {
    if (splitk > 1) {
        switch (bn) {
            case 32: return launch_tc<32, CODES_TMA, true, KA>(tx, tc, p, splitk, st);
            case 64: return launch_tc<64, CODES_TMA, true, KA>(tx, tc, p, splitk, st);
            case 128: return launch_tc<128, CODES_TMA, true, KA>(tx, tc, p, splitk, st);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
        case 32: return launch_tc<32, CODES_TMA, false, KA>(tx, tc, p, 1, st);
        case 64: return launch_tc<64, CODES_TMA, false, KA>(tx, tc, p, 1, st);
        case 128: return launch_tc<128, CODES_TMA, false, KA>(tx, tc, p, 1, st);
        default: return cudaErrorInvalidValue;
    }
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

cudaError_t launch_gemm_packed2_tc(const PackedArgs &a, int tile, int splitk_req, cudaStream_t st) {
    if (!gemm_packed2_tc_supported(a)) return cudaErrorNotSupported;
    TcPackedParams p{};
    p.codes = a.codes;
    p.scales = a.scales;
    p.y = a.y;
    p.M = (int)a.M;
    p.rows = (int)a.rows;
    p.cols = (int)a.cols;
    p.rowbytes = (a.cols + 3) / 4;
    const bool codes_tma = (a.cols % 64 == 0) && (reinterpret_cast<uintptr_t>(a.codes) % 16 == 0);
    // two swizzle atoms (128 fields) per stage when the rows are whole 128-field steps
    const int ka = (codes_tma && a.cols % 128 == 0) ? 2 : 1;
    p.ktiles = (int)((a.cols + 64 * ka - 1) / (64 * ka));
    uint16_t h[4];
    for (int i = 0; i < 4; ++i) fp16_exact(a.cb[i], &h[i]);
    p.cb16[0] = h[0] | ((uint32_t)h[1] << 16);
    p.cb16[1] = h[2] | ((uint32_t)h[3] << 16);
    // enough CTAs to cover the SMs: narrower W tiles when there are few rows, then
    // split K over a cluster of up to 8 CTAs (each keeping at least 4 k-tiles)
    const int64_t mt = (a.M + BM - 1) / BM;
    int bn = tile;
    if (bn == 0) {
        bn = 128;
        while (bn > 32 && ((a.rows + bn - 1) / bn) * mt < 120) bn /= 2;
    }
    const int64_t ctas = ((a.rows + bn - 1) / bn) * mt;
    int splitk = splitk_req;
    if (splitk == 0) splitk = (ctas < 100 && p.ktiles >= 16) ? 2 : 1;  // measured best on GB300
    CUtensorMap tx, tc;
    cudaError_t e = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.x, (uint64_t)a.cols, (uint64_t)a.M,
                                 (uint64_t)a.cols * 2, KATOM, BM, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    if (codes_tma) {
        e = make_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, (uint64_t)p.rowbytes, (uint64_t)a.rows,
                         (uint64_t)p.rowbytes, 16 * ka, (uint32_t)bn, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (e != cudaSuccess) return e;
        return ka == 2 ? launch_tc_bn<true, 2>(bn, splitk, tx, tc, p, st) : launch_tc_bn<true, 1>(bn, splitk, tx, tc, p, st);
    }
    tc = tx;  // unused by the kernel variant that loads code bytes itself
    return launch_tc_bn<false, 1>(bn, splitk, tx, tc, p, st);
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
