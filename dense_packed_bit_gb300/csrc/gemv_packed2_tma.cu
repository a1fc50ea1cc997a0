// gemv_packed2_tma.cu -- 2-bit GEMV with the code rows brought into shared
// memory by TMA and the tensor-core decode.
//
// "Kernel 0112", sections "What is being measured" and "What the kernel costs
// in a whole token": the 12,288 x 1,536 2-bit GEMV streams 4.5 MiB of weights
// and launches too few threads to keep enough reads in flight.  Here a CTA
// streams consecutive 64-row blocks (all of K) through a 2-deep shared-memory
// ring: thread 0 issues the TMA copies of the first two blocks before the
// kernel waits on anything (128-byte boxes with the 128-byte swizzle, so the
// later 16-byte shared loads of 8 different rows hit 8 different bank groups),
// then the CTA stages x while the bytes travel, and each finished block frees
// its slot for the block after next.  One warp per 256-field slab decodes its
// slab of each block (four 16-row MMA blocks) with the exact fp16 encoding of
// gemv_packed2_mma.cu and mma.sync; its x-dependent B operands and the sum of
// x are built once per CTA; the warps' partial sums are added in a fixed
// order through shared memory.  Few, long-lived CTAs per call keep loads in
// flight while they compute, and leave room for the next calls' CTAs when
// calls overlap through programmatic dependent launch.
//
// Requirements: cols % 512 == 0 (whole 128-byte boxes), cols <= 4096 (one
// warp per slab, at most 16 warps), 16-byte aligned codes and x, an affine
// codebook.
#include "gemv_mma.cuh"
#include "mm_internal.h"
#include "tmap.h"

#include <mutex>

namespace mm {

__device__ unsigned int g_gemv_tma_err;

namespace {

using namespace gemv_mma;

constexpr int ROWS = 64, RB = 4, BOX = 128 * ROWS;  // bytes of one 128-byte-wide box of 64 rows
constexpr int RING = 2;                              // 64-row blocks in flight per CTA

// A CTA handles `nblk` consecutive 64-row blocks: block i+1's TMA copies are in
// flight while block i is multiplied, the x-dependent B operands and the sum
// of x are built once per CTA, and each block's partial sums are combined over
// the slab warps in a fixed order.
__global__ void __launch_bounds__(512) gemv2_tma_kernel(const __grid_constant__ CUtensorMap tmC, const PackedArgs a,
                                                        const int prefetch, const int nblk) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    const int KW = blockDim.x >> 5;       // warps = 256-field slabs = cols / 256
    const int nbox = (int)(a.cols >> 9);  // 128-byte boxes per row
    const int stage_bytes = nbox * BOX;
    uint8_t *tiles = smem;  // [RING][nbox][64 rows][128 B], swizzled
    uint32_t *xw32 = reinterpret_cast<uint32_t *>(smem + RING * stage_bytes);
    float *red = reinterpret_cast<float *>(xw32 + (a.cols >> 1));  // [KW][65]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + ((KW * 65 + 1) & ~1));

    const int lane = threadIdx.x & 31, kw = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int blk0 = blockIdx.x * nblk;
    const int nrowblk = (int)((a.rows + ROWS - 1) / ROWS);
    const int my_blocks = min(nblk, nrowblk - blk0);

    if (threadIdx.x == 0) {
        for (int r = 0; r < RING; ++r) mbar_init(&full[r], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int i) {  // block i of this CTA into ring slot i % RING
        uint8_t *dst = tiles + (i % RING) * stage_bytes;
        mbar_arrive_expect_tx(&full[i % RING], (uint32_t)stage_bytes);
        for (int b = 0; b < nbox; ++b) tma_load_2d(dst + b * BOX, &tmC, &full[i % RING], b * 128, (blk0 + i) * ROWS);
    };
    auto issue_first = [&] {
        if (threadIdx.x == 0)
            for (int i = 0; i < RING && i < my_blocks; ++i) issue(i);
    };
    if (prefetch >= 1) {
        issue_first();
        // chained calls: the next call may launch only once this one has passed its wait,
        // so at most one call runs ahead (its weight loads) instead of a queue of parked ones
        if (prefetch == 1) pdl_wait();
        pdl_launch_dependents();
    } else {
        pdl_wait();
        issue_first();
        pdl_launch_dependents();
    }

    // ---- x -> xw[(chunk*8 + g)*4 + i] = (x[64c+16i+g], x[64c+16i+g+8]) while the codes travel
    {
        const int ne = (int)(a.cols >> 1);
        constexpr int XB = 4;
        for (int e0 = threadIdx.x; e0 < ne; e0 += XB * blockDim.x) {
            uint16_t lo[XB], hi[XB];
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                const int e = e0 + u * blockDim.x;
                if (e < ne) {
                    const int k = 64 * (e >> 5) + 16 * (e & 3) + ((e >> 2) & 7);
                    lo[u] = __ldg(a.x + k);
                    hi[u] = __ldg(a.x + k + 8);
                }
            }
#pragma unroll
            for (int u = 0; u < XB; ++u) {
                const int e = e0 + u * blockDim.x;
                if (e < ne) xw32[e] = (uint32_t)lo[u] | ((uint32_t)hi[u] << 16);
            }
        }
    }
    __syncthreads();

    // ---- per-CTA constants of slab kw: B operands (x masked to this thread's column) and sum x
    const int c = 4 * kw + t, box = c >> 3, cc = c & 7;
    const uint4 xv = reinterpret_cast<const uint4 *>(xw32)[c * 8 + g];
    uint32_t bop[2][8][2];
    float dx[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int wp = 0; wp < 2; ++wp)
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint32_t oh = (g == s) ? 0x3C003C00u : 0u;
            bop[wp][s][0] = hmul2_bits(word_of(xv, 2 * wp), oh);
            bop[wp][s][1] = hmul2_bits(word_of(xv, 2 * wp + 1), oh);
            const uint32_t one = slot_ones(s, true);
            mma16816(dx[s & 1], one, one, one, one, bop[wp][s][0], bop[wp][s][1]);
        }
    const float sc0 = col_scale<true>(2 * t), sc1 = col_scale<true>(2 * t + 1);
    float sx = __fadd_rn(__fmul_rn(__fadd_rn(dx[0][0], dx[1][0]), sc0), __fmul_rn(__fadd_rn(dx[0][1], dx[1][1]), sc1));
    sx += __shfl_xor_sync(0xffffffffu, sx, 1);
    sx += __shfl_xor_sync(0xffffffffu, sx, 2);
    if (lane == 0) red[kw * 65 + 64] = sx;
    const float c0 = a.cb[0], dd = a.cb[1] - a.cb[0];

    bool ok = true;
    for (int i = 0; i < my_blocks; ++i) {
        const int slot = i % RING;
        if (!mbar_wait(&full[slot], (i / RING) & 1)) {
            atomicExch(&g_gemv_tma_err, kDevErrWaitFull);
            ok = false;  // every thread of the CTA times out on the same copy
        }
        float d[RB][2][4];
#pragma unroll
        for (int b = 0; b < RB; ++b)
#pragma unroll
            for (int z = 0; z < 2; ++z) d[b][z][0] = d[b][z][1] = d[b][z][2] = d[b][z][3] = 0.f;
        if (ok) {
            const uint8_t *tb = tiles + slot * stage_bytes + box * BOX + ((cc ^ g) << 4);
            uint4 q[RB][2];  // rows 16b + g and 16b + g + 8 (both have row % 8 == g)
#pragma unroll
            for (int b = 0; b < RB; ++b)
#pragma unroll
                for (int h = 0; h < 2; ++h) q[b][h] = *reinterpret_cast<const uint4 *>(tb + (16 * b + g + 8 * h) * 128);
#pragma unroll
            for (int wp = 0; wp < 2; ++wp) {
                uint32_t w[RB][4], ws[RB][4];
#pragma unroll
                for (int b = 0; b < RB; ++b) {
                    w[b][0] = word_of(q[b][0], 2 * wp);
                    w[b][1] = word_of(q[b][1], 2 * wp);
                    w[b][2] = word_of(q[b][0], 2 * wp + 1);
                    w[b][3] = word_of(q[b][1], 2 * wp + 1);
#pragma unroll
                    for (int u = 0; u < 4; ++u) ws[b][u] = w[b][u] >> 10;
                }
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const uint32_t m = slot_mask(s);
#pragma unroll
                    for (int b = 0; b < RB; ++b) {
                        const uint32_t *src = s < 5 ? w[b] : ws[b];
                        mma16816(d[b][s & 1], slot_operand<true>(src[0], m), slot_operand<true>(src[1], m),
                                 slot_operand<true>(src[2], m), slot_operand<true>(src[3], m), bop[wp][s][0],
                                 bop[wp][s][1]);
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < RB; ++b)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = __fadd_rn(__fmul_rn(__fadd_rn(d[b][0][2 * h], d[b][1][2 * h]), sc0),
                                    __fmul_rn(__fadd_rn(d[b][0][2 * h + 1], d[b][1][2 * h + 1]), sc1));
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                if (t == 0) red[kw * 65 + 16 * b + g + 8 * h] = v;
            }
        __syncthreads();  // partial sums written; every warp is done with ring slot `slot`
        if (threadIdx.x == 0 && ok && i + RING < my_blocks) issue(i + RING);
        if (threadIdx.x < ROWS && ok) {
            const int r = threadIdx.x;
            const int64_t row = (int64_t)(blk0 + i) * ROWS + r;
            float s1 = red[r], sxa = red[64];
            for (int k = 1; k < KW; ++k) {
                s1 += red[k * 65 + r];
                sxa += red[k * 65 + 64];
            }
            if (row < a.rows) a.y[row] = h2f(a.scales[row]) * __fadd_rn(__fmul_rn(c0, sxa), __fmul_rn(dd, s1));
        }
        __syncthreads();  // the next block may overwrite the partial sums
        if (!ok) break;
    }
    // copies that missed their wait must land before the shared memory is released
    if (!ok && threadIdx.x == 0)
        for (int i = 0; i < RING && i < my_blocks; ++i)
            if (!mbar_wait(&full[i], 0) && !mbar_wait(&full[i], 1)) atomicExch(&g_gemv_tma_err, kDevErrDrain);
}

}  // namespace

bool gemv_tma_supported(const PackedArgs &a) {
    return a.cols % 512 == 0 && a.cols <= 4096 && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 && a.rows < ((int64_t)1 << 31);
}

cudaError_t launch_gemv_tma(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    if (!gemv_tma_supported(a)) return cudaErrorNotSupported;
    const int64_t rowbytes = a.cols / 4;
    CUtensorMap tm;
    cudaError_t e = make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, (uint64_t)rowbytes, (uint64_t)a.rows,
                                 (uint64_t)rowbytes, 128, ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(gemv2_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 180 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int kw = (int)(a.cols / 256);
    const int64_t nrowblk = (a.rows + ROWS - 1) / ROWS;
    const int nblk = cfg.blocks_per_cta > 0 ? cfg.blocks_per_cta : 1;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((nrowblk + nblk - 1) / nblk));
    lc.blockDim = dim3(32 * kw);
    lc.dynamicSmemBytes = 1024 + (size_t)RING * (a.cols / 512) * BOX + (size_t)a.cols * 2 + (size_t)kw * 65 * 4 + 64;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    return cudaLaunchKernelEx(&lc, gemv2_tma_kernel, tm, a, prefetch, nblk);
}

unsigned int gemv_tma_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_gemv_tma_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_gemv_tma_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
