// gemv_packed2_rows.cu -- 2-bit GEMV, SIMT affine decode, code tiles staged
// by TMA and one lane per row.
//
// "Kernel 0112", sections "What is being measured" and "The four variants":
// the 12,288 x 1,536 GEMV is bound by how fast 18.9 M fields a call become
// products.  This kernel keeps everything but the decode off the hot loop:
//
//  * a CTA streams 128-row blocks of code rows through a TMA ring (128-byte
//    boxes with the 128-byte swizzle); lane l of every warp owns rows l, l+32,
//    l+64, l+96 of the block, so a row's partial sum never crosses lanes and
//    needs no shuffles;
//  * warp w owns the 64-field chunks w, w+8, w+16, ... of every row: for each
//    code word it reads the word's 16 fp16 x values once (shared-memory
//    broadcast, all lanes the same address) and applies them to its four rows;
//  * the eight warps' partial sums of a row, and of sum x, are added in warp
//    order through shared memory (reproducible bit for bit), into one of two
//    buffers by block parity so that a block needs a single barrier.
//
// Decode (exact).  One LOP3 keeps two fields of a code word, at bits q and
// 16 + q with q <= 8, and the two 16-bit halves read as fp16 are the
// subnormals c 2^(q-24); fields 5-7 and 13-15 take the word shifted right by
// 10 first.  Each half is multiplied by its field's fp16 x with fma.rn.f32.f16
// (fp16 inputs, fp32 accumulator; the product c x 2^(q-24) has at most 13
// significant bits, so it is exact) into one of five fp32 accumulators, one
// per q; at the end they are scaled by 2^(24-q) (exact) and added.  Half the
// integer operations of masking every field into an fp32 word for a packed
// f32x2 FMA (1.36 against 1.67 us per 12,288 x 1,536 matrix on GB300), for
// the same instruction count.  sum x runs through the same FMAs with every
// field equal to 1 and is reduced in the same order, so a row of zero-entry
// fields gives exactly 0.
//
// Requirements: cols % 512 == 0, cols <= 4096, 16-byte aligned codes, an
// affine codebook (zero entry, if any, at field 0, 1 or 2).  The batched form
// at the end of the file runs many matrices in one launch.
#include "gemv_mixed.cuh"
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tmap.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {

__device__ unsigned int g_gemv_rows_err;

namespace {

constexpr int ROWS = 128;          // rows per block: one TMA box height
constexpr int BOX = 128 * ROWS;    // bytes of one 128-byte-wide box of 128 rows
constexpr int NWARPS = 8, NTHREADS = 32 * NWARPS;
constexpr int RPL = ROWS / 32;     // rows per lane

// CPW: 64-field chunks per warp (cols = 512 CPW), a template parameter so that the
// chunk loops unroll completely.
template <int CPW>
__global__ void __launch_bounds__(NTHREADS) gemv2_rows_kernel(const __grid_constant__ CUtensorMap tmC,
                                                              const PackedArgs a, const int prefetch, const int nblk,
                                                              const int ring) {
    extern __shared__ uint8_t smem_raw[];
    // set by a thread whose bounded wait for block i ran out, in slot i & 1 (the next block may
    // already be waiting while a slower thread reads this block's slot after the barrier)
    __shared__ int s_fail[2];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    constexpr int cols = 512 * CPW;
    constexpr int nbox = CPW;     // 128-byte boxes per row
    constexpr int stage_bytes = nbox * BOX;
    uint8_t *tiles = smem;                                                       // [ring][nbox][128 rows][128 B]
    float4 *xs = reinterpret_cast<float4 *>(smem + (size_t)ring * stage_bytes);  // prepared x, cols floats
    float *redx = reinterpret_cast<float *>(xs + (cols >> 2));  // [NWARPS] sum x partials
    float *redb = redx + NWARPS;                                   // [2][NWARPS][ROWS]: row partials, by block parity
    uint64_t *full = reinterpret_cast<uint64_t *>(redb + 2 * NWARPS * ROWS);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int blk0 = blockIdx.x * nblk;
    const int nrowblk = (int)((a.rows + ROWS - 1) / ROWS);
    const int my_blocks = min(nblk, nrowblk - blk0);
    const bool leader = threadIdx.x == 0;

    if (leader) {
        s_fail[0] = 0;
        s_fail[1] = 0;
        for (int r = 0; r < ring; ++r) mbar_init(&full[r], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int i) {  // block i of this CTA into ring slot i % ring
        uint8_t *dst = tiles + (size_t)(i % ring) * stage_bytes;
        mbar_arrive_expect_tx(&full[i % ring], (uint32_t)stage_bytes);
        for (int b = 0; b < nbox; ++b) tma_load_2d(dst + b * BOX, &tmC, &full[i % ring], b * 128, (blk0 + i) * ROWS);
    };
    const int first = min(ring, my_blocks);
    if (prefetch >= 1) {
        if (leader) {
            tma_prefetch_desc(&tmC);
            for (int i = 0; i < first; ++i) issue(i);
        }
        // chained calls: the next call may launch only once this one has passed its wait,
        // so at most one call runs ahead (its weight loads) instead of a queue of parked ones
        if (prefetch == 1) pdl_wait();
        pdl_launch_dependents();
    } else {
        pdl_wait();
        if (leader) {
            tma_prefetch_desc(&tmC);
            for (int i = 0; i < first; ++i) issue(i);
        }
        pdl_launch_dependents();
    }

    // ---- x (fp16) -> shared memory as it is
    uint4 *xr = reinterpret_cast<uint4 *>(xs);
    for (int g = threadIdx.x; g < (cols >> 3); g += NTHREADS) xr[g] = __ldg(reinterpret_cast<const uint4 *>(a.x) + g);
    __syncthreads();

    // ---- this warp's sum of x over its chunks, by the same FMAs as the rows (every field 1)
    {
        float ax[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < CPW; ++m)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint4 *xq = xr + 2 * (4 * (warp + NWARPS * m) + u);
                const uint4 xa = xq[0], xb = xq[1];
                const uint32_t X[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
                word_mixed(0x55555555u, X, ax);
            }
        if (lane == 0) redx[warp] = mixed_total(ax);
    }
    const float c0 = a.cb[0], dd = a.cb[1] - a.cb[0];
    float sxr = 0.f;  // sum x (threads 0..127), set at the first block

    bool ok = true;
    int waited = 0;
    for (int i = 0; i < my_blocks && ok; ++i) {
        const int slot = i % ring;
        // scale of this thread's row (threads 0..127), read while the codes travel
        float scl = 0.f;
        const int64_t row = (int64_t)(blk0 + i) * ROWS + threadIdx.x;
        if (threadIdx.x < ROWS && row < a.rows) scl = __half2float(__ushort_as_half(a.scales[row]));
        if (!mbar_wait_sleep(&full[slot], (i / ring) & 1)) {
            atomicExch(&g_gemv_rows_err, kDevErrWaitFull);
            s_fail[i & 1] = 1;  // the bytes read below are then garbage, but every access stays in bounds
        }
        const uint8_t *tile = tiles + (size_t)slot * stage_bytes;
        float acc[RPL][5];
#pragma unroll
        for (int j = 0; j < RPL; ++j)
#pragma unroll
            for (int c5 = 0; c5 < 5; ++c5) acc[j][c5] = 0.f;
#pragma unroll
        for (int m = 0; m < CPW; ++m) {
            const int c = warp + NWARPS * m;  // chunk c lives in box m, at chunk position warp of the box
            const uint8_t *bp = tile + m * BOX + ((warp ^ (lane & 7)) << 4);  // rows lane + 32 j: row % 8 == lane % 8
            uint4 q[RPL];
#pragma unroll
            for (int j = 0; j < RPL; ++j) q[j] = *reinterpret_cast<const uint4 *>(bp + (lane + 32 * j) * 128);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint4 *xq = xr + 2 * (4 * c + u);
                const uint4 xa = xq[0], xb = xq[1];
                const uint32_t X[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
                for (int j = 0; j < RPL; ++j) {
                    const uint32_t w = u == 0 ? q[j].x : u == 1 ? q[j].y : u == 2 ? q[j].z : q[j].w;
                    word_mixed(w, X, acc[j]);
                }
            }
        }
        float *red = redb + (i & 1) * NWARPS * ROWS;
#pragma unroll
        for (int j = 0; j < RPL; ++j) red[warp * ROWS + lane + 32 * j] = mixed_total(acc[j]);
        __syncthreads();  // partial sums written; every warp is done with ring slot `slot`
        ok = reinterpret_cast<volatile int *>(s_fail)[i & 1] == 0;
        if (!ok) break;  // taken by every thread: the flag was read after the barrier
        waited = i + 1;
        if (leader && i + ring < my_blocks) issue(i + ring);
        if (threadIdx.x < ROWS) {
            const int r = threadIdx.x;
            if (i == 0) {
                sxr = redx[0];
                for (int k = 1; k < NWARPS; ++k) sxr += redx[k];
            }
            float s1 = red[r];
            for (int k = 1; k < NWARPS; ++k) s1 += red[k * ROWS + r];
            if (row < a.rows) a.y[row] = scl * __fadd_rn(__fmul_rn(c0, sxr), __fmul_rn(dd, s1));
        }
        // no second barrier: the next block writes the other half of the double-buffered partial
        // sums, and this half is rewritten only after the next block's barrier
    }
    // copies in flight after a failed wait must land before the shared memory is released
    if (!ok && leader) {
        const int issued = min(my_blocks, waited + ring);
        for (int j = waited; j < issued; ++j)
            if (!mbar_wait(&full[j % ring], (j / ring) & 1)) atomicExch(&g_gemv_rows_err, kDevErrDrain);
    }
}

// ---------------------------------------------------------------- batches of matrices
//
// y_b = scale_b (c0 sum x_b + d W_b x_b) for b < batch in one launch: a persistent grid,
// each CTA taking a contiguous run of the batch's 128-row blocks, so that it meets one or
// two matrices and prepares x only when the matrix changes (never, when every matrix
// shares one x); the code blocks stream through a two-stage ring by 3-D TMA
// (coordinates: byte in row, row, matrix).  Per block the arithmetic is the kernel's
// above, in the same order, so each y_b equals bit for bit what one staged call gives.
// One launch instead of one per matrix removes the per-call launch and ramp cost.

struct BatchArgs {
    const uint16_t *scales;
    int64_t scales_stride;  // entries between matrices
    const uint16_t *x;
    int64_t x_stride;       // entries between matrices; 0: one x for every matrix
    float *y;
    int64_t y_stride;       // entries between matrices
    int64_t rows;
    int64_t nrowblk;        // 128-row blocks per matrix
    int64_t total;          // blocks of the batch
    float c0, dd;           // codebook[0], codebook[1] - codebook[0]
};

template <int CPW>
__global__ void __launch_bounds__(NTHREADS) gemv2_batched_kernel(const __grid_constant__ CUtensorMap tmC,
                                                                 const BatchArgs a, const int ring) {
    extern __shared__ uint8_t smem_raw[];
    // set by a thread whose bounded wait for block i ran out, in slot i & 1 (the next block may
    // already be waiting while a slower thread reads this block's slot after the barrier)
    __shared__ int s_fail[2];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    constexpr int cols = 512 * CPW;
    constexpr int nbox = CPW;
    constexpr int stage_bytes = nbox * BOX;
    uint8_t *tiles = smem;
    float4 *xs = reinterpret_cast<float4 *>(smem + (size_t)ring * stage_bytes);
    float *redx = reinterpret_cast<float *>(xs + (cols >> 2));        // [NWARPS] sum x partials
    float *redb = redx + NWARPS;                                         // [2][NWARPS][ROWS]
    uint64_t *full = reinterpret_cast<uint64_t *>(redb + 2 * NWARPS * ROWS);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool leader = threadIdx.x == 0;
    const int64_t per = (a.total + gridDim.x - 1) / gridDim.x;
    const int64_t g0 = (int64_t)blockIdx.x * per;
    const int my = (int)(a.total - g0 < per ? (a.total - g0 > 0 ? a.total - g0 : 0) : per);

    if (leader) {
        s_fail[0] = 0;
        s_fail[1] = 0;
        for (int r = 0; r < ring; ++r) mbar_init(&full[r], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int i) {  // block g0 + i into ring slot i % ring
        const int64_t g = g0 + i;
        const int b = (int)(g / a.nrowblk), rb = (int)(g % a.nrowblk);
        uint8_t *dst = tiles + (size_t)(i % ring) * stage_bytes;
        mbar_arrive_expect_tx(&full[i % ring], (uint32_t)stage_bytes);
        for (int k = 0; k < nbox; ++k) tma_load_3d(dst + k * BOX, &tmC, &full[i % ring], k * 128, rb * ROWS, b);
    };
    if (leader) {
        tma_prefetch_desc(&tmC);
        for (int i = 0; i < min(ring, my); ++i) issue(i);
    }

    float sxr = 0.f;                      // sum x of the prepared x (threads 0..127)
    int64_t xb = -1;                      // matrix whose x is prepared (0 for a shared x)
    bool new_x = false;
    bool ok = true;
    int waited = 0;
    for (int i = 0; i < my && ok; ++i) {
        const int64_t g = g0 + i;
        const int64_t b = g / a.nrowblk;
        const int rb = (int)(g % a.nrowblk);
        const int64_t xsel = a.x_stride ? b : 0;
        if (xsel != xb) {
            if (i > 0) __syncthreads();  // the previous block's reducers are done with the sum-x slots
            // x of matrix b -> prepared fp32 (as in the kernel above); the previous block's
            // readers of xs and red passed its last barrier
            const uint16_t *xp16 = a.x + xsel * a.x_stride;
            uint4 *xr = reinterpret_cast<uint4 *>(xs);
            for (int gg = threadIdx.x; gg < (cols >> 3); gg += NTHREADS) xr[gg] = __ldg(reinterpret_cast<const uint4 *>(xp16) + gg);
            __syncthreads();
            float ax5[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < CPW; ++m)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint4 *xq = xr + 2 * (4 * (warp + NWARPS * m) + u);
                    const uint4 xa = xq[0], xb2 = xq[1];
                    const uint32_t X[8] = {xa.x, xa.y, xa.z, xa.w, xb2.x, xb2.y, xb2.z, xb2.w};
                    word_mixed(0x55555555u, X, ax5);
                }
            if (lane == 0) redx[warp] = mixed_total(ax5);
            xb = xsel;
            new_x = true;
        }
        const int slot = i % ring;
        float scl = 0.f;
        const int64_t row = (int64_t)rb * ROWS + threadIdx.x;
        if (threadIdx.x < ROWS && row < a.rows) scl = __half2float(__ushort_as_half(a.scales[b * a.scales_stride + row]));
        if (!mbar_wait_sleep(&full[slot], (i / ring) & 1)) {
            atomicExch(&g_gemv_rows_err, kDevErrWaitFull);
            s_fail[i & 1] = 1;  // the bytes read below are then garbage, but every access stays in bounds
        }
        const uint8_t *tile = tiles + (size_t)slot * stage_bytes;
        float acc[RPL][5];
#pragma unroll
        for (int j = 0; j < RPL; ++j)
#pragma unroll
            for (int k = 0; k < 5; ++k) acc[j][k] = 0.f;
        const uint4 *xr = reinterpret_cast<const uint4 *>(xs);
#pragma unroll
        for (int m = 0; m < CPW; ++m) {
            const int c = warp + NWARPS * m;
            const uint8_t *bp = tile + m * BOX + ((warp ^ (lane & 7)) << 4);
            uint4 q[RPL];
#pragma unroll
            for (int j = 0; j < RPL; ++j) q[j] = *reinterpret_cast<const uint4 *>(bp + (lane + 32 * j) * 128);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint4 *xq = xr + 2 * (4 * c + u);
                const uint4 xa = xq[0], xb2 = xq[1];
                const uint32_t X[8] = {xa.x, xa.y, xa.z, xa.w, xb2.x, xb2.y, xb2.z, xb2.w};
#pragma unroll
                for (int j = 0; j < RPL; ++j) {
                    const uint32_t w = u == 0 ? q[j].x : u == 1 ? q[j].y : u == 2 ? q[j].z : q[j].w;
                    word_mixed(w, X, acc[j]);
                }
            }
        }
        float *red = redb + (i & 1) * NWARPS * ROWS;
#pragma unroll
        for (int j = 0; j < RPL; ++j) red[warp * ROWS + lane + 32 * j] = mixed_total(acc[j]);
        __syncthreads();  // partial sums written; every warp is done with ring slot `slot`
        ok = reinterpret_cast<volatile int *>(s_fail)[i & 1] == 0;
        if (!ok) break;  // taken by every thread: the flag was read after the barrier
        waited = i + 1;
        if (leader && i + ring < my) issue(i + ring);
        if (threadIdx.x < ROWS) {
            const int r = threadIdx.x;
            if (new_x) {
                sxr = redx[0];
                for (int k = 1; k < NWARPS; ++k) sxr += redx[k];
            }
            float s1 = red[r];
            for (int k = 1; k < NWARPS; ++k) s1 += red[k * ROWS + r];
            if (row < a.rows)
                a.y[b * a.y_stride + row] = scl * __fadd_rn(__fmul_rn(a.c0, sxr), __fmul_rn(a.dd, s1));
        }
        new_x = false;
        // no second barrier: the next block writes the other half of the double-buffered partial sums,
        // and this half is rewritten only after the next block's barrier
    }
    // copies in flight after a failed wait must land before the shared memory is released
    if (!ok && leader) {
        const int issued = min(my, waited + ring);
        for (int j = waited; j < issued; ++j)
            if (!mbar_wait(&full[j % ring], (j / ring) & 1)) atomicExch(&g_gemv_rows_err, kDevErrDrain);
    }
}

size_t rows_smem_bytes(int64_t cols, int ring) {
    return 1024 + (size_t)ring * (size_t)(cols / 512) * BOX + (size_t)cols * 4 + (2 * NWARPS * ROWS + NWARPS) * 4 +
           (size_t)ring * 8;
}

}  // namespace

bool gemv_rows_supported(const PackedArgs &a) {
    return a.cols % 512 == 0 && a.cols <= 4096 && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 && a.rows < ((int64_t)1 << 31) - ROWS;
}

cudaError_t launch_gemv_rows(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    if (!gemv_rows_supported(a)) return cudaErrorNotSupported;
    const int64_t rowbytes = a.cols / 4;
    CUtensorMap tm;
    cudaError_t e = make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, (uint64_t)rowbytes, (uint64_t)a.rows,
                                 (uint64_t)rowbytes, 128, ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const int cpw = (int)(a.cols / 512);
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        const void *fns[8] = {(const void *)gemv2_rows_kernel<1>, (const void *)gemv2_rows_kernel<2>,
                              (const void *)gemv2_rows_kernel<3>, (const void *)gemv2_rows_kernel<4>,
                              (const void *)gemv2_rows_kernel<5>, (const void *)gemv2_rows_kernel<6>,
                              (const void *)gemv2_rows_kernel<7>, (const void *)gemv2_rows_kernel<8>};
        for (const void *f : fns)
            if (attr_err == cudaSuccess)
                attr_err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int nblk = cfg.blocks_per_cta > 0 ? cfg.blocks_per_cta : 1;
    int ring = nblk >= 2 ? 2 : 1;
    if (rows_smem_bytes(a.cols, ring) > 200 * 1024) ring = 1;
    const int64_t nrowblk = (a.rows + ROWS - 1) / ROWS;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((nrowblk + nblk - 1) / nblk));
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = rows_smem_bytes(a.cols, ring);
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    switch (cpw) {
        case 1: return cudaLaunchKernelEx(&lc, gemv2_rows_kernel<1>, tm, a, prefetch, nblk, ring);
        case 2: return cudaLaunchKernelEx(&lc, gemv2_rows_kernel<2>, tm, a, prefetch, nblk, ring);
        case 3: return cudaLaunchKernelEx(&lc, gemv2_rows_kernel<3>, tm, a, prefetch, nblk, ring);
        case 4: return cudaLaunchKernelEx(&lc, gemv2_rows_kernel<4>, tm, a, prefetch, nblk, ring);
        case 5: return cudaLaunchKernelEx(&lc, gemv2_rows_kernel<5>, tm, a, prefetch, nblk, ring);
        case 6: return cudaLaunchKernelEx(&lc, gemv2_rows_kernel<6>, tm, a, prefetch, nblk, ring);
        case 7: return cudaLaunchKernelEx(&lc, gemv2_rows_kernel<7>, tm, a, prefetch, nblk, ring);
        default: return cudaLaunchKernelEx(&lc, gemv2_rows_kernel<8>, tm, a, prefetch, nblk, ring);
    }
}

bool gemv_batched_supported(const PackedBatch &p) {
    return p.cols % 512 == 0 && p.cols <= 4096 && (reinterpret_cast<uintptr_t>(p.codes) % 16) == 0 &&
           p.codes_stride % 16 == 0 && (reinterpret_cast<uintptr_t>(p.x) % 16) == 0 && p.x_stride % 8 == 0 &&
           p.rows < ((int64_t)1 << 31) - ROWS && p.batch < ((int64_t)1 << 31) && codebook_is_affine(p.cb);
}

cudaError_t launch_gemv_batched(const PackedBatch &p, cudaStream_t st) {
    if (!gemv_batched_supported(p)) return cudaErrorNotSupported;
    const int64_t rowbytes = p.cols / 4;
    CUtensorMap tm;
    cudaError_t e = make_tmap_3d(CU_TENSOR_MAP_DATA_TYPE_UINT8, &tm, p.codes, (uint64_t)rowbytes, (uint64_t)p.rows,
                                 (uint64_t)p.batch, (uint64_t)rowbytes, (uint64_t)p.codes_stride, 128, ROWS,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const int cpw = (int)(p.cols / 512);
    constexpr int kSmemLimit = 224 * 1024;  // the opt-in maximum less the static flag and slack
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        const void *fns[8] = {(const void *)gemv2_batched_kernel<1>, (const void *)gemv2_batched_kernel<2>,
                              (const void *)gemv2_batched_kernel<3>, (const void *)gemv2_batched_kernel<4>,
                              (const void *)gemv2_batched_kernel<5>, (const void *)gemv2_batched_kernel<6>,
                              (const void *)gemv2_batched_kernel<7>, (const void *)gemv2_batched_kernel<8>};
        for (const void *f : fns)
            if (attr_err == cudaSuccess)
                attr_err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // two CTAs per SM with a two-stage ring each: the decode is issue bound, and 8 warps per
    // SM (one CTA with a deeper ring) measured 1.97 us per 12,288 x 1,536 matrix against
    // 1.63 us for single calls at 16 warps per SM
    int ring = 2;
    int per_sm = rows_smem_bytes(p.cols, ring) * 2 <= (size_t)kSmemLimit ? 2 : 1;
    while (ring > 1 && rows_smem_bytes(p.cols, ring) > (size_t)kSmemLimit) --ring;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    BatchArgs a{p.scales, p.scales_stride, p.x, p.x_stride, p.y, p.y_stride, p.rows, (p.rows + ROWS - 1) / ROWS, 0,
                p.cb[0], p.cb[1] - p.cb[0]};
    a.total = a.nrowblk * p.batch;
    const int64_t grid = a.total < (int64_t)per_sm * sms ? a.total : (int64_t)per_sm * sms;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = rows_smem_bytes(p.cols, ring);
    lc.stream = st;
    switch (cpw) {
        case 1: return cudaLaunchKernelEx(&lc, gemv2_batched_kernel<1>, tm, a, ring);
        case 2: return cudaLaunchKernelEx(&lc, gemv2_batched_kernel<2>, tm, a, ring);
        case 3: return cudaLaunchKernelEx(&lc, gemv2_batched_kernel<3>, tm, a, ring);
        case 4: return cudaLaunchKernelEx(&lc, gemv2_batched_kernel<4>, tm, a, ring);
        case 5: return cudaLaunchKernelEx(&lc, gemv2_batched_kernel<5>, tm, a, ring);
        case 6: return cudaLaunchKernelEx(&lc, gemv2_batched_kernel<6>, tm, a, ring);
        case 7: return cudaLaunchKernelEx(&lc, gemv2_batched_kernel<7>, tm, a, ring);
        default: return cudaLaunchKernelEx(&lc, gemv2_batched_kernel<8>, tm, a, ring);
    }
}

unsigned int gemv_rows_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_gemv_rows_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_gemv_rows_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
