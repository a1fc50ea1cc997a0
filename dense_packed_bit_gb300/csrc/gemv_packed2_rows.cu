// gemv_packed2_rows.cu -- 2-bit GEMV, SIMT affine decode, code tiles staged
// by TMA and one lane per row.
//
// "Kernel 0112", sections "What is being measured" and "The four variants":
// the 12,288 x 1,536 GEMV is bound by how fast 18.9 M fields a call become
// products.  The affine decode of gemv_packed2.cu needs one LOP3 per field and
// one packed f32x2 FMA per two fields; this kernel keeps everything else off
// the hot loop:
//
//  * a CTA streams 128-row blocks of code rows through a TMA ring (128-byte
//    boxes with the 128-byte swizzle); lane l of every warp owns rows l, l+32,
//    l+64, l+96 of the block, so a row's partial sum never crosses lanes and
//    needs no shuffles;
//  * warp w owns the 64-field chunks w, w+8, w+16, ... of every row: for each
//    code word it reads the 16 prepared x values once (shared-memory broadcast,
//    all lanes the same address) and applies them to its four rows;
//  * the eight warps' partial sums of a row, and of sum x, are added in warp
//    order through shared memory (reproducible bit for bit).
//
// Decode (exact; see gemv_packed2.cu): the field at bit p of a code word,
// masked in place and read as fp32 bits, is c 2^(p-149); x is prepared as
// x 2^(111-p), so each fma.rn.f32x2 adds c x 2^-38 exactly.  sum x runs
// through the same packed FMAs with every field equal to 1 and is reduced in
// the same order, so a row of zero-entry fields gives exactly 0.
//
// Requirements: cols % 512 == 0, cols <= 4096, 16-byte aligned codes, an
// affine codebook (zero entry, if any, at field 0, 1 or 2).
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

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

__device__ __forceinline__ float2 field_pair(uint32_t w, uint32_t m0, uint32_t m1) {
    return make_float2(__uint_as_float(w & m0), __uint_as_float(w & m1));
}

// 16 fields of one code word against the 16 prepared x values of its position.
__device__ __forceinline__ float2 word_fma(uint32_t w, const float4 &x0, const float4 &x1, const float4 &x2,
                                           const float4 &x3, float2 acc) {
    acc = ffma2(field_pair(w, 0x3u, 0xCu), make_float2(x0.x, x0.y), acc);
    acc = ffma2(field_pair(w, 0x30u, 0xC0u), make_float2(x0.z, x0.w), acc);
    acc = ffma2(field_pair(w, 0x300u, 0xC00u), make_float2(x1.x, x1.y), acc);
    acc = ffma2(field_pair(w, 0x3000u, 0xC000u), make_float2(x1.z, x1.w), acc);
    acc = ffma2(field_pair(w, 0x30000u, 0xC0000u), make_float2(x2.x, x2.y), acc);
    acc = ffma2(field_pair(w, 0x300000u, 0xC00000u), make_float2(x2.z, x2.w), acc);
    const uint32_t h = w >> 16;  // fields 12..15 now at bits 8..15
    acc = ffma2(field_pair(h, 0x300u, 0xC00u), make_float2(x3.x, x3.y), acc);
    acc = ffma2(field_pair(h, 0x3000u, 0xC000u), make_float2(x3.z, x3.w), acc);
    return acc;
}

// CPW: 64-field chunks per warp (cols = 512 CPW), a template parameter so that the
// chunk loops unroll completely.
template <int CPW>
__global__ void __launch_bounds__(NTHREADS) gemv2_rows_kernel(const __grid_constant__ CUtensorMap tmC,
                                                              const PackedArgs a, const int prefetch, const int nblk,
                                                              const int ring) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_fail;  // set by a thread whose bounded wait ran out; read after a barrier
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    constexpr int cols = 512 * CPW;
    constexpr int nbox = CPW;     // 128-byte boxes per row
    constexpr int stage_bytes = nbox * BOX;
    uint8_t *tiles = smem;                                                       // [ring][nbox][128 rows][128 B]
    float4 *xs = reinterpret_cast<float4 *>(smem + (size_t)ring * stage_bytes);  // prepared x, cols floats
    float *red = reinterpret_cast<float *>(xs + (cols >> 2));                    // [NWARPS][ROWS], then sum x [NWARPS]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + NWARPS * ROWS + NWARPS);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int blk0 = blockIdx.x * nblk;
    const int nrowblk = (int)((a.rows + ROWS - 1) / ROWS);
    const int my_blocks = min(nblk, nrowblk - blk0);
    const bool leader = threadIdx.x == 0;

    if (leader) {
        s_fail = 0;
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

    // ---- x -> prepared fp32 in shared memory: field f of its code word is read at bit
    // p = 2 (f & 15) for (f & 15) < 12, else 2 (f & 15) - 16 (after the word's shift by 16)
    for (int g = threadIdx.x; g < (cols >> 3); g += NTHREADS) {
        const uint4 hv = __ldg(reinterpret_cast<const uint4 *>(a.x) + g);
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int j = (8 * g + i) & 15;
            const int p = j < 12 ? 2 * j : 2 * j - 16;
            v[i] = __half2float(__ushort_as_half((uint16_t)(hw[i >> 1] >> (16 * (i & 1))))) * pow2f(111 - p);
        }
        xs[2 * g] = make_float4(v[0], v[1], v[2], v[3]);
        xs[2 * g + 1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();

    // ---- this warp's sum of x over its chunks, by the same packed FMAs as the rows
    {
        float2 ax = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < CPW; ++m)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 *xp = xs + 16 * (warp + NWARPS * m) + 4 * u;
                ax = word_fma(0x55555555u, xp[0], xp[1], xp[2], xp[3], ax);
            }
        if (lane == 0) red[NWARPS * ROWS + warp] = ax.x + ax.y;
    }
    const float c0 = a.cb[0], dd = a.cb[1] - a.cb[0];
    const float two38 = 274877906944.0f;  // 2^38
    float sxr = 0.f;                      // sum x (threads 0..127), set at the first block

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
            s_fail = 1;  // the bytes read below are then garbage, but every access stays in bounds
        }
        const uint8_t *tile = tiles + (size_t)slot * stage_bytes;
        float2 acc[RPL];
#pragma unroll
        for (int j = 0; j < RPL; ++j) acc[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < CPW; ++m) {
            const int c = warp + NWARPS * m;  // chunk c lives in box m, at chunk position warp of the box
            const uint8_t *bp = tile + m * BOX + ((warp ^ (lane & 7)) << 4);  // rows lane + 32 j: row % 8 == lane % 8
            uint4 q[RPL];
#pragma unroll
            for (int j = 0; j < RPL; ++j) q[j] = *reinterpret_cast<const uint4 *>(bp + (lane + 32 * j) * 128);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 *xp = xs + 16 * c + 4 * u;
                const float4 x0 = xp[0], x1 = xp[1], x2 = xp[2], x3 = xp[3];
#pragma unroll
                for (int j = 0; j < RPL; ++j) {
                    const uint32_t w = u == 0 ? q[j].x : u == 1 ? q[j].y : u == 2 ? q[j].z : q[j].w;
                    acc[j] = word_fma(w, x0, x1, x2, x3, acc[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < RPL; ++j) red[warp * ROWS + lane + 32 * j] = acc[j].x + acc[j].y;
        __syncthreads();  // partial sums written; every warp is done with ring slot `slot`
        ok = *reinterpret_cast<volatile int *>(&s_fail) == 0;
        if (!ok) break;  // taken by every thread: the flag was read after the barrier
        waited = i + 1;
        if (leader && i + ring < my_blocks) issue(i + ring);
        if (threadIdx.x < ROWS) {
            const int r = threadIdx.x;
            if (i == 0) {
                sxr = red[NWARPS * ROWS];
                for (int k = 1; k < NWARPS; ++k) sxr += red[NWARPS * ROWS + k];
            }
            float s1 = red[r];
            for (int k = 1; k < NWARPS; ++k) s1 += red[k * ROWS + r];
            if (row < a.rows) a.y[row] = scl * __fadd_rn(__fmul_rn(c0, sxr * two38), __fmul_rn(dd, s1 * two38));
        }
        __syncthreads();  // the next block may overwrite the partial sums
    }
    // copies in flight after a failed wait must land before the shared memory is released
    if (!ok && leader) {
        const int issued = min(my_blocks, waited + ring);
        for (int j = waited; j < issued; ++j)
            if (!mbar_wait(&full[j % ring], (j / ring) & 1)) atomicExch(&g_gemv_rows_err, kDevErrDrain);
    }
}

size_t rows_smem_bytes(int64_t cols, int ring) {
    return 1024 + (size_t)ring * (size_t)(cols / 512) * BOX + (size_t)cols * 4 + (NWARPS * ROWS + NWARPS) * 4 +
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
