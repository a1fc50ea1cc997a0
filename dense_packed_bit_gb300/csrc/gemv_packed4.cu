// gemv_packed4.cu -- y = diag(scale) . W . x for 4-bit packed W with a
// 16-entry fp32 codebook (sm_103a).
//
// "Kernel 0112", section "What the kernel costs in a whole token": the 4-bit
// weight-reading kernels of the same model (0099, 0105) are the fastest
// measured on the pages and make the largest in-model contributions; "More
// Stumbling, This Time in the Browser": the packed NF4 path.  Format: element
// k of a row is in byte floor(k/2), low nibble first; the field selects one of
// 16 codebook entries, which the per-row fp16 scale multiplies.
//
// A 16-entry codebook such as NF4 has no affine or fp16-exact form, so each
// field must fetch an fp32 entry.  The fast kernel makes that fetch a
// shared-memory load of a table indexed by the whole code byte: entry b holds
// (codebook[b & 15], codebook[b >> 4]), the two fields' values, which one packed
// f32x2 FMA multiplies by the two x values.  The table is replicated for the 16
// lanes of a half-warp ([byte][lane % 16], 32 KiB): a 64-bit load is served per
// half-warp, and every lane of a half-warp then reads its own bank pair,
// whatever the byte values, so the lookups never conflict.
//
//  * 64-row blocks of code rows arrive by TMA (128-byte boxes = 256 fields,
//    128-byte swizzle) through a one- or two-slot ring;
//  * lane l of every warp owns rows l and l + 32 of the block; warp w owns the
//    16-byte chunk w of every box, so it reads the 32 prepared x values of a
//    chunk once (shared-memory broadcast) for its two rows;
//  * the eight warps' partial sums of a row are added in warp order through
//    shared memory (reproducible bit for bit).
//
// The generic kernel takes any shape and alignment: one warp per row, lanes
// striding over the row's bytes, codebook in shared memory.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tmap.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {

__device__ unsigned int g_gemv4_err;

namespace {

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// ------------------------------------------------------------------ generic

__global__ void __launch_bounds__(256) gemv4_generic_kernel(const Packed4Args a) {
    __shared__ float cb[16];
    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) cb[i] = a.cb[i];  // constant indices: read from the parameter bank
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    pdl_wait();
    if (row >= a.rows) return;
    const int64_t rowbytes = (a.cols + 1) >> 1;
    const uint8_t *rp = a.codes + row * rowbytes;
    float acc = 0.f;
    for (int64_t b = lane; b < rowbytes; b += 32) {
        const uint32_t byte = rp[b];
        const int64_t k = 2 * b;
        acc = fmaf(cb[byte & 15u], h2f(a.x[k]), acc);
        if (k + 1 < a.cols) acc = fmaf(cb[byte >> 4], h2f(a.x[k + 1]), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) a.y[row] = h2f(a.scales[row]) * acc;
}

// ------------------------------------------------------------------ TMA-staged table decode

constexpr int ROWS = 64;          // rows per block: one TMA box height
constexpr int BOX = 128 * ROWS;   // bytes of one 128-byte-wide box of 64 rows
constexpr int NWARPS_MAX = 16;
constexpr int RPL = ROWS / 32;    // rows per lane

// CPW = boxes per row = cols / 256; NW warps, warp w takes the 16-byte chunks c = w, w + NW, ...
// of every row (chunk c is chunk c % 8 of box c / 8), CPW * 8 / NW of them.
template <int CPW, int NW>
__global__ void __launch_bounds__(32 * NW) gemv4_lut_kernel(const __grid_constant__ CUtensorMap tmC,
                                                             const Packed4Args a, const int prefetch, const int nblk,
                                                             const int ring) {
    extern __shared__ uint8_t smem_raw[];
    // the byte table lives in static shared memory: its address is a link-time constant, so
    // a lookup needs only the byte offset in a register (base folded into the load)
    __shared__ __align__(128) float2 lut[256 * 16];  // [byte][lane % 16]
    __shared__ int s_fail;  // set by a thread whose bounded wait ran out; read after a barrier
    __shared__ float cbs[16];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    constexpr int cols = 256 * CPW;
    constexpr int stage_bytes = CPW * BOX;
    uint8_t *tiles = smem;                                                         // [ring][CPW][64 rows][128 B]
    float4 *xs = reinterpret_cast<float4 *>(smem + (size_t)ring * stage_bytes);  // cols floats
    float *red = reinterpret_cast<float *>(xs + cols / 4);                                   // [NW][ROWS]
    uint64_t *full = reinterpret_cast<uint64_t *>(red + NW * ROWS);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int blk0 = blockIdx.x * nblk;
    const int nrowblk = (int)((a.rows + ROWS - 1) / ROWS);
    const int my_blocks = min(nblk, nrowblk - blk0);
    const bool leader = threadIdx.x == 0;

    if (leader) {
        s_fail = 0;
        for (int r = 0; r < ring; ++r) mbar_init(&full[r], 1);
        fence_mbar_init();
#pragma unroll
        for (int c = 0; c < 16; ++c) cbs[c] = a.cb[c];  // constant indices: read from the parameter bank
    }
    __syncthreads();
    auto issue = [&](int i) {  // block i of this CTA into ring slot i % ring
        uint8_t *dst = tiles + (size_t)(i % ring) * stage_bytes;
        mbar_arrive_expect_tx(&full[i % ring], (uint32_t)stage_bytes);
        for (int b = 0; b < CPW; ++b) tma_load_2d(dst + b * BOX, &tmC, &full[i % ring], b * 128, (blk0 + i) * ROWS);
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

    // ---- byte -> (entry of the low field, entry of the high field), one copy per half-warp lane
    for (int e = threadIdx.x; e < 256 * 16; e += 32 * NW) {
        const int b = e >> 4;
        lut[e] = make_float2(cbs[b & 15], cbs[b >> 4]);
    }
    // ---- x -> fp32 in shared memory
    for (int g = threadIdx.x; g < cols / 8; g += 32 * NW) {
        const uint4 hv = __ldg(reinterpret_cast<const uint4 *>(a.x) + g);
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = h2f((uint16_t)(hw[i >> 1] >> (16 * (i & 1))));
        xs[2 * g] = make_float4(v[0], v[1], v[2], v[3]);
        xs[2 * g + 1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    __syncthreads();

    const uint32_t lane_off = (uint32_t)(lane & 15) * 8u;  // byte offset of this lane's copy of an entry
    const uint8_t *lut_bytes = reinterpret_cast<const uint8_t *>(lut);
    bool ok = true;
    int waited = 0;
    for (int i = 0; i < my_blocks && ok; ++i) {
        const int slot = i % ring;
        float scl = 0.f;  // scale of this thread's row (threads 0..63), read while the codes travel
        const int64_t row = (int64_t)(blk0 + i) * ROWS + threadIdx.x;
        if (threadIdx.x < ROWS && row < a.rows) scl = h2f(a.scales[row]);
        if (!mbar_wait_sleep(&full[slot], (i / ring) & 1)) {
            atomicExch(&g_gemv4_err, kDevErrWaitFull);
            s_fail = 1;  // the bytes read below are then garbage, but every access stays in bounds
        }
        const uint8_t *tile = tiles + (size_t)slot * stage_bytes;
        // two accumulators per row (even and odd bytes of each word) shorten the FMA chains;
        // the four table entries of a word are loaded before its FMAs
        float2 acc[RPL][2];
#pragma unroll
        for (int j = 0; j < RPL; ++j) acc[j][0] = acc[j][1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < CPW * 8 / NW; ++m) {
            // chunk c = warp + NW m: 16 bytes = 32 fields of rows lane + 32 j (row % 8 == lane % 8)
            const int c = warp + NW * m;
            const uint8_t *bp = tile + (c >> 3) * BOX + (((c & 7) ^ (lane & 7)) << 4);
            uint4 q[RPL];
#pragma unroll
            for (int j = 0; j < RPL; ++j) q[j] = *reinterpret_cast<const uint4 *>(bp + (lane + 32 * j) * 128);
            const float4 *xp = xs + c * 8;
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                const float4 xa = xp[2 * wd], xb = xp[2 * wd + 1];  // fields 8 wd .. 8 wd + 7 of the chunk
                const float2 xx[4] = {make_float2(xa.x, xa.y), make_float2(xa.z, xa.w), make_float2(xb.x, xb.y),
                                      make_float2(xb.z, xb.w)};
                float2 e[RPL][4];
#pragma unroll
                for (int j = 0; j < RPL; ++j) {
                    const uint32_t w = wd == 0 ? q[j].x : wd == 1 ? q[j].y : wd == 2 ? q[j].z : q[j].w;
                    // byte k of w times 128 (the entry stride), or'ed with the lane's offset: bits 7..14
                    // hold the byte and bits 3..6 the lane, so the sum is a bitwise or
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t sh = k == 0 ? (w << 7) : (w >> (8 * k - 7));
                        const uint32_t off = (sh & 0x7F80u) | lane_off;
                        e[j][k] = *reinterpret_cast<const float2 *>(lut_bytes + off);
                    }
                }
#pragma unroll
                for (int j = 0; j < RPL; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[j][k & 1] = ffma2(e[j][k], xx[k], acc[j][k & 1]);
            }
        }
#pragma unroll
        for (int j = 0; j < RPL; ++j)
            red[warp * ROWS + lane + 32 * j] = (acc[j][0].x + acc[j][0].y) + (acc[j][1].x + acc[j][1].y);
        __syncthreads();  // partial sums written; every warp is done with ring slot `slot`
        ok = *reinterpret_cast<volatile int *>(&s_fail) == 0;
        if (!ok) break;  // taken by every thread: the flag was read after the barrier
        waited = i + 1;
        if (leader && i + ring < my_blocks) issue(i + ring);
        if (threadIdx.x < ROWS) {
            float s = red[threadIdx.x];
            for (int k = 1; k < NW; ++k) s += red[k * ROWS + threadIdx.x];
            if (row < a.rows) a.y[row] = scl * s;
        }
        __syncthreads();  // the next block may overwrite the partial sums
    }
    // copies in flight after a failed wait must land before the shared memory is released
    if (!ok && leader) {
        const int issued = min(my_blocks, waited + ring);
        for (int j = waited; j < issued; ++j)
            if (!mbar_wait(&full[j % ring], (j / ring) & 1)) atomicExch(&g_gemv4_err, kDevErrDrain);
    }
}

// dynamic shared memory (the 32 KiB byte table is static)
size_t lut_smem_bytes(int64_t cols, int ring) {
    return 1024 + (size_t)ring * (size_t)(cols / 256) * BOX + (size_t)cols * 4 + NWARPS_MAX * ROWS * 4 +
           (size_t)ring * 8;
}

// 16 warps when the chunks split evenly over them (an even number of boxes), else 8
template <int CPW>
cudaError_t launch_lut(cudaLaunchConfig_t &lc, const CUtensorMap &tm, const Packed4Args &a, int prefetch, int nblk,
                       int ring) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    constexpr int NW = (CPW % 2 == 0) ? 16 : 8;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(gemv4_lut_kernel<CPW, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        160 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    lc.blockDim = dim3(32 * NW);
    return cudaLaunchKernelEx(&lc, gemv4_lut_kernel<CPW, NW>, tm, a, prefetch, nblk, ring);
}

}  // namespace

bool gemv4_lut_supported(const Packed4Args &a) {
    return a.cols % 256 == 0 && a.cols <= 4096 && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 && a.rows < ((int64_t)1 << 31) - ROWS;
}

cudaError_t launch_gemv_packed4(const Packed4Args &a, const Gemv4Config &cfg, cudaStream_t st) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
    if (!cfg.staging) {
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3((unsigned)((a.rows + 7) / 8));
        lc.blockDim = dim3(256);
        lc.stream = st;
        lc.attrs = attr;
        lc.numAttrs = 1;
        return cudaLaunchKernelEx(&lc, gemv4_generic_kernel, a);
    }
    if (!gemv4_lut_supported(a)) return cudaErrorNotSupported;
    const int64_t rowbytes = a.cols / 2;
    CUtensorMap tm;
    cudaError_t e = make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, (uint64_t)rowbytes, (uint64_t)a.rows,
                                 (uint64_t)rowbytes, 128, ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const int nblk = cfg.blocks_per_cta > 0 ? cfg.blocks_per_cta : 1;
    int ring = nblk >= 2 ? 2 : 1;
    if (lut_smem_bytes(a.cols, ring) > 160 * 1024) ring = 1;
    const int64_t nrowblk = (a.rows + ROWS - 1) / ROWS;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((nrowblk + nblk - 1) / nblk));
    lc.dynamicSmemBytes = lut_smem_bytes(a.cols, ring);
    lc.stream = st;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    switch (a.cols / 256) {
        case 1: return launch_lut<1>(lc, tm, a, prefetch, nblk, ring);
        case 2: return launch_lut<2>(lc, tm, a, prefetch, nblk, ring);
        case 3: return launch_lut<3>(lc, tm, a, prefetch, nblk, ring);
        case 4: return launch_lut<4>(lc, tm, a, prefetch, nblk, ring);
        case 5: return launch_lut<5>(lc, tm, a, prefetch, nblk, ring);
        case 6: return launch_lut<6>(lc, tm, a, prefetch, nblk, ring);
        case 7: return launch_lut<7>(lc, tm, a, prefetch, nblk, ring);
        case 8: return launch_lut<8>(lc, tm, a, prefetch, nblk, ring);
        case 9: return launch_lut<9>(lc, tm, a, prefetch, nblk, ring);
        case 10: return launch_lut<10>(lc, tm, a, prefetch, nblk, ring);
        case 11: return launch_lut<11>(lc, tm, a, prefetch, nblk, ring);
        case 12: return launch_lut<12>(lc, tm, a, prefetch, nblk, ring);
        case 13: return launch_lut<13>(lc, tm, a, prefetch, nblk, ring);
        case 14: return launch_lut<14>(lc, tm, a, prefetch, nblk, ring);
        case 15: return launch_lut<15>(lc, tm, a, prefetch, nblk, ring);
        default: return launch_lut<16>(lc, tm, a, prefetch, nblk, ring);
    }
}

unsigned int gemv4_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_gemv4_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_gemv4_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
