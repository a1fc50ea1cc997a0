// gemv_packed2_fp8.cu -- 2-bit GEMV whose multiply-accumulate runs on the fp8
// tensor-core path (mma.sync m16n8k32, e4m3 x e5m2 operands, fp32 accumulators).
//
// "Kernel 0112", sections "What is being measured" and "What the kernel costs
// in a whole token": the 12,288 x 1,536 GEMV streams 4.5 MiB of 2-bit codes
// and is bound by how fast they can be read and turned into products.  The
// fp16 tensor-core decode (gemv_packed2_mma.cu) spends two instructions per
// pair of fields; here a single AND turns four fields into four exact fp8
// operands, so the integer pipe is no longer the limit.
//
// Codes as e4m3.  An e4m3 byte with exponent field 0 or 1 is worth its low
// four bits, read as an integer, times 2^-9.  Masking a code byte with 0x03
// keeps field 0 and gives c * 2^-9; masking with 0x0C keeps field 1 and gives
// c * 2^-7.  The word shifted right by 4 yields fields 2 and 3 the same way.
// One 32-bit word (16 fields) becomes four A registers with one shift and
// four ANDs.  Fields read with 0x03 and with 0x0C go to two separate sets of
// MMAs and accumulators ("set A" and "set B") whose powers of two are undone
// after the loop.
//
// x as e5m2.  e5m2 is the top byte of an fp16, so truncating an fp16 value to
// its top byte gives an exact e5m2 piece and an exact fp16 remainder; four
// such pieces hold an fp16 value exactly when all of its bits lie at or above
// 2^-16.  That holds for |x| >= 2^-6 ("window 0", x itself); smaller values
// are multiplied by 2^18 first ("window 1"), which covers the rest of the fp16
// range down to 2^-24.  Each value lives in one window; B column n carries
// piece n & 3 of window n >> 2, and the other window's columns are zero.
// After the k loop column n is scaled by 2^9 (set A) or 2^7 (set B) times
// 2^-18 for window 1; all of these scalings are exact.
//
// Affine codebooks (codebook[c] = c0 + c*d): the MMAs give S1 = sum c_k x_k.
// sum x comes from the same MMAs with every field equal to 1, at the same row
// position of the 16-row MMA block, reduced in the same order, and
// y = scale * (c0 * sum x + d * S1).  A row whose fields all hold the zero
// entry c_z in {0, 1, 2} then gives S1 == c_z * sum x exactly and y == 0.
//
// Layout: a CTA streams 64-row blocks of code rows through a TMA ring (one or
// two slots; 128-byte boxes with the 128-byte swizzle).  Warp kw owns the
// 256-field slab kw of every row; its lanes (g, t) load the 16-byte chunk
// 4 kw + t of rows 16 b + g and 16 b + g + 8.  The x pieces are built once per
// CTA, cooperatively, straight into the B fragment order in shared memory.
//
// Requirements: cols % 512 == 0, cols <= 4096, 16-byte aligned codes and x,
// an affine codebook (zero entry, if any, at field 0, 1 or 2).
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tmap.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {

__device__ unsigned int g_gemv_fp8_err;

namespace {

constexpr int ROWS = 64;         // rows per block: one TMA box height
constexpr int BOX = 128 * ROWS;  // bytes of one 128-byte-wide box of 64 rows
constexpr int RB = ROWS / 16;    // 16-row MMA blocks per block
constexpr int RED = 81;          // floats per warp in the reduction area: 64 rows, 16 sum-x positions, pad

__device__ __forceinline__ void mma_e4m3_e5m2(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    // not volatile: a pure function of its operands, so the compiler may interleave
    // independent accumulator chains
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e5m2.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// 2^e as fp32
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Scale of accumulator column n: 2^9 (set A) or 2^7 (set B), times 2^-18 for window 1.
__device__ __forceinline__ float column_scale(int n, bool set_b) {
    return pow2f((set_b ? 7 : 9) - (n >= 4 ? 18 : 0));
}

// Row sum of a thread's two columns of both sets, fixed order, no contraction.
__device__ __forceinline__ float combine(float a0, float a1, float b0, float b1, float sa0, float sa1, float sb0,
                                         float sb1) {
    return __fadd_rn(__fadd_rn(__fmul_rn(a0, sa0), __fmul_rn(a1, sa1)),
                     __fadd_rn(__fmul_rn(b0, sb0), __fmul_rn(b1, sb1)));
}

__device__ __forceinline__ float quad_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// Exact e5m2 pieces of the two fp16 values in v.  win0 gets 0xFFFF in each half
// whose value lies in window 0 (|x| >= 2^-6); p[i] holds piece i of each value
// (window 1 values scaled by 2^18) in the top byte of its half.
__device__ __forceinline__ void split_x2(uint32_t v, uint32_t (&p)[4], uint32_t &win0) {
    const __half2 h = *reinterpret_cast<const __half2 *>(&v);
    win0 = __hge2_mask(__habs2(h), __float2half2_rn(0.015625f));
    const uint32_t k512 = 0x60006000u;  // fp16x2 (512, 512)
    const uint32_t s = hmul2_bits(hmul2_bits(v, k512), k512);
    uint32_t r = (v & win0) | (s & ~win0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        p[i] = r & 0xFF00FF00u;
        r = hsub2_bits(r, p[i]);
    }
}

// Builds the B fragments of the whole K extent in shared memory.  Fragment word
// (slab s, pair p, lane 4g + t, j) holds piece g of x at fields
// 256 s + 64 t + 16 p + off_j + 4 e (e = 0..3 in its bytes), off = {0, 2, 1, 3}:
// j = 0, 1 feed set A (fields 4e, 4e + 2 of a code word), j = 2, 3 set B.
// A unit is one (s, p, t, j); the cols / 4 units fall two to a thread (cols / 8 threads).
__device__ __forceinline__ void build_b_fragments(const uint16_t *xs, uint32_t *bfrag) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {  // cols / 4 units over cols / 8 threads
        const int u = threadIdx.x + k * blockDim.x;
        const int j = u & 3, t = (u >> 2) & 3, sp = u >> 4;  // sp = slab * 4 + pair
        const int off = (j == 0) ? 0 : (j == 1) ? 2 : (j == 2) ? 1 : 3;
        const int s = sp >> 2, p = sp & 3;
        const int f = 256 * s + 64 * t + 16 * p + off;
        const uint32_t v01 = (uint32_t)xs[f] | ((uint32_t)xs[f + 4] << 16);
        const uint32_t v23 = (uint32_t)xs[f + 8] | ((uint32_t)xs[f + 12] << 16);
        uint32_t p01[4], p23[4], w01, w23;
        split_x2(v01, p01, w01);
        split_x2(v23, p23, w23);
        const uint32_t wmask = __byte_perm(w01, w23, 0x7531);  // 0xFF per value in window 0
        uint32_t *dst = bfrag + (size_t)sp * 128 + t * 4 + j;  // + 16 g for lane 4g + t
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t bytes = __byte_perm(p01[i], p23[i], 0x7531);
            dst[16 * i] = bytes & wmask;         // column i: window 0
            dst[16 * (4 + i)] = bytes & ~wmask;  // column 4 + i: window 1
        }
    }
}

__global__ void __launch_bounds__(512) gemv2_fp8_kernel(const __grid_constant__ CUtensorMap tmC, const PackedArgs a,
                                                        const int prefetch, const int nblk, const int ring) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_fail;  // set by any thread whose bounded wait ran out; read after a barrier
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    const int cols = (int)a.cols;
    const int KW = blockDim.x >> 5;  // warps = 256-field slabs
    const int nbox = cols >> 9;      // 128-byte boxes per row
    const int stage_bytes = nbox * BOX;
    uint8_t *tiles = smem;                                                         // [ring][nbox][64][128], swizzled
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + ring * stage_bytes);       // x, cols halves
    uint32_t *bfrag = reinterpret_cast<uint32_t *>(xs + cols);                    // 2 * cols words
    float *red = reinterpret_cast<float *>(bfrag + 2 * cols);                     // [KW][RED]
    uint64_t *bars = reinterpret_cast<uint64_t *>(red + ((KW * RED + 1) & ~1));  // full[ring], xbar
    uint64_t *xbar = bars + ring;

    const int lane = threadIdx.x & 31, kw = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int blk0 = blockIdx.x * nblk;
    const int nrowblk = (int)((a.rows + ROWS - 1) / ROWS);
    const int my_blocks = min(nblk, nrowblk - blk0);
    const bool leader = threadIdx.x == 0;

    if (leader) {
        s_fail = 0;
        for (int r = 0; r < ring; ++r) mbar_init(&bars[r], 1);
        mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int i) {  // block i of this CTA into ring slot i % ring
        uint8_t *dst = tiles + (i % ring) * stage_bytes;
        mbar_arrive_expect_tx(&bars[i % ring], (uint32_t)stage_bytes);
        for (int b = 0; b < nbox; ++b) tma_load_2d(dst + b * BOX, &tmC, &bars[i % ring], b * 128, (blk0 + i) * ROWS);
    };
    auto issue_x = [&] {
        mbar_arrive_expect_tx(xbar, (uint32_t)cols * 2);
        bulk_load(xs, a.x, (uint32_t)cols * 2, xbar);
    };
    const int first = min(ring, my_blocks);
    if (prefetch >= 1) {
        if (leader) {
            for (int i = 0; i < first; ++i) issue(i);
            if (prefetch == 2) issue_x();
        }
        // chained calls: the next call may launch only once this one has passed its wait,
        // so at most one call runs ahead (its weight loads) instead of a queue of parked ones
        if (prefetch == 1) {
            pdl_wait();
            if (leader) issue_x();
        }
        pdl_launch_dependents();
    } else {
        pdl_wait();
        if (leader) {
            for (int i = 0; i < first; ++i) issue(i);
            issue_x();
        }
        pdl_launch_dependents();
    }

    // scale of this thread's row of the first block (threads 0..63 finish the rows)
    float scl = 0.f;
    if (threadIdx.x < ROWS) {
        const int64_t row = (int64_t)blk0 * ROWS + threadIdx.x;
        if (row < a.rows) scl = __half2float(__ushort_as_half(a.scales[row]));
    }

    // Every thread takes the same path through the barriers below: a wait that ran
    // out only marks s_fail (the bytes read are then garbage but in bounds), and the
    // flag is acted on after the next barrier, where all threads see the same value.
    if (!mbar_wait_sleep(xbar, 0)) {
        atomicExch(&g_gemv_fp8_err, kDevErrWaitFull);
        s_fail = 1;
    }
    build_b_fragments(xs, bfrag);
    __syncthreads();
    bool ok = *reinterpret_cast<volatile int *>(&s_fail) == 0;

    // this warp's B fragments: pair p -> (set A b0, set A b1, set B b0, set B b1)
    uint4 bf[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) bf[p] = reinterpret_cast<const uint4 *>(bfrag)[(kw * 4 + p) * 32 + lane];
    const float sa0 = column_scale(2 * t, false), sa1 = column_scale(2 * t + 1, false);
    const float sb0 = column_scale(2 * t, true), sb1 = column_scale(2 * t + 1, true);
    {
        // sum x at each of the 16 row positions: the same MMAs with every field 1
        float dxa[4] = {0.f, 0.f, 0.f, 0.f}, dxb[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t one_a = 0x01010101u, one_b = 0x04040404u;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            mma_e4m3_e5m2(dxa, one_a, one_a, one_a, one_a, bf[p].x, bf[p].y);
            mma_e4m3_e5m2(dxb, one_b, one_b, one_b, one_b, bf[p].z, bf[p].w);
        }
        const float lo = quad_sum(combine(dxa[0], dxa[1], dxb[0], dxb[1], sa0, sa1, sb0, sb1));
        const float hi = quad_sum(combine(dxa[2], dxa[3], dxb[2], dxb[3], sa0, sa1, sb0, sb1));
        if (t == 0) {
            red[kw * RED + 64 + g] = lo;
            red[kw * RED + 72 + g] = hi;
        }
    }
    const float c0 = a.cb[0], dd = a.cb[1] - a.cb[0];
    const int chunk = 4 * kw + t, box = chunk >> 3, cc = chunk & 7;
    float sxr = 0.f;  // sum x for this thread's row position (threads 0..63), set at block 0

    int waited = 0;  // blocks whose copies have landed
    for (int i = 0; i < my_blocks && ok; ++i) {
        const int slot = i % ring;
        if (!mbar_wait_sleep(&bars[slot], (i / ring) & 1)) {
            atomicExch(&g_gemv_fp8_err, kDevErrWaitFull);
            s_fail = 1;
        }
        const uint8_t *tb = tiles + slot * stage_bytes + box * BOX + ((cc ^ g) << 4);
        // rows 16b + g and 16b + g + 8 of the 16-row blocks (all have row % 8 == g, hence
        // the same swizzle), two blocks per pass so that four accumulator chains interleave
#pragma unroll
        for (int b0 = 0; b0 < RB; b0 += 2) {
            uint4 q0[2], q8[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                q0[h] = *reinterpret_cast<const uint4 *>(tb + (16 * (b0 + h) + g) * 128);
                q8[h] = *reinterpret_cast<const uint4 *>(tb + (16 * (b0 + h) + g + 8) * 128);
            }
            float da[2][4], db[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k = 0; k < 4; ++k) da[h][k] = db[h][k] = 0.f;
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t u0 = p == 0 ? q0[h].x : p == 1 ? q0[h].y : p == 2 ? q0[h].z : q0[h].w;
                    const uint32_t u8 = p == 0 ? q8[h].x : p == 1 ? q8[h].y : p == 2 ? q8[h].z : q8[h].w;
                    const uint32_t v0 = u0 >> 4, v8 = u8 >> 4;
                    mma_e4m3_e5m2(da[h], u0 & 0x03030303u, u8 & 0x03030303u, v0 & 0x03030303u, v8 & 0x03030303u,
                                  bf[p].x, bf[p].y);
                    mma_e4m3_e5m2(db[h], u0 & 0x0C0C0C0Cu, u8 & 0x0C0C0C0Cu, v0 & 0x0C0C0C0Cu, v8 & 0x0C0C0C0Cu,
                                  bf[p].z, bf[p].w);
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float lo = quad_sum(combine(da[h][0], da[h][1], db[h][0], db[h][1], sa0, sa1, sb0, sb1));
                const float hi = quad_sum(combine(da[h][2], da[h][3], db[h][2], db[h][3], sa0, sa1, sb0, sb1));
                if (t == 0) {
                    red[kw * RED + 16 * (b0 + h) + g] = lo;
                    red[kw * RED + 16 * (b0 + h) + g + 8] = hi;
                }
            }
        }
        __syncthreads();  // partial sums written; every warp is done with ring slot `slot`
        ok = *reinterpret_cast<volatile int *>(&s_fail) == 0;
        if (!ok) break;  // taken by every thread: the flag was read after the barrier
        waited = i + 1;
        if (leader && i + ring < my_blocks) issue(i + ring);
        if (threadIdx.x < ROWS) {
            const int r = threadIdx.x;
            if (i == 0) {
                sxr = red[64 + (r & 15)];
                for (int k = 1; k < KW; ++k) sxr += red[k * RED + 64 + (r & 15)];
            }
            float s1 = red[r];
            for (int k = 1; k < KW; ++k) s1 += red[k * RED + r];
            const int64_t row = (int64_t)(blk0 + i) * ROWS + r;
            if (row < a.rows) a.y[row] = scl * __fadd_rn(__fmul_rn(c0, sxr), __fmul_rn(dd, s1));
            const int64_t nrow = row + ROWS;
            if (i + 1 < my_blocks && nrow < a.rows) scl = __half2float(__ushort_as_half(a.scales[nrow]));
        }
        __syncthreads();  // the next block may overwrite the partial sums
    }
    // copies in flight after a failed wait must land before the shared memory is released
    if (!ok && leader) {
        if (!mbar_wait(xbar, 0)) atomicExch(&g_gemv_fp8_err, kDevErrDrain);
        const int issued = min(my_blocks, waited + ring);
        for (int j = waited; j < issued; ++j)
            if (!mbar_wait(&bars[j % ring], (j / ring) & 1)) atomicExch(&g_gemv_fp8_err, kDevErrDrain);
    }
}

}  // namespace

bool gemv_fp8_supported(const PackedArgs &a) {
    return a.cols % 512 == 0 && a.cols <= 4096 && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 && a.rows < ((int64_t)1 << 31);
}

cudaError_t launch_gemv_fp8(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    if (!gemv_fp8_supported(a)) return cudaErrorNotSupported;
    const int64_t rowbytes = a.cols / 4;
    CUtensorMap tm;
    cudaError_t e = make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, (uint64_t)rowbytes, (uint64_t)a.rows,
                                 (uint64_t)rowbytes, 128, ROWS, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(gemv2_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int kw = (int)(a.cols / 256);
    const int64_t nrowblk = (a.rows + ROWS - 1) / ROWS;
    const int nblk = cfg.blocks_per_cta > 0 ? cfg.blocks_per_cta : 1;
    const int ring = nblk >= 2 ? 2 : 1;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((nrowblk + nblk - 1) / nblk));
    lc.blockDim = dim3(32 * kw);
    lc.dynamicSmemBytes = 1024 + (size_t)ring * (a.cols / 512) * BOX + (size_t)a.cols * 2 + (size_t)a.cols * 8 +
                          (size_t)((kw * RED + 1) & ~1) * 4 + (size_t)(ring + 1) * 8;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    return cudaLaunchKernelEx(&lc, gemv2_fp8_kernel, tm, a, prefetch, nblk, ring);
}

unsigned int gemv_fp8_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_gemv_fp8_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_gemv_fp8_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
