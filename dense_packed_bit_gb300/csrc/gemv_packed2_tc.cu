// gemv_packed2_tc.cu -- 2-bit GEMV on the tcgen05 tensor cores: the decoded
// codes are the A operand in tensor memory, the activation vector is the B
// operand in shared memory, fp8 x fp8 products, fp32 accumulation in TMEM.
//
// "Kernel 0112", sections "What is being measured" and "What the kernel costs
// in a whole token": the 12,288 x 1,536 GEMV streams 4.5 MiB of 2-bit codes.
// Turning 18.9 M fields per call into products is the expensive part; here
// the CUDA cores only mask bits and the tensor cores do the rest.
//
// Codes as e4m3 (A).  An e4m3 byte whose exponent field is 0 or 1 is worth its
// low four bits, read as an integer, times 2^-9.  For a 32-bit code word w
// (fields f = 0..15 at bits 2f..2f+1), the four registers
//     w & 0x03030303,  w & 0x0C0C0C0C,  (w >> 4) & 0x03030303,  (w >> 4) & 0x0C0C0C0C
// hold fields {0,4,8,12}, {1,5,9,13}, {2,6,10,14}, {3,7,11,15} as exact e4m3
// values c 2^-9 (set 0: the first and third register) or c 2^-7 (set 1).
// Thread r of the four decode warps owns TMEM lane r, i.e. row r of the
// 128-row A tile, and stores these registers there with tcgen05.st: TMEM
// column 4q + j (word q, register j) holds K positions 16q + 4j + e, which
// carry fields 16q + 4e + j (e = 0..3, one per byte).
//
// x as e5m2 (B).  e5m2 is the top byte of an fp16, so cutting an fp16 value
// to its top byte leaves an exact e5m2 piece and an exact fp16 remainder; four
// pieces hold the value exactly when all of its bits lie at or above 2^-16,
// true for |x| >= 2^-6 ("window 0"); smaller values are scaled by 2^18 first
// ("window 1"), which reaches down to the smallest fp16 subnormal.  B has 16
// rows: row 8 s + 4 v + i carries piece i of window v of the x value that
// meets K position k when k belongs to set s, and 0 otherwise.  So D column n
// of a row sums c x over one (set, window, piece); it is scaled by 2^9 or 2^7
// (set) and by 2^-18 for window 1, all exact, and the 16 columns are added in
// a fixed order.
//
// Affine codebooks (codebook[c] = c0 + c d): the MMAs give S1 = sum c_k x_k
// per row.  Lane 127 of every tile is not a weight row: its thread stores the
// bytes of an all-ones field pattern, so D row 127 is sum x, formed by the
// very same MMA instructions and reduced in the same order as the weight rows.
// y = scale (c0 sum x + d S1); a row whose fields all hold the zero entry
// c_z in {0, 1, 2} has S1 == c_z sum x exactly and gives y == 0.  A tile
// therefore covers 127 rows.
//
// Roles (6 warps): warps 0-3 decode and run the epilogue, warp 4 lane 0 issues
// the TMA copies of the code boxes (128 bytes x 128 rows, 128-byte swizzle)
// into a ring, warp 5 lane 0 issues the MMAs (M = 128, N = 16, K = 32) per
// 128-field stage from a 3-deep TMEM ring and commits each stage to the
// barrier that frees it; two TMEM accumulators let the epilogue of a tile run
// while the next tile is multiplied.
//
// Requirements: cols % 512 == 0, cols <= 8192, 16-byte aligned codes and x,
// an affine codebook (zero entry, if any, at field 0, 1 or 2).
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tmap.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {

__device__ unsigned int g_gemv_tc_err;

namespace {

constexpr int LANES = 128, TR = 127;  // TMEM lanes per tile; weight rows per tile (lane 127: sum x)
constexpr int BOXB = 128 * LANES;     // bytes of one code box: 128 bytes (512 fields) x 128 rows
constexpr int ASTAGES = 3;            // TMEM stages of A (128 fields = 32 columns each)
constexpr int TMEM_COLS = 128;        // D0 (0-15), D1 (16-31), A stages (32-127)
constexpr int NDEC = 128, NTHREADS = NDEC + 64;
constexpr int PRODUCER_WARP = 4, MMA_WARP = 5;
constexpr uint32_t IDESC = make_idesc(0 /* e4m3 */, 1 /* e5m2 */, 16, 128);

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

// Exact e5m2 pieces of the two fp16 values in v: win0 gets 0xFFFF in each half whose
// value lies in window 0 (|x| >= 2^-6); p[i] holds piece i of each value (window 1
// values scaled by 2^18) in the top byte of its half.
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

// B tile: 16 rows x cols bytes, K-major with the 128-byte swizzle, in blocks of
// 128 K positions (16 rows x 128 bytes = 2 KiB, 8-row groups 1 KiB apart).
// Word c of row n (K positions 4c .. 4c+3) lives at:
__device__ __forceinline__ uint32_t btile_offset(int n, int c) {
    const int w = c & 31, chunk = w >> 2;
    return (uint32_t)((c >> 5) * 2048 + (n >> 3) * 1024 + (n & 7) * 128 + ((chunk ^ (n & 7)) << 4) + 4 * (w & 3));
}

// One unit per TMEM column c = 4q + j of A: the 4 x values meeting its K positions
// (fields 16q + 4e + j), split into pieces, written to the 16 B rows.
__device__ __forceinline__ void build_b_tile(const uint16_t *xs, uint8_t *btile, int cols, int tid, int nthreads) {
    for (int c = tid; c < (cols >> 2); c += nthreads) {
        const int q = c >> 2, j = c & 3, set = j & 1;
        const int f = 16 * q + j;
        const uint32_t v01 = (uint32_t)xs[f] | ((uint32_t)xs[f + 4] << 16);
        const uint32_t v23 = (uint32_t)xs[f + 8] | ((uint32_t)xs[f + 12] << 16);
        uint32_t p01[4], p23[4], w01, w23;
        split_x2(v01, p01, w01);
        split_x2(v23, p23, w23);
        const uint32_t wmask = __byte_perm(w01, w23, 0x7531);  // 0xFF per value in window 0
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t bytes = __byte_perm(p01[i], p23[i], 0x7531);
            const int n0 = 8 * set + i, n1 = 8 * set + 4 + i, z0 = 8 * (1 - set) + i, z1 = z0 + 4;
            *reinterpret_cast<uint32_t *>(btile + btile_offset(n0, c)) = bytes & wmask;
            *reinterpret_cast<uint32_t *>(btile + btile_offset(n1, c)) = bytes & ~wmask;
            *reinterpret_cast<uint32_t *>(btile + btile_offset(z0, c)) = 0u;
            *reinterpret_cast<uint32_t *>(btile + btile_offset(z1, c)) = 0u;
        }
    }
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f8f6f4
__device__ __forceinline__ void umma_f8_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(IDESC), "r"(accumulate)
        : "memory");
}

// Row sum of the 16 accumulator columns, fixed order, no contraction: column n is
// scaled by 2^9 (set 0) or 2^7 (set 1), times 2^-18 for window 1.
__device__ __forceinline__ float row_sum(const float (&v)[16]) {
    float s = 0.f;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
        const int e = ((n >> 3) ? 7 : 9) - (((n >> 2) & 1) ? 18 : 0);
        s = __fadd_rn(s, __fmul_rn(v[n], __int_as_float((127 + e) << 23)));
    }
    return s;
}

struct Bars {
    uint64_t xbar;
    uint64_t dfull[2], dempty[2];
    uint64_t afull[ASTAGES], aempty[ASTAGES];
    uint64_t last;
    uint32_t tmem_slot;
    int fail;
    float sx[2];
    uint64_t bfull[1];  // [bring], followed by bempty[bring]
};

__global__ void __launch_bounds__(NTHREADS) gemv2_tc_kernel(const __grid_constant__ CUtensorMap tmC, const PackedArgs a,
                                                           const int prefetch, const int tiles_per_cta,
                                                           const int bring) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    const int cols = (int)a.cols;
    const int nbox = cols >> 9;    // code boxes per tile
    const int nst = cols >> 7;     // 128-field stages per tile
    uint8_t *boxes = smem;                                                    // [bring][128 rows][128 B]
    uint8_t *btile = boxes + (size_t)bring * BOXB;                            // cols * 16 bytes
    uint16_t *xs = reinterpret_cast<uint16_t *>(btile + (size_t)cols * 16);  // cols halves
    Bars *bb = reinterpret_cast<Bars *>(xs + cols);
    uint64_t *bfull = bb->bfull, *bempty = bb->bfull + bring;
    volatile int *fail = &bb->fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = (a.rows + TR - 1) / TR;
    const int64_t tile0 = (int64_t)blockIdx.x * tiles_per_cta;
    const int my_tiles = (int)min((int64_t)tiles_per_cta, ntiles - tile0);

    if (tid == 0) {
        mbar_init(&bb->xbar, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bb->dfull[i], 1);
            mbar_init(&bb->dempty[i], NDEC / 32);
        }
        for (int i = 0; i < ASTAGES; ++i) {
            mbar_init(&bb->afull[i], NDEC / 32);
            mbar_init(&bb->aempty[i], 1);
        }
        for (int i = 0; i < bring; ++i) {
            mbar_init(&bfull[i], 1);
            mbar_init(&bempty[i], NDEC / 32);
        }
        mbar_init(&bb->last, 1);
        bb->fail = 0;
        fence_mbar_init();
    }
    if (warp == PRODUCER_WARP) {
        tmem_alloc(&bb->tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bb->tmem_slot;

    // A failed bounded wait marks the CTA; later waits then return at once and every
    // role skips its remaining work but still reaches the barriers below.
    auto wait = [&](uint64_t *bar, uint32_t parity, unsigned code) -> bool {
        if (*fail) return false;
        if (mbar_wait_sleep(bar, parity)) return true;
        *fail = 1;
        atomicExch(&g_gemv_tc_err, code);
        return false;
    };

    // ---------------------------------------------------------------- prologue: x -> B tile
    int issued_boxes = 0;
    auto issue_box = [&](int gb) {  // box gb of this CTA: tile gb / nbox, column block gb % nbox
        const int s = gb % bring;
        mbar_arrive_expect_tx(&bfull[s], (uint32_t)BOXB);
        tma_load_2d(boxes + (size_t)s * BOXB, &tmC, &bfull[s], (gb % nbox) * 128,
                    (int)((tile0 + gb / nbox) * TR));
    };
    const int total_boxes = my_tiles * nbox;
    auto issue_x = [&] {
        mbar_arrive_expect_tx(&bb->xbar, (uint32_t)cols * 2);
        bulk_load(xs, a.x, (uint32_t)cols * 2, &bb->xbar);
    };
    if (prefetch >= 1) {
        if (warp == PRODUCER_WARP && lane == 0) {
            tma_prefetch_desc(&tmC);
            for (; issued_boxes < min(bring, total_boxes); ++issued_boxes) issue_box(issued_boxes);
            if (prefetch == 2) issue_x();
        }
        // chained calls: the next call may launch only once this one has passed its wait,
        // so at most one call runs ahead (its weight loads) instead of a queue of parked ones
        if (prefetch == 1) {
            pdl_wait();
            if (warp == PRODUCER_WARP && lane == 0) issue_x();
        }
        pdl_launch_dependents();
    } else {
        pdl_wait();
        if (warp == PRODUCER_WARP && lane == 0) {
            tma_prefetch_desc(&tmC);
            for (; issued_boxes < min(bring, total_boxes); ++issued_boxes) issue_box(issued_boxes);
            issue_x();
        }
        pdl_launch_dependents();
    }
    if (!mbar_wait_sleep(&bb->xbar, 0)) {
        *fail = 1;
        atomicExch(&g_gemv_tc_err, kDevErrWaitFull);
    }
    build_b_tile(xs, btile, cols, tid, NTHREADS);
    fence_proxy_async_smem();
    __syncthreads();

    if (warp == PRODUCER_WARP) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            for (; issued_boxes < total_boxes; ++issued_boxes) {
                const int s = issued_boxes % bring;
                if (!wait(&bempty[s], ((issued_boxes / bring) - 1) & 1, kDevErrWaitEmpty)) break;
                issue_box(issued_boxes);
            }
            // every issued copy lands before the CTA can exit
            for (int gb = max(0, issued_boxes - bring); gb < issued_boxes; ++gb)
                if (!mbar_wait_sleep(&bfull[gb % bring], (gb / bring) & 1)) atomicExch(&g_gemv_tc_err, kDevErrDrain);
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t b_base = smem_u32(btile);
            int g = 0;  // stage counter over all tiles of this CTA
            bool ok = true;
            for (int t = 0; t < my_tiles && ok; ++t) {
                const int db = t & 1;
                if (t >= 2 && !wait(&bb->dempty[db], ((t >> 1) - 1) & 1, kDevErrWaitEmpty)) break;
                for (int s = 0; s < nst; ++s, ++g) {
                    const int as = g % ASTAGES;
                    if (!wait(&bb->afull[as], (g / ASTAGES) & 1, kDevErrWaitFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f8_tmem_a(tmem + 16 * db, tmem + 32 + 32 * as + 8 * k,
                                       sdesc_kmajor_sw128(b_base + s * 2048 + 32 * k), (s > 0 || k > 0) ? 1u : 0u);
                    umma_commit(&bb->aempty[as]);
                }
                if (ok) umma_commit(&bb->dfull[db]);
            }
            // every issued MMA completes before TMEM is released
            umma_commit(&bb->last);
            if (!mbar_wait_sleep(&bb->last, 0)) atomicExch(&g_gemv_tc_err, kDevErrWaitMma);
        }
    } else {
        // ------------------------------------------------------------ decode + epilogue
        const int r = tid;  // TMEM lane = tile row
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const float c0 = a.cb[0], dd = a.cb[1] - a.cb[0];
        int g = 0, gb = 0;
        for (int t = 0; t < my_tiles; ++t) {
            const int64_t row = (tile0 + t) * TR + r;
            const bool real = r < TR && row < a.rows;
            const float scl = real ? __half2float(__ushort_as_half(a.scales[row])) : 0.f;
            bool ok = __all_sync(0xffffffffu, *fail == 0);  // warp-uniform from here on
            for (int s = 0; s < nst && ok; ++s, ++g) {
                const int bs = gb % bring;
                if ((s & 3) == 0) ok = __all_sync(0xffffffffu, wait(&bfull[bs], (gb / bring) & 1, kDevErrWaitFull));
                const int as = g % ASTAGES;
                if (ok && g >= ASTAGES)
                    ok = __all_sync(0xffffffffu, wait(&bb->aempty[as], ((g / ASTAGES) - 1) & 1, kDevErrWaitMma));
                if (!ok) break;
                uint32_t v[32];
                if (r == TR) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = (i & 1) ? 0x04040404u : 0x01010101u;
                } else {
                    // 32 code bytes of this row: 16-byte chunks 2(s&3), 2(s&3)+1 of the box
                    const uint8_t *rowp = boxes + (size_t)bs * BOXB + r * 128;
                    const int ch = 2 * (s & 3);
                    const uint4 q0 = *reinterpret_cast<const uint4 *>(rowp + ((ch ^ (r & 7)) << 4));
                    const uint4 q1 = *reinterpret_cast<const uint4 *>(rowp + (((ch + 1) ^ (r & 7)) << 4));
                    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t hi = w[q] >> 4;
                        v[4 * q + 0] = w[q] & 0x03030303u;
                        v[4 * q + 1] = w[q] & 0x0C0C0C0Cu;
                        v[4 * q + 2] = hi & 0x03030303u;
                        v[4 * q + 3] = hi & 0x0C0C0C0Cu;
                    }
                }
                tmem_st32(tmem + lane_base + 32 + 32 * as, v);
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bb->afull[as]);
                if ((s & 3) == 3) {  // this warp is done reading the box (nst is a multiple of 4)
                    if (lane == 0) mbar_arrive(&bempty[bs]);
                    ++gb;
                }
            }
            // epilogue of tile t
            const int db = t & 1;
            float v[16];
            if (ok) ok = __all_sync(0xffffffffu, wait(&bb->dfull[db], (t >> 1) & 1, kDevErrWaitMma));
            if (ok) {
                tc_fence_after_sync();
                tmem_ld16(tmem + lane_base + 16 * db, v);
                tc_fence_before_sync();
            }
            __syncwarp();
            if (lane == 0 && ok) mbar_arrive(&bb->dempty[db]);
            const float s1 = ok ? row_sum(v) : 0.f;
            if (r == TR) bb->sx[db] = s1;
            bar_sync(1, NDEC);  // sum x of this tile is in shared memory; taken by all decode warps
            if (!*fail && real) a.y[row] = scl * __fadd_rn(__fmul_rn(c0, bb->sx[db]), __fmul_rn(dd, s1));
            if (__any_sync(0xffffffffu, *fail != 0)) {
                // skip the rest (a warp-uniform decision), but keep the number of named-barrier
                // passes equal across the decode warps
                for (int tt = t + 1; tt < my_tiles; ++tt) bar_sync(1, NDEC);
                break;
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == PRODUCER_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

bool gemv_tc_supported(const PackedArgs &a) {
    return a.cols % 512 == 0 && a.cols <= 8192 && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 && a.rows < ((int64_t)1 << 31) - 128;
}

static size_t tc_smem_bytes(int64_t cols, int bring) {
    return 1024 + (size_t)bring * BOXB + (size_t)cols * 16 + (size_t)cols * 2 + sizeof(Bars) + (size_t)2 * bring * 8;
}

cudaError_t launch_gemv_tc(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    if (!gemv_tc_supported(a)) return cudaErrorNotSupported;
    const int64_t rowbytes = a.cols / 4;
    CUtensorMap tm;
    cudaError_t e = make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, (uint64_t)rowbytes, (uint64_t)a.rows,
                                 (uint64_t)rowbytes, 128, LANES, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(gemv2_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // code-box ring: as deep as one tile (at most 4 boxes), less when shared memory is short
    int bring = (int)std::min<int64_t>(4, a.cols / 512);
    while (bring > 2 && tc_smem_bytes(a.cols, bring) > 200 * 1024) --bring;
    if (tc_smem_bytes(a.cols, bring) > 227 * 1024) return cudaErrorNotSupported;
    const int64_t ntiles = (a.rows + TR - 1) / TR;
    const int tpc = cfg.blocks_per_cta > 0 ? cfg.blocks_per_cta : 1;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((ntiles + tpc - 1) / tpc));
    lc.blockDim = dim3(NTHREADS);
    // at least 48 KiB per CTA: no more than four CTAs share an SM, so their TMEM
    // allocations (128 columns each) always fit in the SM's 512 columns
    lc.dynamicSmemBytes = std::max<size_t>(tc_smem_bytes(a.cols, bring), 48 * 1024);
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = cfg.pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    return cudaLaunchKernelEx(&lc, gemv2_tc_kernel, tm, a, prefetch, tpc, bring);
}

unsigned int gemv_tc_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_gemv_tc_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_gemv_tc_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
