// gemv_packed2_mxf4.cu -- 2-bit GEMV on the tcgen05 tensor cores with packed fp4
// (e2m1) operands: the codes are the A operand in tensor memory as they stand,
// two integer operations per eight fields, and the activations are the B
// operand as exact fp4 digits.
//
// "Kernel 0112", sections "What is being measured" and "The kernel": a
// 12,288 x 1,536 matrix of 2-bit weights times 1,536 inputs, dominated by
// reading the 4.5 MiB of weights.  Here the CUDA cores only move bits; the
// products and sums run in kind::mxf4 MMAs (M = 128, N = 16, K = 64).
//
// Codes as e2m1 (A).  A 2-bit field c in the low two bits of a nibble is the
// e2m1 value c / 2 (0, 0.5, 1, 1.5).  For a 32-bit code word w (fields f =
// 0..15 at bits 2f..2f+1), w & 0x33333333 holds fields 0, 2, .., 14 in its
// nibbles 0..7 and (w >> 2) & 0x33333333 fields 1, 3, .., 15.  Thread r of the
// four decode warps owns TMEM lane r (row r of the 128-row A tile) and stores
// the two words of code word q of a 256-field stage in TMEM columns 2q and
// 2q + 1.  With packed fp4 in TMEM, column c of a lane holds K positions
// 8c .. 8c + 7 (nibble i = K position 8c + i), so K position 16q + 8h + i of a
// stage carries field 16q + 2i + h.
//
// x as e2m1 digits (B).  A finite fp16 value times 2^24 is an integer T with
// |T| < 2^40.  Its balanced radix-8 digits d_j (j = 0..13, each in -4..4) give
// x = sum_j (d_j / 2) 2^(3j - 23), and d_j / 2 is an exact e2m1 value.  B row j
// (piece j) holds d_j / 2 of the x value that meets each K position; rows 14
// and 15 are zero.  All block scales are 1 (ue8m0 127), so every D column is
// an exact sum: D[r][j] = sum_k (c_k / 2)(d_jk / 2), a multiple of 1/4 below
// 2^14 for 1,536 fields.
//
// Affine codebooks (codebook[c] = c0 + c d).  Lane 127 of every tile stores an
// all-ones pattern (every nibble 1.0), so D row 127 is S_j = sum_k d_jk / 2,
// formed by the same MMAs; a tile therefore covers 127 weight rows.  Then
//     y = scale * sum_j 2^(3j - 23) (c0 S_j + 2 d D_j),
// and each bracket is exact for a codebook of small dyadic values such as
// {-2, -1, 0, 1}: the only rounding is the fp32 sum over the 14 pieces and the
// scale.  A row whose fields all hold the zero entry c_z has D_j = (c_z/2) S_j
// and gives y == 0 exactly.  A non-finite x makes every y of that matrix NaN.
//
// Roles (11 warps).  Two decode warpgroups (warps 0-3, 4-7) take the
// 256-field stages of a tile alternately, each thread one TMEM lane (row): it
// reads its row's code bytes from the box in shared memory, stores the two
// words per code word to a TMEM stage with tcgen05.st, and hands the stage to
// the MMA warp one decode later (the store completes meanwhile).  Warp 8 is
// the producer: lane 0 issues the TMA copies of the code boxes (128 bytes x
// 128 rows, 128-byte swizzle) into a ring, and after a tile's last box the
// warp loads that tile's scales into a small shared ring, so that no decode
// warp ever waits on a global load.  Warps 9 and 10 lane 0 each issue the MMAs
// of one warpgroup's stages into their own accumulator of the tile and commit
// each stage to the barrier that frees its TMEM stage; the epilogue adds the
// two accumulators (exactly: both are small multiples of 1/4).  Two tile
// buffers let the epilogue of a tile, run by warpgroup (tile % 2), overlap the
// next tile.  The decode warps and the MMA warps build the B tile, once per
// matrix.  A CTA takes a contiguous run of the (matrix, tile) pairs of a
// strided batch.
//
// Requirements: cols % 512 == 0, cols <= 4096, 16-byte aligned codes (and
// codes stride), an affine codebook.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tmap.h"

#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

namespace mm {

__device__ unsigned int g_gemv_mxf4_err;

namespace {

constexpr int LANES = 128, TR = 127;  // TMEM lanes per tile; weight rows per tile (lane 127: piece sums)
constexpr int BOXB = 128 * LANES;     // bytes of one code box: 128 bytes (512 fields) x 128 rows
constexpr int NPIECE = 14;            // radix-8 digits of x * 2^24
constexpr int NCOL = 16;              // MMA N: the pieces and two zero columns
constexpr int ASTAGES = 4;            // TMEM stages of A, 256 fields (32 columns) each
constexpr int TMEM_COLS = 256;        // D [0,64) (tile buffer db, issuer p at 16 (2 db + p)), SFA [64,72),
                                      // SFB [72,80), A [128,256)
constexpr int D_COL = 0, SFA_COL = 64, SFB_COL = 72, A_COL = 128;
constexpr int NWG = 2;                // decode warpgroups and MMA issuers, taking alternate stages
constexpr int NDEC = 128 * NWG, NTHREADS = NDEC + 32 * (1 + NWG), NBUILD = NDEC + 32 * NWG;
constexpr int PRODUCER_WARP = 4 * NWG, MMA_WARP = PRODUCER_WARP + 1;  // MMA warps MMA_WARP + p, p < NWG
constexpr int SRING = 4;              // tiles whose scales the producer has staged in shared memory
// kind::mxf4 instruction descriptor: A and B e2m1 (code 1), N >> 3 at bit 17, ue8m0 block
// scales (bit 23), M >> 4 at bit 24, scale-factor ids 0, K = 64
constexpr uint32_t IDESC = (1u << 7) | (1u << 10) | ((uint32_t)(NCOL >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);
constexpr uint32_t kUnitScales = 0x7F7F7F7Fu;  // ue8m0 2^0 in every byte
constexpr uint32_t kOnesRow = 0x22222222u;     // e2m1 1.0 in every nibble

struct Mxf4Args {
    const uint16_t *scales;
    int64_t scales_stride;
    const uint16_t *x;
    int64_t x_stride;  // 0: one x for every matrix
    float *y;
    int64_t y_stride;
    int64_t batch, rows, cols;
    float c0, d;  // codebook[c] = c0 + c d
};

// The 14 e2m1 digit nibbles of an fp16 value (nibble j = piece j), and whether it is finite.
// x 2^24 = M 2^sh with M < 2^11; sh = 3 q0 + r, so the balanced radix-8 digits of u = M 2^r
// (< 2^13: five digits in -3..4) sit at pieces q0 .. q0 + 4 (q0 <= 9).  Adding 3 to each of
// the five octal digits, w = u + 3 (1 + 8 + 64 + 512 + 4096), makes every digit of w, t, equal
// to the wanted digit plus 3, carries included.  The five t go to nibbles and are mapped at
// once: d = t - 3 (x >= 0) or 3 - t (x < 0), stored as the e2m1 value d / 2, i.e. sign in bit 3
// and |d| (0..4) in bits 0-2.  Per nibble, (t | 8) - 3 = t + 5 and 11 - t never borrow.
__device__ __forceinline__ uint64_t x_nibbles(uint32_t h, bool &finite) {
    const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
    finite = e != 31u;
    const uint32_t M = e ? (m | 1024u) : m;
    const uint32_t sh = e ? e - 1u : 0u;
    const uint32_t q0 = (sh * 43u) >> 7;  // sh / 3 for sh <= 29
    const uint32_t w = (M << (sh - 3u * q0)) + 14043u;
    const uint32_t t = (w & 7u) | ((w << 1) & 0x70u) | ((w << 2) & 0x700u) | ((w << 3) & 0x7000u) |
                       ((w << 4) & 0x70000u);
    const uint32_t tp5 = (t | 0x88888u) - 0x33333u;  // t + 5: the code of 8 | (t - 3)
    const uint32_t m11 = 0xBBBBBu - t;               // 11 - t: the code of 8 | (3 - t)
    uint32_t code;
    if (h & 0x8000u) {  // d = 3 - t: negative for t >= 4
        const uint32_t ge4 = ((t >> 2) & 0x11111u) * 15u;
        code = (tp5 & ge4) | (m11 & 0x77777u & ~ge4);
    } else {            // d = t - 3: negative for t <= 2
        const uint32_t ge3 = ((tp5 >> 3) & 0x11111u) * 15u;
        code = (tp5 & 0x77777u & ge3) | (m11 & ~ge3);
    }
    return (uint64_t)code << (4u * q0);
}

// a[e] nibble n -> a[n] nibble e for an 8 x 8 block of nibbles (three butterfly stages).
__device__ __forceinline__ void transpose_nibbles8(uint32_t (&a)[8]) {
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const uint32_t t = ((a[e] >> 4) ^ a[e + 1]) & 0x0F0F0F0Fu;
        a[e + 1] ^= t;
        a[e] ^= t << 4;
    }
#pragma unroll
    for (int e = 0; e < 8; e += (e & 1) ? 3 : 1) {  // 0, 1, 4, 5
        const uint32_t t = ((a[e] >> 8) ^ a[e + 2]) & 0x00FF00FFu;
        a[e + 2] ^= t;
        a[e] ^= t << 8;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t t = ((a[e] >> 16) ^ a[e + 4]) & 0x0000FFFFu;
        a[e + 4] ^= t;
        a[e] ^= t << 16;
    }
}

// B tile: NCOL rows x cols K positions, packed fp4, K-major with the 128-byte swizzle, in
// chunks of 256 K positions (NCOL rows x 128 bytes = 2 KiB, 8-row groups 1 KiB apart).  One
// unit per 32-bit word of the rows: word j of chunk s holds K positions 8j .. 8j + 7, which meet
// fields 16 (j >> 1) + (j & 1) + 2i (i = 0..7) of that chunk; the eight values' digit nibbles
// are transposed so that row n's word holds digit n of each, in K order.
__device__ __forceinline__ bool build_b_tile(const uint16_t *xs, uint8_t *btile, int cols, int bt, int nbt) {
    bool finite = true;
    for (int u = bt; u < (cols >> 3); u += nbt) {
        const int s = u >> 5, j = u & 31;
        const int base = (s << 8) + ((j >> 1) << 4) + (j & 1);
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bool f;
            const uint64_t v = x_nibbles(xs[base + 2 * i], f);
            finite = finite && f;
            lo[i] = (uint32_t)v;
            hi[i] = (uint32_t)(v >> 32);
        }
        transpose_nibbles8(lo);
        transpose_nibbles8(hi);
        uint8_t *cb = btile + s * 2048 + 4 * (j & 3);
        const int c = j >> 2;  // the word's 16-byte chunk in the 128-byte row
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            *reinterpret_cast<uint32_t *>(cb + n * 128 + ((c ^ n) << 4)) = lo[n];
            *reinterpret_cast<uint32_t *>(cb + 1024 + n * 128 + ((c ^ n) << 4)) = hi[n];
        }
    }
    return finite;
}

// x (cols fp16 values, cols % 512 == 0) into shared memory with coalesced loads that are all in
// flight at once: 16-byte loads when x is 16-byte aligned, 2-byte loads otherwise.
__device__ __forceinline__ void stage_x(const uint16_t *x, uint16_t *xs, int cols, int bt, int nbt) {
    if ((reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        const uint4 *src = reinterpret_cast<const uint4 *>(x);
        uint4 *dst = reinterpret_cast<uint4 *>(xs);
        for (int i = bt; i < (cols >> 3); i += nbt) dst[i] = __ldg(src + i);
    } else {
#pragma unroll 4
        for (int i = bt; i < cols; i += nbt) xs[i] = __ldg(x + i);
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

__device__ __forceinline__ void tmem_st8(uint32_t taddr, uint32_t v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"r"(taddr), "r"(v)
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

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::mxf4 with block scales read from tensor memory
__device__ __forceinline__ void umma_mxf4_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t sfa,
                                                 uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], [%1], %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(IDESC), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Named barrier over the B-tile builders (decode warps and the MMA warp) that also returns
// whether any of them passed `pred`.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

struct Bars {
    uint64_t dfull[2], dempty[2];
    uint64_t afull[ASTAGES], aempty[ASTAGES];
    uint64_t sfull[SRING], sempty[SRING];
    uint64_t last;
    uint32_t tmem_slot;
    int fail;
    float sx[2][NPIECE];
    uint16_t sbuf[SRING][128];  // the scales of a tile's 127 rows, staged by the producer warp
    uint64_t bfull[1];          // [bring], followed by bempty[bring]
};

__global__ void __launch_bounds__(NTHREADS, 2) gemv2_mxf4_kernel(const __grid_constant__ CUtensorMap tmC,
                                                             const Mxf4Args a, const int prefetch,
                                                             const int tiles_per_cta, const int bring) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    const int cols = (int)a.cols;
    const int nbox = cols >> 9;  // code boxes per tile
    const int nst = cols >> 8;   // 256-field stages per tile
    uint8_t *boxes = smem;                                  // [bring][128 rows][128 B]
    uint8_t *btile = boxes + (size_t)bring * BOXB;          // cols * 8 bytes
    uint16_t *xs = reinterpret_cast<uint16_t *>(btile + (size_t)cols * 8);  // cols fp16
    Bars *bb = reinterpret_cast<Bars *>(xs + cols);
    uint64_t *bfull = bb->bfull, *bempty = bb->bfull + bring;
    volatile int *fail = &bb->fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t ntiles = (a.rows + TR - 1) / TR;
    const int64_t total = ntiles * a.batch;
    const int64_t g0 = (int64_t)blockIdx.x * tiles_per_cta;
    const int my_tiles = (int)min((int64_t)tiles_per_cta, total - g0);

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bb->dfull[i], NWG);  // each MMA issuer commits its share of the tile
            mbar_init(&bb->dempty[i], 4);  // the four warps of the tile's epilogue warpgroup
        }
        for (int i = 0; i < ASTAGES; ++i) {
            mbar_init(&bb->afull[i], 4);   // the four warps of the stage's warpgroup
            mbar_init(&bb->aempty[i], 1);
        }
        for (int i = 0; i < bring; ++i) {
            mbar_init(&bfull[i], 1);
            mbar_init(&bempty[i], NDEC / 32);  // every decode warp reads half a box
        }
        for (int i = 0; i < SRING; ++i) {
            mbar_init(&bb->sfull[i], 32);  // every producer lane stores its share of the scales
            mbar_init(&bb->sempty[i], 4);  // the epilogue warpgroup's four warps
        }
        mbar_init(&bb->last, NWG);
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

    // A failed bounded wait marks the CTA; later waits then return at once and every role
    // skips its remaining work but still reaches the barriers below.
    auto wait = [&](uint64_t *bar, uint32_t parity, unsigned code) -> bool {
        if (*fail) return false;
        if (mbar_wait_sleep(bar, parity)) return true;
        *fail = 1;
        atomicExch(&g_gemv_mxf4_err, code);
        return false;
    };
    // the pipeline's short hand-offs (decode <-> MMA, a box that has landed): spinning tries,
    // same limit; a suspending wait measured ~300 ns per stage on GB300 even when the phase
    // had completed long before
    auto spin = [&](uint64_t *bar, uint32_t parity, unsigned code) -> bool {
        if (*fail) return false;
        if (mbar_wait(bar, parity)) return true;
        *fail = 1;
        atomicExch(&g_gemv_mxf4_err, code);
        return false;
    };

    const int total_boxes = my_tiles * nbox;
    if (warp == PRODUCER_WARP) {
        // ------------------------------------------------------------ TMA producer
        // codes may be loaded before the wait on the previous kernel unless they may be
        // written by it (prefetch 0)
        if (prefetch == 0) pdl_wait();
        if (lane == 0) tma_prefetch_desc(&tmC);
        int issued = 0;
        for (; issued < total_boxes; ++issued) {
            const int slot = issued % bring;
            bool okp = true;
            if (lane == 0 && issued >= bring) okp = wait(&bempty[slot], ((issued / bring) - 1) & 1, kDevErrWaitEmpty);
            if (!__shfl_sync(0xffffffffu, okp, 0)) break;
            const int tl = issued / nbox;  // tile of this CTA
            const int gt = (int)g0 + tl, mt = gt / (int)ntiles, row0 = (gt - mt * (int)ntiles) * TR;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bfull[slot], (uint32_t)BOXB);
                tma_load_3d(boxes + (size_t)slot * BOXB, &tmC, &bfull[slot], (issued % nbox) * 128, row0, mt);
            }
            if (issued % nbox == nbox - 1) {
                // the tile's scales, loaded once its boxes are on their way (its epilogue comes
                // after all of them), so that no decode warp ever waits on a global load
                const int ss = tl % SRING;
                bool oks = true;
                if (lane == 0 && tl >= SRING) oks = wait(&bb->sempty[ss], ((tl / SRING) - 1) & 1, kDevErrWaitEmpty);
                if (!__shfl_sync(0xffffffffu, oks, 0)) break;
                const uint16_t *sc = a.scales + (int64_t)mt * a.scales_stride;
#pragma unroll
                for (int i = lane; i < 128; i += 32) {
                    const int64_t rr = (int64_t)row0 + i;
                    bb->sbuf[ss][i] = (i < TR && rr < a.rows) ? __ldg(sc + rr) : (uint16_t)0;
                }
                mbar_arrive(&bb->sfull[ss]);
            }
        }
        // every issued copy lands before the CTA can exit
        if (lane == 0)
            for (int gb = max(0, issued - bring); gb < issued; ++gb)
                if (!mbar_wait_sleep(&bfull[gb % bring], (gb / bring) & 1)) atomicExch(&g_gemv_mxf4_err, kDevErrDrain);
        if (prefetch == 2) pdl_launch_dependents();
    } else {
        // ------------------------------------------------------------ B builders: decode warps + MMA warp
        const int bt = warp >= MMA_WARP ? NDEC + 32 * (warp - MMA_WARP) + lane : tid;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        if (warp < 4) {  // unit block scales of A and B in this warp's lanes
            tmem_st8(tmem + lane_base + SFA_COL, kUnitScales);
            tmem_st8(tmem + lane_base + SFB_COL, kUnitScales);
            tmem_wait_st();
        }
        // x and y belong to the previous kernel until it has finished (independent calls
        // promise they do not)
        if (prefetch < 2) pdl_wait();
        // the next call may launch once this one has passed its wait: at most one chained call
        // runs ahead (its weight loads) instead of a queue of parked ones
        if (prefetch == 2 || warp == MMA_WARP) pdl_launch_dependents();
        // decode role state (warps 0-3)
        const int r = tid & 127;  // TMEM lane = tile row
        const int wg = tid >> 7;  // decode warpgroup (warps 0-3, 4-7)
        const uint32_t b_base = smem_u32(btile);
        int t = 0;  // tiles of this CTA started
        while (t < my_tiles) {
            const int64_t mat = (g0 + t) / ntiles;  // the matrix whose x the B tile holds
            int seg = my_tiles - t;                  // tiles sharing this x
            if (a.x_stride != 0) seg = (int)min((int64_t)seg, (mat + 1) * ntiles - (g0 + t));
            stage_x(a.x + mat * a.x_stride, xs, cols, bt, NBUILD);
            bar_sync(2, NBUILD);
            const bool finite = build_b_tile(xs, btile, cols, bt, NBUILD);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            const bool nonfinite = bar_red_or(1, NBUILD, !finite);
            tc_fence_after_sync();
            if (warp >= MMA_WARP) {
                // -------------------------------------------------------- MMA issuers
                // Issuer p multiplies the stages s = p, p + 2, .. (those of decode warpgroup p)
                // into its own accumulator of the tile; the epilogue adds the two (exactly).
                const int p = warp - MMA_WARP;
                if (lane == 0) {
                    bool ok = true;
                    for (int tt = t; tt < t + seg && ok; ++tt) {
                        const int db = tt & 1;
                        if (tt >= 2 && !spin(&bb->dempty[db], ((tt >> 1) - 1) & 1, kDevErrWaitEmpty)) break;
                        const uint32_t d = tmem + D_COL + 16 * (2 * db + p);
                        for (int s = p; s < nst; s += NWG) {
                            const int g = tt * nst + s;
                            const int as = g % ASTAGES;
                            if (!spin(&bb->afull[as], (g / ASTAGES) & 1, kDevErrWaitFull)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after_sync();
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                umma_mxf4_tmem_a(d, tmem + A_COL + 32 * as + 8 * k,
                                                 sdesc_kmajor_sw128(b_base + s * 2048 + 32 * k), tmem + SFA_COL,
                                                 tmem + SFB_COL, (s > p || k > 0) ? 1u : 0u);
                            umma_commit(&bb->aempty[as]);
                        }
                        if (ok) umma_commit(&bb->dfull[db]);
                    }
                }
                __syncwarp();
            } else {
                // -------------------------------------------------------- decode + epilogue
                // Warpgroup wg decodes the stages s = wg, wg + 2, .. of every tile (a box's two
                // stages go to the two warpgroups) and runs the epilogue of the tiles tt with
                // tt % 2 == wg, so one warpgroup's epilogue overlaps the other's decode.
                const float c0 = a.c0, two_d = 2.0f * a.d;
                for (int tt = t; tt < t + seg; ++tt) {
                    const int64_t gt = g0 + tt;
                    const int64_t mt = gt / ntiles;  // this tile's matrix (a shared x spans several)
                    const int64_t row = (gt % ntiles) * TR + r;
                    const bool mine = (tt & 1) == wg;  // this warpgroup's epilogue
                    const bool real = mine && r < TR && row < a.rows;
                    bool ok = __all_sync(0xffffffffu, *fail == 0);  // warp-uniform from here on
                    // each stage's TMEM store completes while the warpgroup decodes its next
                    // stage: the stage is handed to the MMA warp one decode later
                    bool pend = false;
                    int pas = 0;
                    for (int s = wg; s < nst && ok; s += NWG) {
                        const int g = tt * nst + s;  // stage of this CTA
                        const int gbx = g >> 1;      // code box of this CTA (two stages each)
                        const int bs = gbx % bring;
                        ok = __all_sync(0xffffffffu, spin(&bfull[bs], (gbx / bring) & 1, kDevErrWaitFull));
                        const int as = g % ASTAGES;
                        if (ok && g >= ASTAGES)
                            ok = __all_sync(0xffffffffu,
                                            spin(&bb->aempty[as], ((g / ASTAGES) - 1) & 1, kDevErrWaitMma));
                        if (!ok) break;
                        uint32_t v[32];
                        if (r == TR) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = kOnesRow;
                        } else {
                            // 64 code bytes of this row: 16-byte chunks 4(s&1) .. 4(s&1)+3 of the box
                            const uint8_t *rowp = boxes + (size_t)bs * BOXB + r * 128;
                            const int ch = 4 * (s & 1);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint4 q = *reinterpret_cast<const uint4 *>(rowp + (((ch + i) ^ (r & 7)) << 4));
                                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    v[8 * i + 2 * j] = w[j] & 0x33333333u;
                                    v[8 * i + 2 * j + 1] = (w[j] >> 2) & 0x33333333u;
                                }
                            }
                        }
                        __syncwarp();  // this warp is done reading its half of the box
                        if (lane == 0) mbar_arrive(&bempty[bs]);
                        if (pend) {
                            tmem_wait_st();
                            tc_fence_before_sync();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bb->afull[pas]);
                        }
                        tmem_st32(tmem + lane_base + A_COL + 32 * as, v);
                        pend = true;
                        pas = as;
                    }
                    if (pend) {
                        tmem_wait_st();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0 && ok) mbar_arrive(&bb->afull[pas]);
                    }
                    if (!mine) continue;
                    // epilogue of tile tt: its scales, staged by the producer warp
                    const int ss = tt % SRING;
                    if (ok) ok = __all_sync(0xffffffffu, spin(&bb->sfull[ss], (tt / SRING) & 1, kDevErrWaitFull));
                    const float scl = ok ? __half2float(__ushort_as_half(bb->sbuf[ss][r])) : 0.f;
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(&bb->sempty[ss]);
                    const int db = tt & 1;
                    float v[16];
                    if (ok) ok = __all_sync(0xffffffffu, spin(&bb->dfull[db], (tt >> 1) & 1, kDevErrWaitMma));
                    if (ok) {
                        float v1[16];
                        tc_fence_after_sync();
                        tmem_ld16(tmem + lane_base + D_COL + 32 * db, v);
                        tmem_ld16(tmem + lane_base + D_COL + 32 * db + 16, v1);
                        tc_fence_before_sync();
#pragma unroll
                        for (int j = 0; j < NPIECE; ++j) v[j] = __fadd_rn(v[j], v1[j]);  // exact: both are small multiples of 1/4
                    }
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(&bb->dempty[db]);
                    if (r == TR) {
#pragma unroll
                        for (int j = 0; j < NPIECE; ++j) bb->sx[db][j] = ok ? v[j] : 0.f;
                    }
                    bar_sync(3 + wg, 128);  // the piece sums of this tile are in shared memory
                    if (!*fail && real) {
                        float acc = 0.f;
#pragma unroll
                        for (int j = 0; j < NPIECE; ++j) {
                            const float p = __fmaf_rn(two_d, v[j], __fmul_rn(c0, bb->sx[db][j]));
                            acc = __fmaf_rn(p, __int_as_float((127 + 3 * j - 23) << 23), acc);
                        }
                        a.y[mt * a.y_stride + row] = nonfinite ? __int_as_float(0x7FC00000) : __fmul_rn(scl, acc);
                    }
                }
            }
            bar_sync(2, NBUILD);  // every MMA reading this B tile has completed (epilogues waited for them)
            t += seg;
        }
        if (warp >= MMA_WARP && lane == 0) {
            // every issued MMA completes before TMEM is released
            umma_commit(&bb->last);
            if (!mbar_wait_sleep(&bb->last, 0)) atomicExch(&g_gemv_mxf4_err, kDevErrWaitMma);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == PRODUCER_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

size_t mxf4_smem_bytes(int64_t cols, int bring) {
    return 1024 + (size_t)bring * BOXB + (size_t)cols * 10 + sizeof(Bars) + (size_t)2 * bring * 8;
}

cudaError_t launch_mxf4(const Mxf4Args &m, const void *codes, int64_t codes_stride, int pdl, int prefetch,
                        int tiles_per_cta, cudaStream_t st) {
    const int64_t rowbytes = m.cols / 4;
    CUtensorMap tm;
    cudaError_t e = make_tmap_3d(CU_TENSOR_MAP_DATA_TYPE_UINT8, &tm, codes, (uint64_t)rowbytes, (uint64_t)m.rows,
                                 (uint64_t)m.batch, (uint64_t)rowbytes,
                                 (uint64_t)(m.batch > 1 ? codes_stride : rowbytes * m.rows), 128, LANES,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(gemv2_mxf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t ntiles = (m.rows + TR - 1) / TR;
    const int64_t total = ntiles * m.batch;
    const int tpc = tiles_per_cta > 0 ? tiles_per_cta : 1;
    const int nbox = (int)(m.cols / 512);
    // code-box ring: a whole tile when a CTA has one, else up to 6 boxes, within 110 KiB so that
    // two CTAs share an SM (their 256 TMEM columns each also fit)
    int bring = std::min<int64_t>(tpc == 1 ? nbox : 6, (int64_t)tpc * nbox);
    bring = std::max(bring, 2);
    while (bring > 2 && mxf4_smem_bytes(m.cols, bring) > 110 * 1024) --bring;
    if (mxf4_smem_bytes(m.cols, bring) > 227 * 1024) return cudaErrorNotSupported;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((total + tpc - 1) / tpc));
    lc.blockDim = dim3(NTHREADS);
    // at least 76 KiB per CTA: no more than two CTAs share an SM, so their TMEM allocations
    // (256 columns each) always fit in the SM's 512 columns
    lc.dynamicSmemBytes = std::max<size_t>(mxf4_smem_bytes(m.cols, bring), 76 * 1024);
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, gemv2_mxf4_kernel, tm, m, prefetch, tpc, bring);
}

}  // namespace

bool gemv_mxf4_supported(const PackedArgs &a) {
    return a.cols % 512 == 0 && a.cols <= 4096 && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
           a.rows < ((int64_t)1 << 31) - 128 && codebook_is_affine(a.cb);
}

bool gemv_batched_mxf4_supported(const PackedBatch &p) {
    PackedArgs a{p.codes, p.scales, p.x, p.y, 1, p.rows, p.cols, {p.cb[0], p.cb[1], p.cb[2], p.cb[3]}};
    const int64_t ntiles = (p.rows + TR - 1) / TR;
    return gemv_mxf4_supported(a) && (p.batch == 1 || p.codes_stride % 16 == 0) &&
           ntiles * p.batch < ((int64_t)1 << 31) && p.batch < ((int64_t)1 << 31);
}

cudaError_t launch_gemv_mxf4(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t st) {
    if (!gemv_mxf4_supported(a)) return cudaErrorNotSupported;
    const Mxf4Args m{a.scales, 0, a.x, 0, a.y, 0, 1, a.rows, a.cols, a.cb[0], a.cb[1] - a.cb[0]};
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    return launch_mxf4(m, a.codes, 0, cfg.pdl, prefetch, cfg.blocks_per_cta, st);
}

cudaError_t launch_gemv_batched_mxf4(const PackedBatch &p, int tiles_per_cta, cudaStream_t st) {
    if (!gemv_batched_mxf4_supported(p)) return cudaErrorNotSupported;
    const Mxf4Args m{p.scales, p.scales_stride, p.x, p.x_stride, p.y, p.y_stride, p.batch, p.rows, p.cols, p.cb[0],
                     p.cb[1] - p.cb[0]};
    int tpc = tiles_per_cta;
    if (tpc <= 0) {
        // one run of tiles per CTA, two CTAs per SM
        int dev = 0, sms = 152;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t total = ((p.rows + TR - 1) / TR) * p.batch;
        tpc = (int)std::max<int64_t>(1, (total + 2 * sms - 1) / (2 * sms));
    }
    return launch_mxf4(m, p.codes, p.codes_stride, 0, 0, tpc, st);
}

unsigned int gemv_mxf4_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_gemv_mxf4_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_gemv_mxf4_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
