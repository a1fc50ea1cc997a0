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
// Roles.  One CTA per SM holds three independent tile pipelines.  Pipeline w has
// its own decode warpgroup (128 threads, one per TMEM lane: thread r reads its
// row's code bytes from the box in shared memory and stores the two words per
// code word to one of four TMEM A stages with tcgen05.st, handing the stage to
// the MMA warp as soon as the store has completed), its own MMA issuer warp
// (lane 0 issues the four MMAs of each stage into the pipeline's accumulator
// and commits them to the barrier that frees the stage), its code-box ring and
// its accumulator; the same warpgroup runs the tile's epilogue.  One producer
// warp issues the TMA copies of every pipeline's code boxes (128 bytes x 128
// rows, 128-byte swizzle) in the order the pipelines take their tiles; one
// scale warp stages each tile's 127 scales in shared memory, so that no decode
// warp ever waits on a global load.  The decode and MMA warps build the B
// tile once per matrix (once per launch when the batch shares x).  A CTA takes
// a contiguous run of the (matrix, tile) pairs of a strided batch; pipeline w
// takes its tiles w, w + 3, ...  Measured on the 64-matrix rotation: three
// pipelines with four A stages each and the immediate hand-off 0.97-1.00 us per
// matrix, four pipelines with three stages 1.00-1.02, the earlier hand-off one
// decode later 1.03-1.06.
//
// Requirements: cols % 512 == 0, cols <= 12,800, 16-byte aligned codes (and
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
constexpr int NWG = 3;                // tile pipelines per CTA (one CTA per SM), one decode warpgroup each
constexpr int ASLOTS = 4;             // TMEM stages of A per pipeline, 256 fields (32 columns) each
constexpr int MAX_RING = 3;           // code boxes per pipeline in shared memory (a 1,536-field tile: 3)
constexpr int TMEM_COLS = 512;        // SFA [0,8), SFB [8,16), accumulator of pipeline w [16 + 16 w, +16),
                                      // A stages of pipeline w [128 + 128 w, +128)
constexpr int SFA_COL = 0, SFB_COL = 8, D_COL = 16, A_COL = 128, A_SPAN = 32 * ASLOTS;
constexpr int NDEC = 128 * NWG, NTHREADS = NDEC + 32 * (2 + NWG), NBUILD = NDEC + 32 * NWG;
constexpr int PRODUCER_WARP = 4 * NWG, MMA_WARP = PRODUCER_WARP + 1;  // MMA warp of pipeline w: MMA_WARP + w
constexpr int SCALE_WARP = MMA_WARP + NWG;
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

// Barriers of one tile pipeline.  All counters of a pipeline are sequence numbers over the
// tiles it has taken (k-th tile: parity k & 1 for the per-tile barriers).
struct Pipe {
    uint64_t bfull[MAX_RING], bempty[MAX_RING];  // code boxes: TMA -> decode
    uint64_t afull[ASLOTS], aempty[ASLOTS];      // TMEM A stages: decode -> MMA
    uint64_t dfull, dempty;                      // accumulator: MMA -> epilogue
    uint64_t sfull, sempty;                      // the tile's scales: producer -> epilogue
    float sx[NPIECE];                            // the piece sums of the tile (TMEM lane 127)
    uint16_t sbuf[128];                          // the scales of the tile's 127 rows
};

struct Bars {
    Pipe pipe[NWG];
    uint64_t last;
    uint32_t tmem_slot;
    int fail;
};

// A CTA takes the tiles g0 .. g0 + my_tiles - 1 (of all matrices of the batch, in order).  A
// segment is a run of them that shares one x (the whole run when x is shared); within a segment
// pipeline w takes the segment's tiles w, w + NWG, w + 2 NWG, ..
__global__ void __launch_bounds__(NTHREADS, 1) gemv2_mxf4_kernel(const __grid_constant__ CUtensorMap tmC,
                                                                const Mxf4Args a, const int prefetch,
                                                                const int tiles_per_cta, const int ring) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    const int cols = (int)a.cols;
    const int nbox = cols >> 9;  // code boxes per tile
    const int nst = cols >> 8;   // 256-field stages per tile (two per box)
    uint8_t *boxes = smem;                                                   // [NWG][ring][128 rows][128 B]
    uint8_t *btile = boxes + (size_t)NWG * ring * BOXB;                     // cols * 8 bytes
    uint16_t *xs = reinterpret_cast<uint16_t *>(btile + (size_t)cols * 8);  // cols fp16
    Bars *bb = reinterpret_cast<Bars *>(xs + cols);
    volatile int *fail = &bb->fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = (int)((a.rows + TR - 1) / TR);  // tiles per matrix; ntiles * batch < 2^31
    const int total = ntiles * (int)a.batch;
    const int g0 = (int)blockIdx.x * tiles_per_cta;
    const int my_tiles = min(tiles_per_cta, total - g0);

    if (tid == 0) {
        for (int w = 0; w < NWG; ++w) {
            Pipe &pp = bb->pipe[w];
            for (int i = 0; i < ring; ++i) {
                mbar_init(&pp.bfull[i], 1);
                mbar_init(&pp.bempty[i], 4);  // the pipeline's four decode warps
            }
            for (int i = 0; i < ASLOTS; ++i) {
                mbar_init(&pp.afull[i], 4);
                mbar_init(&pp.aempty[i], 1);
            }
            mbar_init(&pp.dfull, 1);
            mbar_init(&pp.dempty, 4);
            mbar_init(&pp.sfull, 32);  // every producer lane stores its share of the scales
            mbar_init(&pp.sempty, 4);
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
        if (mbar_try_wait(bar, parity)) return true;
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait(bar, parity)) {
            __nanosleep(32);
            if (global_ns() - t0 > kWaitLimitNs) {
                *fail = 1;
                atomicExch(&g_gemv_mxf4_err, code);
                return false;
            }
        }
        return true;
    };
    // waits of the roles off the decode's critical path (MMA issuers, producer, scales): they
    // sleep between tries, so that their polling leaves the issue slots to the decode warps
    auto nap = [&](uint64_t *bar, uint32_t parity, unsigned code) -> bool {
        if (*fail) return false;
        if (mbar_try_wait(bar, parity)) return true;
        const unsigned long long t0 = global_ns();
        unsigned ns = 32;
        while (!mbar_try_wait(bar, parity)) {
            __nanosleep(ns);
            ns = ns < 256 ? 2 * ns : 256;
            if (global_ns() - t0 > kWaitLimitNs) {
                *fail = 1;
                atomicExch(&g_gemv_mxf4_err, code);
                return false;
            }
        }
        return true;
    };
    auto seg_len = [&](int t) -> int {  // tiles from CTA tile t that share its x
        int seg = my_tiles - t;
        if (a.x_stride != 0) {
            const int gt = g0 + t;
            seg = min(seg, (gt / ntiles + 1) * ntiles - gt);
        }
        return seg;
    };

    if (warp == SCALE_WARP) {
        // ------------------------------------------------------------ scales
        // each tile's 127 scales into its pipeline's buffer, in the order the pipelines take
        // their tiles, so that no decode warp ever waits on a global load (a tile's epilogue
        // comes long after its first stage)
        int kbase[NWG];
#pragma unroll
        for (int w = 0; w < NWG; ++w) kbase[w] = 0;
        bool ok = true;
        for (int t = 0; t < my_tiles && ok;) {
            const int seg = seg_len(t);
            for (int rd = 0; rd * NWG < seg && ok; ++rd) {
#pragma unroll
                for (int w = 0; w < NWG; ++w) {
                    if (rd * NWG + w >= seg || !ok) continue;
                    Pipe &pp = bb->pipe[w];
                    const int k = kbase[w] + rd;
                    bool oks = true;
                    if (lane == 0 && k >= 1) oks = nap(&pp.sempty, (k - 1) & 1, kDevErrWaitEmpty);
                    ok = __shfl_sync(0xffffffffu, oks, 0);
                    if (!ok) continue;
                    const int gt = g0 + t + rd * NWG + w, mt = gt / ntiles, row0 = (gt - mt * ntiles) * TR;
                    const uint16_t *sc = a.scales + (int64_t)mt * a.scales_stride;
                    uint16_t v4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int e = lane + 32 * i;
                        const int64_t rr = (int64_t)row0 + e;
                        v4[i] = (e < TR && rr < a.rows) ? __ldg(sc + rr) : (uint16_t)0;
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) pp.sbuf[lane + 32 * i] = v4[i];
                    mbar_arrive(&pp.sfull);
                }
            }
#pragma unroll
            for (int w = 0; w < NWG; ++w) kbase[w] += seg > w ? (seg - w + NWG - 1) / NWG : 0;
            t += seg;
        }
    } else if (warp == PRODUCER_WARP) {
        // ------------------------------------------------------------ producer
        // codes may be loaded before the wait on the previous kernel unless they may be
        // written by it (prefetch 0)
        if (prefetch == 0) pdl_wait();
        if (lane == 0) tma_prefetch_desc(&tmC);
        int kbase[NWG], nq[NWG];  // tiles each pipeline took in earlier segments; boxes issued to it
        int pslot[NWG], pphase[NWG];  // the ring slot of a pipeline's next box, and that slot's use parity
#pragma unroll
        for (int w = 0; w < NWG; ++w) kbase[w] = nq[w] = pslot[w] = pphase[w] = 0;
        bool ok = true;
        for (int t = 0; t < my_tiles && ok;) {
            const int seg = seg_len(t);
            for (int rd = 0; rd * NWG < seg && ok; ++rd) {
                for (int b = 0; b < nbox && ok; ++b) {
#pragma unroll
                    for (int w = 0; w < NWG; ++w) {
                        if (rd * NWG + w >= seg || !ok) continue;
                        Pipe &pp = bb->pipe[w];
                        const int q = nq[w];  // this pipeline's box number
                        const int slot = pslot[w];
                        bool okp = true;
                        if (lane == 0 && q >= ring) okp = nap(&pp.bempty[slot], pphase[w] ^ 1, kDevErrWaitEmpty);
                        ok = __shfl_sync(0xffffffffu, okp, 0);
                        if (!ok) continue;
                        const int gt = g0 + t + rd * NWG + w, mt = gt / ntiles, row0 = (gt - mt * ntiles) * TR;
                        if (lane == 0) {
                            mbar_arrive_expect_tx(&pp.bfull[slot], (uint32_t)BOXB);
                            tma_load_3d(boxes + ((size_t)w * ring + slot) * BOXB, &tmC, &pp.bfull[slot], b * 128, row0,
                                        mt);
                        }
                        nq[w] = q + 1;
                        if (++pslot[w] == ring) {
                            pslot[w] = 0;
                            pphase[w] ^= 1;
                        }
                    }
                }
            }
#pragma unroll
            for (int w = 0; w < NWG; ++w) kbase[w] += seg > w ? (seg - w + NWG - 1) / NWG : 0;
            t += seg;
        }
        // every issued copy lands before the CTA can exit
        if (lane == 0) {
#pragma unroll
            for (int w = 0; w < NWG; ++w)
                for (int q = max(0, nq[w] - ring); q < nq[w]; ++q)
                    if (!mbar_wait_sleep(&bb->pipe[w].bfull[q % ring], (q / ring) & 1))
                        atomicExch(&g_gemv_mxf4_err, kDevErrDrain);
        }
        if (prefetch == 2) pdl_launch_dependents();
    } else {
        // ------------------------------------------------------------ B builders: decode + MMA warps
        const bool is_mma = warp >= MMA_WARP;  // (the scale warp took the branch above)
        const int w = is_mma ? warp - MMA_WARP : warp >> 2;  // this warp's pipeline
        const int bt = is_mma ? NDEC + 32 * (warp - MMA_WARP) + lane : tid;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        Pipe &pp = bb->pipe[w];
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
        const int r = tid & 127;  // TMEM lane = tile row
        const uint32_t a_base = tmem + A_COL + A_SPAN * w, d_tm = tmem + D_COL + 16 * w;
        const uint32_t b_base = smem_u32(btile);
        const uint8_t *myboxes = boxes + (size_t)w * ring * BOXB;
        int kbase = 0;  // tiles this pipeline took in earlier segments
        // ring positions, carried over tiles and segments: the MMA issuer's next A stage and its
        // use parity; the decode's current box (slot, fill parity) and next A stage
        int m_aslot = 0, m_aphase = 0;
        int d_bslot = -1, d_bphase = 0, d_aslot = 0, d_aphase = 0, d_g = 0;
        for (int t = 0; t < my_tiles;) {
            const int seg = seg_len(t);
            const int mat = (g0 + t) / ntiles;  // the matrix whose x the B tile holds
            stage_x(a.x + (int64_t)mat * a.x_stride, xs, cols, bt, NBUILD);
            bar_sync(2, NBUILD);
            const bool finite = build_b_tile(xs, btile, cols, bt, NBUILD);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            const bool nonfinite = bar_red_or(1, NBUILD, !finite);
            tc_fence_after_sync();
            const int nk = seg > w ? (seg - w + NWG - 1) / NWG : 0;  // tiles of this segment for pipeline w
            if (is_mma) {
                // -------------------------------------------------------- MMA issuer of pipeline w
                if (lane == 0) {
                    bool ok = true;
                    for (int kk = 0; kk < nk && ok; ++kk) {
                        const int k = kbase + kk;
                        if (k >= 1 && !nap(&pp.dempty, (k - 1) & 1, kDevErrWaitEmpty)) break;
                        for (int s = 0; s < nst; ++s) {
                            const int as = m_aslot;
                            const bool got = nap(&pp.afull[as], m_aphase, kDevErrWaitFull);
                            if (++m_aslot == ASLOTS) {
                                m_aslot = 0;
                                m_aphase ^= 1;
                            }
                            if (!got) {
                                ok = false;
                                break;
                            }
                            tc_fence_after_sync();
#pragma unroll
                            for (int k4 = 0; k4 < 4; ++k4)
                                umma_mxf4_tmem_a(d_tm, a_base + 32 * as + 8 * k4,
                                                 sdesc_kmajor_sw128(b_base + s * 2048 + 32 * k4), tmem + SFA_COL,
                                                 tmem + SFB_COL, (s > 0 || k4 > 0) ? 1u : 0u);
                            umma_commit(&pp.aempty[as]);
                        }
                        if (ok) umma_commit(&pp.dfull);
                    }
                }
                __syncwarp();
            } else {
                // -------------------------------------------------------- decode + epilogue of pipeline w
                const float c0 = a.c0, two_d = 2.0f * a.d;
                for (int kk = 0; kk < nk; ++kk) {
                    const int k = kbase + kk;
                    const int gt = g0 + t + w + kk * NWG;
                    const int mt = gt / ntiles;
                    const int64_t row = (int64_t)(gt - mt * ntiles) * TR + r;
                    const bool real = r < TR && row < a.rows;
                    bool ok = __all_sync(0xffffffffu, *fail == 0);  // warp-uniform from here on
                    for (int s = 0; s < nst && ok; ++s) {
                        if ((s & 1) == 0) {  // a new box
                            if (++d_bslot == ring) {
                                d_bslot = 0;
                                d_bphase ^= 1;
                            }
                            ok = __all_sync(0xffffffffu, spin(&pp.bfull[d_bslot], d_bphase, kDevErrWaitFull));
                        }
                        const int slot = d_bslot, as = d_aslot;
                        if (ok && d_g >= ASLOTS)
                            ok = __all_sync(0xffffffffu, spin(&pp.aempty[as], d_aphase ^ 1, kDevErrWaitMma));
                        ++d_g;
                        if (++d_aslot == ASLOTS) {
                            d_aslot = 0;
                            d_aphase ^= 1;
                        }
                        if (!ok) break;
                        uint32_t v[32];
                        if (r == TR) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = kOnesRow;
                        } else {
                            // 64 code bytes of this row: 16-byte chunks 4(s&1) .. 4(s&1)+3 of the box
                            const uint8_t *rowp = myboxes + (size_t)slot * BOXB + r * 128;
                            const int ch = 4 * (s & 1);
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint4 c4 = *reinterpret_cast<const uint4 *>(rowp + (((ch + i) ^ (r & 7)) << 4));
                                const uint32_t cw[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    v[8 * i + 2 * j] = cw[j] & 0x33333333u;
                                    v[8 * i + 2 * j + 1] = (cw[j] >> 2) & 0x33333333u;
                                }
                            }
                        }
                        if (s & 1) {  // this warp is done reading the box
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&pp.bempty[slot]);
                        }
                        // the stage goes to the MMA warp as soon as its store has completed (handing
                        // it over one decode later, to overlap the store, measured slower: the MMAs
                        // then started a stage later and the A stages ran out first)
                        tmem_st32(a_base + lane_base + 32 * as, v);
                        tmem_wait_st();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&pp.afull[as]);
                    }
                    // epilogue: the tile's scales (staged by the producer) and accumulator
                    if (ok) ok = __all_sync(0xffffffffu, spin(&pp.sfull, k & 1, kDevErrWaitFull));
                    const float scl = ok ? __half2float(__ushort_as_half(pp.sbuf[r])) : 0.f;
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(&pp.sempty);
                    float v[16];
                    if (ok) ok = __all_sync(0xffffffffu, spin(&pp.dfull, k & 1, kDevErrWaitMma));
                    if (ok) {
                        tc_fence_after_sync();
                        tmem_ld16(d_tm + lane_base, v);
                        tc_fence_before_sync();
                    }
                    __syncwarp();
                    if (lane == 0 && ok) mbar_arrive(&pp.dempty);
                    if (r == TR) {
#pragma unroll
                        for (int j = 0; j < NPIECE; ++j) pp.sx[j] = ok ? v[j] : 0.f;
                    }
                    bar_sync(3 + w, 128);  // the piece sums of this tile are in shared memory
                    if (!*fail && real) {
                        float acc = 0.f;
#pragma unroll
                        for (int j = 0; j < NPIECE; ++j) {
                            const float p = __fmaf_rn(two_d, v[j], __fmul_rn(c0, pp.sx[j]));
                            acc = __fmaf_rn(p, __int_as_float((127 + 3 * j - 23) << 23), acc);
                        }
                        a.y[(int64_t)mt * a.y_stride + row] =
                            nonfinite ? __int_as_float(0x7FC00000) : __fmul_rn(scl, acc);
                    }
                }
            }
            bar_sync(2, NBUILD);  // every MMA reading this B tile has completed (epilogues waited for them)
            kbase += nk;
            t += seg;
        }
        if (is_mma && lane == 0) {
            // every issued MMA completes before TMEM is released
            umma_commit(&bb->last);
            if (!mbar_wait_sleep(&bb->last, 0)) atomicExch(&g_gemv_mxf4_err, kDevErrWaitMma);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == PRODUCER_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

size_t mxf4_smem_bytes(int64_t cols, int ring) {
    return 1024 + (size_t)NWG * ring * BOXB + (size_t)cols * 10 + sizeof(Bars);
}

constexpr int64_t kMxf4MaxCols = 12800;

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
    const int tpc = tiles_per_cta > 0 ? tiles_per_cta : NWG;
    const int nbox = (int)(m.cols / 512);
    // code boxes per pipeline: a whole tile of boxes when shared memory holds them, at least two
    int ring = std::min(MAX_RING, std::max(nbox, 2));
    while (ring > 2 && mxf4_smem_bytes(m.cols, ring) > 227 * 1024) --ring;
    if (mxf4_smem_bytes(m.cols, ring) > 227 * 1024) return cudaErrorNotSupported;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((total + tpc - 1) / tpc));
    lc.blockDim = dim3(NTHREADS);
    // at least 116 KiB: one CTA per SM, whose 512 TMEM columns are the SM's whole tensor memory
    lc.dynamicSmemBytes = std::max<size_t>(mxf4_smem_bytes(m.cols, ring), 116 * 1024);
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, gemv2_mxf4_kernel, tm, m, prefetch, tpc, ring);
}

}  // namespace

// cols: a multiple of 512 whose x digit tile, x and two code boxes per pipeline fit shared memory
// (cols <= 12,800: the transposed 1,536 x 12,288 shape included); every per-digit sum stays exact
// (multiples of 1/4 below 3 cols < 2^22)
bool gemv_mxf4_supported(const PackedArgs &a) {
    return a.cols % 512 == 0 && a.cols <= kMxf4MaxCols && (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 &&
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

cudaError_t launch_gemv_batched_mxf4(const PackedBatch &p, int tiles_per_cta, const GemvConfig &cfg, cudaStream_t st) {
    if (!gemv_batched_mxf4_supported(p)) return cudaErrorNotSupported;
    const Mxf4Args m{p.scales, p.scales_stride, p.x, p.x_stride, p.y, p.y_stride, p.batch, p.rows, p.cols, p.cb[0],
                     p.cb[1] - p.cb[0]};
    int tpc = tiles_per_cta;
    if (tpc <= 0) {
        // one run of tiles per CTA and SM, a multiple of the pipelines
        int dev = 0, sms = 152;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t total = ((p.rows + TR - 1) / TR) * p.batch;
        tpc = (int)std::max<int64_t>(NWG, (total + sms - 1) / sms);
        tpc = (tpc + NWG - 1) / NWG * NWG;
    }
    const int prefetch = !cfg.pdl ? 0 : cfg.independent ? 2 : cfg.weights_static ? 1 : 0;
    return launch_mxf4(m, p.codes, p.codes_stride, cfg.pdl, prefetch, tpc, st);
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
