// gemm_packed2_tcr.cu -- Y = X . (diag(scale) W)^T for a short batch of tokens,
// the decoded weights held in tensor memory as the A operand of tcgen05.mma.
//
// "More Stumbling, This Time in the Browser", sections "This time, in a
// browser" and "The attractive ideas that went away": the 16-layer ternary
// encoder multiplies the activations of 2 x 111 tokens by packed ternary
// weights (3072 x 768 and 768 x 3072).  The contraction is laid out as
//
//     D[f][t] = sum_k Wdec[f][k] . X[t][k]       (f: output feature, t: token)
//     Y[t][f] = scale_f . D[f][t]
//
// with 128 features per CTA as the MMA's M, one tile of ntok tokens (a multiple
// of 16) as its N, fp16 x fp16 products (exact) and fp32 accumulation in
// tensor memory.  A CTA owns a contiguous share of the K atoms (64 fields
// each); the CTAs of a (1, 1, S) cluster split K.  Per atom, through a ring of
// R stages:
//   * the TMA warp brings the atom's X tile (ntok rows x 64 fp16, 128-byte
//     swizzle: the K-major B operand);
//   * eight decode warps read the code bytes themselves (8 bytes of one row per
//     thread and atom, prefetched four atoms ahead into registers), turn them
//     into fp16 weights in registers and store them with tcgen05.st into the
//     stage's 32 TMEM columns: the thread of TMEM lane f owns weight row f, the
//     two warps of a lane quarter take one half of the atom each, and column c
//     of a stage holds the fp16 pair of K positions 2c (low half) and 2c + 1.
//     Two atoms' stores are waited for at once, and the next atom is decoded
//     while they complete;
//   * one thread issues the atom's 4 MMAs (K = 16), A from TMEM and B from
//     shared memory, and commits them to the barrier that frees the stage.
// Only X passes through shared memory; the decoded weights go straight from
// registers to tensor memory, so no shared-memory bandwidth is spent on storing
// and re-reading them.  (A timeline of the first version, which brought the code
// bytes by TMA in boxes of 16-byte rows and waited for each atom's TMEM store
// before decoding the next, showed ~0.4 us per atom spent in the decode warps
// and about 1 us of TMA issue before the first X tile: per-product time grew
// with the atoms per CTA, not with N or the CTA count.)
//
// Decode without tables.  A code byte b holds fields c0..c3 at bits 2i, 2i+1.
// Multiplications by sums of powers of two move the fields to byte lanes:
// (b & 0x33) * 0x1001 puts c0 at bit 0 and c2 at bit 16, (b & 0xCC) * 0x40040
// puts c1 at bit 8 and c3 at bit 24 (the shifted copies never overlap, so
// nothing carries), and a mask keeps those four 2-bit groups.  s * 0x11 +
// 0x40404040 turns them into the byte selectors (c, c + 4) of prmt: with L
// holding the low bytes of the four fp16 codebook entries and H their high
// bytes, prmt(L, H, sel) is the fp16 pair (cb[c0], cb[c1]) and
// prmt(L, H, sel >> 16) the pair (cb[c2], cb[c3]).  Exact for any codebook whose
// four entries are fp16 numbers.
//
// Epilogue.  Alone (S = 1), the thread of lane f scales its feature and stores
// it at every token of the tile: at a fixed token the 32 lanes of a warp write
// 32 consecutive floats.  In a cluster, every CTA writes its partial tile to its
// own shared memory as [t][f]; CTA z then adds, for its 128 / S features and
// every token, the S partials in rank order (deterministic), scales and stores,
// with the remote loads (ld.shared::cluster) of 16 / S tokens in flight at once.
// (Pushing the partials to their owners with st.shared::cluster instead left
// each CTA's tensor-memory release 15-25 us late on GB300.)
//
// With programmatic dependent launch the prologue and, when the weights are
// promised static, the first atoms' code loads and their decode run before
// the wait on the previous kernel; X is read and Y written only after it.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tmap.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {

__device__ unsigned int g_tcr_err;

namespace {

constexpr int FM = 128;                 // features per CTA: the MMA's M, one per TMEM lane
constexpr int KATOM = 64;               // fields per atom (one 128-byte swizzled row of X)
constexpr int NDEC = 256;               // eight decode / epilogue warps
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_DEC0 = 2;
constexpr int NTHREADS = 64 + NDEC;
constexpr int TMEM_COLS = 512;          // the whole tensor memory: one CTA per SM
constexpr int ACC_COLS = 256;           // accumulator (ntok <= 256 columns)
constexpr int RMAX = 8;                 // ring stages, 32 TMEM columns each after the accumulator
constexpr int PREF = 4;                 // atoms of code bytes a decode thread holds ahead
constexpr int PSTR = FM + 4;            // staged partial tile [t][f]: row stride in floats
constexpr int SMEM_MIN = 116 * 1024;    // more than half an SM's shared memory: one CTA per SM
constexpr int SMEM_LIMIT = 227 * 1024;

struct TcrParams {
    const uint8_t *codes;
    const uint16_t *scales;
    float *y;
    int M, rows, cols;
    int rowbytes;
    int atoms;  // K atoms of 64 fields
    int ntok;   // tokens per tile = MMA N (multiple of 16, 16..256) = X box rows
    int R;      // ring stages
    int pdl, weights_static;
    int vec;    // rows % 4 == 0 and 16-byte aligned Y: float4 stores in the cluster epilogue
    uint32_t lo4, hi4;  // low / high bytes of the four fp16 codebook entries (byte i: entry i)
};

// Shared-memory plan: R stages of X tiles, reused in a cluster for the staged
// partial tile ([t][f], rows of PSTR floats); barriers; the tile's scales.
struct TcrPlan {
    int stage, bar_off, scale_off, total;
    __host__ __device__ TcrPlan(int ntok, int R, int S) {
        stage = ntok * 128;  // a multiple of 2048: every X tile 1024-byte aligned
        const int ring = R * stage;
        const int partial = S > 1 ? ntok * PSTR * 4 : 0;
        bar_off = ((ring > partial ? ring : partial) + 1023) / 1024 * 1024;
        scale_off = bar_off + ((4 * RMAX + 1) * 8 + 8 + 15) / 16 * 16;  // barriers, TMEM slot, flag
        total = scale_off + FM * 4 + 1024;  // + alignment slack of the dynamic allocation
        if (total < SMEM_MIN) total = SMEM_MIN;
    }
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The 16 fields of code word w as 8 fp16 pairs: out[2i] = (cb[field 4i], cb[field 4i + 1]),
// out[2i + 1] = (cb[field 4i + 2], cb[field 4i + 3]), the lower K position in the low half.
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t lo4, uint32_t hi4, uint32_t *out) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = w >> (8 * i);
        const uint32_t s = (((x & 0x33u) * 0x1001u) | ((x & 0xCCu) * 0x40040u)) & 0x03030303u;
        const uint32_t sel = s * 0x11u + 0x40404040u;
        out[2 * i] = prmt(lo4, hi4, sel);
        out[2 * i + 1] = prmt(lo4, hi4, sel >> 16);
    }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 accumulator columns of this warp's lane quarter (16 when only 16 are left)
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, int ncols, float (&v)[32]) {
    if (ncols >= 32) {
        tmem_ld32(taddr, v);
    } else {
        uint32_t r[16];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr)
            : "memory");
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
#pragma unroll
        for (int i = 16; i < 32; ++i) v[i] = 0.f;
    }
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16: A is 128 lanes x 16 fp16 in 8 TMEM columns
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

template <int S>  // CTAs of the cluster that split K (1: no cluster)
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_packed2_tcr_kernel(const __grid_constant__ CUtensorMap tmX, const TcrParams p) {
    constexpr bool CLUSTER = S > 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    const int z = CLUSTER ? (int)blockIdx.z : 0;
    const int a0 = (int)((int64_t)z * p.atoms / S), a1 = (int)((int64_t)(z + 1) * p.atoms / S);
    const int kc = a1 - a0;
    const int R = p.R;
    const TcrPlan L(p.ntok, R, S);
    const int xbytes = p.ntok * 128;
    uint64_t *xfull = reinterpret_cast<uint64_t *>(smem + L.bar_off);  // X tile landed
    uint64_t *afull = xfull + 2 * RMAX;                                 // decoded weights in TMEM
    uint64_t *empty = afull + RMAX;                                     // the stage's MMAs completed
    uint64_t *done = empty + RMAX;                                      // every MMA completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *fail = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *sscale = reinterpret_cast<float *>(smem + L.scale_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int f0 = blockIdx.x * FM, t0 = blockIdx.y * p.ntok;

    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&xfull[r], 1);
            mbar_init(&afull[r], NDEC / 32);
            mbar_init(&empty[r], 1);
        }
        mbar_init(done, 1);
        *fail = 0;
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // A wait that runs out marks the CTA; later waits return at once and every role skips
    // its remaining work but still reaches the barriers below.
    auto wait = [&](uint64_t *bar, uint32_t parity, unsigned code) -> bool {
        if (*fail) return false;
        if (mbar_wait(bar, parity)) return true;
        *fail = 1;
        atomicExch(&g_tcr_err, code);
        return false;
    };

    if (warp == WARP_TMA) {
        // ---------------------------------------------------------------- TMA
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            pdl_wait();  // X may be the previous kernel's output
            // the next call may launch once this one has passed its wait (not before: a chain
            // of calls would otherwise park every later call's CTAs on the SMs)
            if (p.pdl) pdl_launch_dependents();
            int nx = 0;  // X copies issued
            for (; nx < kc; ++nx) {
                const int s = nx % R;
                if (nx >= R && !wait(&empty[s], ((nx / R) - 1) & 1, kDevErrWaitEmpty)) break;
                mbar_arrive_expect_tx(&xfull[s], (uint32_t)xbytes);
                tma_load_2d(smem + s * L.stage, &tmX, &xfull[s], (a0 + nx) * KATOM, t0);
            }
            // every issued copy lands before this CTA's shared memory is reused or released
            for (int i = nx > R ? nx - R : 0; i < nx; ++i)
                if (!mbar_wait(&xfull[i % R], (i / R) & 1)) atomicExch(&g_tcr_err, kDevErrDrain);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc(kFmtF16, kFmtF16, (uint32_t)p.ntok, FM);
            for (int i = 0; i < kc; ++i) {
                const int s = i % R;
                const uint32_t ph = (i / R) & 1;
                if (!wait(&afull[s], ph, kDevErrWaitFull) || !wait(&xfull[s], ph, kDevErrWaitFull)) break;
                tc_fence_after_sync();
                const uint32_t xb = smem_u32(smem + s * L.stage);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_f16_ta(tmem, tmem + (uint32_t)(ACC_COLS + 32 * s + 8 * ks), sdesc_kmajor_sw128(xb + 32 * ks),
                                idesc, (i > 0 || ks > 0) ? 1u : 0u);
                // a commit costs about two MMA issues: only where atom i + R will reuse the stage
                if (i + R < kc) umma_commit(&empty[s]);
            }
            // every issued MMA completes before the accumulator is read or TMEM released
            umma_commit(done);
            if (!mbar_wait(done, 0)) atomicExch(&g_tcr_err, kDevErrWaitMma);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- decode, epilogue
        const int d = tid - 64;                 // 0 .. NDEC - 1
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        const int h = (warp - WARP_DEC0) >> 2;  // which half of each atom
        const int f = 32 * q + lane;            // weight row = TMEM lane
        const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
        // code bytes of this thread's row and half, PREF atoms ahead; rows past the end read nothing
        const bool real = f0 + f < p.rows;
        const uint8_t *crow = p.codes + (real ? (int64_t)(f0 + f) * p.rowbytes + (int64_t)a0 * 16 + 8 * h : 0);
        auto load_codes = [&](int i) -> uint2 {
            return (real && i < kc) ? __ldg(reinterpret_cast<const uint2 *>(crow + 16 * i)) : make_uint2(0u, 0u);
        };
        // codes and scales are weights: read after the same wait as X unless promised static
        if (!p.weights_static) pdl_wait();
        uint2 pre[PREF];
#pragma unroll
        for (int u = 0; u < PREF; ++u) pre[u] = load_codes(u);
        if (h == 0) sscale[f] = real ? h2f(p.scales[f0 + f]) : 0.f;
        // decoded atoms in four register buffers: two atoms' TMEM stores are in flight per wait,
        // and the next atom is decoded while they complete
        uint32_t rb[4][16];
        decode_word(pre[0].x, p.lo4, p.hi4, rb[0]);
        decode_word(pre[0].y, p.lo4, p.hi4, rb[0] + 8);
        pre[0] = load_codes(PREF);
        bool bad = false;
        int s_prev = 0;  // stage of the stored atom not yet announced
        for (int i0 = 0; i0 < kc && !bad; i0 += PREF) {
#pragma unroll
            for (int u = 0; u < PREF; ++u) {
                const int i = i0 + u;
                if (i >= kc) break;
                const int s = i % R;
                // the stage's TMEM columns are free once the MMAs of atom i - R have completed;
                // one decision per warp: the TMEM store is a warp-wide instruction
                if (i >= R && !__all_sync(0xffffffffu, wait(&empty[s], ((i / R) - 1) & 1, kDevErrWaitEmpty))) {
                    bad = true;
                    break;
                }
                tc_fence_after_sync();
                tmem_st16(tmem + lane_addr + (uint32_t)(ACC_COLS + 32 * s + 16 * h), rb[u]);
                if (i + 1 < kc) {
                    // buffer (u + 1) % 4 was last stored two atoms ago, before the previous wait
                    const uint2 c = pre[(u + 1) % PREF];
                    decode_word(c.x, p.lo4, p.hi4, rb[(u + 1) % 4]);
                    decode_word(c.y, p.lo4, p.hi4, rb[(u + 1) % 4] + 8);
                    pre[(u + 1) % PREF] = load_codes(i + 1 + PREF);
                }
                if ((u & 1) || i == kc - 1) {
                    tmem_wait_st();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (u & 1) mbar_arrive(&afull[s_prev]);
                        mbar_arrive(&afull[s]);
                    }
                } else {
                    s_prev = s;
                }
            }
        }
        bar_sync(1, NDEC);  // the scales are in shared memory
        pdl_wait();         // Y may still be read by the previous kernel
        if (!mbar_wait(done, 0)) {
            *fail = 1;
            atomicExch(&g_tcr_err, kDevErrWaitMma);
        }
        tc_fence_after_sync();
        const bool ok = !*fail;
        if (!CLUSTER) {
            const float sc = sscale[f];
            const int feat = f0 + f;
            for (int c0 = 32 * h; c0 < p.ntok; c0 += 64) {
                float v[32];
                tmem_ld_cols(tmem + lane_addr + (uint32_t)c0, p.ntok - c0, v);
                if (ok && feat < p.rows)
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int t = t0 + c0 + j;
                        if (c0 + j < p.ntok && t < p.M) p.y[(int64_t)t * p.rows + feat] = v[j] * sc;
                    }
            }
        }
        (void)d;
    }

    if constexpr (CLUSTER) {
        const bool ok = !*fail;
        float *part = reinterpret_cast<float *>(smem);  // the ring: every copy landed, every MMA done
        if (warp >= WARP_DEC0) {
            // partial tile -> own shared memory as [t][f]: at a fixed token a warp writes 32
            // consecutive floats
            const int q = warp & 3, h = (warp - WARP_DEC0) >> 2, f = 32 * q + lane;
            const uint32_t lane_addr = (uint32_t)(32 * q) << 16;
            for (int c0 = 32 * h; c0 < p.ntok; c0 += 64) {
                float v[32];
                tmem_ld_cols(tmem + lane_addr + (uint32_t)c0, p.ntok - c0, v);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < p.ntok) part[(c0 + j) * PSTR + f] = ok ? v[j] : 0.f;
            }
        }
        __syncwarp();
        cluster_sync();  // every partial tile is staged and visible to the cluster
        // CTA z adds, for its FM / S features and every token, the S partials in rank order;
        // thread (g, tl) takes 4 features and every LANES_T-th token, TB tokens per batch, and
        // LANES_T * TB = 128 tokens per pass: at most two passes (ntok <= 256).  The sums are
        // kept in registers; the CTA arrives at the closing cluster barrier (release: its remote
        // loads have been performed, so no peer can pass the barrier and exit while one of them
        // still reads its shared memory) before it stores Y, so the release does not wait for
        // the global stores.
        constexpr int FS = FM / S, GROUPS = FS / 4, LANES_T = NDEC / GROUPS, TB = 16 / S;
        static_assert(LANES_T * TB == 128, "two passes cover 256 tokens");
        const int d = tid - 64;
        const int g = d % GROUPS, tl = d / GROUPS;
        const int fl = z * FS + 4 * g;
        float4 res[2][TB];
        if (warp >= WARP_DEC0) {
            const uint32_t base = smem_u32(part) + (uint32_t)(fl * 4);
            uint32_t peer[S];
#pragma unroll
            for (int r = 0; r < S; ++r) peer[r] = cluster_map(base, (uint32_t)r);
#pragma unroll
            for (int it = 0; it < 2; ++it) {
                float4 v[TB][S];
#pragma unroll
                for (int u = 0; u < TB; ++u) {
                    const int t = tl + it * 128 + u * LANES_T;
#pragma unroll
                    for (int r = 0; r < S; ++r)
                        if (t < p.ntok && t0 + t < p.M && ok) v[u][r] = ld_cluster_v4(peer[r] + (uint32_t)(t * PSTR * 4));
                }
#pragma unroll
                for (int u = 0; u < TB; ++u) {
                    const int t = tl + it * 128 + u * LANES_T;
                    if (t >= p.ntok || t0 + t >= p.M || !ok) continue;
                    float4 acc = v[u][0];
#pragma unroll
                    for (int r = 1; r < S; ++r) {
                        acc.x += v[u][r].x;
                        acc.y += v[u][r].y;
                        acc.z += v[u][r].z;
                        acc.w += v[u][r].w;
                    }
                    res[it][u] = acc;
                }
            }
        }
        __syncwarp();
        cluster_arrive();
        if (warp >= WARP_DEC0) {
            const float4 sc = *reinterpret_cast<const float4 *>(sscale + fl);
            const int fg = f0 + fl;
#pragma unroll
            for (int it = 0; it < 2; ++it)
#pragma unroll
                for (int u = 0; u < TB; ++u) {
                    const int t = tl + it * 128 + u * LANES_T;
                    if (t >= p.ntok || t0 + t >= p.M || !ok) continue;
                    float *yrow = p.y + (int64_t)(t0 + t) * p.rows + fg;
                    const float4 acc = res[it][u];
                    const float r4[4] = {acc.x * sc.x, acc.y * sc.y, acc.z * sc.z, acc.w * sc.w};
                    if (p.vec && fg + 3 < p.rows) {
                        *reinterpret_cast<float4 *>(yrow) = make_float4(r4[0], r4[1], r4[2], r4[3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            if (fg + j < p.rows) yrow[j] = r4[j];
                    }
                }
        }
        __syncwarp();
        cluster_wait();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int S>
cudaError_t launch_tcr(const CUtensorMap &tx, const TcrParams &p, int ftiles, int ttiles, int smem, cudaStream_t st) {
    constexpr bool CLUSTER = S > 1;
    auto kern = gemm_packed2_tcr_kernel<S>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] { attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT); });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)ftiles, (unsigned)ttiles, (unsigned)S);
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = (size_t)smem;
    lc.stream = st;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (CLUSTER) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = (unsigned)S;
        ++n;
    }
    if (p.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    lc.attrs = attr;
    lc.numAttrs = n;
    return cudaLaunchKernelEx(&lc, kern, tx, p);
}

bool fp16_bits(float v, uint16_t *bits) {
    const __half hv = __float2half_rn(v);
    if (__half2float(hv) != v) return false;
    *bits = *reinterpret_cast<const uint16_t *>(&hv);
    return true;
}

int round16(int64_t v) { return (int)((v + 15) / 16 * 16); }

}  // namespace

bool gemm_packed2_tcr_supported(const PackedArgs &a) {
    uint16_t b;
    for (int i = 0; i < 4; ++i)
        if (!fp16_bits(a.cb[i], &b)) return false;
    return a.cols % KATOM == 0 && (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 && a.M < (1 << 30) && a.rows < (1 << 30) &&
           a.cols < (1 << 30) && (a.rows + FM - 1) / FM < 65536 && (a.M + 15) / 16 < 65536;
}

// Tokens per tile and cluster split: the (ntok, S) with the least estimated time among
// grids that run in one wave (CTAs within the clusters of S the GPU can hold at once,
// from the occupancy calculator).  Estimate, fitted to the ternary encoder shapes on
// GB300: 0.49 us per atom of a CTA's K share (a chain of MMA issues at ~105 cycles
// each, the decode and the stage hand-offs) plus 0.055 us per KB of partial tile a CTA
// reads from its peers ((S - 1) / S of 128 x ntok floats).
void gemm_packed2_tcr_shape(int64_t M, int64_t rows, int64_t cols, const int capacity[4], int *ntok_out,
                            int *split_out) {
    const int atoms = (int)(cols / KATOM);
    const int64_t ftiles = (rows + FM - 1) / FM;
    double best = 1e30;
    int bn = round16(M < 256 ? M : 256), bs = 1;
    for (int T = 1; T <= 64; ++T) {
        const int ntok = round16((M + T - 1) / T);
        if (ntok > 256 || ntok < 16) continue;
        if ((M + ntok - 1) / ntok != T) continue;  // this tiling is reached with fewer tiles
        for (int si = 0, S = 1; si < 4; ++si, S *= 2) {
            if (S > atoms) break;
            const int64_t ctas = ftiles * T * S;
            const int64_t waves = (ctas + capacity[si] - 1) / (capacity[si] > 0 ? capacity[si] : 1);
            const int kc = (atoms + S - 1) / S;
            const double kb = 128.0 * ntok * 4.0 / 1024.0 * (S - 1) / S;
            const double cost = (double)waves * (0.49 * kc + 0.055 * kb);
            if (cost < best - 1e-9) {
                best = cost;
                bn = ntok;
                bs = S;
            }
        }
    }
    *ntok_out = bn;
    *split_out = bs;
}

// CTAs of this kernel the GPU holds at once in clusters of 1, 2, 4, 8 (one CTA per SM),
// from the occupancy calculator, once per device.
static cudaError_t cluster_capacity(int sms, int cap[4]) {
    static std::mutex mu;
    static int cached[64][4];
    static bool have[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!have[dev]) {
        cached[dev][0] = sms;
        for (int si = 1; si < 4; ++si) {
            const int S = 1 << si;
            cudaLaunchConfig_t lc = {};
            lc.gridDim = dim3(1, 1, (unsigned)S);
            lc.blockDim = dim3(NTHREADS);
            lc.dynamicSmemBytes = SMEM_MIN;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = (unsigned)S;
            lc.attrs = attr;
            lc.numAttrs = 1;
            int n = 0;
            const void *k = si == 1 ? (const void *)gemm_packed2_tcr_kernel<2>
                          : si == 2 ? (const void *)gemm_packed2_tcr_kernel<4>
                                    : (const void *)gemm_packed2_tcr_kernel<8>;
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
            if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, k, &lc);
            if (e != cudaSuccess) return e;
            cached[dev][si] = n * S;
        }
        have[dev] = true;
    }
    for (int si = 0; si < 4; ++si) cap[si] = cached[dev][si];
    return cudaSuccess;
}

cudaError_t launch_gemm_packed2_tcr(const PackedArgs &a, int ntok_req, int splitk_req, int pdl, int weights_static,
                                    cudaStream_t st) {
    if (!gemm_packed2_tcr_supported(a)) return cudaErrorNotSupported;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    TcrParams p{};
    p.codes = a.codes;
    p.scales = a.scales;
    p.y = a.y;
    p.M = (int)a.M;
    p.rows = (int)a.rows;
    p.cols = (int)a.cols;
    p.rowbytes = (int)(a.cols / 4);
    p.atoms = (int)(a.cols / KATOM);
    int ntok = ntok_req, splitk = splitk_req;
    if (!ntok || !splitk) {
        int cap[4];
        e = cluster_capacity(sms, cap);
        if (e != cudaSuccess) return e;
        int an = 0, as = 0;
        gemm_packed2_tcr_shape(a.M, a.rows, a.cols, cap, &an, &as);
        if (!ntok) ntok = an;
        if (!splitk) splitk = as;
    }
    if (ntok < 16 || ntok > 256 || ntok % 16 || splitk < 1 || splitk > 8 || (splitk & (splitk - 1)) ||
        splitk > p.atoms)
        return cudaErrorInvalidValue;
    p.ntok = ntok;
    p.vec = (a.rows % 4 == 0) && (reinterpret_cast<uintptr_t>(a.y) % 16 == 0);
    p.pdl = pdl;
    p.weights_static = pdl ? weights_static : 0;
    uint16_t hb[4];
    for (int i = 0; i < 4; ++i) fp16_bits(a.cb[i], &hb[i]);
    p.lo4 = 0;
    p.hi4 = 0;
    for (int i = 0; i < 4; ++i) {
        p.lo4 |= (uint32_t)(hb[i] & 0xFFu) << (8 * i);
        p.hi4 |= (uint32_t)(hb[i] >> 8) << (8 * i);
    }
    // the deepest ring that fits, up to RMAX stages and no deeper than the CTA's share of K
    const int kc_max = (p.atoms + splitk - 1) / splitk;
    int R = RMAX < kc_max ? RMAX : kc_max;
    if (R < 1) R = 1;
    while (R > 1 && TcrPlan(ntok, R, splitk).total > SMEM_LIMIT) --R;
    const TcrPlan L(ntok, R, splitk);
    if (L.total > SMEM_LIMIT) return cudaErrorInvalidValue;
    p.R = R;
    CUtensorMap tx;
    e = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.x, (uint64_t)a.cols, (uint64_t)a.M,
                     (uint64_t)a.cols * 2, KATOM, (uint32_t)ntok, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const int ftiles = (int)((a.rows + FM - 1) / FM), ttiles = (int)((a.M + ntok - 1) / ntok);
    switch (splitk) {
        case 1: return launch_tcr<1>(tx, p, ftiles, ttiles, L.total, st);
        case 2: return launch_tcr<2>(tx, p, ftiles, ttiles, L.total, st);
        case 4: return launch_tcr<4>(tx, p, ftiles, ttiles, L.total, st);
        default: return launch_tcr<8>(tx, p, ftiles, ttiles, L.total, st);
    }
}

unsigned int gemm_packed2_tcr_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_tcr_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_tcr_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
