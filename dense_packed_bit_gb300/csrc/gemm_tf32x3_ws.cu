// gemm_tf32x3_ws.cu -- warp-specialised, persistent 3xTF32 GEMM on tcgen05.
//
// The GEMM of "I built a GPT-2 in the browser...", section "The kernel sweep"
// (C = A.B forward, dA = dC.B^T and dB = A^T.dC backward), in fp32 accuracy by
// the three-term split of Ootomo and Yokota (IJHPCA 2022):
//
//     a.b ~= a_hi.b_hi + a_hi.b_lo + a_lo.b_hi,
//     a_hi = a with its 13 low mantissa bits cleared, a_lo = a - a_hi (exact).
//
// The tf32 MMA reads the top 19 bits of each fp32 container, so a raw fp32
// tile that is already in the operand layout *is* the hi operand and only
// its lo tile has to be computed.  Operands are K-major with the 64-byte
// swizzle (rows of 16 fp32 along K; 16-byte chunk c of row r at chunk
// c ^ ((r >> 1) & 3)).  A K-contiguous operand arrives that way from TMA and
// its lo tile is the element-wise map at the same offsets; an M/N-contiguous
// operand arrives as an unswizzled [k][m] tile and the lo pass writes both
// its hi and lo tiles transposed (4 conflict-free column reads, one 16-byte
// conflict-free store per tile).
//
// Roles (one CTA per SM, persistent over output tiles of 128 x 256 per CTA,
// or 256 x 256 per pair of CTAs):
//   warp 0      one thread issues the TMA loads of each 16-deep k-slab of
//               op(A) (128 x 16) and op(B) (256 x 16) into a ring of 3 or
//               4 stages (as many as fit in shared memory);
//   warp 1      one thread issues 2 x 3 tcgen05.mma kind::tf32 (M = 128,
//               N = 256, K = 8) per slab into one of two TMEM accumulators
//               and commits each slab to the barrier that frees its stage;
//               with CTA pairs (cta_group::2, a cluster of 2) the even CTA's
//               thread issues M = 256 MMAs over both CTAs' tiles -- each CTA
//               holds its 128 rows of op(A) and 128 of the 256 rows of op(B)
//               -- and its commits arrive on the barriers of both CTAs;
//   warps 2-5   compute lo = a - a_hi for each landed slab (and transpose
//               M/N-contiguous operands into the K-major layout);
//   warps 6-9   drain a finished accumulator (tcgen05.ld) into C with edge
//               masks while the MMAs of the next tile run in the other one.
// In a pair, the lo-pass and epilogue warps of both CTAs report to the even
// CTA's barriers (one arrival per warp, after fence.proxy.async for the lo
// tiles the peer's tensor core reads).
// Every wait is bounded; a wait that runs out records an error, raises a CTA
// flag that the other roles poll, and the CTA drains its copies and MMAs,
// frees its TMEM and returns.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tf32x3_split.cuh"
#include "tmap.h"

#include <mutex>

namespace mm {

__device__ unsigned int g_tf32ws_err;

namespace {

constexpr int BM = 128, BK = 16, NACC = 2;
constexpr int ACC_COLS = 256;                 // TMEM columns per accumulator (N of a tile <= 256)
constexpr int A_BYTES = BM * BK * 4;          // 8 KiB: one CTA's 128 x 16 fp32 A tile
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_CONV0 = 2, NCONV = 128, WARP_EPI0 = 6;
constexpr int NTHREADS = 320;
constexpr int TMEM_COLS = NACC * ACC_COLS;    // 512: the whole tensor memory of the SM
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr int MAX_STAGES = 6;
constexpr int EPI_TMA_BYTES = 4 * 32 * 128;   // CTA pairs: a 32 x 32 fp32 block per epilogue warp for TMA stores

// Shared-memory plan of one stage of one CTA.  CG CTAs share a tile of
// (128 CG) x BN: each holds 128 rows of op(A) and BN / CG rows of op(B).  A
// K-contiguous operand keeps raw (= hi) and lo tiles; an M/N-contiguous one
// keeps its raw [k][m] tile plus K-major hi and lo.  Every tile is a multiple
// of 512 bytes, the period of the 64-byte swizzle.
template <bool A_KC, bool B_KC, int CG, int BN>
struct Plan {
    static constexpr int BNC = BN / CG;                 // B rows held by one CTA
    static_assert(BN % 16 == 0 && BNC % 8 == 0 && BN <= ACC_COLS, "MMA N: a multiple of 16, at most 256");
    static_assert((BNC * BK * 4) % 512 == 0, "tiles keep the swizzle period");
    static constexpr int B_BYTES = BNC * BK * 4;
    static constexpr int RAW_BYTES = A_BYTES + B_BYTES;  // bytes TMA brings per stage
    static constexpr int A_REGION = (A_KC ? 2 : 3) * A_BYTES;
    static constexpr int B_REGION = (B_KC ? 2 : 3) * B_BYTES;
    static constexpr int STAGE_BYTES = A_REGION + B_REGION;
    static constexpr int RAW_A = 0, HI_A = A_KC ? 0 : A_BYTES, LO_A = A_KC ? A_BYTES : 2 * A_BYTES;
    static constexpr int RAW_B = A_REGION, HI_B = A_REGION + (B_KC ? 0 : B_BYTES),
                         LO_B = A_REGION + (B_KC ? B_BYTES : 2 * B_BYTES);
    static constexpr int EPI = CG == 2 ? EPI_TMA_BYTES : 0;
    static constexpr int FIXED = EPI + (3 * MAX_STAGES + 2 * NACC + 2) * 8 + 16 + 1024;
    static constexpr int S_FIT = (SMEM_LIMIT - FIXED) / STAGE_BYTES;
    static constexpr int STAGES = S_FIT < MAX_STAGES ? S_FIT : MAX_STAGES;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI + (3 * STAGES + 2 * NACC + 2) * 8 + 16 + 1024;
    static_assert(STAGES >= 3, "at least three stages");
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
};

struct WsParams {
    int M, N, K;
    int tiles_m, tiles;  // tiles = output tiles x ksplit work units
    int ksplit;          // K slices per output tile (1: no split)
    float *C;
    int64_t ldc;
    float *ws;           // ksplit > 1: slice s of every output tile goes to ws + s M N (row-major, ld N)
    // stream-K: unit c (a CTA, or a pair) takes slabs [c sk_w, (c + 1) sk_w) of the tiles' K
    // ranges laid end to end; a tile's segment that starts its K range adds the other
    // segments' partial tiles (slot of their unit, in K order) once their flags are set
    int sk, sk_w, sk_total;
    float *sk_slots;        // [unit][rank][128][BN] fp32
    unsigned int *sk_flags; // [unit][rank], zeroed before the launch
    int c_tma;              // CTA pairs: C is stored through shared memory by TMA (tmC valid)
    const float *bias;      // epilogue of C: + bias[column] (null: none), then GELU when act
    int act;
};

// Work unit t: output tile t / ksplit, K slice t % ksplit (slabs [kt0, kt1)).
struct Unit {
    int mn, s, kt0, kt1;
};

__device__ __forceinline__ Unit unit_of(int t, const WsParams &p, int KT) {
    Unit u;
    u.s = t % p.ksplit;
    u.mn = t / p.ksplit;
    u.kt0 = (int)((int64_t)u.s * KT / p.ksplit);
    u.kt1 = (int)((int64_t)(u.s + 1) * KT / p.ksplit);
    return u;
}

// The work of unit `cid` as a sequence of segments, identical for every role: work units
// cid, cid + ncl, ... or, with stream-K, the pieces of its slab range cut at tile boundaries.
template <bool SK>
__device__ __forceinline__ int seg_begin(const WsParams &p, int cid) { return SK ? cid * p.sk_w : cid; }

template <bool SK>
__device__ __forceinline__ bool seg_next(const WsParams &p, int KT, int cid, int ncl, int &cur, Unit &u) {
    if (!SK) {
        if (cur >= p.tiles) return false;
        u = unit_of(cur, p, KT);
        cur += ncl;
        return true;
    }
    const int r1 = min((cid + 1) * p.sk_w, p.sk_total);
    if (cur >= r1) return false;
    u.mn = cur / KT;
    u.kt0 = cur - u.mn * KT;
    u.kt1 = min(KT, u.kt0 + (r1 - cur));
    u.s = 0;
    cur += u.kt1 - u.kt0;
    return true;
}

// Record an error and raise the abort flag of this CTA and, in a pair, of its peer.
template <int CG>
__device__ __forceinline__ void fail(volatile int *abort_flag, unsigned int code) {
    atomicExch(&g_tf32ws_err, code);
    *abort_flag = 1;
    if constexpr (CG == 2)
        st_cluster_u32(cluster_map(smem_u32(const_cast<int *>(abort_flag)), cluster_ctarank() ^ 1u), 1u);
}

// One arrival on the barrier at `bar`'s offset in CTA 0 of the pair (or this CTA).
template <int CG>
__device__ __forceinline__ void arrive_leader(uint64_t *bar) {
    if constexpr (CG == 2) mbar_arrive_cluster(cluster_map(smem_u32(bar), 0));
    else mbar_arrive(bar);
}

// Stream-K flags in global memory: set with release, polled with acquire (device scope),
// the wait bounded like every other wait here.
__device__ __forceinline__ void flag_set(unsigned int *f) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(1u) : "memory");
}

__device__ __forceinline__ bool flag_wait(const unsigned int *f) {
    const unsigned long long t0 = global_ns();
    while (true) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
        if (v) return true;
        if (global_ns() - t0 > kWaitLimitNs) return false;
        __nanosleep(64);
    }
}

template <bool A_KC, bool B_KC, int CG, int BN, bool SK>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tf32x3_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const WsParams p) {
    using P = Plan<A_KC, B_KC, CG, BN>;
    constexpr int STAGES = P::STAGES, STAGE_BYTES = P::STAGE_BYTES, BNC = P::BNC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    uint8_t *epi_stage = smem + STAGES * STAGE_BYTES;  // CTA pairs: [4 warps][32 rows][128 B], 128-byte swizzled
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + P::EPI);  // TMA -> lo pass
    uint64_t *conv = full + STAGES;    // lo passes -> MMA (CTA 0's, one arrival per lo-pass warp of the pair)
    uint64_t *empty = conv + STAGES;   // MMA -> TMA (every CTA's, by commit)
    uint64_t *accf = empty + STAGES;   // MMA -> epilogue (every CTA's, by commit)
    uint64_t *acce = accf + NACC;      // epilogues -> MMA (CTA 0's, one arrival per epilogue warp of the pair)
    uint64_t *last = acce + NACC;
    uint64_t *epi = last + 1;          // the 128 epilogue threads of this CTA (stream-K slot hand-off)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(epi + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = (p.K + BK - 1) / BK;
    const uint32_t rank = CG == 2 ? cluster_ctarank() : 0u;
    const int cid = blockIdx.x / CG, ncl = gridDim.x / CG;

    if (warp == WARP_MMA) {
        if constexpr (CG == 2) {
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&conv[s], 4 * CG);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(&accf[b], 1);
            mbar_init(&acce[b], 4 * CG);
        }
        mbar_init(last, 1);
        mbar_init(epi, 128);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync();
    else __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == WARP_TMA) {
        if (lane == 0) {
            int it = 0;  // slabs issued so far (ring position)
            bool stop = false;
            int cur = seg_begin<SK>(p, cid);
            Unit u;
            while (!stop && seg_next<SK>(p, KT, cid, ncl, cur, u)) {
                const int m0 = (u.mn % p.tiles_m) * (BM * CG) + BM * (int)rank;
                const int nb = (u.mn / p.tiles_m) * BN + BNC * (int)rank;
                for (int kt = u.kt0; kt < u.kt1; ++kt) {
                    const int s = it % STAGES;
                    const uint32_t use = it / STAGES;
                    if (*abort_flag) { stop = true; break; }
                    if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1)) {
                        fail<CG>(abort_flag, kDevErrWaitEmpty);
                        stop = true;
                        break;
                    }
                    uint8_t *st = smem + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s], P::RAW_BYTES);
                    const int k0 = kt * BK;
                    if (A_KC) tma_load_2d(st + P::RAW_A, &tmA, &full[s], k0, m0);
                    else tma_load_2d(st + P::RAW_A, &tmA, &full[s], m0, k0);
                    if (B_KC) tma_load_2d(st + P::RAW_B, &tmB, &full[s], k0, nb);
                    else tma_load_2d(st + P::RAW_B, &tmB, &full[s], nb, k0);
                    ++it;
                }
            }
            // every copy issued must land before this CTA's shared memory is released
            for (int s = 0; s < STAGES && s < it; ++s) {
                const int lastit = s + ((it - 1 - s) / STAGES) * STAGES;
                if (!mbar_wait(&full[s], (uint32_t)(lastit / STAGES) & 1)) {
                    atomicExch(&g_tf32ws_err, kDevErrDrain);
                    break;
                }
            }
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = make_idesc(kFmtTF32, kFmtTF32, BN, BM * CG);
            constexpr uint16_t all = (uint16_t)((1u << CG) - 1u);
            int it = 0, tc = 0;
            bool stop = false;
            int cur = seg_begin<SK>(p, cid);
            Unit u;
            for (; !stop && seg_next<SK>(p, KT, cid, ncl, cur, u); ++tc) {
                const int b = tc % NACC;
                const uint32_t ause = tc / NACC;
                if (*abort_flag) break;
                if (ause > 0 && !mbar_wait(&acce[b], (ause - 1) & 1)) {
                    fail<CG>(abort_flag, kDevErrWaitEmpty);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + (uint32_t)(b * ACC_COLS);
                for (int kt = u.kt0; kt < u.kt1; ++kt, ++it) {
                    const int s = it % STAGES;
                    const uint32_t use = it / STAGES;
                    if (*abort_flag) { stop = true; break; }
                    if (!mbar_wait(&conv[s], use & 1)) {
                        fail<CG>(abort_flag, kDevErrWaitFull);
                        stop = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t st = smem_u32(smem + s * STAGE_BYTES);
#pragma unroll
                    for (int ks = 0; ks < BK / 8; ++ks) {
                        // 8 tf32 of K are 32 bytes along the swizzled 64-byte rows
                        const uint32_t o = 32u * ks;
                        const uint64_t ah = sdesc_make(st + P::HI_A + o, 16, 512, kSdescSw64);
                        const uint64_t al = sdesc_make(st + P::LO_A + o, 16, 512, kSdescSw64);
                        const uint64_t bh = sdesc_make(st + P::HI_B + o, 16, 512, kSdescSw64);
                        const uint64_t bl = sdesc_make(st + P::LO_B + o, 16, 512, kSdescSw64);
                        const uint32_t acc0 = (kt > u.kt0 || ks > 0) ? 1u : 0u;
                        if constexpr (CG == 2) {
                            umma_tf32_pair(d, ah, bh, idesc, acc0);
                            umma_tf32_pair(d, ah, bl, idesc, 1u);
                            umma_tf32_pair(d, al, bh, idesc, 1u);
                        } else {
                            umma_tf32(d, ah, bh, idesc, acc0);
                            umma_tf32(d, ah, bl, idesc, 1u);
                            umma_tf32(d, al, bh, idesc, 1u);
                        }
                    }
                    if constexpr (CG == 2) umma_commit_pair(&empty[s], all);
                    else umma_commit(&empty[s]);
                }
                if (!stop) {
                    if constexpr (CG == 2) umma_commit_pair(&accf[b], all);
                    else umma_commit(&accf[b]);
                }
            }
            // every MMA issued must be complete before the tensor memory is freed
            if constexpr (CG == 2) umma_commit_pair(last, 1);
            else umma_commit(last);
            if (!mbar_wait(last, 0)) atomicExch(&g_tf32ws_err, kDevErrWaitMma);
        }
    } else if (warp < WARP_EPI0) {
        // lo pass (and transposes of M/N-contiguous operands)
        const int ct = threadIdx.x - 32 * WARP_CONV0;
        int it = 0;
        bool stop = false;
        int cur = seg_begin<SK>(p, cid);
        Unit u;
        while (!stop && seg_next<SK>(p, KT, cid, ncl, cur, u)) {
            for (int kt = u.kt0; kt < u.kt1; ++kt, ++it) {
                const int s = it % STAGES;
                const uint32_t use = it / STAGES;
                if (*abort_flag) { stop = true; break; }
                if (!mbar_wait(&full[s], use & 1)) {
                    fail<CG>(abort_flag, kDevErrWaitFull);
                    stop = true;
                    break;
                }
                uint8_t *st = smem + s * STAGE_BYTES;
                if (A_KC) tf32x3::lo_in_place_layout<A_BYTES, NCONV>(st + P::RAW_A, st + P::LO_A, ct);
                else tf32x3::split_transpose<BM, NCONV>(st + P::RAW_A, st + P::HI_A, st + P::LO_A, ct);
                if (B_KC) tf32x3::lo_in_place_layout<P::B_BYTES, NCONV>(st + P::RAW_B, st + P::LO_B, ct);
                else tf32x3::split_transpose<BNC, NCONV>(st + P::RAW_B, st + P::HI_B, st + P::LO_B, ct);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) arrive_leader<CG>(&conv[s]);
            }
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31 of this CTA
        const int q = warp & 3;
        const int et = threadIdx.x - 32 * WARP_EPI0;  // 0..127
        uint32_t epi_phase = 0;
        auto epi_sync = [&] {  // all 128 epilogue threads, bounded
            mbar_arrive(epi);
            if (!mbar_wait(epi, epi_phase & 1)) fail<CG>(abort_flag, kDevErrWaitFull);
            ++epi_phase;
        };
        int tc = 0;
        int cur = seg_begin<SK>(p, cid);
        Unit u;
        for (; seg_next<SK>(p, KT, cid, ncl, cur, u); ++tc) {
            const int b = tc % NACC;
            const uint32_t ause = tc / NACC;
            if (*abort_flag) break;
            if (!mbar_wait_sleep(&accf[b], ause & 1)) {
                fail<CG>(abort_flag, kDevErrWaitMma);
                break;
            }
            tc_fence_after_sync();
            const int m0 = (u.mn % p.tiles_m) * (BM * CG) + BM * (int)rank, n0 = (u.mn / p.tiles_m) * BN;

            const uint32_t base = tmem + (uint32_t)(b * ACC_COLS) + ((uint32_t)(32 * q) << 16);
            // stream-K: a segment that does not start its tile's K range leaves its partial tile
            // in its unit's slot; the one that starts it adds the later segments' slots in K order
            const bool sk_part = SK && u.kt0 > 0;
            const bool sk_fix = SK && u.kt0 == 0 && u.kt1 < KT;
            int c_last = cid;
            if (sk_fix) {
                c_last = ((u.mn + 1) * KT - 1) / p.sk_w;
                bool ok = true;
                if (et == 0)
                    for (int c = cid + 1; c <= c_last && ok; ++c)
                        ok = flag_wait(p.sk_flags + c * CG + rank);
                if (!ok) fail<CG>(abort_flag, kDevErrWaitFull);
                epi_sync();  // every slot to be read is complete
            }
            // the output, this K slice's part of the workspace, or this unit's stream-K slot.  Each
            // thread stores its own row (a warp instruction touches 32 rows): staging 32 x 32
            // blocks through shared memory for row-coalesced stores measured slower on GB300
            // (2048^3: 76 against 68 us), four times the store instructions costing more
            const int lrow = 32 * q + lane, row = m0 + lrow;
            float *out = sk_part ? p.sk_slots + ((int64_t)cid * CG + rank) * BM * BN
                         : p.ws  ? p.ws + (int64_t)u.s * p.M * p.N : p.C;
            const int64_t ld = sk_part ? (int64_t)BN : p.ws ? (int64_t)p.N : p.ldc;
            const bool vec = (ld % 4 == 0) && ((reinterpret_cast<uintptr_t>(out) & 15) == 0);
            float *crow = sk_part ? out + (int64_t)lrow * BN : out + (int64_t)row * ld + n0;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                // bias of this chunk's 32 columns, one per lane, loaded while TMEM is read
                float bl = 0.0f;
                if (p.bias && !p.ws && n0 + c0 + lane < p.N) bl = __ldg(p.bias + n0 + c0 + lane);
                tmem_ld32(base + (uint32_t)c0, v);
                if (sk_part) {
                    // the whole 128 x BN partial tile, unmasked: the slot is private to this unit
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(crow + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    continue;
                }
                for (int c = cid + 1; c <= c_last; ++c) {
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.sk_slots + ((int64_t)c * CG + rank) * BM * BN + (int64_t)lrow * BN + c0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 a = __ldcg(src + j);
                        v[4 * j] += a.x;
                        v[4 * j + 1] += a.y;
                        v[4 * j + 2] += a.z;
                        v[4 * j + 3] += a.w;
                    }
                }
                // columns of this chunk inside the tile (the last chunk of a 240-wide tile has 16)
                const int w = BN - c0 < 32 ? BN - c0 : 32;
                if (!p.ws) {  // K slices: the reduce kernel applies bias and act; stream-K: the fixup writes C
                    if (p.act) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = gelu_tanh_f(v[j] + __shfl_sync(0xffffffffu, bl, j));
                    } else if (p.bias) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xffffffffu, bl, j);
                    }
                }
                if (CG == 2 && p.c_tma && !p.ws) {
                    // the warp's 32 x 32 block to its swizzled staging buffer (16-byte chunk k of
                    // row i at k ^ (i % 8), conflict-free), then one TMA store that clips at M, N
                    uint8_t *stg = epi_stage + q * 4096;
                    if (lane == 0) bulk_wait_read_all();  // the previous block has left the buffer
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<float4 *>(stg + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && m0 + 32 * q < p.M && n0 + c0 < p.N) {
                        tma_store_2d(&tmC, stg, n0 + c0, m0 + 32 * q);
                        bulk_commit();
                    }
                    continue;
                }
                if (row < p.M && n0 + c0 < p.N) {
                    if (vec && w == 32 && n0 + c0 + 32 <= p.N) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(crow + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < w && n0 + c0 + j < p.N) crow[c0 + j] = v[j];
                    }
                }
            }
            if (sk_part) {
                // the slot's stores are visible device-wide before its flag is
                __threadfence();
                epi_sync();
                if (et == 0) flag_set(p.sk_flags + cid * CG + rank);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) arrive_leader<CG>(&acce[b]);
        }
        // TMA stores of C complete before the CTA's shared memory is released
        if (CG == 2 && lane == 0) bulk_wait_all();
    }

    tc_fence_before_sync();
    if constexpr (CG == 2) cluster_sync();
    else __syncthreads();
    tc_fence_after_sync();
    if (warp == WARP_MMA) {
        if constexpr (CG == 2) tmem_dealloc_pair(tmem, TMEM_COLS);
        else tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <bool A_KC, bool B_KC, int CG, int BN, bool SK>
cudaError_t launch_ws1(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const WsParams &p,
                       int grid, cudaStream_t s) {
    auto kern = gemm_tf32x3_ws_kernel<A_KC, B_KC, CG, BN, SK>;
    constexpr int smem = Plan<A_KC, B_KC, CG, BN>::SMEM_BYTES;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = CG == 2 ? 1 : 0;
    return cudaLaunchKernelEx(&lc, kern, ta, tb, tc, p);
}

// C = sum over the ksplit slices of the workspace, added in slice order (bit-reproducible).
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ ws, float *__restrict__ C,
                                                            int64_t ldc, int M, int N, int ksplit,
                                                            const float *__restrict__ bias, int act) {
    // the sum of the slices in slice order, then the layer's bias and activation when given
    auto fin = [&](float z, int64_t col) {
        if (bias) z += __ldg(bias + col);
        return act ? gelu_tanh_f(z) : z;
    };
    const int64_t MN = (int64_t)M * N;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    const bool vec = (N % 4 == 0) && (ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(C) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(ws) & 15) == 0);
    if (vec) {
        const float4 *w4 = reinterpret_cast<const float4 *>(ws);
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < MN / 4; i += step) {
            float4 acc = w4[i];
            for (int s = 1; s < ksplit; ++s) {
                const float4 v = w4[(int64_t)s * (MN / 4) + i];
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const int64_t row = (4 * i) / N, col = (4 * i) % N;
            if (bias || act) acc = make_float4(fin(acc.x, col), fin(acc.y, col + 1), fin(acc.z, col + 2), fin(acc.w, col + 3));
            *reinterpret_cast<float4 *>(C + row * ldc + col) = acc;
        }
    } else {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < MN; i += step) {
            float acc = ws[i];
            for (int s = 1; s < ksplit; ++s) acc += ws[(int64_t)s * MN + i];
            C[(i / N) * ldc + i % N] = (bias || act) ? fin(acc, i % N) : acc;
        }
    }
}

template <bool A_KC, bool B_KC, int CG, int BN>
cudaError_t launch_ws(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc, const WsParams &p, int grid,
                      cudaStream_t s) {
    return p.sk ? launch_ws1<A_KC, B_KC, CG, BN, true>(ta, tb, tc, p, grid, s)
                : launch_ws1<A_KC, B_KC, CG, BN, false>(ta, tb, tc, p, grid, s);
}

template <int CG, int BN>
cudaError_t launch_ws_cg(const GemmArgs &g, int sms, int ksplit, float *ws, cudaStream_t s) {
    constexpr int BNC = BN / CG;
    CUtensorMap ta, tb;
    cudaError_t e;
    // K-contiguous operands: 16 x rows boxes, 64-byte swizzle (the MMA operand layout);
    // M/N-contiguous: rows x 16 boxes, unswizzled (transposed by the lo pass)
    if (!g.transA)
        e = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.K, g.M, g.lda * 4, BK, BM,
                         CU_TENSOR_MAP_SWIZZLE_64B);
    else
        e = make_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.M, g.K, g.lda * 4, BM, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    if (g.transB)
        e = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.K, g.N, g.ldb * 4, BK, BNC,
                         CU_TENSOR_MAP_SWIZZLE_64B);
    else
        e = make_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.N, g.K, g.ldb * 4, BNC, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    const int tiles_m = (int)((g.M + BM * CG - 1) / (BM * CG)), tiles_n = (int)((g.N + BN - 1) / BN);
    const bool sk = ksplit == kStreamK && ws;
    float *const sk_ws = ws;
    if (ksplit < 2) ws = nullptr;
    WsParams p{(int)g.M, (int)g.N, (int)g.K, tiles_m, tiles_m * tiles_n * (ws ? ksplit : 1), ws ? ksplit : 1,
               g.C, g.ldc, ws, 0, 0, 0, nullptr, nullptr, 0, g.bias, g.act};
    // C through TMA stores (CTA pairs): 16-byte aligned C, ldc a multiple of 4
    CUtensorMap tc = ta;
    if (CG == 2 && (reinterpret_cast<uintptr_t>(g.C) & 15) == 0 && g.ldc % 4 == 0 &&
        make_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.C, g.N, g.M, g.ldc * 4, 32, 32,
                     CU_TENSOR_MAP_SWIZZLE_128B) == cudaSuccess)
        p.c_tma = 1;
    const int units = sms / CG;
    int grid = CG * (p.tiles < units ? p.tiles : units);
    if (sk) {
        const int KT = (int)((g.K + BK - 1) / BK);
        p.sk = 1;
        p.sk_total = tiles_m * tiles_n * KT;
        p.sk_w = (p.sk_total + units - 1) / units;
        const int used = (p.sk_total + p.sk_w - 1) / p.sk_w;
        p.sk_slots = sk_ws;
        p.sk_flags = reinterpret_cast<unsigned int *>(sk_ws + (int64_t)used * CG * BM * BN);
        e = cudaMemsetAsync(p.sk_flags, 0, (size_t)used * CG * sizeof(unsigned int), s);
        if (e != cudaSuccess) return e;
        grid = CG * used;
        ws = nullptr;  // no second kernel
    }
    if (!g.transA && !g.transB) e = launch_ws<true, false, CG, BN>(ta, tb, tc, p, grid, s);
    else if (!g.transA && g.transB) e = launch_ws<true, true, CG, BN>(ta, tb, tc, p, grid, s);
    else if (g.transA && !g.transB) e = launch_ws<false, false, CG, BN>(ta, tb, tc, p, grid, s);
    else e = launch_ws<false, true, CG, BN>(ta, tb, tc, p, grid, s);
    if (e != cudaSuccess || !ws) return e;
    const int64_t work = (g.M * g.N + 3) / 4;
    const int64_t blocks = (work + 255) / 256;
    splitk_reduce_kernel<<<(unsigned)(blocks < 4 * sms ? blocks : 4 * sms), 256, 0, s>>>(ws, g.C, g.ldc, (int)g.M,
                                                                                        (int)g.N, ksplit, g.bias, g.act);
    return cudaGetLastError();
}

}  // namespace

static cudaError_t sm_count(int *sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    return e;
}

cudaError_t launch_gemm_tf32x3_ws(const GemmArgs &g, int pair, cudaStream_t s) {
    return launch_gemm_tf32x3_ws_splitk(g, pair, 1, nullptr, s);
}

cudaError_t launch_gemm_tf32x3_ws_splitk(const GemmArgs &g, int pair, int ksplit, float *ws, cudaStream_t s) {
    if (!gemm_tf32x3_supported(g)) return cudaErrorNotSupported;
    int sms = 0;
    cudaError_t e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    // 256 columns per tile: a 240-wide pair tile (72 tiles of a 2048^2 output on 76
    // pairs instead of 64) measured no faster on GB300, the MMA time not shrinking with N
    return pair ? launch_ws_cg<2, 256>(g, sms, ksplit, ws, s) : launch_ws_cg<1, 256>(g, sms, ksplit, ws, s);
}

// Automatic K split.  Tiles that leave more than half of the persistent grid idle: split-K,
// as many slices as keep every tile's slices within one wave, at least 4 slabs of 16 per
// slice, at most 16.  Several waves of tiles with a costly partial last wave: stream-K.
static int gemm_splitk_auto_shape(int64_t M, int64_t N, int64_t K, int pair, int sms);

// The shape's choice (below), raised to the K slices that keep every accumulation within the
// 3xTF32 accuracy margin: a K longer than kTf32x3MaxK never runs stream-K nor one slice.
int gemm_splitk_auto(int64_t M, int64_t N, int64_t K, int pair, int sms) {
    const int64_t need = (K + kTf32x3MaxK - 1) / kTf32x3MaxK;
    const int s = gemm_splitk_auto_shape(M, N, K, pair, sms);
    if (need <= 1) return s;
    const int64_t r = s == kStreamK || s < need ? need : s;
    return r > 16 ? 16 : (int)r;
}

static int gemm_splitk_auto_shape(int64_t M, int64_t N, int64_t K, int pair, int sms) {
    const int cg = pair ? 2 : 1;
    const int64_t tiles = ((M + 128 * cg - 1) / (128 * cg)) * ((N + 255) / 256);
    const int64_t kt = (K + BK - 1) / BK;
    const int64_t units = sms / cg;
    if (tiles >= units) {
        // stream-K when the last wave is partial enough to cost more than 5% (4 waves' worth of
        // units for 256 pair tiles on 76 pairs: +12% measured), each unit keeps 8 slabs, and a
        // tile has at least 64 slabs (K >= 1024): with 48 (8192 x 3072 x 768, 384 pair tiles)
        // the fixups measured slower than the partial last wave (154 against 149 us)
        const int64_t waves = (tiles + units - 1) / units;
        return (waves * units * 100 > tiles * 105 && tiles * kt >= 8 * units && kt >= 64) ? kStreamK : 1;
    }
    int64_t s = units / tiles;
    if (s >= 2) {
        if (s > kt / 4) s = kt / 4;
        if (s > 16) s = 16;
        return s < 1 ? 1 : (int)s;
    }
    // between half a wave and a wave (64 pair tiles of 2048^3 on 76 pairs): no split; stream-K
    // measured slower there, all 152 SMs running each slab ~11% slower than 128
    return 1;
}

// Workspace floats of a split: split-K slices, or the stream-K slots and flags.
int64_t gemm_splitk_workspace_floats(int64_t M, int64_t N, int64_t K, int pair, int split, int sms) {
    if (split >= 2) return (int64_t)split * M * N;
    if (split != kStreamK) return 0;
    const int cg = pair ? 2 : 1;
    const int64_t tiles = ((M + 128 * cg - 1) / (128 * cg)) * ((N + 255) / 256);
    const int64_t total = tiles * ((K + BK - 1) / BK);
    const int64_t units = sms / cg;
    const int64_t w = (total + units - 1) / units;
    const int64_t used = (total + w - 1) / w;
    return used * cg * BM * 256 + (used * cg + 3) / 4 * 4;  // slots, then one flag word per CTA
}

unsigned int gemm_tf32x3_ws_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_tf32ws_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_tf32ws_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
