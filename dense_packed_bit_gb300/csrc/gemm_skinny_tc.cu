// gemm_skinny_tc.cu -- fp32 GEMM with few rows of C (M <= 64) on the tcgen05 tensor
// cores, in fp32 accuracy (3xTF32), the K range split over a thread-block cluster.
//
// "I built a GPT-2 in the browser, then made it 2.6x-12.1x faster", section "The
// kernel sweep": the MLP up-projection of 64 tokens, C = A . B with A 64 x 768 and
// B 768 x 3072.  A kernel of 128 x 256 output tiles has 12 tiles for 152 SMs.  Here
// the product is computed transposed,
//
//     D[f][t] = sum_k op(B)[k][f] . op(A)[t][k]      (f: column of C, t: row of C),
//
// with 128 columns of C per CTA as the MMA's M and all (up to 64) rows of C as its
// N, so that no MMA row is padding, and the K range of each 128-column tile cut over
// the S CTAs of a (S, 1, 1) cluster (64 x 768 x 3072: 24 tiles x S = 6, 144 CTAs).
// fp32 accuracy comes from the three-term split of tf32x3_split.cuh: the raw fp32
// tile is the hi operand, a lo pass writes the lo tile, and each 8-deep k-step
// issues hi.hi + hi.lo + lo.hi.
//
// Roles (320 threads, one CTA per SM):
//   warp 0      one thread issues the TMA loads of each 16-deep slab of the CTA's K
//               share into a landing ring of 12 slabs: op(B)^T as 128 columns x 16
//               (K-major with the 64-byte swizzle when B is stored transposed, else an
//               unswizzled [16][128] box) and op(A) as 64 rows x 16 (the same two
//               forms);
//   warp 1      allocates 64 tensor-memory columns; one thread issues 2 x 3
//               tcgen05.mma kind::tf32 (M = 128, N = 64, K = 8) per slab and commits
//               each slab to the barrier that frees its operand stage;
//   warps 2-9   the lo pass of each slab: the landed boxes become K-major hi and lo
//               tiles in one of three operand stages (M/N-contiguous boxes transposed)
//               and the landing slot goes back to the TMA thread at once, so that a
//               CTA's whole K share is in flight from the start (a timeline of the
//               first version, whose MMAs read the landed box itself as the hi operand,
//               showed each slot's refill waiting for the MMAs: 0.38 us per slab);
//               then the epilogue: the thread of TMEM lane f writes
//               column f of the CTA's partial tile to shared memory as [t][f]; after
//               a cluster barrier, CTA r adds, for its share of the tile, the S
//               partial tiles in rank order through distributed shared memory
//               (ld.shared::cluster: deterministic, no workspace), applies bias and
//               GELU, and stores whole rows of C; a second cluster barrier keeps every
//               partial tile alive until its peers have read it.
// Every wait is bounded; a wait that runs out records an error, and the CTA skips its
// remaining work but still arrives at both cluster barriers and frees its tensor
// memory only after its MMAs have completed.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tf32x3_split.cuh"
#include "tmap.h"

#include <mutex>

namespace mm {

__device__ unsigned int g_skinny_tc_err;

namespace {

constexpr int FM = 128;                  // columns of C per CTA: the MMA's M, one per TMEM lane
constexpr int TN = 64;                   // rows of C (at most 64): the MMA's N
constexpr int BK = tf32x3::BK;           // fp32 of K per slab
constexpr int NCONV = 256;               // lo-pass and epilogue threads (warps 2-9)
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_CONV0 = 2;
constexpr int NTHREADS = 64 + NCONV;
constexpr int TMEM_COLS = 64;            // the accumulator: TN fp32 columns
constexpr int MAX_SPLIT = 8;
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr int F_BYTES = FM * BK * 4;     // 8 KiB: a 128 x 16 fp32 tile
constexpr int T_BYTES = TN * BK * 4;     // 4 KiB: a 64 x 16 fp32 tile
constexpr int PART_BYTES = TN * FM * 4;  // 32 KiB: the partial tile [t][f]
// Landing ring: units of UNIT slabs, one TMA copy per operand and unit, freed as soon as the
// lo pass has read them, so that a CTA's whole K share (10 slabs for 64 x 768 x 3072 in
// clusters of 5) is in flight at once.  Operand ring: the K-major hi and lo tiles of a slab,
// freed by the MMAs' commit.  (Units of 2 and 4 slabs, fewer copies to issue, measured
// slower on 64 x 768 x 3072: 14.2 and 14.6 against 12.9 us per call.)
constexpr int UNIT = 1;                           // slabs per landing unit
constexpr int PRE_ISSUE = 16;                     // units issued before the tensor-memory allocation
                                                  // (at most the landing ring)
constexpr int UF_BYTES = UNIT * F_BYTES;          // op(B)^T: [16 UNIT k][128 f] or [128 f][16 UNIT k]
constexpr int UT_BYTES = UNIT * T_BYTES;          // op(A): [16 UNIT k][64 t] or [64 t][16 UNIT k]
constexpr int RAW_BYTES = UF_BYTES + UT_BYTES;
constexpr int OP_BYTES = 2 * (F_BYTES + T_BYTES);
constexpr int HI_F = 0, LO_F = F_BYTES, HI_T = 2 * F_BYTES, LO_T = 2 * F_BYTES + T_BYTES;
constexpr int OPS = 3;
constexpr int MAX_RAWS = 16;
constexpr int BARS = 2 * MAX_RAWS * 8 + 2 * OPS * 8 + 8 + 16;  // landing, operand, accumulator barriers;
                                                                // slot, flag
constexpr int RAWS_FIT = (SMEM_LIMIT - 1024 - BARS - OPS * OP_BYTES) / RAW_BYTES;
constexpr int RAWS = RAWS_FIT < MAX_RAWS ? RAWS_FIT : MAX_RAWS;
constexpr int OP_OFF = RAWS * RAW_BYTES;  // the operand ring, later the partial tile
constexpr int BAR_OFF = OP_OFF + OPS * OP_BYTES;
constexpr int SMEM_BYTES = BAR_OFF + BARS + 1024;  // + alignment slack of the dynamic allocation
static_assert(OPS * OP_BYTES >= PART_BYTES, "the partial tile fits the operand ring");
static_assert(RAWS >= 2 && SMEM_BYTES <= SMEM_LIMIT, "shared memory");

struct SkParams {
    int M, N, K;
    int S;  // CTAs per cluster: the K split
    float *C;
    int64_t ldc;
    const float *bias;  // + bias[column] (null: none), then GELU when act
    int act;
};

// The tile's partial sums of this CTA's float4 tasks [lo, hi): the SS partial tiles of the
// cluster added in rank order (deterministic), bias and GELU, stored to C.  The remote loads
// of 16 / SS tasks are in flight at once (one round for 64 x 768 x 3072 with SS = 5).
template <int SS>
__device__ __forceinline__ void reduce_store(const SkParams &p, uint32_t part_base, int n0, int lo, int hi) {
    constexpr int TPB = 16 / SS;
    const int ct = threadIdx.x;
    const bool vec = (p.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
    for (int i0 = lo + ct; i0 < hi; i0 += TPB * NTHREADS) {
        float4 pv[TPB][SS];
#pragma unroll
        for (int u = 0; u < TPB; ++u) {
            const int i = i0 + u * NTHREADS;  // task i: row i / 32, quad i % 32 of the [t][f] tile
            if (i < hi) {
#pragma unroll
                for (int r = 0; r < SS; ++r)
                    pv[u][r] = ld_cluster_v4(cluster_map(part_base + (uint32_t)(i * 16), (uint32_t)r));
            }
        }
#pragma unroll
        for (int u = 0; u < TPB; ++u) {
            const int i = i0 + u * NTHREADS;
            const int t = i / (FM / 4), col = n0 + 4 * (i % (FM / 4));
            if (i >= hi || col >= p.N) continue;
            float z[4] = {pv[u][0].x, pv[u][0].y, pv[u][0].z, pv[u][0].w};
#pragma unroll
            for (int r = 1; r < SS; ++r) {  // rank order: the same sum on every call
                z[0] += pv[u][r].x;
                z[1] += pv[u][r].y;
                z[2] += pv[u][r].z;
                z[3] += pv[u][r].w;
            }
            const int w = p.N - col < 4 ? p.N - col : 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (p.bias && j < w) z[j] += __ldg(p.bias + col + j);
                if (p.act) z[j] = gelu_tanh_f(z[j]);
            }
            float *crow = p.C + (int64_t)t * p.ldc + col;
            if (vec && w == 4) {
                *reinterpret_cast<float4 *>(crow) = make_float4(z[0], z[1], z[2], z[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (j < w) crow[j] = z[j];
            }
        }
    }
}

template <bool F_KC, bool T_KC>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_skinny_tc_kernel(const __grid_constant__ CUtensorMap tmF, const __grid_constant__ CUtensorMap tmT,
                          const SkParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    uint8_t *ops = smem + OP_OFF;
    float *part = reinterpret_cast<float *>(ops);  // [TN][FM], over the operand ring once the MMAs are done
    uint64_t *rfull = reinterpret_cast<uint64_t *>(smem + BAR_OFF);  // TMA -> lo pass
    uint64_t *rfree = rfull + MAX_RAWS;                             // lo pass -> TMA
    uint64_t *ofull = rfree + MAX_RAWS;                             // lo pass -> MMA
    uint64_t *ofree = ofull + OPS;                                  // MMA -> lo pass
    uint64_t *accf = ofree + OPS;                                   // MMA -> epilogue
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accf + 1);
    volatile int *fail_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.S;
    const uint32_t rank = cluster_ctarank();
    const int n0 = (int)(blockIdx.x / S) * FM;
    const int KT = (p.K + BK - 1) / BK;
    const int kt0 = (int)((int64_t)rank * KT / S), nk = (int)((int64_t)(rank + 1) * KT / S) - kt0;
    const int nu = (nk + UNIT - 1) / UNIT;  // landing units; the last may reach past this CTA's K
                                            // share, and those slabs are never multiplied

    // one unit's two boxes into landing slot u % RAWS
    auto issue = [&](int u) {
        const int s = u % RAWS, k0 = (kt0 + UNIT * u) * BK;
        uint8_t *st = smem + s * RAW_BYTES;
        mbar_arrive_expect_tx(&rfull[s], RAW_BYTES);
        if (F_KC) tma_load_2d(st, &tmF, &rfull[s], k0, n0);
        else tma_load_2d(st, &tmF, &rfull[s], n0, k0);
        if (T_KC) tma_load_2d(st + UF_BYTES, &tmT, &rfull[s], k0, 0);
        else tma_load_2d(st + UF_BYTES, &tmT, &rfull[s], 0, k0);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < RAWS; ++s) {
            mbar_init(&rfull[s], 1);
            mbar_init(&rfree[s], NCONV / 32);
        }
        for (int c = 0; c < OPS; ++c) {
            mbar_init(&ofull[c], NCONV / 32);
            mbar_init(&ofree[c], 1);
        }
        mbar_init(accf, 1);
        *fail_flag = 0;
        fence_mbar_init();
        // the first landing ring's worth of copies goes out before anything else: the DRAM
        // latency of the first slab then overlaps the tensor-memory allocation and the barrier
        for (int u = 0; u < nu && u < PRE_ISSUE && u < RAWS; ++u) issue(u);
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&](unsigned int code) {
        atomicExch(&g_skinny_tc_err, code);
        *fail_flag = 1;
    };

    if (warp == WARP_TMA) {
        if (lane == 0) {
            int it = nu < PRE_ISSUE ? nu : PRE_ISSUE;  // units issued
            if (it > RAWS) it = RAWS;
            for (; it < nu; ++it) {
                if (*fail_flag) break;
                if (it >= RAWS && !mbar_wait(&rfree[it % RAWS], (uint32_t)(it / RAWS - 1) & 1)) {
                    fail(kDevErrWaitEmpty);
                    break;
                }
                issue(it);
            }
            // every copy issued lands before the shared memory is reused or released
            for (int s = 0; s < RAWS && s < it; ++s) {
                const int lastit = s + ((it - 1 - s) / RAWS) * RAWS;
                if (!mbar_wait(&rfull[s], (uint32_t)(lastit / RAWS) & 1)) {
                    atomicExch(&g_skinny_tc_err, kDevErrDrain);
                    break;
                }
            }
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(kFmtTF32, kFmtTF32, TN, FM);
            for (int it = 0; it < nk; ++it) {
                const int c = it % OPS;
                const uint32_t use = it / OPS;
                if (*fail_flag) break;
                if (!mbar_wait(&ofull[c], use & 1)) {
                    fail(kDevErrWaitFull);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t st = smem_u32(ops + c * OP_BYTES);
#pragma unroll
                for (int ks = 0; ks < BK / 8; ++ks) {
                    // 8 tf32 of K are 32 bytes along the swizzled 64-byte rows
                    const uint32_t o = 32u * ks;
                    const uint64_t fh = sdesc_make(st + HI_F + o, 16, 512, kSdescSw64);
                    const uint64_t fl = sdesc_make(st + LO_F + o, 16, 512, kSdescSw64);
                    const uint64_t th = sdesc_make(st + HI_T + o, 16, 512, kSdescSw64);
                    const uint64_t tl = sdesc_make(st + LO_T + o, 16, 512, kSdescSw64);
                    const uint32_t acc0 = (it > 0 || ks > 0) ? 1u : 0u;
                    umma_tf32(tmem, fh, th, idesc, acc0);
                    umma_tf32(tmem, fh, tl, idesc, 1u);
                    umma_tf32(tmem, fl, th, idesc, 1u);
                }
                umma_commit(&ofree[c]);
            }
            // every MMA issued has completed when accf fires (also after a failure, so that
            // the tensor memory is never freed under a running MMA)
            umma_commit(accf);
            if (!mbar_wait_sleep(accf, 0)) atomicExch(&g_skinny_tc_err, kDevErrWaitMma);
        }
    } else {
        // ---------------------------------------------------------------- lo pass
        // slab j of a landed unit -> K-major hi and lo tiles of an operand stage; the landing
        // unit is handed back as soon as its last slab has been read
        const int ct = threadIdx.x - 32 * WARP_CONV0;
        for (int it = 0; it < nk; ++it) {
            const int u = it / UNIT, j = it % UNIT, s = u % RAWS, c = it % OPS;
            if (*fail_flag) break;
            if (!mbar_wait(&rfull[s], (uint32_t)(u / RAWS) & 1) ||
                (it >= OPS && !mbar_wait(&ofree[c], (uint32_t)(it / OPS - 1) & 1))) {
                fail(kDevErrWaitFull);
                break;
            }
            const uint8_t *raw = smem + s * RAW_BYTES;
            uint8_t *op = ops + c * OP_BYTES;
            if (F_KC) tf32x3::split_rows<FM, UNIT * BK, NCONV>(raw, j, op + HI_F, op + LO_F, ct);
            else tf32x3::split_transpose<FM, NCONV>(raw + j * F_BYTES, op + HI_F, op + LO_F, ct);
            if (T_KC) tf32x3::split_rows<TN, UNIT * BK, NCONV>(raw + UF_BYTES, j, op + HI_T, op + LO_T, ct);
            else tf32x3::split_transpose<TN, NCONV>(raw + UF_BYTES + j * T_BYTES, op + HI_T, op + LO_T, ct);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (j == UNIT - 1 || it == nk - 1) mbar_arrive(&rfree[s]);
                mbar_arrive(&ofull[c]);
            }
        }
        // ---------------------------------------------------------------- partial tile
        // the warp of lane quarter q reads TMEM lanes 32 q .. 32 q + 31 (columns f of C), the
        // rows of C of its half; after a failure the tile is written as zeros, so that the peers
        // read defined values
        if (!mbar_wait_sleep(accf, 0)) fail(kDevErrWaitMma);
        tc_fence_after_sync();
        {
            const int q = warp & 3, f = 32 * q + lane;
            const bool have = nk > 0 && !*fail_flag;
            for (int c0 = 32 * ((warp - WARP_CONV0) / 4); c0 < TN; c0 += 32 * (NCONV / 128)) {
                float v[32];
                if (have) {
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0, v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;  // a rank without K slabs adds zeros
                }
#pragma unroll
                for (int j = 0; j < 32; ++j) part[(c0 + j) * FM + f] = v[j];
            }
        }
    }

    // every CTA's partial tile is written (release / acquire at cluster scope)
    tc_fence_before_sync();
    cluster_sync();

    if (!*fail_flag) {
        // ---------------------------------------------------------------- reduction and C
        // CTA `rank` owns the float4 tasks [lo, hi) of the tile's rows x 32 column quads, taken
        // by all 320 threads; a warp's lanes take consecutive quads, i.e. 512 contiguous bytes
        // of a row of C.  (Pushing each CTA's rows to their owner with one bulk copy per peer
        // instead measured slower: 12.8 against 11.2 us per 64 x 768 x 3072 call.)
        const int rows = p.M < TN ? p.M : TN;
        const int tasks = rows * (FM / 4);
        const int lo = (int)((int64_t)rank * tasks / S), hi = (int)((int64_t)(rank + 1) * tasks / S);
        const uint32_t part_base = smem_u32(part);
        switch (S) {
            case 1: reduce_store<1>(p, part_base, n0, lo, hi); break;
            case 2: reduce_store<2>(p, part_base, n0, lo, hi); break;
            case 3: reduce_store<3>(p, part_base, n0, lo, hi); break;
            case 4: reduce_store<4>(p, part_base, n0, lo, hi); break;
            case 5: reduce_store<5>(p, part_base, n0, lo, hi); break;
            case 6: reduce_store<6>(p, part_base, n0, lo, hi); break;
            case 7: reduce_store<7>(p, part_base, n0, lo, hi); break;
            default: reduce_store<8>(p, part_base, n0, lo, hi); break;
        }
    }

    // no CTA leaves while a peer may still read its partial tile
    cluster_sync();
    tc_fence_after_sync();
    if (warp == WARP_MMA) tmem_dealloc(tmem, TMEM_COLS);
}

template <bool F_KC, bool T_KC>
cudaError_t launch_sk(const CUtensorMap &tf, const CUtensorMap &tt, const SkParams &p, int tiles, cudaStream_t s) {
    auto kern = gemm_skinny_tc_kernel<F_KC, T_KC>;
    constexpr int smem = SMEM_BYTES;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)(tiles * p.S));
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, tf, tt, p);
}

// Clusters of s CTAs of this kernel the GPU holds at once (one CTA per SM; a cluster stays
// within a GPC, so 24 clusters of 5 fit on GB300 where 24 of 6 do not), cached per s.
int active_clusters(int s) {
    static std::mutex mu;
    static int cache[MAX_SPLIT + 1] = {0};
    std::lock_guard<std::mutex> lock(mu);
    if (cache[s] == 0) {
        auto kern = gemm_skinny_tc_kernel<false, true>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3((unsigned)(s * 64));
        lc.blockDim = dim3(NTHREADS);
        lc.dynamicSmemBytes = SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)s;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        int n = 0;
        cache[s] = cudaOccupancyMaxActiveClusters(&n, kern, &lc) == cudaSuccess && n > 0 ? n : -1;
    }
    return cache[s];
}

}  // namespace

// The K split: the most CTAs per 128-column tile (at most 8, a portable cluster, and at least
// two 16-deep slabs each) whose clusters all fit on the GPU at once -- a second wave of
// clusters measured ~70% slower (64 x 768 x 3072: 5 -> 11.2 us, 6 -> 19 us).
int gemm_skinny_tc_split(int64_t M, int64_t N, int64_t K, int sms) {
    (void)M;
    const int64_t tiles = (N + FM - 1) / FM, kt = (K + BK - 1) / BK;
    int64_t s = sms / tiles;
    if (s > MAX_SPLIT) s = MAX_SPLIT;
    if (s > kt / 2) s = kt / 2;
    for (; s > 1; --s) {
        const int n = active_clusters((int)s);
        if (n < 0 || tiles <= n) break;  // no figure: the SM count alone
    }
    return s < 1 ? 1 : (int)s;
}

// M <= 64 rows of C, the TMA operand rules of the 3xTF32 kernels (16-byte aligned A and
// B, lda and ldb multiples of 4), K within the 3xTF32 accuracy margin.
bool gemm_skinny_tc_supported(const GemmArgs &g) {
    return g.M >= 1 && g.M <= TN && g.K <= kTf32x3MaxK && gemm_tf32x3_supported(g) &&
           (g.N + FM - 1) / FM * MAX_SPLIT < ((int64_t)1 << 31);
}

cudaError_t launch_gemm_skinny_tc(const GemmArgs &g, int split, cudaStream_t s) {
    if (!gemm_skinny_tc_supported(g) || split < 0 || split > MAX_SPLIT) return cudaErrorNotSupported;
    int dev = 0, sms = 152;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int S = split > 0 ? split : gemm_skinny_tc_split(g.M, g.N, g.K, sms);
    CUtensorMap tf, tt;
    // unswizzled boxes of one landing unit (16 UNIT of K), in the operand's stored orientation:
    // op(B)^T, 128 columns of C: [128][16 UNIT] when B is stored transposed (K contiguous),
    // else [16 UNIT][128]; op(A), 64 rows of C (rows past M read as zeros): [64][16 UNIT] or
    // [16 UNIT][64]
    if (g.transB)
        e = make_tmap_2d(&tf, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.K, g.N, g.ldb * 4, UNIT * BK, FM,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        e = make_tmap_2d(&tf, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.N, g.K, g.ldb * 4, FM, UNIT * BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    if (!g.transA)
        e = make_tmap_2d(&tt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.K, g.M, g.lda * 4, UNIT * BK, TN,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        e = make_tmap_2d(&tt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.M, g.K, g.lda * 4, TN, UNIT * BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    const SkParams p{(int)g.M, (int)g.N, (int)g.K, S, g.C, g.ldc, g.bias, g.act};
    const int tiles = (int)((g.N + FM - 1) / FM);
    if (g.transB) return g.transA ? launch_sk<true, false>(tf, tt, p, tiles, s) : launch_sk<true, true>(tf, tt, p, tiles, s);
    return g.transA ? launch_sk<false, false>(tf, tt, p, tiles, s) : launch_sk<false, true>(tf, tt, p, tiles, s);
}

unsigned int gemm_skinny_tc_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_skinny_tc_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_skinny_tc_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
