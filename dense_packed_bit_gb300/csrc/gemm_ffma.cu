// gemm_ffma.cu -- C = op(A) . op(B), fp32 FFMA, TMA-staged and register-blocked.
//
// "I built a GPT-2 in the browser...", section "The kernel sweep": Step 1
// stages 16 x 16 tiles of A and B in workgroup memory, Step 2 gives each
// thread a 4 x 4 register block so each shared load feeds 4 multiply-adds;
// section "The three things that didn't work": an 8 x 8 block lost on Apple
// hardware through register spills, and 128-bit vector loads won 1.37x.
// "More Stumbling, This Time in the Browser", "Four answers per worker":
// register blocks of outputs, edge masks for partial tiles, one fixed
// accumulation order along k.
//
// GB300 design: a CTA computes a 128 x 128 tile of C with 8 consumer warps
// (8 x 8 outputs per thread, 128-bit shared loads, the multiply-adds as packed
// f32x2 FMAs where an operand read along m or n supplies the pairs -- two
// outputs per instruction, each rounded once as by FFMA: identical bits, at
// 2048^3 NN 13 %, TN 8 % and TT 14 % faster) and one producer warp that
// streams 128 x 32 k-slabs of A and B into a 4-stage shared-memory ring with
// TMA, each stage guarded by a "full" mbarrier (TMA transaction bytes) and an
// "empty" mbarrier (one arrival per consumer thread).  Operands whose
// contiguous dimension is K are loaded with the 128-byte swizzle and read
// along k as float4s; operands contiguous along M/N are loaded unswizzled and
// read along M/N.  The thread-to-row maps are chosen per layout so every
// 128-bit shared load of a warp is bank-conflict free.  Out-of-range parts of
// edge tiles read as zeros (TMA fill) and are masked at the store.
//
// Stream-K tail (launch_gemm_ffma_streamk, with a workspace).  One CTA per SM
// and 128 x 128 tiles leave the last wave partly idle whenever the tile count
// is not a multiple of the SM count (2048^2: 256 tiles on 152 SMs, 1.68 waves,
// the SMs busy 84% of the time).  The first floor(T / G) * G tiles (G = the CTAs
// the GPU holds at once) run whole, one per CTA; the k-steps of the remaining
// tiles, laid end to end, are cut evenly over G more CTAs, so every SM ends
// with the same number of k-steps.  A CTA's share of the tail covers at most two
// tiles (it is shorter than one tile's K range); for each it leaves the partial
// tile of its k-steps in its own workspace slot, and a second kernel adds each
// tile's partial tiles in K order (bit-reproducible) and stores C.  (No bias or
// activation on this form.)
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tmap.h"

#include <mutex>

namespace mm {

__device__ unsigned int g_ffma_err;

namespace {

constexpr int BM = 128, BN = 128, BK = 32, STAGES = 4;
constexpr int NCONS = 256;
constexpr int NTHREADS = NCONS + 32;
constexpr int TILE_BYTES = BM * BK * 4;  // 16 KiB per operand per stage
constexpr int STAGE_BYTES = 2 * TILE_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

struct FfmaParams {
    int M, N, K;
    float *C;
    int64_t ldc;
    const float *bias;  // C = act(op(A) op(B) + bias): bias per column or null, act 1 = GELU (tanh)
    int act;
    // stream-K tail (the SK instantiation only): tiles are numbered row-major over tiles_n
    // columns of tiles; blocks below dp_tiles compute tile blockIdx.x whole, block dp_tiles + j
    // (j < sk_ctas) the k-steps [j I / sk_ctas, (j + 1) I / sk_ctas) of the I = sk_iters k-steps
    // of tiles dp_tiles, dp_tiles + 1, ... laid end to end, into workspace slots 2 j and 2 j + 1
    int tiles_n, dp_tiles, sk_ctas;
    int64_t sk_iters;
    float *ws;
};

constexpr int WS_TILE = BM * BN;  // floats per workspace slot: one partial tile, row-major

// One piece of a CTA's work: k-steps [ka, kb) of a tile, into C (slot < 0) or a workspace slot.
struct Piece {
    int tile, ka, kb, slot;
};

// The pieces of stream-K CTA j: its share [s, e) of the tail's k-steps, cut at tile boundaries.
__device__ __forceinline__ int sk_pieces(const FfmaParams &p, int KT, int j, Piece *pc) {
    const int64_t s = (int64_t)j * p.sk_iters / p.sk_ctas, e = (int64_t)(j + 1) * p.sk_iters / p.sk_ctas;
    if (e <= s) return 0;
    const int u0 = (int)(s / KT), u1 = (int)((e - 1) / KT);
    int n = 0;
    for (int u = u0; u <= u1 && n < 2; ++u, ++n) {
        const int64_t lo = (int64_t)u * KT;
        pc[n].tile = p.dp_tiles + u;
        pc[n].ka = (int)((s > lo ? s : lo) - lo);
        pc[n].kb = (int)((e < lo + KT ? e : lo + KT) - lo);
        pc[n].slot = 2 * j + n;
    }
    return n;
}

// A_KC: the A tile sits in shared memory as [m][k] (k contiguous, 128-byte
// swizzled); otherwise as [k][m].  B_KC: B tile as [n][k] swizzled; else [k][n].
template <bool A_KC, bool B_KC, bool SK>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_ffma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const FfmaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *empty = full + STAGES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KT = (p.K + BK - 1) / BK;
    // this CTA's pieces: one whole tile, or (stream-K tail) up to two partial ones
    Piece pc[2];
    int npc = 1;  // a compile-time 1 without the tail, so the plain kernel keeps its one k loop
    if constexpr (SK) {
        const int b = (int)blockIdx.x;
        if (b < p.dp_tiles) pc[0] = Piece{b, 0, KT, -1};
        else npc = sk_pieces(p, KT, b - p.dp_tiles, pc);
    } else {
        pc[0] = Piece{0, 0, KT, -1};  // the tile is (blockIdx.y, blockIdx.x)
    }
    const int tiles_n = p.tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCONS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCONS / 32) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmA);
            tma_prefetch_desc(&tmB);
            int issued = 0;  // k-steps issued over all pieces: the ring position
            bool stop = false;
            for (int q = 0; q < (SK ? npc : 1) && !stop; ++q) {
                const int m0 = SK ? (pc[q].tile / tiles_n) * BM : (int)blockIdx.y * BM;
                const int n0 = SK ? (pc[q].tile % tiles_n) * BN : (int)blockIdx.x * BN;
                for (int kt = pc[q].ka; kt < pc[q].kb; ++kt) {
                    const int s = issued % STAGES;
                    const uint32_t round = issued / STAGES;
                    if (issued >= STAGES && !mbar_wait(&empty[s], (round - 1) & 1)) {
                        atomicExch(&g_ffma_err, kDevErrWaitEmpty);
                        stop = true;
                        break;
                    }
                    uint8_t *st = smem + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                    const int k0 = kt * BK;
                    if (A_KC) tma_load_2d(st, &tmA, &full[s], k0, m0);
                    else tma_load_2d(st, &tmA, &full[s], m0, k0);
                    if (B_KC) tma_load_2d(st + TILE_BYTES, &tmB, &full[s], k0, n0);
                    else tma_load_2d(st + TILE_BYTES, &tmB, &full[s], n0, k0);
                    ++issued;
                }
            }
            // every issued copy must land before this CTA's shared memory is released
            for (int kt = issued > STAGES ? issued - STAGES : 0; kt < issued; ++kt)
                if (!mbar_wait(&full[kt % STAGES], (kt / STAGES) & 1)) {
                    atomicExch(&g_ffma_err, kDevErrDrain);
                    break;
                }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const int wm = warp & 3, wn = warp >> 2, tr = lane >> 3, tc = lane & 7;
    int rowA[8], colB[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        rowA[i] = A_KC ? wm * 32 + tr + 4 * i : wm * 32 + (i < 4 ? 4 * tr + i : 16 + 4 * tr + (i - 4));
        colB[i] = B_KC ? wn * 64 + tc + 8 * i : wn * 64 + (i < 4 ? 4 * tc + i : 32 + 4 * tc + (i - 4));
    }

    int used = 0;  // k-steps consumed over all pieces: the ring position
    for (int q = 0; q < (SK ? npc : 1); ++q) {
        const int m0 = SK ? (pc[q].tile / tiles_n) * BM : (int)blockIdx.y * BM;
        const int n0 = SK ? (pc[q].tile % tiles_n) * BN : (int)blockIdx.x * BN;
        float acc[8][8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

        for (int kt = pc[q].ka; kt < pc[q].kb; ++kt, ++used) {
            const int s = used % STAGES;
            if (!mbar_wait(&full[s], (used / STAGES) & 1)) {
                atomicExch(&g_ffma_err, kDevErrWaitFull);
                return;
            }
            const float *As = reinterpret_cast<const float *>(smem + s * STAGE_BYTES);
            const float *Bs = reinterpret_cast<const float *>(smem + s * STAGE_BYTES + TILE_BYTES);
#pragma unroll 2
            for (int kg = 0; kg < BK / 4; ++kg) {
                float a[8][4], b[8][4];
                if (A_KC) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int m = rowA[i];
                        const float4 v = reinterpret_cast<const float4 *>(As + m * BK)[kg ^ (m & 7)];
                        a[i][0] = v.x; a[i][1] = v.y; a[i][2] = v.z; a[i][3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const float *row = As + (4 * kg + kk) * BM + wm * 32 + 4 * tr;
                        const float4 v0 = *reinterpret_cast<const float4 *>(row);
                        const float4 v1 = *reinterpret_cast<const float4 *>(row + 16);
                        a[0][kk] = v0.x; a[1][kk] = v0.y; a[2][kk] = v0.z; a[3][kk] = v0.w;
                        a[4][kk] = v1.x; a[5][kk] = v1.y; a[6][kk] = v1.z; a[7][kk] = v1.w;
                    }
                }
                if (B_KC) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = colB[j];
                        const float4 v = reinterpret_cast<const float4 *>(Bs + n * BK)[kg ^ (n & 7)];
                        b[j][0] = v.x; b[j][1] = v.y; b[j][2] = v.z; b[j][3] = v.w;
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const float *row = Bs + (4 * kg + kk) * BN + wn * 64 + 4 * tc;
                        const float4 v0 = *reinterpret_cast<const float4 *>(row);
                        const float4 v1 = *reinterpret_cast<const float4 *>(row + 32);
                        b[0][kk] = v0.x; b[1][kk] = v0.y; b[2][kk] = v0.z; b[3][kk] = v0.w;
                        b[4][kk] = v1.x; b[5][kk] = v1.y; b[6][kk] = v1.z; b[7][kk] = v1.w;
                    }
                }
                // Packed f32x2 FMAs pair the outputs along the operand whose values one 16-byte shared
                // load already leaves in adjacent registers: B read along n pairs columns (2 jp, 2 jp + 1),
                // A read along m pairs rows; with both read along k, packing would cost a move per pair
                // and plain FFMAs measured faster.
                if constexpr (!B_KC) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
#pragma unroll
                            for (int jp = 0; jp < 4; ++jp)
                                fma2_bcast(acc[i][2 * jp], acc[i][2 * jp + 1], a[i][kk], b[2 * jp][kk], b[2 * jp + 1][kk]);
                } else if constexpr (!A_KC) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int j = 0; j < 8; ++j)
#pragma unroll
                            for (int ip = 0; ip < 4; ++ip)
                                fma2_bcast(acc[2 * ip][j], acc[2 * ip + 1][j], b[j][kk], a[2 * ip][kk], a[2 * ip + 1][kk]);
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i][kk], b[j][kk], acc[i][j]);
                }
            }
            mbar_arrive(&empty[s]);
        }

        if (SK && pc[q].slot >= 0) {
            // ------------------------------------------------ partial tile -> its workspace slot
            float *wt = p.ws + (int64_t)pc[q].slot * WS_TILE;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float *wrow = wt + rowA[i] * BN;
                if constexpr (!B_KC) {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        *reinterpret_cast<float4 *>(wrow + colB[4 * h]) =
                            make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) wrow[colB[j]] = acc[i][j];
                }
            }
            continue;
        }

        // ---------------------------------------------------- epilogue (masked)
        const bool vec_ok = !B_KC && (p.ldc % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0);
        if (p.bias || p.act) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int n = n0 + colB[j];
                const float bj = (p.bias && n < p.N) ? __ldg(p.bias + n) : 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float z = acc[i][j] + bj;
                    acc[i][j] = p.act ? gelu_tanh_f(z) : z;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int m = m0 + rowA[i];
            if (m >= p.M) continue;
            float *crow = p.C + (int64_t)m * p.ldc;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = n0 + colB[4 * h];
                if (vec_ok && n + 3 < p.N) {
                    *reinterpret_cast<float4 *>(crow + n) =
                        make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
                } else {
#pragma unroll
                    for (int j = 4 * h; j < 4 * h + 4; ++j) {
                        const int nj = n0 + colB[j];
                        if (nj < p.N) crow[nj] = acc[i][j];
                    }
                }
            }
        }
    }  // pieces
}

// The stream-K CTA whose share of the tail's k-steps holds k-step i: the largest j with
// floor(j I / G) <= i.
__device__ __forceinline__ int sk_cta_of(int64_t i, int64_t I, int G) {
    return (int)(((i + 1) * G + I - 1) / I) - 1;
}

constexpr int RED_ROWS = 8;  // rows of a tile per reduce CTA (32 threads x 4 columns per row)

// C for the tail tiles: each tile's partial tiles added in K order (the order of the CTAs that
// computed them), masked at M and N.
__global__ void __launch_bounds__(256) ffma_sk_reduce_kernel(const FfmaParams p, int KT) {
    const int u = (int)blockIdx.x / (BM / RED_ROWS), strip = (int)blockIdx.x % (BM / RED_ROWS);
    const int row = strip * RED_ROWS + ((int)threadIdx.x >> 5), c4 = 4 * ((int)threadIdx.x & 31);
    const int tile = p.dp_tiles + u;
    const int m = (tile / p.tiles_n) * BM + row, n = (tile % p.tiles_n) * BN + c4;
    if (m >= p.M || n >= p.N) return;
    const int64_t I = p.sk_iters;
    const int G = p.sk_ctas;
    const int ja = sk_cta_of((int64_t)u * KT, I, G), jb = sk_cta_of((int64_t)(u + 1) * KT - 1, I, G);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = ja; j <= jb; ++j) {
        const int first = (int)((int64_t)j * I / G / KT);  // the first tail tile CTA j touches
        const int slot = 2 * j + (u - first);
        const float4 v = *reinterpret_cast<const float4 *>(p.ws + (int64_t)slot * WS_TILE + row * BN + c4);
        if (j == ja) {
            acc = v;
        } else {
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
    }
    const float r[4] = {acc.x, acc.y, acc.z, acc.w};
    float *crow = p.C + (int64_t)m * p.ldc;
    if (n + 3 < p.N && p.ldc % 4 == 0 && (reinterpret_cast<uintptr_t>(p.C) & 15) == 0) {
        *reinterpret_cast<float4 *>(crow + n) = make_float4(r[0], r[1], r[2], r[3]);
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if (n + c < p.N) crow[n + c] = r[c];
    }
}

template <bool A_KC, bool B_KC, bool SK>
cudaError_t launch_ffma(const CUtensorMap &ta, const CUtensorMap &tb, const FfmaParams &p, cudaStream_t s) {
    auto kern = gemm_ffma_kernel<A_KC, B_KC, SK>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;
    if constexpr (SK) {
        kern<<<(unsigned)(p.dp_tiles + p.sk_ctas), NTHREADS, SMEM_BYTES, s>>>(ta, tb, p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        const int KT = (p.K + BK - 1) / BK;
        const int tail = (int)(p.sk_iters / KT);
        ffma_sk_reduce_kernel<<<(unsigned)(tail * (BM / RED_ROWS)), 256, 0, s>>>(p, KT);
    } else {
        dim3 grid((unsigned)((p.N + BN - 1) / BN), (unsigned)((p.M + BM - 1) / BM));
        kern<<<grid, NTHREADS, SMEM_BYTES, s>>>(ta, tb, p);
    }
    return cudaGetLastError();
}

cudaError_t make_ffma_tmaps(const GemmArgs &g, CUtensorMap *ta, CUtensorMap *tb) {
    cudaError_t e;
    if (!g.transA)
        e = make_tmap_2d(ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.K, g.M, g.lda * 4, BK, BM,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    else
        e = make_tmap_2d(ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.A, g.M, g.K, g.lda * 4, BM, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    if (!g.transB)
        e = make_tmap_2d(tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.N, g.K, g.ldb * 4, BN, BK,
                         CU_TENSOR_MAP_SWIZZLE_NONE);
    else
        e = make_tmap_2d(tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.B, g.K, g.N, g.ldb * 4, BK, BN,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    return e;
}

template <bool SK>
cudaError_t launch_ffma_layout(const GemmArgs &g, const CUtensorMap &ta, const CUtensorMap &tb, const FfmaParams &p,
                               cudaStream_t s) {
    if (!g.transA && !g.transB) return launch_ffma<true, false, SK>(ta, tb, p, s);
    if (!g.transA && g.transB) return launch_ffma<true, true, SK>(ta, tb, p, s);
    if (g.transA && !g.transB) return launch_ffma<false, false, SK>(ta, tb, p, s);
    return launch_ffma<false, true, SK>(ta, tb, p, s);
}

}  // namespace

bool ffma_streamk_plan(int64_t M, int64_t N, int64_t K, int ctas, int max_tail_pct, FfmaStreamKPlan *plan) {
    *plan = FfmaStreamKPlan{};
    if (M < 1 || N < 1 || K < 1 || ctas < 2) return false;
    const int64_t tn = (N + BN - 1) / BN, T = ((M + BM - 1) / BM) * tn, KT = (K + BK - 1) / BK;
    const int64_t rem = T % ctas;
    // no tail, or one that nearly fills its wave: nothing to gain
    if (rem == 0 || rem * 100 > (int64_t)ctas * max_tail_pct) return false;
    const int64_t I = rem * KT;
    int64_t sk = I / kFfmaStreamKMinSteps;  // every share at least kFfmaStreamKMinSteps k-steps
    if (sk > ctas) sk = ctas;
    // a share no longer than one tile's K range (so it touches at most two tiles) and at least two
    if (sk < rem || sk < 2 || T - rem > (int64_t)1 << 30 || I > ((int64_t)1 << 40)) return false;
    plan->tiles_n = (int)tn;
    plan->dp_tiles = (int)(T - rem);
    plan->sk_ctas = (int)sk;
    plan->sk_iters = I;
    plan->workspace_floats = 2 * sk * WS_TILE;
    return true;
}

bool gemm_ffma_supported(const GemmArgs &g) {
    const int64_t lim = (int64_t)1 << 30;
    return (reinterpret_cast<uintptr_t>(g.A) % 16) == 0 && (reinterpret_cast<uintptr_t>(g.B) % 16) == 0 &&
           g.lda % 4 == 0 && g.ldb % 4 == 0 && g.M < lim && g.N < lim && g.K < lim && (g.N + BN - 1) / BN < 65536 &&
           (g.M + BM - 1) / BM < 65536;
}

cudaError_t launch_gemm_ffma(const GemmArgs &g, int tile, cudaStream_t s) {
    (void)tile;
    if (!gemm_ffma_supported(g)) return cudaErrorNotSupported;
    CUtensorMap ta, tb;
    cudaError_t e = make_ffma_tmaps(g, &ta, &tb);
    if (e != cudaSuccess) return e;
    FfmaParams p{(int)g.M, (int)g.N, (int)g.K, g.C, g.ldc, g.bias, g.act};
    return launch_ffma_layout<false>(g, ta, tb, p, s);
}

cudaError_t launch_gemm_ffma_streamk(const GemmArgs &g, const FfmaStreamKPlan &plan, float *ws, cudaStream_t s) {
    if (!gemm_ffma_supported(g) || g.bias || g.act) return cudaErrorNotSupported;
    if (plan.sk_ctas < 2) return launch_gemm_ffma(g, 0, s);
    CUtensorMap ta, tb;
    cudaError_t e = make_ffma_tmaps(g, &ta, &tb);
    if (e != cudaSuccess) return e;
    FfmaParams p{(int)g.M, (int)g.N, (int)g.K, g.C, g.ldc, g.bias, g.act,
                 plan.tiles_n, plan.dp_tiles, plan.sk_ctas, plan.sk_iters, ws};
    return launch_ffma_layout<true>(g, ta, tb, p, s);
}

unsigned int gemm_ffma_take_device_error(cudaStream_t s, cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaStreamSynchronize(s);
    if (*err != cudaSuccess) return 0;
    *err = cudaMemcpyFromSymbol(&v, g_ffma_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_ffma_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
