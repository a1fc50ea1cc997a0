// attention_fa2.cu -- scaled dot-product attention, forward and backward, in the
// Flash-Attention-2 form, fp32 on the CUDA cores (sm_103a).
//
// "I built a GPT-2 in the browser, then made it 2.6x-12.1x faster", section
// "Flash Attention 2": one workgroup per (batch, head, tile of query rows), the
// keys and values walked in blocks, the online-softmax state (running maximum
// m, running sum l, unnormalised output O) kept in registers across the blocks;
// the forward stores L = m + log(l) per query row and the backward rebuilds
// P = exp(S - L) from q and k instead of keeping the attention matrix.
//
// Layout: Q, K, V, O, dO, dQ, dK, dV are [heads][T][64] fp32 row-major (a batch
// of B sequences of H heads is B H heads), L is [heads][T] fp32 (natural log).
//
// GB300 form.  A CTA of 256 threads owns a 64-row tile; 64-row tiles of the
// other operands pass through shared memory.  Every 64 x 64 x 64 product
// C[i][j] += sum_t A[i][t] B[t][j] reads its operands as A^T and B, both stored
// [t][...] with rows padded to 68 words: thread (ty, tx) = (tid / 16, tid % 16)
// holds C[4 ty + r][4 tx + c] and reads per t one 16-byte vector of each
// (A^T's shared by the half-warp, a broadcast), multiplying with packed f32x2
// FMAs.  So a tile is stored in whichever orientation its products read it --
// "natural" [row][d] or "transposed" [d][row] (the copy does the transpose) --
// and the probabilities P and dS are written from registers in the orientation
// the next product needs.  The 16 threads of a half-warp hold whole rows of S:
// the softmax's row maximum and row sum are 4-step shuffles within it.  Scores
// are kept in base-2 units (scale * log2(e) folded into one multiply), so each
// probability is one exp2.
//
// Tiles stream through two shared-memory buffers by 4-byte cp.async, the next
// block's copies in flight while the current one is multiplied.  With a causal
// mask query tile j meets j + 1 key blocks, so a CTA takes the tile pair
// (j, n - 1 - j): every CTA then does n + 1 blocks of work (n tiles per head)
// instead of 1 .. n.
//
// The backward is split in two kernels so that every gradient is a sum in a
// fixed order (no atomics): one CTA per key tile (pair) accumulates dK and dV
// over the query tiles, one CTA per query tile (pair) accumulates dQ over the
// key tiles; both rebuild S, P and dS = P (dP - D), D_i = dO_i . O_i, from
// identical products in identical order.  Causal attention skips the blocks
// above the diagonal.
#include "mm_common.cuh"
#include "mm_internal.h"

#include <math.h>

namespace mm {

namespace {

constexpr int HD = 64;      // head dimension
constexpr int BT = 64;      // rows per tile (queries or keys)
constexpr int TS = BT + 4;  // padded shared-memory row: 16-byte aligned, 4 banks of skew
constexpr int TILE = BT * TS;
constexpr int NT = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// acc[r][c] += sum_t At[t][4 ty + r] B[t][4 tx + c], t = 0..63 in order
__device__ __forceinline__ void mm64(float (&acc)[4][4], const float *At, const float *B, int ty, int tx) {
#pragma unroll 8
    for (int t = 0; t < BT; ++t) {
        const float4 a = *reinterpret_cast<const float4 *>(At + t * TS + 4 * ty);
        const float4 b = *reinterpret_cast<const float4 *>(B + t * TS + 4 * tx);
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            fma2_bcast(acc[r][0], acc[r][1], av[r], b.x, b.y);
            fma2_bcast(acc[r][2], acc[r][3], av[r], b.z, b.w);
        }
    }
}

// two independent products in one loop (twice the independent FMA chains per step)
__device__ __forceinline__ void mm64_2(float (&c1)[4][4], const float *At1, const float *B1, float (&c2)[4][4],
                                       const float *At2, const float *B2, int ty, int tx) {
#pragma unroll 4
    for (int t = 0; t < BT; ++t) {
        const float4 a1 = *reinterpret_cast<const float4 *>(At1 + t * TS + 4 * ty);
        const float4 b1 = *reinterpret_cast<const float4 *>(B1 + t * TS + 4 * tx);
        const float4 a2 = *reinterpret_cast<const float4 *>(At2 + t * TS + 4 * ty);
        const float4 b2 = *reinterpret_cast<const float4 *>(B2 + t * TS + 4 * tx);
        const float av1[4] = {a1.x, a1.y, a1.z, a1.w}, av2[4] = {a2.x, a2.y, a2.z, a2.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            fma2_bcast(c1[r][0], c1[r][1], av1[r], b1.x, b1.y);
            fma2_bcast(c2[r][0], c2[r][1], av2[r], b2.x, b2.y);
            fma2_bcast(c1[r][2], c1[r][3], av1[r], b1.z, b1.w);
            fma2_bcast(c2[r][2], c2[r][3], av2[r], b2.z, b2.w);
        }
    }
}

__device__ __forceinline__ void cp_async4(float *dst, const float *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// rows row0 .. row0 + 63 of a [T][64] matrix into a tile, asynchronously (the caller commits
// and waits), natural ([row][d]) or transposed ([d][row]); rows past T read 0 (not read)
template <bool TRANS>
__device__ __forceinline__ void load_tile(float *dst, const float *src, int64_t row0, int T) {
    for (int e = threadIdx.x; e < BT * HD; e += NT) {
        const int r = e >> 6, d = e & 63;
        const int64_t row = row0 + r;
        cp_async4(dst + (TRANS ? d * TS + r : r * TS + d), row < T ? src + row * HD + d : src, row < T ? 4 : 0);
    }
}

// the query (or key) tiles of CTA b: tile b alone, or with a causal mask the pair (b, n - 1 - b)
__device__ __forceinline__ int tiles_of(int b, int n, int causal, int (&t)[2]) {
    t[0] = b;
    if (!causal) return 1;
    t[1] = n - 1 - b;
    return t[1] != b ? 2 : 1;
}

__device__ __forceinline__ float half_max(float v) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

struct AttnArgs {
    const float *Q, *K, *V, *O, *dO, *L;
    float *Out, *Lout, *dQ, *dK, *dV;
    int T, causal;
    float scale, scale2;  // scale, and scale * log2(e)
};

__device__ __forceinline__ bool allowed(int i, int k, int T, int causal) {
    return i < T && k < T && (!causal || k <= i);
}

// tile value v[r][c] (row 4 ty + r, column 4 tx + c) into a natural or a transposed tile
__device__ __forceinline__ void store_n(float *dst, const float (&v)[4][4], int ty, int tx) {
#pragma unroll
    for (int r = 0; r < 4; ++r)
        *reinterpret_cast<float4 *>(dst + (4 * ty + r) * TS + 4 * tx) = make_float4(v[r][0], v[r][1], v[r][2], v[r][3]);
}
__device__ __forceinline__ void store_t(float *dst, const float (&v)[4][4], int ty, int tx) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<float4 *>(dst + (4 * tx + c) * TS + 4 * ty) = make_float4(v[0][c], v[1][c], v[2][c], v[3][c]);
}

// D_i = dO_i . O_i for rows i = q0 + 4 ty + r (global dO and O, 4 columns per thread)
__device__ __forceinline__ void row_dots(const AttnArgs &a, int64_t head, int q0, int ty, int tx, float (&Drow)[4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + 4 * ty + r;
        float p = 0.f;
        if (i < a.T) {
            const int64_t base = (head * a.T + i) * HD + 4 * tx;
#pragma unroll
            for (int c = 0; c < 4; ++c) p = fmaf(__ldg(a.dO + base + c), __ldg(a.O + base + c), p);
        }
        Drow[r] = half_sum(p);
    }
}

// P and dS of the block (query tile q0, key tile k0) in registers, from S = Q K^T and
// dP = dO V^T (Qt, Kt, dOt, Vt transposed tiles)
__device__ __forceinline__ void probs_and_dS(const AttnArgs &a, int q0, int k0, const float *Qt, const float *Kt,
                                             const float *dOt, const float *Vt, const float (&L2)[4],
                                             const float (&Drow)[4], float (&p)[4][4], float (&ds)[4][4], int ty,
                                             int tx) {
    float dp[4][4] = {};
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) p[r][c] = 0.f;
    mm64_2(p, Qt, Kt, dp, dOt, Vt, ty, tx);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + 4 * ty + r;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int k = k0 + 4 * tx + c;
            p[r][c] = allowed(i, k, a.T, a.causal) ? exp2f(p[r][c] * a.scale2 - L2[r]) : 0.f;
            ds[r][c] = p[r][c] * (dp[r][c] - Drow[r]);
        }
    }
}

__device__ __forceinline__ void load_L2(const AttnArgs &a, int64_t head, int q0, int ty, float (&L2)[4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + 4 * ty + r;
        L2[r] = i < a.T ? __ldg(a.L + head * a.T + i) * kLog2e : 0.f;
    }
}

// ---------------------------------------------------------------- forward
// The online-softmax update of one query tile for one key block: scores s (rows 4 ty + r of the
// tile at q0, keys k0 + 4 tx + c) in, probabilities out (in s); state m, l, o rescaled.
__device__ __forceinline__ void softmax_step(const AttnArgs &a, int q0, int k0, float (&s)[4][4], float (&m)[4],
                                             float (&l)[4], float (&o)[4][4], int ty, int tx) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + 4 * ty + r;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int k = k0 + 4 * tx + c;
            s[r][c] = allowed(i, k, a.T, a.causal) ? s[r][c] * a.scale2 : -INFINITY;
            mx = fmaxf(mx, s[r][c]);
        }
        const float mnew = fmaxf(m[r], half_max(mx));
        // a row with no allowed key yet (only rows past T) keeps zero weights
        const float alpha = mnew == -INFINITY ? 1.f : exp2f(m[r] - mnew);
        float ls = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            s[r][c] = mnew == -INFINITY ? 0.f : exp2f(s[r][c] - mnew);  // now P
            ls += s[r][c];
            o[r][c] *= alpha;
        }
        l[r] = l[r] * alpha + ls;
        m[r] = mnew;
    }
}

__device__ __forceinline__ void store_out(const AttnArgs &a, int64_t head, int q0, const float (&m)[4],
                                          const float (&l)[4], const float (&o)[4][4], int ty, int tx) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + 4 * ty + r;
        const float lrow = half_sum(l[r]);
        if (i >= a.T) continue;
        const float inv = 1.f / lrow;
        float *orow = a.Out + (head * a.T + i) * HD + 4 * tx;
#pragma unroll
        for (int c = 0; c < 4; ++c) orow[c] = o[r][c] * inv;
        if (tx == 0) a.Lout[head * a.T + i] = (m[r] + log2f(lrow)) * kLn2;
    }
}

// A CTA walks the key blocks once for its tile (pair): with a causal mask the lower tile of a
// pair (j < n - 1 - j) needs blocks 0 .. j, the upper one 0 .. n - 1 - j; both share every K
// and V block they have in common, and their two products per block run as independent chains.
__global__ void __launch_bounds__(NT, 1) attn_fwd_kernel(const AttnArgs a) {
    extern __shared__ __align__(16) float sm[];
    // Qt of tile 0 and 1, Pt of tile 0 and 1, [2 buffers][Kt, V]
    float *Qt0 = sm, *Qt1 = sm + TILE, *Pt0 = sm + 2 * TILE, *Pt1 = sm + 3 * TILE, *KV = sm + 4 * TILE;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    const int T = a.T;
    const int64_t head = blockIdx.y;
    const float *Qh = a.Q + head * T * HD, *Kh = a.K + head * T * HD, *Vh = a.V + head * T * HD;
    int tl[2];
    const int nt = tiles_of(blockIdx.x, (T + BT - 1) / BT, a.causal, tl);
    const int q0a = tl[0] * BT, q0b = nt == 2 ? tl[1] * BT : q0a;
    // keys past a tile's last query are masked (causal)
    const int kend_a = a.causal ? min(T, q0a + BT) : T, kend_b = a.causal ? min(T, q0b + BT) : T;
    const int kend = max(kend_a, kend_b);
    load_tile<true>(Qt0, Qh, q0a, T);
    if (nt == 2) load_tile<true>(Qt1, Qh, q0b, T);
    load_tile<true>(KV, Kh, 0, T);
    load_tile<false>(KV + TILE, Vh, 0, T);
    cp_commit();
    float m0[4], l0[4], o0[4][4], m1[4], l1[4], o1[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        m0[r] = m1[r] = -INFINITY;
        l0[r] = l1[r] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) o0[r][c] = o1[r][c] = 0.f;
    }
    for (int k0 = 0, buf = 0; k0 < kend; k0 += BT, buf ^= 1) {
        cp_wait_all();
        __syncthreads();  // this block's K, V (and Q) landed; the other buffer and P are free
        if (k0 + BT < kend) {
            load_tile<true>(KV + (buf ^ 1) * 2 * TILE, Kh, k0 + BT, T);
            load_tile<false>(KV + (buf ^ 1) * 2 * TILE + TILE, Vh, k0 + BT, T);
        }
        cp_commit();
        const float *Kt = KV + buf * 2 * TILE, *Vs = Kt + TILE;
        const bool two = nt == 2 && k0 < kend_b, one = k0 < kend_a;  // block-uniform
        float s0[4][4] = {}, s1[4][4] = {};
        if (one && two) {
            mm64_2(s0, Qt0, Kt, s1, Qt1, Kt, ty, tx);
        } else if (one) {
            mm64(s0, Qt0, Kt, ty, tx);
        } else {
            mm64(s1, Qt1, Kt, ty, tx);
        }
        if (one) {
            softmax_step(a, q0a, k0, s0, m0, l0, o0, ty, tx);
            store_t(Pt0, s0, ty, tx);
        }
        if (two) {
            softmax_step(a, q0b, k0, s1, m1, l1, o1, ty, tx);
            store_t(Pt1, s1, ty, tx);
        }
        __syncthreads();  // P complete
        if (one && two) {
            mm64_2(o0, Pt0, Vs, o1, Pt1, Vs, ty, tx);
        } else if (one) {
            mm64(o0, Pt0, Vs, ty, tx);
        } else {
            mm64(o1, Pt1, Vs, ty, tx);
        }
    }
    cp_wait_all();  // (an empty group when the last block had no successor)
    store_out(a, head, q0a, m0, l0, o0, ty, tx);
    if (nt == 2) store_out(a, head, q0b, m1, l1, o1, ty, tx);
}

// ---------------------------------------------------------------- backward: dK, dV per key tile
__global__ void __launch_bounds__(NT, 1) attn_bwd_dkdv_kernel(const AttnArgs a) {
    extern __shared__ __align__(16) float sm[];
    // Kt, Vt; P, dS (natural); [2 buffers][Qt, Q, dOt, dO]
    float *Kt = sm, *Vt = sm + TILE, *Pn = sm + 2 * TILE, *dSn = sm + 3 * TILE, *QD = sm + 4 * TILE;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    const int T = a.T;
    const int64_t head = blockIdx.y;
    const int64_t off = head * T * HD;
    auto load_q = [&](float *dst, int q0) {
        load_tile<true>(dst, a.Q + off, q0, T);
        load_tile<false>(dst + TILE, a.Q + off, q0, T);
        load_tile<true>(dst + 2 * TILE, a.dO + off, q0, T);
        load_tile<false>(dst + 3 * TILE, a.dO + off, q0, T);
    };
    int tl[2];
    const int nt = tiles_of(blockIdx.x, (T + BT - 1) / BT, a.causal, tl);
    for (int w = 0; w < nt; ++w) {
        const int k0 = tl[w] * BT;
        // causal: query tiles from the one holding row k0 on (earlier queries see none of these keys)
        const int qstart = a.causal ? k0 : 0;
        __syncthreads();  // the previous key tile's buffers are no longer read
        load_tile<true>(Kt, a.K + off, k0, T);
        load_tile<true>(Vt, a.V + off, k0, T);
        load_q(QD, qstart);
        cp_commit();
        float dv[4][4] = {}, dk[4][4] = {};
        for (int q0 = qstart, buf = 0; q0 < T; q0 += BT, buf ^= 1) {
            cp_wait_all();
            __syncthreads();  // this tile's Q, dO landed; the other buffer, P and dS are free
            if (q0 + BT < T) load_q(QD + (buf ^ 1) * 4 * TILE, q0 + BT);
            cp_commit();
            const float *Qt = QD + buf * 4 * TILE, *Qn = Qt + TILE, *dOt = Qt + 2 * TILE, *dOn = Qt + 3 * TILE;
            float L2[4], Drow[4], p[4][4], ds[4][4];
            load_L2(a, head, q0, ty, L2);
            row_dots(a, head, q0, ty, tx, Drow);
            probs_and_dS(a, q0, k0, Qt, Kt, dOt, Vt, L2, Drow, p, ds, ty, tx);
            store_n(Pn, p, ty, tx);
            store_n(dSn, ds, ty, tx);
            __syncthreads();  // P and dS complete
            // dV[k][d] += sum_i P[i][k] dO[i][d], dK[k][d] += sum_i dS[i][k] Q[i][d]
            mm64_2(dv, Pn, dOn, dk, dSn, Qn, ty, tx);
        }
        cp_wait_all();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int k = k0 + 4 * ty + r;
            if (k >= T) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                a.dV[off + (int64_t)k * HD + 4 * tx + c] = dv[r][c];
                a.dK[off + (int64_t)k * HD + 4 * tx + c] = dk[r][c] * a.scale;
            }
        }
    }
}

// ---------------------------------------------------------------- backward: dQ per query tile
__global__ void __launch_bounds__(NT, 1) attn_bwd_dq_kernel(const AttnArgs a) {
    extern __shared__ __align__(16) float sm[];
    // Qt, dOt; dS (transposed); [2 buffers][Kt, Vt, K]
    float *Qt = sm, *dOt = sm + TILE, *dSt = sm + 2 * TILE, *KV = sm + 3 * TILE;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    const int T = a.T;
    const int64_t head = blockIdx.y;
    const int64_t off = head * T * HD;
    auto load_k = [&](float *dst, int k0) {
        load_tile<true>(dst, a.K + off, k0, T);
        load_tile<true>(dst + TILE, a.V + off, k0, T);
        load_tile<false>(dst + 2 * TILE, a.K + off, k0, T);
    };
    int tl[2];
    const int nt = tiles_of(blockIdx.x, (T + BT - 1) / BT, a.causal, tl);
    for (int w = 0; w < nt; ++w) {
        const int q0 = tl[w] * BT;
        __syncthreads();  // the previous query tile's buffers are no longer read
        load_tile<true>(Qt, a.Q + off, q0, T);
        load_tile<true>(dOt, a.dO + off, q0, T);
        load_k(KV, 0);
        cp_commit();
        float L2[4], Drow[4];
        load_L2(a, head, q0, ty, L2);
        row_dots(a, head, q0, ty, tx, Drow);
        float dq[4][4] = {};
        const int kend = a.causal ? min(T, q0 + BT) : T;
        for (int k0 = 0, buf = 0; k0 < kend; k0 += BT, buf ^= 1) {
            cp_wait_all();
            __syncthreads();  // this block's K, V landed; the other buffer and dS are free
            if (k0 + BT < kend) load_k(KV + (buf ^ 1) * 3 * TILE, k0 + BT);
            cp_commit();
            const float *Kt = KV + buf * 3 * TILE, *Vt = Kt + TILE, *Kn = Kt + 2 * TILE;
            float p[4][4], ds[4][4];
            probs_and_dS(a, q0, k0, Qt, Kt, dOt, Vt, L2, Drow, p, ds, ty, tx);
            store_t(dSt, ds, ty, tx);
            __syncthreads();  // dS complete
            mm64(dq, dSt, Kn, ty, tx);  // dQ[i][d] += sum_k dS[i][k] K[k][d]
        }
        cp_wait_all();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = q0 + 4 * ty + r;
            if (i >= T) continue;
#pragma unroll
            for (int c = 0; c < 4; ++c) a.dQ[off + (int64_t)i * HD + 4 * tx + c] = dq[r][c] * a.scale;
        }
    }
}

constexpr int FWD_SMEM = 8 * TILE * 4;    // Qt and Pt of both tiles, two buffers of Kt and V
constexpr int DKDV_SMEM = 12 * TILE * 4;  // Kt, Vt, P, dS, two buffers of Qt, Q, dOt, dO
constexpr int DQ_SMEM = 9 * TILE * 4;     // Qt, dOt, dSt, two buffers of Kt, Vt, K

cudaError_t set_smem_once() {
    static cudaError_t err = [] {
        cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DKDV_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
        return e;
    }();
    return err;
}

}  // namespace

bool attention_supported(int64_t heads, int64_t T, int64_t D) {
    return D == HD && T >= 1 && T <= (1 << 24) && heads >= 1 && heads <= 65535;
}

cudaError_t launch_attention_fwd(const float *Q, const float *K, const float *V, float *O, float *L, int64_t heads,
                                 int64_t T, int causal, float scale, cudaStream_t st) {
    const cudaError_t e = set_smem_once();
    if (e != cudaSuccess) return e;
    AttnArgs a{Q, K, V, nullptr, nullptr, nullptr, O, L, nullptr, nullptr, nullptr, (int)T, causal, scale,
               scale * kLog2e};
    const int n = (int)((T + BT - 1) / BT);
    const dim3 grid((unsigned)(causal ? (n + 1) / 2 : n), (unsigned)heads);
    attn_fwd_kernel<<<grid, NT, FWD_SMEM, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attention_bwd(const float *Q, const float *K, const float *V, const float *O, const float *dO,
                                 const float *L, float *dQ, float *dK, float *dV, int64_t heads, int64_t T, int causal,
                                 float scale, cudaStream_t st) {
    const cudaError_t e = set_smem_once();
    if (e != cudaSuccess) return e;
    AttnArgs a{Q, K, V, O, dO, L, nullptr, nullptr, dQ, dK, dV, (int)T, causal, scale, scale * kLog2e};
    const int n = (int)((T + BT - 1) / BT);
    const dim3 grid((unsigned)(causal ? (n + 1) / 2 : n), (unsigned)heads);
    attn_bwd_dkdv_kernel<<<grid, NT, DKDV_SMEM, st>>>(a);
    cudaError_t e2 = cudaGetLastError();
    if (e2 != cudaSuccess) return e2;
    attn_bwd_dq_kernel<<<grid, NT, DQ_SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mm
