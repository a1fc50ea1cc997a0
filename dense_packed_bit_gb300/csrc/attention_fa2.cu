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
// GB300 form.  A CTA of 256 threads owns a 64-row tile; K/V (or Q/dO) tiles of
// 64 rows pass through shared memory, rows padded to 65 words so that every
// access of the products below -- by rows or by columns -- falls on distinct
// banks or is a broadcast.  Thread (ty, tx) = (tid / 16, tid % 16) holds
// outputs (ty + 16 r, tx + 16 c), r, c = 0..3, of every 64 x 64 product, so
// the 16 threads of a half-warp hold whole rows: the softmax's row maximum and
// row sum are 4-step shuffles within the half-warp.  Scores are kept in base-2
// units (scale * log2(e) folded into one multiply), so each probability is one
// exp2.
//
// The backward is split in two kernels so that every gradient is a sum in a
// fixed order (no atomics): one CTA per key tile accumulates dK and dV over the
// query tiles, one CTA per query tile accumulates dQ over the key tiles; both
// rebuild P and dS = P (dP - D) with D_i = dO_i . O_i from identical products,
// in identical order.  Causal attention skips the blocks above the diagonal.
#include "mm_common.cuh"
#include "mm_internal.h"

#include <math.h>

namespace mm {

namespace {

constexpr int HD = 64;     // head dimension
constexpr int BT = 64;     // rows per tile (queries or keys)
constexpr int TS = BT + 1; // padded shared-memory row
constexpr int TILE = BT * TS;
constexpr int NT = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// acc[r][c] += sum_t a(ty + 16 r, t) b(t, tx + 16 c), t = 0..63 in order
template <class FA, class FB>
__device__ __forceinline__ void mm64(float (&acc)[4][4], int ty, int tx, FA a, FB b) {
#pragma unroll 4
    for (int t = 0; t < BT; ++t) {
        float av[4], bv[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) av[r] = a(ty + 16 * r, t);
#pragma unroll
        for (int c = 0; c < 4; ++c) bv[c] = b(t, tx + 16 * c);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
}

// rows row0 .. row0 + 63 of a [T][64] matrix into a padded tile; rows past T read 0
__device__ __forceinline__ void load_tile(float *dst, const float *src, int64_t row0, int T) {
    for (int e = threadIdx.x; e < BT * HD; e += NT) {
        const int r = e >> 6, d = e & 63;
        const int64_t row = row0 + r;
        dst[r * TS + d] = row < T ? __ldg(src + row * HD + d) : 0.f;
    }
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

// ---------------------------------------------------------------- forward
__global__ void __launch_bounds__(NT, 3) attn_fwd_kernel(const AttnArgs a) {
    extern __shared__ float sm[];
    float *Qs = sm, *Ks = sm + TILE, *Vs = sm + 2 * TILE, *Ps = sm + 3 * TILE;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    const int T = a.T;
    const int64_t head = blockIdx.y;
    const int q0 = blockIdx.x * BT;
    const float *Qh = a.Q + head * T * HD, *Kh = a.K + head * T * HD, *Vh = a.V + head * T * HD;
    load_tile(Qs, Qh, q0, T);

    float m[4], l[4], o[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) o[r][c] = 0.f;
    }
    const int kend = a.causal ? min(T, q0 + BT) : T;  // keys past the tile's last query are masked
    for (int k0 = 0; k0 < kend; k0 += BT) {
        __syncthreads();  // the previous block's K, V and P are no longer read
        load_tile(Ks, Kh, k0, T);
        load_tile(Vs, Vh, k0, T);
        __syncthreads();
        float s[4][4] = {};
        mm64(s, ty, tx, [&](int i, int t) { return Qs[i * TS + t]; }, [&](int t, int j) { return Ks[j * TS + t]; });
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = q0 + ty + 16 * r;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int k = k0 + tx + 16 * c;
                s[r][c] = allowed(i, k, T, a.causal) ? s[r][c] * a.scale2 : -INFINITY;
                mx = fmaxf(mx, s[r][c]);
            }
            const float mnew = fmaxf(m[r], half_max(mx));
            // a row with no allowed key yet (only rows past T) keeps zero weights
            const float alpha = mnew == -INFINITY ? 1.f : exp2f(m[r] - mnew);
            float ls = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float p = mnew == -INFINITY ? 0.f : exp2f(s[r][c] - mnew);
                Ps[(ty + 16 * r) * TS + tx + 16 * c] = p;
                ls += p;
                o[r][c] *= alpha;
            }
            l[r] = l[r] * alpha + ls;
            m[r] = mnew;
        }
        __syncthreads();  // P complete
        mm64(o, ty, tx, [&](int i, int t) { return Ps[i * TS + t]; }, [&](int t, int d) { return Vs[t * TS + d]; });
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + ty + 16 * r;
        const float lrow = half_sum(l[r]);
        if (i >= T) continue;
        const float inv = 1.f / lrow;
        float *orow = a.Out + (head * T + i) * HD;
#pragma unroll
        for (int c = 0; c < 4; ++c) orow[tx + 16 * c] = o[r][c] * inv;
        if (tx == 0) a.Lout[head * T + i] = (m[r] + log2f(lrow)) * kLn2;
    }
}

// D_i = dO_i . O_i for the thread's rows ty + 16 r of the tile at q0 (dOs holds the dO tile)
__device__ __forceinline__ void row_dots(const AttnArgs &a, int64_t head, int q0, const float *dOs, int ty, int tx,
                                         float (&Drow)[4]) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + ty + 16 * r;
        float p = 0.f;
        if (i < a.T) {
            const float *orow = a.O + (head * a.T + i) * HD;
#pragma unroll
            for (int c = 0; c < 4; ++c) p = fmaf(dOs[(ty + 16 * r) * TS + tx + 16 * c], __ldg(orow + tx + 16 * c), p);
        }
        Drow[r] = half_sum(p);
    }
}

// P and dS of the (query tile q0, key tile k0) block, into Ps and dSs as [i][k]
__device__ __forceinline__ void probs_and_dS(const AttnArgs &a, int q0, int k0, const float *Qs, const float *dOs,
                                             const float *Ks, const float *Vs, const float (&L2)[4],
                                             const float (&Drow)[4], float *Ps, float *dSs, int ty, int tx) {
    float s[4][4] = {}, dp[4][4] = {};
    mm64(s, ty, tx, [&](int i, int t) { return Qs[i * TS + t]; }, [&](int t, int j) { return Ks[j * TS + t]; });
    mm64(dp, ty, tx, [&](int i, int t) { return dOs[i * TS + t]; }, [&](int t, int j) { return Vs[j * TS + t]; });
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + ty + 16 * r;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int k = k0 + tx + 16 * c;
            const float p = allowed(i, k, a.T, a.causal) ? exp2f(s[r][c] * a.scale2 - L2[r]) : 0.f;
            Ps[(ty + 16 * r) * TS + tx + 16 * c] = p;
            dSs[(ty + 16 * r) * TS + tx + 16 * c] = p * (dp[r][c] - Drow[r]);
        }
    }
}

// ---------------------------------------------------------------- backward: dK, dV per key tile
__global__ void __launch_bounds__(NT, 2) attn_bwd_dkdv_kernel(const AttnArgs a) {
    extern __shared__ float sm[];
    float *Ks = sm, *Vs = sm + TILE, *Qs = sm + 2 * TILE, *dOs = sm + 3 * TILE, *Ps = sm + 4 * TILE,
          *dSs = sm + 5 * TILE;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    const int T = a.T;
    const int64_t head = blockIdx.y;
    const int k0 = blockIdx.x * BT;
    const int64_t off = head * T * HD;
    load_tile(Ks, a.K + off, k0, T);
    load_tile(Vs, a.V + off, k0, T);
    float dv[4][4] = {}, dk[4][4] = {};
    // causal: query tiles from the one holding row k0 on (earlier queries see none of these keys)
    for (int q0 = a.causal ? k0 : 0; q0 < T; q0 += BT) {
        __syncthreads();  // the previous tile's Q, dO, P and dS are no longer read
        load_tile(Qs, a.Q + off, q0, T);
        load_tile(dOs, a.dO + off, q0, T);
        __syncthreads();
        float L2[4], Drow[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = q0 + ty + 16 * r;
            L2[r] = i < T ? __ldg(a.L + head * T + i) * kLog2e : 0.f;
        }
        row_dots(a, head, q0, dOs, ty, tx, Drow);
        probs_and_dS(a, q0, k0, Qs, dOs, Ks, Vs, L2, Drow, Ps, dSs, ty, tx);
        __syncthreads();  // P and dS complete
        mm64(dv, ty, tx, [&](int k, int t) { return Ps[t * TS + k]; }, [&](int t, int d) { return dOs[t * TS + d]; });
        mm64(dk, ty, tx, [&](int k, int t) { return dSs[t * TS + k]; }, [&](int t, int d) { return Qs[t * TS + d]; });
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int k = k0 + ty + 16 * r;
        if (k >= T) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            a.dV[off + (int64_t)k * HD + tx + 16 * c] = dv[r][c];
            a.dK[off + (int64_t)k * HD + tx + 16 * c] = dk[r][c] * a.scale;
        }
    }
}

// ---------------------------------------------------------------- backward: dQ per query tile
__global__ void __launch_bounds__(NT, 2) attn_bwd_dq_kernel(const AttnArgs a) {
    extern __shared__ float sm[];
    float *Qs = sm, *dOs = sm + TILE, *Ks = sm + 2 * TILE, *Vs = sm + 3 * TILE, *dSs = sm + 4 * TILE,
          *Ps = sm + 5 * TILE;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    const int T = a.T;
    const int64_t head = blockIdx.y;
    const int q0 = blockIdx.x * BT;
    const int64_t off = head * T * HD;
    load_tile(Qs, a.Q + off, q0, T);
    load_tile(dOs, a.dO + off, q0, T);
    __syncthreads();
    float L2[4], Drow[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + ty + 16 * r;
        L2[r] = i < T ? __ldg(a.L + head * T + i) * kLog2e : 0.f;
    }
    row_dots(a, head, q0, dOs, ty, tx, Drow);
    float dq[4][4] = {};
    const int kend = a.causal ? min(T, q0 + BT) : T;
    for (int k0 = 0; k0 < kend; k0 += BT) {
        __syncthreads();  // the previous block's K, V and dS are no longer read
        load_tile(Ks, a.K + off, k0, T);
        load_tile(Vs, a.V + off, k0, T);
        __syncthreads();
        probs_and_dS(a, q0, k0, Qs, dOs, Ks, Vs, L2, Drow, Ps, dSs, ty, tx);
        __syncthreads();  // dS complete
        mm64(dq, ty, tx, [&](int i, int t) { return dSs[i * TS + t]; }, [&](int t, int d) { return Ks[t * TS + d]; });
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + ty + 16 * r;
        if (i >= T) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) a.dQ[off + (int64_t)i * HD + tx + 16 * c] = dq[r][c] * a.scale;
    }
}

constexpr int FWD_SMEM = 4 * TILE * 4;  // Q, K, V, P
constexpr int BWD_SMEM = 6 * TILE * 4;  // six tiles

cudaError_t set_smem_once() {
    static cudaError_t err = [] {
        cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BWD_SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BWD_SMEM);
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
    const dim3 grid((unsigned)((T + BT - 1) / BT), (unsigned)heads);
    attn_fwd_kernel<<<grid, NT, FWD_SMEM, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attention_bwd(const float *Q, const float *K, const float *V, const float *O, const float *dO,
                                 const float *L, float *dQ, float *dK, float *dV, int64_t heads, int64_t T, int causal,
                                 float scale, cudaStream_t st) {
    const cudaError_t e = set_smem_once();
    if (e != cudaSuccess) return e;
    AttnArgs a{Q, K, V, O, dO, L, nullptr, nullptr, dQ, dK, dV, (int)T, causal, scale, scale * kLog2e};
    const dim3 grid((unsigned)((T + BT - 1) / BT), (unsigned)heads);
    attn_bwd_dkdv_kernel<<<grid, NT, BWD_SMEM, st>>>(a);
    cudaError_t e2 = cudaGetLastError();
    if (e2 != cudaSuccess) return e2;
    attn_bwd_dq_kernel<<<grid, NT, BWD_SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mm
