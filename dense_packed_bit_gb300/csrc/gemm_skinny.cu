// gemm_skinny.cu -- C = act(op(A) . op(B) + bias), fp32 FFMA, for products with few rows
// (the GPT-2 MLP at small batch: 64 x 768 x 3072), without any workspace.
//
// "I built a GPT-2 in the browser...", section "The kernel sweep": shared-memory
// tiles loaded cooperatively and a 4 x 4 block of outputs per thread in registers;
// "More Stumbling, This Time in the Browser", section "Four answers per worker":
// edge masks and one fixed accumulation order per output.
//
// A product with short M has few output tiles, so one CTA per tile leaves most of
// the GPU idle (64 x 3072 in 64 x 64 tiles: 48 tiles on 152 SMs).  Here the K
// range of each tile is cut over the S CTAs of a thread-block cluster (1, 1, S):
// CTA rank r multiplies K chunks [r c, (r + 1) c) of 32 into a 64 x 64 partial
// tile in its shared memory; after a cluster barrier rank r adds, for its share
// of the tile's outputs, the S partial tiles in rank order (read through
// distributed shared memory), applies the bias and activation, and stores C.
// Every output is therefore the same sum in the same order on every call, and no
// global scratch is touched.  A second cluster barrier keeps every CTA's partial
// tile alive until its peers have read it.
//
// Loads: each chunk of op(A) (64 x 32) and op(B) (32 x 64) is copied by the 256
// threads with the stored matrix's contiguous dimension fastest (coalesced for
// every layout) by cp.async -- 16 bytes per copy when both operands are 16-byte
// aligned with leading dimensions a multiple of four, else 4 -- into shared tiles
// of a 4-stage ring, kept in the
// stored orientation (conflict-free copies), three chunks in flight while one is
// multiplied.
//
// Multiply: thread (tm, tn) owns rows 4 tm .. 4 tm + 3 and four columns: 4 tn .. 4 tn + 3
// when op(B) is kept [k][n] (one 16-byte read gives them), tn + 16 j when it is kept
// [n][k] (then sixteen rows of stride 36 words fall on distinct bank quads).  Every
// operand is read 16 bytes at a time, four k per read along a k-contiguous row, so a
// warp spends three shared-memory wavefronts per k on 16 FMA instructions and the
// FMA pipe, not shared memory, bounds the loop.
#include "mm_common.cuh"
#include "mm_internal.h"

#include <algorithm>
#include <mutex>

namespace mm {
namespace {

constexpr int SB = 64, SKC = 32, NT = 256;  // tile edge, K chunk, threads
constexpr int MAX_SPLIT = 8;                // portable cluster size
constexpr int NSTAGE = 4;                   // chunks in the cp.async ring
constexpr int KP = SKC + 4;                 // padded row of a k-contiguous tile (16-byte rows)
constexpr int OPF = SB * KP;                // floats of one operand chunk (either orientation)
constexpr int SMEM_BYTES = 2 * NSTAGE * OPF * 4;  // 72 KiB (the 16 KiB partial tile reuses it)

// 4-byte asynchronous copy global -> shared; src_bytes 0 zero-fills the destination (the
// source address is then not read).
__device__ __forceinline__ void cp_async4(void *dst, const float *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
// 16-byte asynchronous copy; the bytes past src_bytes (0, 4, 8, 12 or 16) are zero-filled
__device__ __forceinline__ void cp_async16(void *dst, const float *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// VEC: both operands are 16-byte aligned with leading dimensions a multiple of four floats,
// so every group of four elements along the stored contiguous dimension is one 16-byte copy
template <bool TA, bool TB, bool VEC>
__global__ void __launch_bounds__(NT) gemm_skinny_kernel(const GemmArgs g, const int chunks_per_rank) {
    extern __shared__ __align__(16) float sm[];
    // each operand chunk is kept in its stored orientation, so that a warp's copies land on
    // consecutive words: op(A) as [k][m] (A stored K x M) or [m][k + pad] (A stored M x K),
    // op(B) as [k][n] (B stored K x N) or [n][k + pad] (B stored N x K); the padded rows keep
    // the multiply's reads across rows on distinct banks
    float *Abuf = sm, *Bbuf = sm + NSTAGE * OPF;
    float (*P)[SB] = reinterpret_cast<float (*)[SB]>(sm);  // the partial tile, once the ring is idle
    const int tid = threadIdx.x, tm = tid >> 4, tn = tid & 15;
    const uint32_t rank = cluster_ctarank();
    const uint32_t S = gridDim.z;  // the cluster spans the grid's z dimension
    const int64_t m0 = (int64_t)blockIdx.y * SB, n0 = (int64_t)blockIdx.x * SB;
    const int64_t nchunks = (g.K + SKC - 1) / SKC;
    const int64_t c0 = (int64_t)rank * chunks_per_rank;
    const int64_t c1 = nchunks < c0 + chunks_per_rank ? nchunks : c0 + chunks_per_rank;

    // chunk c of op(A) and op(B) into stage st: element e = tid + 256 i of each 64 x 32 block,
    // the stored matrix's contiguous dimension fastest; elements outside the matrices read 0
    // the 16-byte groups: group e = tid + 256 i (i = 0, 1) of each operand chunk, rows of 8
    // groups when k is the contiguous dimension, of 16 groups when m (n) is
    auto issue_vec = [&](int64_t c, int st) {
        const int64_t k0 = c * SKC;
        float *as = Abuf + st * OPF, *bs = Bbuf + st * OPF;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int e = tid + NT * i;
            int mm, kk, nn, kb;
            if (TA) { kk = e >> 4; mm = (e & 15) * 4; } else { mm = e >> 3; kk = (e & 7) * 4; }
            if (TB) { nn = e >> 3; kb = (e & 7) * 4; } else { kb = e >> 4; nn = (e & 15) * 4; }
            const int64_t m = m0 + mm, ka = k0 + kk, n = n0 + nn, kq = k0 + kb;
            // elements of the group inside the matrix (a prefix of the group)
            const int64_t ra = TA ? (ka < g.K ? g.M - m : 0) : (m < g.M ? g.K - ka : 0);
            const int64_t rb = TB ? (n < g.N ? g.K - kq : 0) : (kq < g.K ? g.N - n : 0);
            const int ba = ra <= 0 ? 0 : ra >= 4 ? 16 : (int)ra * 4;
            const int bb = rb <= 0 ? 0 : rb >= 4 ? 16 : (int)rb * 4;
            float *da = TA ? as + kk * SB + mm : as + mm * KP + kk;
            float *db = TB ? bs + nn * KP + kb : bs + kb * SB + nn;
            cp_async16(da, ba ? (TA ? g.A + ka * g.lda + m : g.A + m * g.lda + ka) : g.A, ba);
            cp_async16(db, bb ? (TB ? g.B + n * g.ldb + kq : g.B + kq * g.ldb + n) : g.B, bb);
        }
    };
    auto issue = [&](int64_t c, int st) {
        if (VEC) {
            issue_vec(c, st);
            return;
        }
        const int64_t k0 = c * SKC;
        float *as = Abuf + st * OPF, *bs = Bbuf + st * OPF;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = tid + NT * i;
            int mm, kk, nn, kb;
            if (TA) { kk = e >> 6; mm = e & 63; } else { mm = e >> 5; kk = e & 31; }
            if (TB) { nn = e >> 5; kb = e & 31; } else { kb = e >> 6; nn = e & 63; }
            const int64_t m = m0 + mm, ka = k0 + kk, n = n0 + nn, kq = k0 + kb;
            const bool ina = m < g.M && ka < g.K, inb = n < g.N && kq < g.K;
            float *da = TA ? as + kk * SB + mm : as + mm * KP + kk;
            float *db = TB ? bs + nn * KP + kb : bs + kb * SB + nn;
            cp_async4(da, ina ? (TA ? g.A + ka * g.lda + m : g.A + m * g.lda + ka) : g.A, ina ? 4 : 0);
            cp_async4(db, inb ? (TB ? g.B + n * g.ldb + kq : g.B + kq * g.ldb + n) : g.B, inb ? 4 : 0);
        }
    };

    float acc[4][4] = {};
    // column jj of this thread
    auto col = [&](int jj) { return TB ? tn + 16 * jj : 4 * tn + jj; };
    const int64_t nc = c1 - c0;
    // NSTAGE - 1 chunks in flight ahead of the one being multiplied (empty groups past the end)
#pragma unroll
    for (int j = 0; j < NSTAGE - 1; ++j) {
        if (j < nc) issue(c0 + j, j);
        cp_async_commit();
    }
    for (int64_t j = 0; j < nc; ++j) {
        cp_async_wait<NSTAGE - 2>();  // chunk j has landed (this thread's copies)
        __syncthreads();              // everyone's copies of chunk j; chunk j - 1 no longer read
        if (j + NSTAGE - 1 < nc) issue(c0 + j + NSTAGE - 1, (int)((j + NSTAGE - 1) % NSTAGE));
        cp_async_commit();
        const int st = (int)(j % NSTAGE);
        const float *as = Abuf + st * OPF, *bs = Bbuf + st * OPF;
#pragma unroll
        for (int kq = 0; kq < SKC; kq += 4) {
            float a[4][4], b[4][4];  // a[i][t] = op(A)[4 tm + i][kq + t], b[t][jj] = op(B)[kq + t][col(jj)]
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if (TA) {
                    const float4 v = *reinterpret_cast<const float4 *>(as + (kq + t) * SB + 4 * tm);
                    a[0][t] = v.x, a[1][t] = v.y, a[2][t] = v.z, a[3][t] = v.w;
                } else {
                    const float4 v = *reinterpret_cast<const float4 *>(as + (4 * tm + t) * KP + kq);
                    a[t][0] = v.x, a[t][1] = v.y, a[t][2] = v.z, a[t][3] = v.w;
                }
                if (TB) {
                    const float4 v = *reinterpret_cast<const float4 *>(bs + col(t) * KP + kq);
                    b[0][t] = v.x, b[1][t] = v.y, b[2][t] = v.z, b[3][t] = v.w;
                } else {
                    const float4 v = *reinterpret_cast<const float4 *>(bs + (kq + t) * SB + 4 * tn);
                    b[t][0] = v.x, b[t][1] = v.y, b[t][2] = v.z, b[t][3] = v.w;
                }
            }
            // packed f32x2 FMAs (two outputs per instruction, each rounded once) pair columns when
            // op(B) is read along n, rows when op(A) is read along m; plain FFMAs otherwise
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                if constexpr (!TB) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int jp = 0; jp < 2; ++jp)
                            fma2_bcast(acc[i][2 * jp], acc[i][2 * jp + 1], a[i][t], b[t][2 * jp], b[t][2 * jp + 1]);
                } else if constexpr (TA) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                        for (int ip = 0; ip < 2; ++ip)
                            fma2_bcast(acc[2 * ip][jj], acc[2 * ip + 1][jj], b[t][jj], a[2 * ip][t], a[2 * ip + 1][t]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(a[i][t], b[t][jj], acc[i][jj]);
                }
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // the ring is idle: the partial tile takes its place
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (TB) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) P[4 * tm + i][col(jj)] = acc[i][jj];
        } else {
            *reinterpret_cast<float4 *>(&P[4 * tm + i][4 * tn]) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
    }
    cluster_sync();  // every partial tile of the cluster is complete and visible

    // rank r adds the S partial tiles for its share of the tile's 1,024 float4 groups
    const int per = (SB * SB / 4 + (int)S - 1) / (int)S;
    const int q0 = (int)rank * per, q1 = SB * SB / 4 < q0 + per ? SB * SB / 4 : q0 + per;
    const uint32_t pbase = smem_u32(&P[0][0]);
    for (int q = q0 + tid; q < q1; q += NT) {
        const int i = q >> 4, j = (q & 15) * 4;
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        for (uint32_t p = 0; p < S; ++p) {
            const float4 v = ld_cluster_v4(cluster_map(pbase + (uint32_t)(i * SB + j) * 4u, p));
            sum.x += v.x;
            sum.y += v.y;
            sum.z += v.z;
            sum.w += v.w;
        }
        const int64_t m = m0 + i;
        if (m >= g.M) continue;
        const float s4[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int64_t n = n0 + j + jj;
            if (n >= g.N) continue;
            float z = s4[jj];
            if (g.bias) z += g.bias[n];
            g.C[m * g.ldc + n] = g.act ? gelu_tanh_f(z) : z;
        }
    }
    cluster_sync();  // peers have read this CTA's partial tile
}

}  // namespace

int gemm_skinny_split(int64_t M, int64_t N, int64_t K, int sms) {
    const int64_t tiles = ((N + SB - 1) / SB) * ((M + SB - 1) / SB);
    const int64_t nchunks = (K + SKC - 1) / SKC;
    // about three CTAs per SM (each holds 64 KiB of shared memory), at most the portable cluster
    int64_t s = std::max<int64_t>(1, (3 * (int64_t)sms) / std::max<int64_t>(1, tiles));
    s = std::min<int64_t>({s, (int64_t)MAX_SPLIT, nchunks});
    // no rank without K: the chunks per rank decide the ranks
    const int64_t per = (nchunks + s - 1) / s;
    return (int)((nchunks + per - 1) / per);
}

bool gemm_skinny_supported(const GemmArgs &g) {
    return (g.M + SB - 1) / SB <= 65535 && (g.N + SB - 1) / SB <= 2147483647;
}

cudaError_t launch_gemm_skinny(const GemmArgs &g, int split, cudaStream_t st) {
    if (!gemm_skinny_supported(g)) return cudaErrorInvalidConfiguration;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t nchunks = (g.K + SKC - 1) / SKC;
    int s = split > 0 ? (int)std::min<int64_t>(split, nchunks) : gemm_skinny_split(g.M, g.N, g.K, sms);
    const int per = (int)((nchunks + s - 1) / s);
    s = (int)((nchunks + per - 1) / per);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)((g.N + SB - 1) / SB), (unsigned)((g.M + SB - 1) / SB), (unsigned)s);
    lc.blockDim = dim3(NT);
    lc.dynamicSmemBytes = SMEM_BYTES;
    lc.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = (unsigned)s;
    lc.attrs = attr;
    lc.numAttrs = 1;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        const void *k[8] = {(const void *)gemm_skinny_kernel<false, false, false>,
                            (const void *)gemm_skinny_kernel<false, true, false>,
                            (const void *)gemm_skinny_kernel<true, false, false>,
                            (const void *)gemm_skinny_kernel<true, true, false>,
                            (const void *)gemm_skinny_kernel<false, false, true>,
                            (const void *)gemm_skinny_kernel<false, true, true>,
                            (const void *)gemm_skinny_kernel<true, false, true>,
                            (const void *)gemm_skinny_kernel<true, true, true>};
        for (const void *f : k) {
            const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            if (e != cudaSuccess) attr_err = e;
        }
    });
    if (attr_err != cudaSuccess) return attr_err;
    const bool vec = ((uintptr_t)g.A % 16 == 0) && ((uintptr_t)g.B % 16 == 0) && g.lda % 4 == 0 && g.ldb % 4 == 0;
    if (vec) {
        if (g.transA && g.transB) return cudaLaunchKernelEx(&lc, gemm_skinny_kernel<true, true, true>, g, per);
        if (g.transA) return cudaLaunchKernelEx(&lc, gemm_skinny_kernel<true, false, true>, g, per);
        if (g.transB) return cudaLaunchKernelEx(&lc, gemm_skinny_kernel<false, true, true>, g, per);
        return cudaLaunchKernelEx(&lc, gemm_skinny_kernel<false, false, true>, g, per);
    }
    if (g.transA && g.transB) return cudaLaunchKernelEx(&lc, gemm_skinny_kernel<true, true, false>, g, per);
    if (g.transA) return cudaLaunchKernelEx(&lc, gemm_skinny_kernel<true, false, false>, g, per);
    if (g.transB) return cudaLaunchKernelEx(&lc, gemm_skinny_kernel<false, true, false>, g, per);
    return cudaLaunchKernelEx(&lc, gemm_skinny_kernel<false, false, false>, g, per);
}

}  // namespace mm
