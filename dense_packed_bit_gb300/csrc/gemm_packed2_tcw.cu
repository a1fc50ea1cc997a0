// gemm_packed2_tcw.cu -- Y = X . (diag(scale) W)^T with the decoded weights as
// the A operand of tcgen05.mma and the short batch of activations as its N.
//
// "More Stumbling, This Time in the Browser", sections "This time, in a
// browser" and "The attractive ideas that went away": the 16-layer ternary
// encoder multiplies the activations of 2 x 111 tokens by packed ternary
// weights.  The batch (M = 222) is short and the weight matrices wide (3072 x
// 768 and 768 x 3072), so the contraction is laid out as
//
//     D[f][t] = sum_k Wdec[f][k] . X[t][k]       (f: output feature, t: token)
//
// with 128 features per CTA as the MMA's M, all tokens of a tile (up to 256,
// a multiple of 16: 224 for 222 tokens) as its N and fp16 x fp16 products
// (exact) accumulated in fp32 in tensor memory.  Y[t][f] = scale_f . D[f][t].
//
// A CTA owns one 128-feature tile, one token tile and a contiguous share of
// the K atoms (64 fields each); the CTAs of a (1, 1, S) cluster split K.  Every
// operand of the share is resident at once -- no ring:
//   * one TMA box brings the CTA's code bytes (128 rows x 16 bytes per atom);
//   * one TMA box per atom brings X (tokens x 64 fp16, 128-byte swizzle);
//   * the 128 threads of warps 0-3 each decode one weight row: every code byte
//     indexes a 256-entry table of its four fields' fp16 codebook entries, and
//     each 16-byte chunk goes to its swizzled place in the K-major A tile;
//   * thread 0 issues 4 MMAs (K = 16) per atom and one commit;
//   * warps 0-3 read the accumulator (feature = TMEM lane, token = column).
// Alone (S = 1) each thread scales its feature and stores Y directly: at a
// fixed token the 32 lanes of a warp write 32 consecutive floats.  In a
// cluster, every CTA stages its partial tile in shared memory as [t][f]; CTA r
// then adds, for its 128 / S features and every token, the S partials in rank
// order (ld.shared::cluster; deterministic), scales and stores.
//
// With programmatic dependent launch the prologue (table, TMEM, barriers) and,
// when the weights are promised static, the code load and decode run before
// the wait on the previous kernel; X is read and Y written only after it.
#include "mm_common.cuh"
#include "mm_internal.h"
#include "tcgen05.cuh"
#include "tmap.h"

#include <cuda_fp16.h>

#include <mutex>

namespace mm {

__device__ unsigned int g_tcw_err;

namespace {

constexpr int FM = 128;          // features per CTA: the MMA's M
constexpr int KATOM = 64;        // fp16 along K per 128-byte swizzled row
constexpr int NDEC = 128;        // decode / MMA / epilogue threads (warps 0-3)
constexpr int NTHREADS = NDEC + 32;  // + the TMA warp
constexpr int W_ATOM = FM * 128;     // 16 KiB of decoded weights per atom
constexpr int PST = FM + 8;          // staged partial tile: [t][f], row stride in floats
constexpr int KC_MAX = 8;            // atoms per CTA (shared-memory bound)
constexpr int SMEM_LIMIT = 227 * 1024;

struct TcwParams {
    const uint8_t *codes;
    const uint16_t *scales;
    float *y;
    int M, rows, cols;
    int atoms;  // K atoms of 64 fields
    int kcmax;  // atoms of the largest share (sizes every CTA's shared-memory plan and the code box)
    int ntok;   // tokens per tile = MMA N (multiple of 16, <= 256) = X box rows
    int pdl, weights_static;
    uint32_t cb16[2];
};

// Shared-memory plan for a CTA holding kc atoms of a tile of ntok tokens in a
// cluster of S CTAs.  After the MMAs the operand region is reused for the
// partial tile: pushed (S slices [owner][t][f], each padded by 8 floats against
// bank conflicts, plus S - 1 receive slots for the slices the peers send) when
// that fits, else staged as one [t][f] tile that the owners read remotely.
struct TcwPlan {
    int w_off, x_off, c_off, region, bar_off, lut_off, scale_off, total;
    int push, slice_floats, recv_off;
    __host__ __device__ TcwPlan(int kc, int ntok, int S) {
        w_off = 0;
        x_off = kc * W_ATOM;
        c_off = x_off + kc * ntok * 128;
        const int ring = c_off + kc * FM * 16;
        constexpr int TAIL = 64 + 256 * 8 + FM * 4 + 1024;  // barriers, table, scales, alignment slack
        push = 0;
        slice_floats = 0;
        recv_off = 0;
        int staged = 0;
        if (S > 1) {
            slice_floats = ntok * (FM / S) + 8;
            const int push_need = (2 * S - 1) * slice_floats * 4;
            const int push_region = ((ring > push_need ? ring : push_need) + 1023) / 1024 * 1024;
            push = push_region + TAIL <= SMEM_LIMIT;
            recv_off = S * slice_floats * 4;
            staged = push ? push_need : ntok * PST * 4;
        }
        region = ((ring > staged ? ring : staged) + 1023) / 1024 * 1024;
        bar_off = region;
        lut_off = bar_off + 64;
        scale_off = lut_off + 256 * 8;
        total = scale_off + FM * 4 + 1024;
    }
};

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// 32 columns of this warp's TMEM lane quarter with the wait inside (tmem_ld32),
// or 16 when only 16 are left in the tile.
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

template <bool CLUSTER>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_packed2_tcw_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmC,
                            const TcwParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_aligned<1024>(smem_raw);
    const int S = gridDim.z, z = blockIdx.z;
    const int a0 = (int)((int64_t)z * p.atoms / S), a1 = (int)((int64_t)(z + 1) * p.atoms / S);
    const int kc = a1 - a0;
    const TcwPlan L(p.kcmax, p.ntok, S);
    uint8_t *sW = smem + L.w_off, *sX = smem + L.x_off, *sC = smem + L.c_off;
    uint64_t *bar_c = reinterpret_cast<uint64_t *>(smem + L.bar_off);  // code bytes landed
    uint64_t *bar_x = bar_c + 1;                                        // X landed
    uint64_t *bar_m = bar_c + 2;                                        // MMAs complete
    uint64_t *bar_r = bar_c + 3;                                        // peers' slices received
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_c + 4);
    int *bad = reinterpret_cast<int *>(tmem_slot + 1);
    uint2 *lut = reinterpret_cast<uint2 *>(smem + L.lut_off);
    float *sscale = reinterpret_cast<float *>(smem + L.scale_off);  // fp32 scales of the tile's features

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int f0 = blockIdx.x * FM, t0 = blockIdx.y * p.ntok;

    // byte -> fp16 codebook entries of its 4 fields, in K order
    for (int b = tid; b < 256; b += NTHREADS) {
        uint32_t h[4];
#pragma unroll
        for (int f = 0; f < 4; ++f) {
            const uint32_t c = (b >> (2 * f)) & 3u;
            h[f] = (p.cb16[c >> 1] >> (16 * (c & 1))) & 0xFFFFu;
        }
        lut[b] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar_c, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_m, 1);
        mbar_init(bar_r, 1);
        *bad = 0;
        fence_mbar_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == NDEC / 32) {
        // ---------------------------------------------------------------- TMA
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmC);
            if (!p.weights_static) pdl_wait();
            mbar_arrive_expect_tx(bar_c, (uint32_t)(p.kcmax * FM * 16));  // the whole box
            tma_load_2d(sC, &tmC, bar_c, a0 * 16, f0);
            pdl_wait();  // X may be the previous kernel's output
            // the next call may launch once this one has passed its wait (not before: a chain
            // of calls would otherwise park every later call's CTAs on the SMs)
            if (p.pdl) pdl_launch_dependents();
            mbar_arrive_expect_tx(bar_x, (uint32_t)(kc * p.ntok * 128));
            for (int a = 0; a < kc; ++a) tma_load_2d(sX + a * p.ntok * 128, &tmX, bar_x, (a0 + a) * KATOM, t0);
            // both copies must land before this CTA's shared memory is released
            if (!mbar_wait(bar_c, 0) || !mbar_wait(bar_x, 0)) atomicExch(&g_tcw_err, kDevErrDrain);
        }
    } else {
        // ---------------------------------------------------------------- decode
        const int f = tid;  // weight row of this thread within the tile
        // the scales are weights too: read after the same wait as the codes
        if (!p.weights_static) pdl_wait();
        sscale[f] = f0 + f < p.rows ? h2f(p.scales[f0 + f]) : 0.f;
        if (!mbar_wait(bar_c, 0)) {
            atomicExch(&g_tcw_err, kDevErrWaitFull);
            *bad = 1;
        } else {
            for (int a = 0; a < kc; ++a) {
                const uint4 v = *reinterpret_cast<const uint4 *>(sC + f * (16 * p.kcmax) + 16 * a);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint8_t *dst = sW + a * W_ATOM + f * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint32_t word = w[cc >> 1] >> (16 * (cc & 1));
                    const uint2 lo = lut[word & 0xFF], hi = lut[(word >> 8) & 0xFF];
                    *reinterpret_cast<uint4 *>(dst + ((cc ^ (f & 7)) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
                }
            }
        }
        fence_proxy_async_smem();
        bar_sync(1, NDEC);
        if (tid == 0) {
            if (*bad || !mbar_wait(bar_x, 0)) {
                atomicExch(&g_tcw_err, kDevErrWaitFull);
                *bad = 1;
            } else {
                tc_fence_after_sync();
                const uint32_t idesc = make_idesc(kFmtF16, kFmtF16, (uint32_t)p.ntok, FM);
                const uint32_t wb = smem_u32(sW), xb = smem_u32(sX);
                for (int a = 0; a < kc; ++a)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        umma_f16(tmem, sdesc_kmajor_sw128(wb + a * W_ATOM + 32 * ks),
                                 sdesc_kmajor_sw128(xb + a * p.ntok * 128 + 32 * ks), idesc,
                                 (a > 0 || ks > 0) ? 1u : 0u);
            }
            umma_commit(bar_m);
        }
        pdl_wait();  // Y may still be read by the previous kernel
        if (!mbar_wait(bar_m, 0)) {
            atomicExch(&g_tcw_err, kDevErrWaitMma);
            *bad = 1;
        }
        tc_fence_after_sync();
        bar_sync(1, NDEC);
        const bool ok = !*bad;
        const int feat = f0 + tid;
        if (!CLUSTER) {
            // feature = lane: at a fixed token a warp stores 32 consecutive floats
            const float sc = sscale[tid];
            for (int c0 = 0; c0 < p.ntok; c0 += 32) {
                float v[32];
                tmem_ld_cols(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, p.ntok - c0, v);
                if (ok && feat < p.rows)
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int t = t0 + c0 + j;
                        if (c0 + j < p.ntok && t < p.M) p.y[(int64_t)t * p.rows + feat] = v[j] * sc;
                    }
            }
        } else if (L.push) {
            // partial tile -> own shared memory as one slice per owner, [owner][t][f - owner fs]
            float *stage = reinterpret_cast<float *>(smem);
            const int fs = FM / S;
            float *dst = stage + (tid / fs) * L.slice_floats + (tid % fs);
            for (int c0 = 0; c0 < p.ntok; c0 += 32) {
                float v[32];
                tmem_ld_cols(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, p.ntok - c0, v);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < p.ntok) dst[(c0 + j) * fs] = ok ? v[j] : 0.f;
            }
            if (tid == 0) mbar_arrive_expect_tx(bar_r, (uint32_t)((S - 1) * L.slice_floats * 4));
            fence_proxy_async_smem();
        } else {
            // partial tile -> own shared memory as [t][f] (operands are consumed)
            float *part = reinterpret_cast<float *>(smem);
            for (int c0 = 0; c0 < p.ntok; c0 += 32) {
                float v[32];
                tmem_ld_cols(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, p.ntok - c0, v);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < p.ntok) part[(c0 + j) * PST + tid] = ok ? v[j] : 0.f;
            }
        }
    }

    if (CLUSTER && L.push) {
        // every CTA's MMAs are done (its operand region may now receive) and its slices staged
        cluster_sync();
        const int fs = FM / S, fz = z * fs;
        const float *stage = reinterpret_cast<const float *>(smem);
        const float *recv = reinterpret_cast<const float *>(smem + L.recv_off);
        const uint32_t slice_bytes = (uint32_t)(L.slice_floats * 4);
        if (tid == 0) {
            // my slice for owner q goes to q's receive slot of rank z (slots skip the owner's own rank)
            for (int q = 0; q < S; ++q) {
                if (q == z) continue;
                const uint32_t slot = (uint32_t)(z < q ? z : z - 1);
                bulk_copy_to_cluster(cluster_map(smem_u32(smem + L.recv_off) + slot * slice_bytes, (uint32_t)q),
                                     stage + q * L.slice_floats, slice_bytes, cluster_map(smem_u32(bar_r), (uint32_t)q));
            }
        }
        if (tid < NDEC) {
            if (!mbar_wait(bar_r, 0)) atomicExch(&g_tcw_err, kDevErrWaitFull);
            // sum the S slices of my features in rank order, scale, store
            const int groups = fs / 4, lanes_t = NDEC / groups;
            const int g = tid % groups, tl = tid / groups;
            const int fl = fz + 4 * g;
            const float4 sc = *reinterpret_cast<const float4 *>(sscale + fl);
            for (int t = tl; t < p.ntok; t += lanes_t) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int r = 0; r < S; ++r) {
                    const float *src = r == z ? stage + z * L.slice_floats : recv + (r < z ? r : r - 1) * L.slice_floats;
                    const float4 v = *reinterpret_cast<const float4 *>(src + t * fs + 4 * g);
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                const int tg = t0 + t;
                if (tg >= p.M) continue;
                float *yrow = p.y + (int64_t)tg * p.rows + f0 + fl;
                const float r4[4] = {acc.x * sc.x, acc.y * sc.y, acc.z * sc.z, acc.w * sc.w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (f0 + fl + j < p.rows) yrow[j] = r4[j];
            }
        }
        // my outgoing copies must finish reading my shared memory before it is released
        if (tid == 0) bulk_commit_and_wait_read();
    } else if (CLUSTER) {
        cluster_sync();  // every partial tile is staged and visible to the cluster
        if (tid < NDEC) {
            // CTA z adds, for its FM / S features and every token, the S partials in rank
            // order, reading the peers' tiles remotely
            constexpr int TB = 4;
            const int fs = FM / S, fz = z * fs;
            const int groups = fs / 4;
            const int lanes_t = NDEC / groups;
            const int g = tid % groups, tl = tid / groups;
            const int fl = fz + 4 * g;
            const float4 sc = *reinterpret_cast<const float4 *>(sscale + fl);
            const uint32_t base = smem_u32(smem) + (uint32_t)(fl * 4);
            for (int tb = tl * TB; tb < p.ntok; tb += lanes_t * TB) {
                float4 acc[TB];
#pragma unroll
                for (int u = 0; u < TB; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q = 0; q < S; ++q) {
                    float4 v[TB];
#pragma unroll
                    for (int u = 0; u < TB; ++u)
                        if (tb + u < p.ntok && t0 + tb + u < p.M)
                            v[u] = ld_cluster_v4(cluster_map(base + (uint32_t)((tb + u) * PST * 4), (uint32_t)q));
#pragma unroll
                    for (int u = 0; u < TB; ++u)
                        if (tb + u < p.ntok && t0 + tb + u < p.M) {
                            acc[u].x += v[u].x;
                            acc[u].y += v[u].y;
                            acc[u].z += v[u].z;
                            acc[u].w += v[u].w;
                        }
                }
#pragma unroll
                for (int u = 0; u < TB; ++u) {
                    const int tg = t0 + tb + u;
                    if (tb + u >= p.ntok || tg >= p.M) continue;
                    float *yrow = p.y + (int64_t)tg * p.rows + f0 + fl;
                    const float r4[4] = {acc[u].x * sc.x, acc[u].y * sc.y, acc[u].z * sc.z, acc[u].w * sc.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (f0 + fl + j < p.rows) yrow[j] = r4[j];
                }
            }
        }
        // peers keep their shared memory alive until every CTA has read it.  The arrive has
        // release semantics so that it waits for this CTA's remote loads to be performed: a
        // load whose value goes unused (a token past M) must not still be reading a peer's
        // shared memory when that peer passes the barrier and exits.
        cluster_sync();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

template <bool CLUSTER>
cudaError_t launch_tcw(const CUtensorMap &tx, const CUtensorMap &tc, const TcwParams &p, int ftiles, int ttiles,
                       int splitk, int smem, cudaStream_t st) {
    auto kern = gemm_packed2_tcw_kernel<CLUSTER>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_LIMIT);
        if (attr_err == cudaSuccess && CLUSTER)
            attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    });
    if (attr_err != cudaSuccess) return attr_err;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)ftiles, (unsigned)ttiles, (unsigned)splitk);
    lc.blockDim = dim3(NTHREADS);
    lc.dynamicSmemBytes = (size_t)smem;
    lc.stream = st;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (CLUSTER) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = (unsigned)splitk;
        ++n;
    }
    if (p.pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    lc.attrs = attr;
    lc.numAttrs = n;
    return cudaLaunchKernelEx(&lc, kern, tx, tc, p);
}

bool fp16_exact_bits(float v, uint16_t *bits) {
    const __half h = __float2half_rn(v);
    if (__half2float(h) != v) return false;
    *bits = *reinterpret_cast<const uint16_t *>(&h);
    return true;
}

int ntok_for(int64_t M) {
    const int64_t r = (M + 15) / 16 * 16;
    return (int)(r < 256 ? r : 256);
}

}  // namespace

// Atoms per CTA and cluster size: the smallest power-of-two split whose share of
// atoms fits in shared memory, then doubled while the grid stays within one CTA
// per SM; 0 when no split up to 16 fits.
int gemm_packed2_tcw_split(int64_t M, int64_t rows, int64_t cols, int sms) {
    const int atoms = (int)(cols / KATOM), ntok = ntok_for(M);
    const int64_t tiles = ((rows + FM - 1) / FM) * ((M + ntok - 1) / ntok);
    for (int s = 1; s <= 16; s *= 2) {
        if (s > atoms) return 0;
        const int kc = (atoms + s - 1) / s;
        if (kc > KC_MAX || TcwPlan(kc, ntok, s).total > SMEM_LIMIT) continue;
        while (s < 16 && 2 * s <= atoms && tiles * 2 * s <= sms) s *= 2;
        return s;
    }
    return 0;
}

bool gemm_packed2_tcw_fits(int64_t M, int64_t cols, int splitk) {
    const int atoms = (int)(cols / KATOM);
    if (splitk < 1 || splitk > 16 || splitk > atoms) return false;
    const int kc = (atoms + splitk - 1) / splitk;
    return kc <= KC_MAX && TcwPlan(kc, ntok_for(M), splitk).total <= SMEM_LIMIT;
}

bool gemm_packed2_tcw_supported(const PackedArgs &a) {
    uint16_t b;
    for (int i = 0; i < 4; ++i)
        if (!fp16_exact_bits(a.cb[i], &b)) return false;
    return a.cols % KATOM == 0 && (reinterpret_cast<uintptr_t>(a.x) % 16) == 0 &&
           (reinterpret_cast<uintptr_t>(a.codes) % 16) == 0 && a.M < (1 << 30) && a.rows < (1 << 30) &&
           a.cols < (1 << 30) && (a.M + 255) / 256 < 65536 && gemm_packed2_tcw_split(a.M, a.rows, a.cols, 152) > 0;
}

cudaError_t launch_gemm_packed2_tcw(const PackedArgs &a, int splitk_req, int pdl, int weights_static,
                                    cudaStream_t st) {
    if (!gemm_packed2_tcw_supported(a)) return cudaErrorNotSupported;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    TcwParams p{};
    p.codes = a.codes;
    p.scales = a.scales;
    p.y = a.y;
    p.M = (int)a.M;
    p.rows = (int)a.rows;
    p.cols = (int)a.cols;
    p.atoms = (int)(a.cols / KATOM);
    p.ntok = ntok_for(a.M);
    p.pdl = pdl;
    p.weights_static = pdl ? weights_static : 0;
    uint16_t h[4];
    for (int i = 0; i < 4; ++i) fp16_exact_bits(a.cb[i], &h[i]);
    p.cb16[0] = h[0] | ((uint32_t)h[1] << 16);
    p.cb16[1] = h[2] | ((uint32_t)h[3] << 16);
    int splitk = splitk_req ? splitk_req : gemm_packed2_tcw_split(a.M, a.rows, a.cols, sms);
    if (splitk < 1 || splitk > 16 || splitk > p.atoms) return cudaErrorInvalidValue;
    const int kc_max = (p.atoms + splitk - 1) / splitk;
    p.kcmax = kc_max;
    const TcwPlan L(kc_max, p.ntok, splitk);
    if (kc_max > KC_MAX || L.total > SMEM_LIMIT) return cudaErrorInvalidValue;
    CUtensorMap tx, tc;
    e = make_tmap_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.x, (uint64_t)a.cols, (uint64_t)a.M,
                     (uint64_t)a.cols * 2, KATOM, (uint32_t)p.ntok, CU_TENSOR_MAP_SWIZZLE_128B);
    if (e != cudaSuccess) return e;
    const uint64_t rowbytes = (uint64_t)a.cols / 4;
    e = make_tmap_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.codes, rowbytes, (uint64_t)a.rows, rowbytes,
                     (uint32_t)(16 * kc_max), FM, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
    const int ftiles = (int)((a.rows + FM - 1) / FM), ttiles = (int)((a.M + p.ntok - 1) / p.ntok);
    if (splitk > 1) return launch_tcw<true>(tx, tc, p, ftiles, ttiles, splitk, L.total, st);
    return launch_tcw<false>(tx, tc, p, ftiles, ttiles, 1, L.total, st);
}

unsigned int gemm_packed2_tcw_take_device_error(cudaError_t *err) {
    unsigned int v = 0;
    *err = cudaMemcpyFromSymbol(&v, g_tcw_err, sizeof(v));
    if (*err == cudaSuccess && v != 0) {
        const unsigned int zero = 0;
        *err = cudaMemcpyToSymbol(g_tcw_err, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mm
