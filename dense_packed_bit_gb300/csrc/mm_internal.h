// mm_internal.h -- host-side interfaces between the C-ABI layer (mm_api.cu)
// and the kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mm {

// ------------------------------------------------------------------ GEMV / packed GEMM

struct PackedArgs {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint16_t *x;  // GEMV: cols entries; GEMM: M x cols
    float *y;           // GEMV: rows entries; GEMM: M x rows
    int64_t M, rows, cols;
    float cb[4];
};

struct GemvConfig {
    int split;          // lanes per row: 4, 8, 16
    int rows_per_lane;  // 1, 2, 4
    int warps;          // warps per CTA
    int dequant;        // 1 select, 2 affine (SIMT), 3 affine (tensor-core mma)
    int pdl;
    int weights_static;
    int independent;
    int staging;        // tensor-core decode: 1 = codes brought to shared memory by TMA
    int blocks_per_cta; // staging and fp8 decode: 64-row blocks each CTA streams through its TMA ring
};

// 4-bit packed GEMV: codes rows x ceil(cols/2) bytes (low nibble first), 16-entry codebook.
struct Packed4Args {
    const uint8_t *codes;
    const uint16_t *scales;
    const uint16_t *x;
    float *y;
    int64_t rows, cols;
    float cb[16];
};

struct Gemv4Config {
    int pdl;
    int weights_static;
    int independent;
    int staging;         // 1 = TMA-staged table decode, 0 = generic kernel
    int blocks_per_cta;  // staging: 64-row blocks each CTA streams through its TMA ring
};

bool gemv4_lut_supported(const Packed4Args &a);
cudaError_t launch_gemv_packed4(const Packed4Args &a, const Gemv4Config &cfg, cudaStream_t s);
unsigned int gemv4_take_device_error(cudaError_t *err);

// True when cb[c] == cb[0] + c * (cb[1] - cb[0]) holds exactly in fp32 for c = 0..3.
bool codebook_is_affine(const float cb[4]);

// A strided batch of 2-bit GEMVs: matrix b's codes at codes + b codes_stride (bytes), its
// scales, x and y at b times the matching stride in entries (x_stride 0: one x for all).
struct PackedBatch {
    const uint8_t *codes;
    int64_t codes_stride;
    const uint16_t *scales;
    int64_t scales_stride;
    const uint16_t *x;
    int64_t x_stride;
    float *y;
    int64_t y_stride;
    int64_t batch, rows, cols;
    float cb[4];
};
// One launch over the whole batch (staged SIMT affine decode): cols % 512 == 0,
// cols <= 4096, 16-byte aligned codes (and codes_stride) and x (x_stride % 8 == 0),
// an affine codebook.
bool gemv_batched_supported(const PackedBatch &p);
cudaError_t launch_gemv_batched(const PackedBatch &p, cudaStream_t s);

// Vectorised path needs cols % 64 == 0, 16-byte aligned codes and x pointers
// and cols small enough for x to sit in shared memory.
bool gemv_vec_supported(const PackedArgs &a);

// Tensor-core GEMV (affine codebooks): cols % 256 == 0, 16-byte aligned codes and x.
bool gemv_mma_supported(const PackedArgs &a);
cudaError_t launch_gemv_mma(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t s);

// Tensor-core GEMV with each CTA's 64 code rows staged in shared memory by TMA:
// cols % 512 == 0, cols <= 4096, 16-byte aligned codes and x.
bool gemv_tma_supported(const PackedArgs &a);
cudaError_t launch_gemv_tma(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t s);
unsigned int gemv_tma_take_device_error(cudaError_t *err);
bool gemv_fp8_supported(const PackedArgs &a);
cudaError_t launch_gemv_fp8(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t s);
unsigned int gemv_fp8_take_device_error(cudaError_t *err);
bool gemv_rows_supported(const PackedArgs &a);
cudaError_t launch_gemv_rows(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t s);
unsigned int gemv_rows_take_device_error(cudaError_t *err);
// 2-bit GEMV on tcgen05 with packed fp4 operands (kind::mxf4): codes in TMEM as e2m1 c/2, x as 14
// exact e2m1 digit pieces; affine codebook, cols % 512 == 0, cols <= 4096, 16-byte aligned codes.
// The batched form runs a strided batch in one launch (tiles_per_cta 0: automatic).
bool gemv_mxf4_supported(const PackedArgs &a);
bool gemv_batched_mxf4_supported(const PackedBatch &p);
cudaError_t launch_gemv_mxf4(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t s);
// cfg: pdl, weights_static and independent as for a single call (the batch is one kernel)
cudaError_t launch_gemv_batched_mxf4(const PackedBatch &p, int tiles_per_cta, const GemvConfig &cfg, cudaStream_t s);
unsigned int gemv_mxf4_take_device_error(cudaError_t *err);
bool gemv_tc_supported(const PackedArgs &a);
cudaError_t launch_gemv_tc(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t s);
unsigned int gemv_tc_take_device_error(cudaError_t *err);

// Launches the GEMV.  Falls back to the bytewise kernel when the vectorised
// path does not apply.  Returns the launch error.
cudaError_t launch_gemv_packed2(const PackedArgs &a, const GemvConfig &cfg, cudaStream_t s);

// Skinny packed GEMM (M >= 1), FFMA on shared-memory tiles: any shape, any codebook.
cudaError_t launch_gemm_packed2(const PackedArgs &a, int tile, cudaStream_t s);

// Skinny packed GEMM on tcgen05 tensor cores: codebook entries exact in fp16,
// cols % 8 == 0, 16-byte aligned X.  tile = W rows per CTA (32, 64, 128) or 0;
// splitk = CTAs of a cluster sharing K (1, 2, 4, 8) or 0 for automatic.
bool gemm_packed2_tc_supported(const PackedArgs &a);
cudaError_t launch_gemm_packed2_tc(const PackedArgs &a, int tile, int splitk, cudaStream_t s);
unsigned int gemm_packed2_tc_take_device_error(cudaError_t *err);

// Skinny packed GEMM with the decoded weights as the MMA's A operand (128 W rows
// per CTA) and the tokens as its N (up to 256): fp16-exact codebook, cols % 64 == 0,
// 16-byte aligned codes and X; K split over a cluster of `splitk` CTAs (0 = auto).
int gemm_packed2_tcw_split(int64_t M, int64_t rows, int64_t cols, int sms);
bool gemm_packed2_tcw_fits(int64_t M, int64_t cols, int splitk);  // a share of K fits one CTA
bool gemm_packed2_tcw_supported(const PackedArgs &a);
cudaError_t launch_gemm_packed2_tcw(const PackedArgs &a, int splitk, int pdl, int weights_static, cudaStream_t s);
unsigned int gemm_packed2_tcw_take_device_error(cudaError_t *err);

// Tile 3: decoded weights in tensor memory as the MMA's A (128 features per CTA as
// M), ntok tokens as N, a pipelined ring over K atoms, K split over a (1, 1, S)
// cluster (S = 1, 2, 4, 8).  fp16-exact codebook, cols % 64 == 0, 16-byte aligned
// codes and X.  ntok = 0 / splitk = 0: automatic (gemm_packed2_tcr_shape).
bool gemm_packed2_tcr_supported(const PackedArgs &a);
// capacity[i]: CTAs the GPU holds at once in clusters of 2^i
void gemm_packed2_tcr_shape(int64_t M, int64_t rows, int64_t cols, const int capacity[4], int *ntok, int *splitk);
cudaError_t launch_gemm_packed2_tcr(const PackedArgs &a, int ntok, int splitk, int pdl, int weights_static,
                                    cudaStream_t s);
unsigned int gemm_packed2_tcr_take_device_error(cudaError_t *err);

// ------------------------------------------------------------------ dense GEMM

struct GemmArgs {
    int transA, transB;
    int64_t M, N, K;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
    // epilogue (the warp-specialised and the plain tiled kernels): C = act(op(A) op(B) + bias),
    // bias one fp32 per column of C or null, act 0 = none, 1 = GELU (tanh form)
    const float *bias = nullptr;
    int act = 0;
};

// GELU in the tanh form GPT-2 uses: z/2 (1 + tanh(u)), u = sqrt(2/pi) (z + 0.044715 z^3).
// Since (1 + tanh(u)) / 2 = 1 / (1 + e^(-2u)), it is z / (1 + e^(-2u)): one exponential and
// one division, no branch, so that a thread's 32 outputs evaluate side by side.  Relative
// error a few ulp where e^(-2u) is moderate; the exponent is capped at 80 so the divisor
// stays below 2^126 (z e^-80 < 2e-35 |z| is the result's size beyond the cap).
__device__ __forceinline__ float gelu_tanh_f(float z) {
    const float u = 0.7978845608028654f * (z + 0.044715f * z * z * z);
    return __fdividef(z, 1.0f + __expf(fminf(-2.0f * u, 80.0f)));
}

// Plain shared-memory tiled FFMA kernel: any sizes, strides and alignment.
cudaError_t launch_gemm_simple(const GemmArgs &g, cudaStream_t s);

// FFMA kernel for few rows of C: 64 x 64 tiles whose K range is split over a thread-block
// cluster of `split` CTAs (0: automatic), partial tiles added in rank order through
// distributed shared memory; any sizes, strides and alignment, no workspace.
int gemm_skinny_split(int64_t M, int64_t N, int64_t K, int sms);
bool gemm_skinny_supported(const GemmArgs &g);
cudaError_t launch_gemm_skinny(const GemmArgs &g, int split, cudaStream_t s);

// Few rows of C on the tensor cores (3xTF32): C computed transposed with 128 columns of C per
// CTA as the MMA's M and the rows (M <= 64) as its N, the K range split over a (split, 1, 1)
// cluster (0: automatic), partial tiles added in rank order through distributed shared
// memory.  Needs the 3xTF32 operand rules and K <= kTf32x3MaxK.
int gemm_skinny_tc_split(int64_t M, int64_t N, int64_t K, int sms);
bool gemm_skinny_tc_supported(const GemmArgs &g);
cudaError_t launch_gemm_skinny_tc(const GemmArgs &g, int split, cudaStream_t s);
unsigned int gemm_skinny_tc_take_device_error(cudaError_t *err);

// TMA-staged register-blocked FFMA kernel.  Needs 16-byte aligned A, B and
// leading dimensions that are multiples of 4.  Returns cudaErrorNotSupported
// when the arguments do not fit.
bool gemm_ffma_supported(const GemmArgs &g);
cudaError_t launch_gemm_ffma(const GemmArgs &g, int tile, cudaStream_t s);

// The same kernel with a stream-K tail: the first dp_tiles 128 x 128 tiles whole, one per CTA,
// then the k-steps of the remaining tiles cut evenly over sk_ctas CTAs (each share shorter than
// one tile's K range), whose partial tiles (two workspace slots of 128 x 128 floats per CTA) a
// second kernel adds in K order into C (no bias or activation).  ffma_streamk_plan gives the split for `ctas` resident
// CTAs (one per SM: the kernel's shared memory admits one), splitting a last wave of at most
// max_tail_pct % of the CTAs; false = no tail to split (the plan is then zero and the plain
// launch runs).
constexpr int kFfmaStreamKMinSteps = 8;     // k-steps of 32 per share, at least
constexpr int kFfmaStreamKAutoTailPct = 85; // automatic: a last wave fuller than this runs as it is
struct FfmaStreamKPlan {
    int tiles_n, dp_tiles, sk_ctas;
    int64_t sk_iters;          // k-steps of the tail tiles, laid end to end
    int64_t workspace_floats;  // 2 * sk_ctas * 128 * 128
};
bool ffma_streamk_plan(int64_t M, int64_t N, int64_t K, int ctas, int max_tail_pct, FfmaStreamKPlan *plan);
cudaError_t launch_gemm_ffma_streamk(const GemmArgs &g, const FfmaStreamKPlan &plan, float *ws, cudaStream_t s);

// 3xTF32 tcgen05 kernels: same operand requirements as the FFMA TMA kernel.
// launch_gemm_tf32x3: one 128 x 128 tile per CTA, two stages, all threads split
// and wait together; launch_gemm_tf32x3_ws: persistent, warp-specialised,
// raw tiles used as the hi operands, 128 x 256 tiles per CTA (pair = 0) or
// 256 x 256 tiles per pair of CTAs sharing each MMA (pair = 1).
bool gemm_tf32x3_supported(const GemmArgs &g);
cudaError_t launch_gemm_tf32x3(const GemmArgs &g, cudaStream_t s);
cudaError_t launch_gemm_tf32x3_ws(const GemmArgs &g, int pair, cudaStream_t s);
// Split-K form: ksplit slices per output tile computed into ws (ksplit * M * N floats,
// 16-byte aligned), then summed in slice order into C by a second kernel.
// ksplit == kStreamK: stream-K instead, ws holding the units' partial-tile slots and flags.
// Attention (attention_fa2.cu): [heads][T][64] fp32, forward O and L, backward dQ/dK/dV.
bool attention_supported(int64_t heads, int64_t T, int64_t D);
cudaError_t launch_attention_fwd(const float *Q, const float *K, const float *V, float *O, float *L, int64_t heads,
                                 int64_t T, int causal, float scale, cudaStream_t st);
cudaError_t launch_attention_bwd(const float *Q, const float *K, const float *V, const float *O, const float *dO,
                                 const float *L, float *dQ, float *dK, float *dV, int64_t heads, int64_t T, int causal,
                                 float scale, cudaStream_t st);

constexpr int kStreamK = -1;

// Longest K one 3xTF32 accumulation may cover.  The tensor core's fp32 accumulation error
// grows like sqrt(K): worst |C - C_ref| / sum_k |a_ik b_kj| measured 3.3e-6 at K = 2048 and
// 5.2e-6 at K = 8192 (N(0, 0.02) operands), so about 7.4e-6 at 16,384 and past the 1e-5
// bound near 3e4.  A longer K runs the FFMA kernels (fp32 FMA, one rounding per step) or,
// in the split entry points, K slices of at most this length added in fp32.
constexpr int64_t kTf32x3MaxK = 16384;
cudaError_t launch_gemm_tf32x3_ws_splitk(const GemmArgs &g, int pair, int ksplit, float *ws, cudaStream_t s);
int gemm_splitk_auto(int64_t M, int64_t N, int64_t K, int pair, int sms);
int64_t gemm_splitk_workspace_floats(int64_t M, int64_t N, int64_t K, int pair, int split, int sms);

// The static scratch of the split-K entry point that allocates nothing: its device
// address on the current device (looked up on the first call per device) and size.
constexpr int64_t kSplitkStaticFloats = 4194304;  // 16 MiB; mm.h states the same limit
cudaError_t splitk_static_scratch(float **ptr, int64_t *floats);

// Per translation unit device error words (read and cleared).
unsigned int gemm_ffma_take_device_error(cudaStream_t s, cudaError_t *err);
unsigned int gemm_tf32x3_take_device_error(cudaError_t *err);
unsigned int gemm_tf32x3_ws_take_device_error(cudaError_t *err);

// Failure-detection probe (wait_probe.cu): one bounded mbarrier wait with a caller-chosen
// limit, arriving first or never; out (device, may be null) receives {completed, ns waited}.
cudaError_t launch_wait_probe(int arrive, unsigned long long limit_ns, unsigned long long *out, cudaStream_t s);
unsigned int wait_probe_take_device_error(cudaError_t *err);

}  // namespace mm
