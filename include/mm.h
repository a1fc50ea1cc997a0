/*
 * mm.h -- C ABI of libmm: fp32 dense GEMM and packed 2-bit GEMV / skinny GEMM
 * on one NVIDIA GB300 (sm_103a).
 *
 * The two operations:
 *
 *  1. Dense fp32 matrix multiply  C = op(A) . op(B), C overwritten.
 *     "I built a GPT-2 in the browser, then made it 2.6x-12.1x faster",
 *     section "The kernel sweep": the matmul that is about 80% of a GPT-2
 *     training step; one output cell per (row, column) walks the inner
 *     dimension summing products.  The forward pass uses C = A.B (NN); the
 *     backward products are dA = dC.B^T (NT) and dB = A^T.dC (TN).
 *     "More Stumbling, This Time in the Browser", section "Four answers per
 *     worker": rows are tokens, columns output features; edge masks cover
 *     partial tiles; each output accumulates along the inner dimension in one
 *     fixed order, so repeated calls give bit-identical results.
 *
 *  2. Packed 2-bit weights times activations:
 *        Y[m][r] = scale_r * sum_k codebook[field(r, k)] * X[m][k]
 *     "Kernel 0112", section "What is being measured": a 12,288 x 1,536
 *     matrix of weights stored in 2 bits each, times a vector of 1,536
 *     inputs; the work is dominated by reading the 4.5 MiB of weights.
 *     The GEMV is the M = 1 case; the skinny GEMM serves a short batch of
 *     rows ("More Stumbling...", the 16-layer ternary encoder on a 111-token
 *     input with 2 questions).
 *
 *  3. Packed 4-bit weights times a vector (GEMV), the same formula with a
 *     16-entry codebook: "Kernel 0112", section "What the kernel costs in a
 *     whole token" (the model's 4-bit weight-reading kernels, the fastest the
 *     pages measure) and "More Stumbling..." (the packed NF4 path).
 *
 * Layouts (all row-major, all pointers DEVICE memory owned by the caller):
 *  - A: M x K (lda >= K), or K x M when transA (lda >= M).
 *  - B: K x N (ldb >= N), or N x K when transB (ldb >= K).
 *  - C: M x N (ldc >= N).  Leading dimensions count elements.
 *  - codes: rows x ceil(cols/4) bytes.  Element k of a row is the 2-bit field
 *    in byte floor(k/4), bits 2*(k mod 4) and 2*(k mod 4)+1 (little-endian
 *    along K).  Fields of the last byte past `cols` are ignored.
 *  - scales: rows fp16 values, passed as their uint16 bit patterns.
 *  - x / X: fp16 bit patterns, x has cols entries, X is M x cols.
 *  - y / Y: fp32, y has rows entries, Y is M x rows.
 *  - 4-bit codes: rows x ceil(cols/2) bytes; element k of a row is the field in
 *    byte floor(k/2), bits 4*(k mod 2)..4*(k mod 2)+3 (low nibble first).  The
 *    pages give no bit order; this is the 2-bit convention carried over.
 *  - codebook: 4 (2-bit) or 16 (4-bit) fp32 values in HOST memory, read
 *    during the call; every entry must be finite.
 *
 * Arithmetic: fp32 accumulation everywhere.  Every output satisfies
 * |y - y_exact| <= 1e-5 * sum_k |term_k|; decoding of 2-bit fields is exact.
 *
 * Calls are asynchronous on `stream` (NULL = the legacy default stream); the
 * return code covers argument checks and launch errors only.  The library
 * keeps no pointer past a call and allocates no device memory in these calls.
 * Operands must not overlap the output.  Calls from several host threads may
 * run concurrently: the library's shared state is one-time setup (kernel
 * attributes, the device check, the driver entry point that encodes tensor
 * maps) done under std::call_once or a mutex; tensor maps are encoded on the
 * host in each call; the last-error message is per thread.
 *
 * Device-side waits are bounded: a wait that runs out sets a device error word
 * and the kernel returns early; mm_check_device_error() reports it as
 * MM_ERR_TIMEOUT.  No kernel traps.
 */
#ifndef MM_H_
#define MM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *mm_stream_t;

typedef enum {
    MM_OK = 0,
    MM_ERR_INVALID_ARG = 1,  /* null pointer, bad size / leading dim, overlap, bad option */
    MM_ERR_UNSUPPORTED = 2,  /* valid request the library cannot run here (e.g. no sm_103 device) */
    MM_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    MM_ERR_TIMEOUT = 4       /* a kernel's bounded device wait ran out (see mm_check_device_error) */
} mm_status;

/* Version of this ABI: major*10000 + minor*100 + patch. */
int mm_version(void);

/* Message for the last non-MM_OK status returned on this host thread. */
const char *mm_last_error(void);

/*
 * Dense fp32 GEMM, C = op(A) . op(B).  M, N, K >= 1.
 * Kernel: M <= 64 with few output tiles, a few-rows kernel whose K range is split
 * over a thread-block cluster -- on the tensor cores (3xTF32) when A and B are
 * 16-byte aligned with lda, ldb multiples of 4 and K <= 16384, else in FFMA; else
 * the 3xTF32 tensor-core kernel when A and B are 16-byte aligned with lda, ldb multiples of 4
 * and K <= 16384 (its accuracy margin: the tensor core's fp32 accumulation error
 * grows like sqrt(K) and would pass the bound near K = 3e4); else the TMA-staged
 * FFMA kernel, or the plain tiled one for operands TMA cannot describe.
 * Errors: MM_ERR_INVALID_ARG for a null pointer, a dimension < 1, a leading
 * dimension below the stored width, or C overlapping A or B.
 */
mm_status mm_gemm_f32(int transA, int transB, int64_t M, int64_t N, int64_t K,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      float *C, int64_t ldc, mm_stream_t stream);

/*
 * y = W . x for a packed 2-bit W (rows x cols) with per-row fp16 scale.
 * rows, cols >= 1.  Errors: MM_ERR_INVALID_ARG for null pointers, sizes < 1,
 * a null codebook, non-finite codebook entries, or y overlapping an input.
 */
mm_status mm_gemv_packed2(const uint8_t *codes, const uint16_t *scales, const uint16_t *x,
                          float *y, int64_t rows, int64_t cols, const float codebook[4],
                          mm_stream_t stream);

/*
 * Y = X . W^T for a packed 2-bit W (rows x cols), X (M x cols) fp16, Y (M x rows) fp32.
 * M, rows, cols >= 1.  Errors as mm_gemv_packed2.
 */
mm_status mm_gemm_packed2(const uint8_t *codes, const uint16_t *scales, const uint16_t *X,
                          float *Y, int64_t M, int64_t rows, int64_t cols,
                          const float codebook[4], mm_stream_t stream);

/*
 * Waits for `stream`, then reads and clears the device error word set by a
 * kernel whose bounded wait ran out.  Returns MM_OK, MM_ERR_TIMEOUT or
 * MM_ERR_CUDA.
 */
mm_status mm_check_device_error(mm_stream_t stream);

/*
 * Failure-detection probe: exercises the path by which a kernel's bounded
 * device wait reports that it ran out, without breaking any computing kernel.
 * One warp initialises an mbarrier expecting one arrival and waits on its first
 * phase through the wait helper every pipelined kernel uses, with the limit
 * limit_ns in place of the kernels' 2 s.  arrive = 1: the warp arrives first and
 * the wait completes at once.  arrive = 0: nothing can complete the phase, so
 * the wait runs out after limit_ns; the kernel records the timeout in its device
 * error word and returns, and the next mm_check_device_error reports
 * MM_ERR_TIMEOUT and clears the word.  The context stays usable.
 * out: NULL, or 2 uint64 in device memory, 8-byte aligned, written by the kernel:
 * out[0] = 1 if the wait completed, 0 if it ran out; out[1] = the nanoseconds it
 * waited (%globaltimer).  limit_ns: 1,000 .. 100,000,000 (1 us .. 0.1 s).
 * Asynchronous on `stream`.  Errors: MM_ERR_INVALID_ARG for arrive not 0 / 1, a
 * limit out of range or a misaligned out; MM_ERR_UNSUPPORTED without an sm_103
 * device; MM_ERR_CUDA if the launch fails.
 */
mm_status mm_probe_bounded_wait(int arrive, uint64_t limit_ns, uint64_t *out, mm_stream_t stream);

/*
 * Scaled dot-product attention of a GPT-2 training step, in the Flash-Attention-2
 * form of "I built a GPT-2 in the browser, then made it 2.6x-12.1x faster",
 * section "Flash Attention 2": per head, S = scale * Q K^T (keys after the query
 * masked when causal = 1), P = softmax over each row of S, O = P V, and
 * L[i] = log sum_k exp(S[i][k]) (the forward's m + log(l)), from which the
 * backward rebuilds P without storing it.
 *
 * Q, K, V, O (and dO, dQ, dK, dV): heads x T x D fp32, row-major, contiguous
 * (a batch of B sequences of H heads is heads = B * H); L: heads x T fp32.  All
 * device memory owned by the caller, 4-byte aligned; outputs must not overlap
 * inputs or each other.  D = 64 (GPT-2's head dimension); T >= 1; causal 0 or
 * 1; scale finite (usually 1 / sqrt(D)).  Asynchronous on `stream`.
 *
 * mm_attention_fwd writes O and L.  mm_attention_bwd takes the forward's O and L
 * and the gradient dO of a loss with respect to O, and writes dQ, dK, dV
 * (every element, so their contents on entry do not matter).  Every output is a
 * sum in a fixed order: bit-reproducible run to run.  Bound, per output, against
 * the fp64 definition: |err| <= 1e-5 * T_out, T_out the sum of the magnitudes of
 * the terms of the output's last contraction with the earlier sums taken in
 * magnitude (O: sum_k P |V|; dV: sum_i P |dO|; dQ, dK: scale sum P (|dP| + |D|)
 * |K| or |Q|, |dP| = sum_d |dO V|, |D| = sum_d |dO O|); L within 1e-5 (1 + |L|).
 * Errors: MM_ERR_INVALID_ARG for NULL or misaligned pointers, sizes < 1, causal
 * not 0/1, a non-finite scale or overlapping outputs; MM_ERR_UNSUPPORTED for
 * D != 64 or T > 2^24 or heads > 65535.
 */
mm_status mm_attention_fwd(const float *Q, const float *K, const float *V, float *O, float *L, int64_t heads,
                           int64_t T, int64_t D, int causal, float scale, mm_stream_t stream);
mm_status mm_attention_bwd(const float *Q, const float *K, const float *V, const float *O, const float *dO,
                           const float *L, float *dQ, float *dK, float *dV, int64_t heads, int64_t T, int64_t D,
                           int causal, float scale, mm_stream_t stream);

/*
 * GPT-2's linear layer with its MLP activation fused into the GEMM epilogue:
 *     C = act(op(A) . op(B) + bias),   bias[n] added to column n of every row.
 * bias: N fp32 values in device memory, or NULL for none.  act: MM_ACT_NONE or
 * MM_ACT_GELU_TANH, gelu(z) = z/2 (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))) (the
 * pages name GPT-2's step but print no activation; this is GPT-2's own).  Same
 * layouts as mm_gemm_f32; |C - C_exact| <= 1.13e-5 (sum_k |a b| + |bias|) +
 * 2^-20 (1 + |z|), z the exact pre-activation (1.13 bounds gelu's slope).  The
 * 3xTF32 tensor-core kernel runs when A, B, C and their leading dimensions are
 * 16-byte aligned, the general kernel otherwise.  Errors: as mm_gemm_f32, plus
 * MM_ERR_INVALID_ARG for an unknown act or C overlapping bias.
 */
enum { MM_ACT_NONE = 0, MM_ACT_GELU_TANH = 1 };
mm_status mm_gemm_f32_bias_act(int transA, int transB, int64_t M, int64_t N, int64_t K,
                               const float *A, int64_t lda, const float *B, int64_t ldb,
                               const float *bias, int act, float *C, int64_t ldc,
                               mm_stream_t stream);

/*
 * mm_gemm_f32_bias_act with the split of mm_gemm_f32_splitk (same splitk values and
 * workspace, sized by mm_gemm_f32_splitk_workspace): K slices add up in the reduce
 * kernel, which then applies bias and act; with stream-K the segment that completes
 * a tile applies them.  Same bound as mm_gemm_f32_bias_act.  Errors: the union of
 * both calls' errors.
 */
mm_status mm_gemm_f32_bias_act_splitk(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                      const float *A, int64_t lda, const float *B, int64_t ldb,
                                      const float *bias, int act, float *C, int64_t ldc, int splitk,
                                      float *workspace, int64_t workspace_floats,
                                      mm_stream_t stream);

/*
 * Split-K form of mm_gemm_f32 for products with fewer output tiles than the GPU
 * has SMs (short M and N, long K: the GPT-2 MLP shapes at small batch; or a
 * last partial wave, such as 2048^3 on CTA pairs).  splitk = 1..16: K is cut into
 * that many slices, every slice of every output tile is computed by its own CTA
 * into `workspace`, then a second kernel adds the slices in slice order into C.
 * splitk = -1: stream-K -- the tiles' K ranges, laid end to end, are cut evenly
 * over the SMs; the CTA holding the start of a tile's K range adds the partial
 * tiles the other CTAs leave in the workspace (in K order, after their flags).
 * splitk = 0: automatic (no split when the tiles fill the GPU, stream-K when they
 * fill more than half of it, split slices otherwise).  Results are
 * bit-reproducible run to run; they may differ from mm_gemm_f32 in the last bits,
 * by summation order.  Same bound |C - C_exact| <= 1e-5 sum|a b|.  Every 3xTF32
 * accumulation stays within K <= 16384 (mm_gemm_f32): the automatic split uses at
 * least ceil(K / 16384) slices, and a split that would exceed it (fewer slices,
 * stream-K with K > 16384, or K beyond 16 slices of 16384) runs the TMA-staged FFMA
 * kernel unsplit, with a workspace need of 0.
 *
 * workspace: caller-owned device memory, 16-byte aligned, at least the number of
 * floats mm_gemm_f32_splitk_workspace reports for the same M, N, K, splitk
 * (splitk * M * N for slices; one 128 x 256 partial tile per CTA plus a flag
 * word for stream-K; 0 when the split resolves to 1, and NULL is then
 * accepted).  It must not overlap A, B or C; its contents on entry do not
 * matter.  Calls sharing one workspace must not overlap on the GPU.  Operands
 * TMA cannot describe (A or B not 16-byte aligned, lda or ldb not a multiple
 * of 4) run the unsplit general kernel and leave the workspace untouched.
 * Errors: as mm_gemm_f32, plus MM_ERR_INVALID_ARG for splitk outside -1..16, a
 * misaligned, overlapping or too small workspace.
 */
mm_status mm_gemm_f32_splitk_workspace(int64_t M, int64_t N, int64_t K, int splitk, int64_t *floats);

/*
 * The split mm_gemm_f32_splitk takes automatically (splitk = 0) for an M x N x K
 * product on a GPU with `sms` SMs, and the workspace floats it needs, without
 * touching any device: *splitk = 1 (no split), 2..16 (K slices) or -1 (stream-K).
 * For sizing workspaces ahead of time on a known GPU (152 SMs on a GB300).
 * Errors: MM_ERR_INVALID_ARG for sizes < 1, sms < 2 or NULL outputs.
 */
mm_status mm_gemm_f32_split_plan(int64_t M, int64_t N, int64_t K, int sms, int *splitk,
                                 int64_t *workspace_floats);
mm_status mm_gemm_f32_splitk(int transA, int transB, int64_t M, int64_t N, int64_t K,
                             const float *A, int64_t lda, const float *B, int64_t ldb,
                             float *C, int64_t ldc, int splitk, float *workspace,
                             int64_t workspace_floats, mm_stream_t stream);

/*
 * mm_gemm_f32_splitk with no workspace argument and no allocation: the partial
 * tiles go to a scratch array of MM_SPLITK_NOALLOC_MAX_FLOATS floats (16 MiB)
 * that the library holds in device memory of every GPU that loads it, until the
 * process exits.  The pages have no counterpart: this is for callers that cannot
 * call cudaMalloc or hand over a workspace where they multiply (device memory
 * owned by another allocator, such as a framework's caching pool that has
 * reserved what it manages; paths where cudaMalloc's device-wide synchronisation
 * is not acceptable).  Nothing here calls cudaMalloc, cudaFree or any
 * allocating routine.
 *
 * Same arguments, result and errors as mm_gemm_f32_splitk, plus
 * MM_ERR_INVALID_ARG when a given split needs more than
 * MM_SPLITK_NOALLOC_MAX_FLOATS floats (splitk * M * N).  An automatic split that
 * would need more takes the most K slices that fit (at least two; M * N * slices
 * <= MM_SPLITK_NOALLOC_MAX_FLOATS), and otherwise runs unsplit; an automatic
 * stream-K split (one 128 x 256 partial tile per CTA: about 5M floats on a
 * 152-SM GB300) never fits and so runs unsplit.  splitk = -1 is refused.  The
 * first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it for the life of
 * the process: make that first call before any stream capture, and do not call
 * this entry point on a device after cudaDeviceReset of that device (the cached
 * address would be stale).  Every call shares the one array and leaves its partial
 * tiles there.  The caller clears nothing: a call writes every partial tile before
 * reading it.  Calls whose kernels overlap on the GPU (on different streams, or
 * from different threads) race on the array and may return wrong results:
 * serialise them.
 */
#define MM_SPLITK_NOALLOC_MAX_FLOATS 4194304
mm_status mm_gemm_f32_splitk_noalloc(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                     const float *A, int64_t lda, const float *B, int64_t ldb,
                                     float *C, int64_t ldc, int splitk, mm_stream_t stream);

/* ------------------------------------------------------------------------
 * Variant selection for sweeps and tests.  A zeroed struct means "automatic".
 * Every variant computes the same operation to the same bound.
 * ------------------------------------------------------------------------ */

enum {
    MM_GEMM_AUTO = 0,    /* 3xTF32 when A, B are 16-byte aligned and lda, ldb are multiples
                            of 4; the plain tiled FFMA kernel otherwise */
    MM_GEMM_FFMA = 1,    /* TMA-staged, register-blocked fp32 FFMA (plain tiled FFMA kernel
                            when the operands cannot be described by TMA) */
    MM_GEMM_TF32X3 = 2   /* fp32 by the three-term tf32 split (hi*hi + hi*lo + lo*hi) on the
                            tcgen05 tensor cores, TMEM accumulators; same operand rules as AUTO */
};

typedef struct {
    int path;      /* MM_GEMM_* */
    int tile;      /* 0 = automatic, else a path-specific tile id.  3xTF32 (MM_GEMM_AUTO
                      or MM_GEMM_TF32X3 with TMA-describable operands): 1 = one 128 x 128
                      tile per CTA, two stages; 2 = persistent warp-specialised kernel,
                      128 x 256 tiles; 3 = the same with pairs of CTAs (a cluster of 2)
                      sharing 256 x 256 tiles.  Automatic: 3 when M > 128, else 2.
                      MM_GEMM_TF32X3 only: 4 = few rows of C on the tensor cores (M <= 64,
                      K <= 16384: C computed transposed, 128 columns of C per CTA as the
                      MMA's M and the rows as its N, the K range split over a cluster of
                      `splitk` CTAs whose partial tiles are added in rank order through
                      distributed shared memory; no workspace).
                      MM_GEMM_FFMA: 4 = the kernel for few rows of C (64 x 64 FFMA tiles
                      whose K range is split over a thread-block cluster of `splitk` CTAs,
                      partial tiles added in rank order through distributed shared memory:
                      no workspace, any alignment).  Automatic (MM_GEMM_AUTO, tile 0): the
                      3xTF32 tile 4 when M <= 64, the 3xTF32 kernel's 128 x 256 tiles would
                      occupy at most a quarter of the SMs and its operand rules and K margin
                      hold; the FFMA tile 4 for such a product otherwise.  Other values are
                      refused. */
    int splitk;    /* tile 4 (MM_GEMM_FFMA or MM_GEMM_TF32X3): CTAs of the cluster sharing
                      K, 1..8; 0 = automatic (FFMA: about three CTAs per SM; 3xTF32: as many
                      as keep every 128-column tile's cluster within one wave, at least two
                      16-deep K slabs each); other paths: must be 0 */
    int reserved[5];
} mm_gemm_opts;

mm_status mm_gemm_f32_ex(int transA, int transB, int64_t M, int64_t N, int64_t K,
                         const float *A, int64_t lda, const float *B, int64_t ldb,
                         float *C, int64_t ldc, mm_stream_t stream, const mm_gemm_opts *opts);

/*
 * mm_gemm_f32_splitk with a choice of kernel.  opts NULL, or opts->path MM_GEMM_AUTO:
 * exactly mm_gemm_f32_splitk.  opts->path MM_GEMM_FFMA: the TMA-staged register-blocked
 * FFMA kernel ("I built a GPT-2 in the browser...", section "The kernel sweep": shared
 * tiles and register blocks; "More Stumbling...", "Four answers per worker": one fixed
 * accumulation order), 128 x 128 tiles, one CTA per SM.  When the tiles do not fill a
 * whole number of waves, the last wave is partly idle (2048^2: 256 tiles on 152 SMs);
 * with a stream-K tail the first floor(T / SMs) * SMs tiles run whole and the k-steps
 * of the rest, laid end to end, are cut evenly over one CTA per SM, each share leaving
 * its partial tiles (at most two) in the workspace, and a second kernel adds each
 * tile's partial tiles in K order into C.  splitk: 0 = a tail when the last wave is
 * at most 85% full, -1 = a tail whenever there is one, 1 = none; other values are
 * refused for this path.  A share is at least 8 k-steps of 32 and at most one tile's
 * K range, or there is no tail.  opts->tile and opts->splitk must be 0.
 * Workspace: mm_gemm_f32_splitk_workspace_ex with the same opts (2 x SMs x 128 x 128
 * floats with a tail, else 0); same rules as mm_gemm_f32_splitk.  Results are
 * bit-reproducible run to run; with a tail they may differ from the unsplit kernel
 * in the last bits (summation order).  Bound |C - C_exact| <= 1e-5 sum|a b| for any
 * K (fp32 FMA, one rounding per step).  Operands TMA cannot describe run the plain
 * tiled kernel unsplit.  Errors: as mm_gemm_f32_splitk, plus MM_ERR_INVALID_ARG for
 * an unknown path, nonzero opts->tile or opts->splitk, or an FFMA splitk outside -1..1.
 */
mm_status mm_gemm_f32_splitk_ex(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                const float *A, int64_t lda, const float *B, int64_t ldb,
                                float *C, int64_t ldc, int splitk, float *workspace,
                                int64_t workspace_floats, mm_stream_t stream,
                                const mm_gemm_opts *opts);

/* The workspace mm_gemm_f32_splitk_ex needs for the same M, N, K, splitk and opts (the
 * device's SM count decides the FFMA tail).  Errors as mm_gemm_f32_splitk_workspace, plus
 * those of mm_gemm_f32_splitk_ex's options. */
mm_status mm_gemm_f32_splitk_workspace_ex(int64_t M, int64_t N, int64_t K, int splitk,
                                          const mm_gemm_opts *opts, int64_t *floats);

/* mm_gemm_f32_split_plan for mm_gemm_f32_splitk_ex's automatic split (splitk = 0) on a GPU
 * with `sms` SMs, without touching a device; for the FFMA path *splitk = -1 (a stream-K
 * tail) or 1 (none). */
mm_status mm_gemm_f32_split_plan_ex(int64_t M, int64_t N, int64_t K, int sms, const mm_gemm_opts *opts,
                                    int *splitk, int64_t *workspace_floats);

enum {
    MM_DEQ_AUTO = 0,     /* MM_DEQ_AFFINE (TMA-staged when the shape allows), MM_DEQ_SELECT
                            when the codebook is not affine: the fastest measured on GB300 for
                            independent and for chained calls */
    MM_DEQ_SELECT = 1,   /* any codebook: per-field select of the entry, fp32 FMA */
    MM_DEQ_AFFINE = 2,   /* codebook[c] = c0 + c*d exactly (and no zero entry at field 3):
                            fields used in place as exact fp32 subnormals in packed f32x2
                            FMAs, y = scale * (c0 * sum x + d * sum c x) */
    MM_DEQ_MMA = 3,      /* same affine condition, cols % 256 == 0: two fields per integer
                            op become an fp16x2 (1 + c 2^(p-10)) from which one fp16x2
                            subtraction leaves c 2^(p-10) exactly; the multiply-adds run as
                            tensor-core mma.sync (fp16 in, fp32 accumulate) */
    MM_DEQ_FP8 = 4,      /* same affine condition, cols % 512 == 0, cols <= 4096, 16-byte
                            aligned codes and x: one AND turns four fields into exact e4m3
                            operands, x is split exactly into e5m2 pieces, and the
                            multiply-adds run as mma.sync m16n8k32 (fp8 in, fp32 accumulate);
                            code rows are staged by TMA, one warp per 256-field slab */
    MM_DEQ_TC = 5,       /* same affine condition, cols % 512 == 0, cols <= 8192, 16-byte
                            aligned codes and x: the e4m3 field bytes are written to tensor
                            memory as the A operand of tcgen05.mma kind::f8f6f4 (M = 128,
                            K = 32), x as exact e5m2 pieces is the B operand in shared memory,
                            fp32 accumulation in tensor memory; 127 rows per tile, the 128th
                            lane forms sum x with the same MMAs */
    MM_DEQ_MXF4 = 6      /* same affine condition, cols % 512 == 0, cols <= 12800, 16-byte
                            aligned codes: a 2-bit field in the low bits of a nibble is the
                            e2m1 value c/2, so two integer ops per eight fields write the codes
                            to tensor memory as the packed-fp4 A operand of tcgen05.mma
                            kind::mxf4 (M = 128, N = 16, K = 64, unit block scales); x * 2^24
                            is split into 14 balanced radix-8 digits, each digit/2 an exact
                            e2m1 value, as 14 B columns, so every per-digit sum is exact and
                            the only rounding is the fp32 sum over the digits; 127 rows per
                            tile, the 128th lane forms the digit sums of x.  A non-finite x
                            gives NaN in every output.  rows_per_lane: 127-row tiles per CTA,
                            which multiplies three at a time (0 = 3); split, warps and staging
                            must be 0 (staging may be -1) */
};

typedef struct {
    int split;           /* SIMT decodes: lanes sharing one row's dot product (4, 8, 16);
                            MM_DEQ_MMA: warps sharing one row's dot product (1, 2, 3, 4, 6);
                            0 = automatic */
    int rows_per_lane;   /* SIMT decodes: rows each lane carries (1, 2, 4);
                            MM_DEQ_MMA: 16-row blocks each warp carries (1, 2, 4);
                            MM_DEQ_FP8: 64-row blocks each CTA streams (1..64);
                            MM_DEQ_TC: 127-row tiles each CTA multiplies (1..64);
                            0 = automatic */
    int warps;           /* warps per CTA: 0 (auto), 1..16 (MM_DEQ_MMA: a multiple of split,
                            at most 8 when rows_per_lane is 2 or 4; MM_DEQ_FP8 and
                            MM_DEQ_TC: must be 0, like split) */
    int dequant;         /* MM_DEQ_* */
    int pdl;             /* 1: launch with programmatic dependent launch so the
                            kernel's prologue overlaps the previous kernel; it
                            still waits for that kernel before reading x */
    int weights_static;  /* 1: promise that codes and scales are not written by
                            work queued before this call, so their loads may start
                            before the wait on the previous kernel (needs pdl) */
    int independent;     /* 1: promise that no work queued before this call writes
                            codes, scales or x, or reads y: the kernel then never
                            waits for the previous kernel (needs pdl), so back-to-back
                            calls over different matrices overlap completely */
    int staging;         /* MM_DEQ_MMA and MM_DEQ_AFFINE: 1 = code rows arrive in shared
                            memory by TMA (cols % 512 == 0, cols <= 4096; split and warps must
                            be 0).  MM_DEQ_MMA: 64-row blocks through a 2-deep ring per CTA,
                            one warp per 256-field slab, rows_per_lane = 64-row blocks per CTA
                            (0 = 4 for independent calls, 1 otherwise).  MM_DEQ_AFFINE:
                            128-row blocks, one lane per row, eight warps splitting K,
                            rows_per_lane = 128-row blocks per CTA (0 = 3 for independent
                            calls, 1 otherwise).  0 = per-warp register loads; negative =
                            automatic (staged for affine calls when the shape allows, the
                            default without options). */
    int reserved[4];
} mm_gemv_opts;

mm_status mm_gemv_packed2_ex(const uint8_t *codes, const uint16_t *scales, const uint16_t *x,
                             float *y, int64_t rows, int64_t cols, const float codebook[4],
                             mm_stream_t stream, const mm_gemv_opts *opts);

typedef struct {
    int tile;       /* 0 = automatic (tile 3 when the codebook entries are exact in fp16,
                       cols % 64 == 0 and codes and X are 16-byte aligned; else tensor
                       cores with W rows as the MMA's N when the entries are exact in
                       fp16, cols % 8 == 0 and X is 16-byte aligned; else FFMA),
                       1 = FFMA kernel,
                       2 = tensor cores with 128 W rows per CTA as the MMA's M and up to
                       256 rows of X as its N, each CTA's share of K resident at once
                       (fp16-exact codebook, cols % 64 == 0, 16-byte aligned codes and
                       X), 3 = tensor cores with 128 W rows per CTA decoded into tensor
                       memory as the MMA's A, ntok rows of X as its N, a pipelined ring
                       over K (same requirements as 2), 32 / 64 / 128 = tensor cores with
                       that many W rows per CTA as the MMA's N, X rows as its M, a
                       pipelined ring over K */
    int splitk;     /* tensor cores: CTAs of one thread-block cluster that split K and add
                       their partial tiles through distributed shared memory in rank
                       order: 0 (auto), 1, 2, 4, 8; tile 2 also 16; tile 3 at most
                       cols / 64 */
    int pdl;        /* tiles 2 and 3 (and 0 when it picks 3): 1 = launch with
                       programmatic dependent launch; the kernel's prologue overlaps the
                       previous kernel, and it still waits for that kernel before reading
                       X or writing Y */
    int weights_static; /* 1 (needs pdl): promise that codes and scales are not written by
                       work queued before this call, so they may be loaded and decoded
                       before that wait */
    int ntok;       /* tile 3: rows of X per CTA (the MMA's N), a multiple of 16 in
                       16..256; 0 = automatic */
    int reserved[3];
} mm_gemm_packed2_opts;

mm_status mm_gemm_packed2_ex(const uint8_t *codes, const uint16_t *scales, const uint16_t *X,
                             float *Y, int64_t M, int64_t rows, int64_t cols,
                             const float codebook[4], mm_stream_t stream,
                             const mm_gemm_packed2_opts *opts);

/*
 * A strided batch of 2-bit GEMVs, y_b = mm_gemv_packed2(W_b, x_b) for b < batch:
 * matrix b's codes at codes + b * codes_stride (bytes), its scales at scales +
 * b * scales_stride, its x at x + b * x_stride (x_stride 0: one x for every matrix)
 * and its y at y + b * y_stride (entries).  With an affine codebook, cols % 512 ==
 * 0, cols <= 12800, 16-byte aligned codes and codes_stride % 16 == 0 the whole batch
 * runs in one launch of the fp4 tensor-core decode (MM_DEQ_MXF4; each y_b equals bit for
 * bit the single MM_DEQ_MXF4 call's); failing that, with 16-byte aligned x and x_stride %
 * 8 == 0, one launch of the staged SIMT affine kernel (each y_b equals bit for bit the
 * staged single call's); other shapes run one call per matrix.  Same tolerance as
 * mm_gemv_packed2.  Errors: as mm_gemv_packed2, plus MM_ERR_INVALID_ARG for batch
 * < 1, a negative stride, strides that do not cover one matrix (batch > 1), or any
 * y overlapping any input.
 */
mm_status mm_gemv_packed2_strided_batched(const uint8_t *codes, int64_t codes_stride,
                                          const uint16_t *scales, int64_t scales_stride,
                                          const uint16_t *x, int64_t x_stride, float *y,
                                          int64_t y_stride, int64_t batch, int64_t rows,
                                          int64_t cols, const float codebook[4],
                                          mm_stream_t stream);

/*
 * mm_gemv_packed2_strided_batched with a decode choice.  opts: NULL (automatic), or a
 * mm_gemv_opts whose dequant is MM_DEQ_AUTO, MM_DEQ_AFFINE (the staged SIMT affine
 * kernel when the shape allows) or MM_DEQ_MXF4 (one launch of the fp4 tensor-core
 * decode over the whole batch: its requirements, plus codes_stride % 16 == 0; each CTA,
 * one per SM, takes rows_per_lane consecutive 127-row tiles of the batch, three at a
 * time, 0 = spread evenly over the SMs).  With the fp4 decode, pdl, weights_static and
 * independent mean what they mean for one mm_gemv_packed2_ex call, the batch being one
 * kernel: independent = 1 promises that nothing this launch reads or writes is written by
 * the kernel before it in the stream, so that launch runs without waiting for it and
 * back-to-back batched launches overlap their first and last CTAs.  Every other field 0
 * (staging may be -1).  Each y_b then equals bit for bit the single MM_DEQ_MXF4 call's.
 * Errors: as mm_gemv_packed2_strided_batched, plus MM_ERR_INVALID_ARG for other options,
 * launch options without the fp4 decode, or a decode the shape does not allow.
 */
mm_status mm_gemv_packed2_strided_batched_ex(const uint8_t *codes, int64_t codes_stride,
                                             const uint16_t *scales, int64_t scales_stride,
                                             const uint16_t *x, int64_t x_stride, float *y,
                                             int64_t y_stride, int64_t batch, int64_t rows,
                                             int64_t cols, const float codebook[4],
                                             mm_stream_t stream, const mm_gemv_opts *opts);

/* ------------------------------------------------------------------ 4-bit GEMV */

/* y[r] = scale_r * sum_k codebook[field4(r, k)] * x[k], r < rows, k < cols.
 * codes: rows x ceil(cols/2) bytes (low nibble first); scales: rows fp16; x: cols
 * fp16; y: rows fp32; codebook: 16 fp32 values in host memory (any finite values,
 * for example a normal-quantile (NF4-style) table).  fp32 products and
 * accumulation, |y - y_exact| <= 1e-5 * sum_k |term_k|; decoding is exact.
 * Errors: MM_ERR_INVALID_ARG for NULL pointers, sizes < 1, a non-finite codebook
 * entry or an output overlapping an input; MM_ERR_UNSUPPORTED on a device other
 * than sm_103; MM_ERR_CUDA for launch failures. */
mm_status mm_gemv_packed4(const uint8_t *codes, const uint16_t *scales, const uint16_t *x, float *y,
                          int64_t rows, int64_t cols, const float codebook[16], mm_stream_t stream);

typedef struct {
    int blocks;          /* staged kernel: 64-row blocks each CTA streams (1..64; 0 = 2 for
                            independent calls, 1 otherwise) */
    int pdl;             /* as in mm_gemv_opts */
    int weights_static;  /* as in mm_gemv_opts */
    int independent;     /* as in mm_gemv_opts */
    int staging;         /* 1: code rows arrive in shared memory by TMA and each code byte
                            indexes a shared-memory table of its two fields' fp32 entries
                            (cols % 256 == 0, cols <= 4096, 16-byte aligned codes and x);
                            0: the generic kernel (any shape); negative: automatic (1 when
                            the shape allows, the default without options) */
    int reserved[3];
} mm_gemv4_opts;

mm_status mm_gemv_packed4_ex(const uint8_t *codes, const uint16_t *scales, const uint16_t *x, float *y,
                             int64_t rows, int64_t cols, const float codebook[16], mm_stream_t stream,
                             const mm_gemv4_opts *opts);

#ifdef __cplusplus
}
#endif

#endif /* MM_H_ */
