/*
 * fp8dl.h — C ABI of the GB300 (sm_103a) FP8 delayed-scaling linear layer.
 *
 * The method (per-tensor FP8 training with delayed scaling, as run by
 * Transformer Engine's te.Linear under a DelayedScaling recipe) is described
 * in "FP8 低精度训练：Transformer Engine 简析" (m.haoling.cc), §三 "FP8技术分析":
 *   - §三.1 "宏观实现框架": one scale per tensor, symmetric linear quantisation;
 *     delayed scaling takes the max of an amax history window and sets
 *     scale = (FP8_MAX / amax) / 2^margin; recipe parameters margin, interval,
 *     fp8_format (forward E4M3, backward E5M2 in HYBRID), amax_history_len.
 *   - §三.3 "FP8框架TE计算流程": inputs and weights are cast to FP8 with the
 *     stored scale, the cast writes its amax into the history, fp8_gemm
 *     computes; at autocast exit the amaxes update history and scale.
 *   - §三.4 "Tensor Core如何进行FP8训练": the GEMM returns a high-precision
 *     result; every dimension is a multiple of 16.
 * MXFP8 (block-scaled FP8) is named by the Transformer Engine README
 * ("亮点": MXFP8 on Blackwell); the pages do not define it.  This library reads
 * it as E4M3 data with one E8M0 (power-of-two) scale per 32 consecutive
 * elements along the reduction axis.
 *
 * Conventions shared by every call
 *   Memory      All pointers are DEVICE pointers owned by the caller, unless a
 *               parameter says "host".  The library allocates no device memory;
 *               where a call needs scratch space the caller passes it in
 *               (see fp8_cast_workspace_size).
 *   Layout      Matrices are row-major and densely packed.  FP8 data are one
 *               byte per element (E4M3 or E5M2 codes).  bf16 is IEEE bfloat16.
 *   GEMMs       Every GEMM is "TN": D[M,N] = A[M,K] * B[N,K]^T, both operands
 *               row-major with K contiguous.  The linear layer uses it three
 *               times: forward Y = X W^T (A = X, B = W), dgrad dX = dY W
 *               (A = dY, B = W^T, the transposed copy of W's cast), wgrad
 *               dW = dY^T X (A = dY^T, B = X^T, the transposed copies).
 *   Shapes      Every dimension must be a positive multiple of 16 (32 for the
 *               MXFP8 calls); otherwise FP8DL_ERR_SHAPE.  Pointers must be
 *               16-byte aligned (FP8DL_ERR_ALIGN).
 *   Streams     Every call is asynchronous on `stream` (NULL = the legacy
 *               default stream) and never synchronises with the host.
 *               Scales are read from device memory, so a training step never
 *               waits for the host.
 *   Errors      Argument checks run on the host before any launch and return a
 *               status; nothing throws across the ABI and no kernel traps.
 *               fp8dl_last_error() returns the calling thread's last message.
 *               GEMM pipelines bound every wait; if a wait runs out the kernel
 *               stops, writes FP8DL_ERR_TIMEOUT into *dev_status (when given)
 *               and returns, leaving D undefined.
 *   Device      The library is built for sm_103a only (GB300).  Calls on any
 *               other device return FP8DL_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef FP8DL_H
#define FP8DL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t. */
typedef struct CUstream_st *fp8dl_stream_t;

typedef enum {
    FP8DL_OK = 0,
    FP8DL_ERR_INVALID_ARG = 1,        /* null pointer, unknown enum, bad recipe   */
    FP8DL_ERR_SHAPE = 2,              /* dimension not a positive multiple of 16  */
    FP8DL_ERR_ALIGN = 3,              /* pointer not 16-byte aligned              */
    FP8DL_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not sm_103             */
    FP8DL_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed        */
    FP8DL_ERR_TIMEOUT = 6,            /* written to *dev_status by a kernel only  */
    FP8DL_ERR_WORKSPACE = 7           /* workspace missing or too small           */
} fp8dl_status;

/* FP8 element formats.  E4M3: bias 7, max 448, no infinity, S.1111.111 = NaN.
 * E5M2: bias 15, max 57344, S.11111.00 = infinity, other S.11111.xx = NaN. */
typedef enum { FP8DL_E4M3 = 0, FP8DL_E5M2 = 1 } fp8dl_fp8_dtype;

/* High-precision element types. */
typedef enum { FP8DL_F32 = 0, FP8DL_BF16 = 1 } fp8dl_hp_dtype;

/* Recipe format: E4M3 everywhere, or HYBRID (E4M3 forward, E5M2 gradients). */
typedef enum { FP8DL_FORMAT_E4M3 = 0, FP8DL_FORMAT_HYBRID = 1 } fp8dl_format;

/* Delayed-scaling recipe (§三.1 "宏观实现框架" lists margin, interval,
 * fp8_format and amax_history_len; "max" is the window algorithm of the
 * Transformer Engine tutorial's HYBRID recipe).  Host struct. */
typedef struct {
    int32_t margin;            /* scale = (FP8_MAX/amax) / 2^margin, 0 <= margin <= 126 */
    int32_t interval;          /* recompute the scale when step % interval == 0, >= 1   */
    int32_t fp8_format;        /* fp8dl_format; informs which slots use E5M2            */
    int32_t amax_history_len;  /* L >= 1, window length of the amax history            */
    int32_t amax_compute_algo; /* 0 = max over the window (the only algorithm)         */
} fp8dl_recipe;

/* ----------------------------------------------------------------------------
 * Scaling state.  One "slot" per scaled tensor (e.g. input, weight and
 * grad_output of each GEMM).  The state of n slots is one caller-allocated
 * device block of fp8dl_scaling_state_bytes(L, n) bytes; slot i starts at
 * byte i * fp8dl_slot_stride(L) and holds
 *     float   scale       offset 0   multiplier used by the next casts
 *     float   scale_inv   offset 4   1/scale, read by the GEMM epilogue
 *     float   amax        offset 8   amax recorded since the last update;
 *                                    casts max their |x| into it atomically
 *     int32   hist_pos    offset 12  next write position in the history ring
 *     int32   fp8_dtype   offset 16  fp8dl_fp8_dtype of the slot (FP8_MAX)
 *     int32   reserved[3]
 *     float   hist[L]     offset 32  amax history ring
 * The block is plain data: saving and restoring it (with the caller's step
 * counter) resumes training bit-identically.
 * ------------------------------------------------------------------------- */
size_t fp8dl_slot_stride(int32_t amax_history_len);
size_t fp8dl_scaling_state_bytes(int32_t amax_history_len, int32_t n_slots);

/* Initialise n_slots slots: scale = scale_inv = 1, amax = 0, hist = 0,
 * hist_pos = 0, fp8_dtype = slot_fp8_dtype[i] (HOST array of n_slots). */
fp8dl_status fp8_scaling_state_init(const fp8dl_recipe *recipe, int32_t n_slots,
                                    const int32_t *slot_fp8_dtype, void *state,
                                    fp8dl_stream_t stream);

/* Delayed scale update of every slot (§三.1 "宏观实现框架", §三.3: at autocast
 * exit the recorded amaxes update the history and the scale).  Per slot:
 *   hist[hist_pos] = amax; hist_pos = (hist_pos + 1) % L; amax = 0;
 *   if (step % interval == 0):
 *       a = max(hist[0..L))
 *       if a > 0 and finite: s = fl32(FP8_MAX / a) / 2^margin
 *           if s > 0 and finite: scale = s, scale_inv = fl32(1 / s)
 *   (otherwise scale and scale_inv keep their values).
 * `step` is the caller's step counter.  One launch for all slots. */
fp8dl_status fp8_update_scale(const fp8dl_recipe *recipe, int32_t n_slots, void *state,
                              int64_t step, fp8dl_stream_t stream);

/* First step: fill every history entry with the slot's recorded amax (from
 * an amax-only cast pass), clear amax, set hist_pos = 0 and derive the scale
 * as above, so the first real cast already uses a data-derived scale. */
fp8dl_status fp8_seed_amax_history(const fp8dl_recipe *recipe, int32_t n_slots, void *state,
                                   fp8dl_stream_t stream);

/* ----------------------------------------------------------------------------
 * Fused cast + amax (+ transpose) (+ bias gradient) (§三.1 / §三.3: the cast
 * to FP8 uses the stored scale and records the tensor's amax).
 *   x        [rows x cols], x_dtype (FP8DL_F32 or FP8DL_BF16)
 *   scale    device float (a slot's scale)
 *   out      [rows x cols] FP8 codes, out[i,j] = enc(fl32(x[i,j] * scale)), or NULL
 *   out_t    [cols x rows] FP8 codes, out_t[j,i] = out[i,j], or NULL
 *   amax     device float, atomically max-ed with max |x| (pre-scale), or NULL
 *   scale_inv_out  device float receiving fl32(1 / *scale), the factor that
 *            decodes these codes, or NULL.  Codes kept past the next scale
 *            update (a weight cast once and reused over micro-batches, §三.3:
 *            the cast is skipped while a cached FP8 copy exists) carry their
 *            own decode factor this way, since the update rewrites the slot's
 *            scale_inv.  Written by a one-thread kernel after the cast.
 *   dbias    [cols] fp32 column sums of x (the bias gradient when x is
 *            grad_output), or NULL; overwritten, not accumulated
 *   workspace/workspace_bytes  scratch of fp8_cast_workspace_size(rows, cols)
 *            bytes, needed only when dbias != NULL
 * Encoding: round to nearest even, saturating to +-FP8_MAX (including
 * infinities); NaN gives a NaN code.  With out, out_t and dbias all NULL the
 * call is an amax-only pass. */
size_t fp8_cast_workspace_size(int64_t rows, int64_t cols);

fp8dl_status fp8_cast_amax_transpose(const void *x, int32_t x_dtype, int64_t rows, int64_t cols,
                                     int32_t out_dtype, const float *scale, uint8_t *out,
                                     uint8_t *out_t, float *amax, float *scale_inv_out, float *dbias,
                                     void *workspace, size_t workspace_bytes, fp8dl_stream_t stream);

/* Grouped cast: the casts of up to 8 tensors (say the two weights of a
 * LayerNormMLP, or the weights of several layers) in one launch, so that the
 * small tensors share one grid instead of each paying a launch, a ramp-up
 * and a tail.  Per tensor the results are exactly those of
 * fp8_cast_amax_transpose without dbias (§三.1 / §三.3: the cast with the
 * stored scale records the tensor's amax).
 *   items  HOST array of n items (1 <= n <= 8), each with its own x
 *          [rows x cols], scale, outputs and amax, as in
 *          fp8_cast_amax_transpose; all share x_dtype and out_dtype.
 *   Argument errors of any item are reported before any launch. */
typedef struct {
    const void *x;          /* [rows x cols] of the call's x_dtype */
    int64_t rows, cols;     /* positive multiples of 16 */
    const float *scale;     /* device float */
    uint8_t *out;           /* [rows x cols] codes, or NULL */
    uint8_t *out_t;         /* [cols x rows] codes, or NULL */
    float *amax;            /* device float, max-ed with max |x|, or NULL */
    float *scale_inv_out;   /* device float receiving fl32(1 / *scale), or NULL */
} fp8dl_cast_item;

fp8dl_status fp8_cast_amax_transpose_multi(int32_t n, const fp8dl_cast_item *items, int32_t x_dtype,
                                           int32_t out_dtype, fp8dl_stream_t stream);

/* The same cast for callers that cannot allocate device memory.  The paper
 * has no counterpart to this call: it exists for callers that only hand the
 * library their input and output buffers (a plugin or custom-op interface
 * whose fixed signature has no workspace argument, or a process whose device
 * memory belongs to another allocator that does not let it call cudaMalloc),
 * so they can neither pass the bias-gradient workspace nor allocate one.
 *   Arguments, layouts and results are those of fp8_cast_amax_transpose,
 *   without workspace/workspace_bytes.
 *   Scratch: the dbias workspace is a 4 MiB array in the library's static
 *   device memory (every GPU that loads the library holds it until the
 *   process exits).  Calls with dbias != NULL need
 *   fp8_cast_workspace_size(rows, cols) <= 4 MiB, i.e.
 *   ceil(rows/128) * cols * 4 <= 4194304; larger ones return
 *   FP8DL_ERR_WORKSPACE before any launch.  The call allocates nothing
 *   (no cudaMalloc, cudaFree or allocating library routine).
 *   First call per device: looks up the array's device address with
 *   cudaGetSymbolAddress (that device current) and caches it; make that first
 *   call before any stream capture.
 *   Sharing: all calls on a device share the one array, which keeps the last
 *   call's contents; each call writes every scratch entry it reads, so no
 *   clearing is needed.  A call enqueues its two launches (partials, then
 *   their reduction) under a library lock, so calls from several host
 *   threads on one stream run one after another on the GPU.  Calls whose
 *   work overlaps on the GPU (different streams not ordered by events) race
 *   on the array and give wrong dbias: put them on one stream. */
fp8dl_status fp8_cast_amax_transpose_noalloc(const void *x, int32_t x_dtype, int64_t rows, int64_t cols,
                                             int32_t out_dtype, const float *scale, uint8_t *out,
                                             uint8_t *out_t, float *amax, float *dbias,
                                             fp8dl_stream_t stream);

/* ----------------------------------------------------------------------------
 * FP8 GEMM with dequantising epilogue (§三.3 fp8_gemm; §三.4 high-precision
 * output, dims multiple of 16):
 *   D[m,n] = round_d( acc[m,n] * fl32(a_scale_inv * b_scale_inv) + bias[n] )
 *   (the product and the bias add are one fp32 fused multiply-add)
 *   acc[m,n] = sum_k A[m,k] * B[n,k] on the tcgen05 tensor cores, fp32 accumulate.
 *     A GEMM with K > 8192 and at least two waves of tiles sums the k-blocks of
 *     every other tile of a CTA (pair) last to first (less DRAM traffic); the
 *     order is fixed by the shape and the GPU's SM count, so repeated calls give
 *     the same bits.
 *   A [M x K] codes of a_dtype, B [N x K] codes of b_dtype (E4M3/E5M2 mixed ok)
 *   a_scale_inv, b_scale_inv   device floats (the operands' slots' scale_inv)
 *   bias       [N] of bias_dtype, or NULL
 *   D          [M x N] of d_dtype (FP8DL_BF16 or FP8DL_F32)
 *   dev_status device int or NULL; set to FP8DL_ERR_TIMEOUT if a pipeline wait
 *              runs out (never reset to 0 by the library). */
fp8dl_status fp8_gemm(const uint8_t *A, int32_t a_dtype, const uint8_t *B, int32_t b_dtype,
                      int64_t M, int64_t N, int64_t K, const float *a_scale_inv,
                      const float *b_scale_inv, const void *bias, int32_t bias_dtype, void *D,
                      int32_t d_dtype, int32_t *dev_status, fp8dl_stream_t stream);

/* FP8 GEMM whose epilogue also applies GELU and the FP8 cast of the result
 * (the fc1 GEMM of a LayerNormMLP).  Delayed scaling knows the cast's scale
 * before the GEMM runs ("FP8 低精度训练：Transformer Engine 简析" §三.1: with the
 * scale known in advance the computation stays in one kernel), so the GELU
 * output never makes an HBM round trip:
 *   H[m,n] = bf16( acc[m,n] * fl32(a_scale_inv * b_scale_inv) + bias[n] )   (as fp8_gemm)
 *   G = bf16( GELU(H) )  (erf form; see fp8_gelu_cast)
 *   q = enc(fl32(G * q_scale)) [M x N], q_t = q^T [N x M], *q_amax max-ed with max |G|
 *   g [M x N] bf16 receives G, or NULL.
 * H is bf16.  Results are identical to fp8_gemm followed by fp8_gelu_cast. */
fp8dl_status fp8_gemm_gelu_cast(const uint8_t *A, int32_t a_dtype, const uint8_t *B, int32_t b_dtype,
                                int64_t M, int64_t N, int64_t K, const float *a_scale_inv,
                                const float *b_scale_inv, const void *bias, int32_t bias_dtype, void *H,
                                int32_t q_dtype, const float *q_scale, uint8_t *q, uint8_t *q_t,
                                float *q_amax, void *g, int32_t *dev_status, fp8dl_stream_t stream);

/* FP8 GEMM whose epilogue applies dGELU and the FP8 cast of the result (the
 * fc2 dgrad GEMM of a LayerNormMLP feeding the fc1 backward), with the fc1
 * bias gradient.  As for fp8_gemm_gelu_cast, the delayed scale of the output
 * is known before the GEMM, so dg never makes an HBM round trip:
 *   dg[m,n] = bf16( acc[m,n] * fl32(a_scale_inv * b_scale_inv) )   (no bias)
 *   dh = bf16( dg * GELU'(h) )  (erf form; see fp8_dgelu_cast), h [M x N] bf16
 *   q = enc(fl32(dh * q_scale)) [M x N], q_t = q^T [N x M], *q_amax max-ed with max |dh|
 *   dbias[n] = sum over m of dh[m,n] (fp32, a fixed order), or NULL
 *   dg and dh [M x N] bf16 receive those tensors, or NULL.
 * workspace: fp8_gemm_dgelu_workspace_size(M, N) bytes (16-byte aligned),
 * needed only when dbias != NULL.  Codes, amax, dg and dh are identical to
 * fp8_gemm followed by fp8_dgelu_cast; dbias agrees within its summation
 * bound (the order of the sum differs).  Needs CTA-pair clusters
 * (FP8DL_ERR_UNSUPPORTED_DEVICE otherwise). */
size_t fp8_gemm_dgelu_workspace_size(int64_t M, int64_t N);

fp8dl_status fp8_gemm_dgelu_cast(const uint8_t *A, int32_t a_dtype, const uint8_t *B, int32_t b_dtype,
                                 int64_t M, int64_t N, int64_t K, const float *a_scale_inv,
                                 const float *b_scale_inv, const void *h, void *dg, int32_t q_dtype,
                                 const float *q_scale, uint8_t *q, uint8_t *q_t, float *q_amax,
                                 float *dbias, void *workspace, size_t workspace_bytes, void *dh,
                                 int32_t *dev_status, fp8dl_stream_t stream);

/* ----------------------------------------------------------------------------
 * MXFP8 quantisation (block-scaled FP8, named by the Transformer Engine
 * README).  x [rows x cols] (bf16 or fp32).  Blocks are 32 consecutive
 * elements; per block: e = the smallest integer with amax_b * 2^-e <= 448,
 * clamped to [-127, 127] (amax_b = 0 gives e = 0); scale byte = e + 127 (E8M0);
 * data = enc_e4m3(fl32(x * 2^-e)).
 *   row_q [rows x cols]: blocks along each row, or NULL
 *   row_s  scales of row_q in the tiled layout below (R = rows, NB = cols/32)
 *   col_q [cols x rows]: blocks along each column, stored transposed (row j
 *         of col_q is column j of x), or NULL
 *   col_s  scales of col_q in the tiled layout (R = cols, NB = rows/32)
 * rows and cols must be multiples of 32.
 *
 * Tiled scale layout (the order the tensor cores read block scales in).  For
 * a matrix of R rows with NB blocks per row, S[r][b] is the scale byte of
 * block b of row r.  Rows are grouped by 128 and blocks by 4; each
 * (row group g, block group h) is one 512-byte tile at byte offset
 * (g * ceil(NB/4) + h) * 512, and inside the tile
 *     byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (b % 4)  holds  S[r][b].
 * Total size: mxfp8_scale_bytes(R, 32*NB).  Entries for rows >= R or blocks
 * >= NB (padding) are written as 127 (2^0).
 *
 * dbias [cols] fp32 receives the column sums of x (the bias gradient when x
 * is grad_output; the te.Linear example has bias=True), in the same pass over
 * x, or NULL; overwritten, not accumulated.  The sum runs in a fixed order,
 * so repeated calls give the same bits.  workspace/workspace_bytes: scratch
 * of fp8_cast_workspace_size(rows, cols) bytes (16-byte aligned), needed
 * only when dbias != NULL (FP8DL_ERR_WORKSPACE otherwise). */
size_t mxfp8_scale_bytes(int64_t rows, int64_t cols);

fp8dl_status mxfp8_quantize(const void *x, int32_t x_dtype, int64_t rows, int64_t cols,
                            uint8_t *row_q, uint8_t *row_s, uint8_t *col_q, uint8_t *col_s,
                            float *dbias, void *workspace, size_t workspace_bytes,
                            fp8dl_stream_t stream);

/* MXFP8 GEMM: D[m,n] = round_d( sum_b 2^(ea[m,b]+eb[n,b]) * sum_{k in b} A[m,k]*B[n,k]
 *                               + bias[n] )
 * A [M x K] E4M3 with scales A_s (tiled layout, R = M, NB = K/32);
 * B [N x K] E4M3 with scales B_s (tiled layout, R = N, NB = K/32), as produced
 * by mxfp8_quantize (row_q/row_s of X and W for the forward GEMM; col_q/col_s
 * for the operands of the gradient GEMMs).  M, N, K multiples of 32.
 * bias, D, dev_status and the order of the k-blocks as for fp8_gemm. */
fp8dl_status mxfp8_gemm(const uint8_t *A, const uint8_t *A_s, const uint8_t *B, const uint8_t *B_s,
                        int64_t M, int64_t N, int64_t K, const void *bias, int32_t bias_dtype,
                        void *D, int32_t d_dtype, int32_t *dev_status, fp8dl_stream_t stream);

/* ----------------------------------------------------------------------------
 * LayerNormMLP pieces.  The Transformer Engine tutorial builds its blocks
 * from te.LayerNormMLP (LayerNorm -> fc1 -> GELU -> fc2), mirrored in plain
 * PyTorch by nn.LayerNorm and nn.GELU (erf form).  Under delayed scaling the
 * scale of each activation's FP8 cast is known before the activation runs
 * ("FP8 低精度训练：Transformer Engine 简析" §三.1), so each activation is fused
 * with the cast of its output (cast semantics as fp8_cast_amax_transpose).
 * All high-precision tensors here are bf16; mu and rsigma are fp32.
 */

/* LayerNorm forward + cast, per row of x [rows x cols] (cols <= 8192):
 *   mu = mean(x), var = mean((x - mu)^2) (biased), rsigma = 1/sqrt(var + eps)
 *   y = bf16((x - mu) * rsigma * gamma + beta)       (fp32 arithmetic)
 *   out = enc(fl32(y * scale)), out_t = out^T, amax max-ed with max |y|
 * gamma, beta [cols] bf16; mu, rsigma [rows] fp32 (for the backward);
 * y [rows x cols] bf16 or NULL; out/out_t/amax nullable as for the cast. */
fp8dl_status fp8_layernorm_cast(const void *x, int64_t rows, int64_t cols, const void *gamma,
                                const void *beta, float eps, int32_t out_dtype, const float *scale,
                                uint8_t *out, uint8_t *out_t, float *amax, float *mu, float *rsigma,
                                void *y, fp8dl_stream_t stream);

/* GELU + cast: g = bf16(0.5 * h * (1 + erf(h / sqrt2))) in fp32 arithmetic, then the
 * cast of g (out, out_t, amax of g).  h [rows x cols] bf16 (the fc1 output);
 * g [rows x cols] bf16 or NULL. */
fp8dl_status fp8_gelu_cast(const void *h, int64_t rows, int64_t cols, int32_t out_dtype,
                           const float *scale, uint8_t *out, uint8_t *out_t, float *amax, void *g,
                           fp8dl_stream_t stream);

/* dGELU + cast: dh = bf16(dg * (0.5 * (1 + erf(h/sqrt2)) + h * exp(-h^2/2) / sqrt(2 pi))),
 * then the cast of dh (E5M2 in HYBRID) with amax, transposed copy and the
 * bias gradient dbias = column sums of dh (workspace as for the cast).
 * dg, h [rows x cols] bf16; dh [rows x cols] bf16 or NULL. */
fp8dl_status fp8_dgelu_cast(const void *dg, const void *h, int64_t rows, int64_t cols, int32_t out_dtype,
                            const float *scale, uint8_t *out, uint8_t *out_t, float *amax, float *dbias,
                            void *workspace, size_t workspace_bytes, void *dh, fp8dl_stream_t stream);

/* LayerNorm backward from the forward's mu and rsigma:
 *   xhat = (x - mu) * rsigma, g = dy * gamma
 *   dx = bf16(rsigma * (g - mean(g) - xhat * mean(g * xhat)))
 *   dgamma = sum_rows dy * xhat, dbeta = sum_rows dy   (fp32 [cols], overwritten)
 * dy, x [rows x cols] bf16, gamma [cols] bf16; workspace of
 * fp8_layernorm_bwd_workspace_size(rows, cols) bytes. */
size_t fp8_layernorm_bwd_workspace_size(int64_t rows, int64_t cols);

fp8dl_status fp8_layernorm_bwd(const void *dy, const void *x, const void *gamma, const float *mu,
                               const float *rsigma, int64_t rows, int64_t cols, void *dx, float *dgamma,
                               float *dbeta, void *workspace, size_t workspace_bytes,
                               fp8dl_stream_t stream);

/* ----------------------------------------------------------------------------
 * Library state. */
/* 1 if `device` is an sm_103 GPU this library can run on, else 0. */
int32_t fp8dl_device_supported(int32_t device);
/* Last error message of the calling thread ("" if none). */
const char *fp8dl_last_error(void);
/* Self-test of failure detection without a GPU fault.  One thread waits,
 * through the same bounded wait the GEMM pipelines use, on a shared-memory
 * barrier phase; if arrive_first is 0 nothing ever completes it, the wait
 * gives up after budget_cycles SM clock cycles (<= 2^32), writes
 * FP8DL_ERR_TIMEOUT into *dev_status and the kernel returns; with
 * arrive_first = 1 the phase completes and *dev_status is set to FP8DL_OK.
 * The CUDA context stays usable either way. */
fp8dl_status fp8dl_wait_selftest(int64_t budget_cycles, int32_t arrive_first, int32_t *dev_status,
                                 fp8dl_stream_t stream);
/* Clock probe (measurement): n_ctas CTAs each write, to out[3 * i .. 3 * i + 2]
 * (device memory, 16-byte aligned, 3 * n_ctas uint64), the id of the SM CTA i
 * ran on, that SM's cycle counter (clock64) and the global nanosecond timer
 * (%globaltimer), read back to back.  Two probes on a stream around some work
 * give each SM's mean clock over it: (cycles_2 - cycles_1) / (ns_2 - ns_1) GHz
 * for an SM seen in both.  One launch; no other effect. */
fp8dl_status fp8dl_clock_probe(uint64_t *out, int32_t n_ctas, fp8dl_stream_t stream);
/* Library version, major*10000 + minor*100 + patch. */
int32_t fp8dl_version(void);
/* Number of kernels this library has enqueued in this process, over all threads
 * and devices (launches that failed are not counted).  A CUDA graph replay
 * launches its captured kernels without calling the library, so it does not
 * count: count one eager step to know what a replayed step launches. */
uint64_t fp8dl_kernel_launches(void);

/* ----------------------------------------------------------------------------
 * Environment switches (testing and diagnosis).  They choose which kernel, tile
 * order or grid runs.  The GEMM switches leave every output bit unchanged,
 * except in a GEMM with K > 8192 and two or more waves of tiles, where they
 * can change which tiles sum K last to first (within the GEMM's error bound;
 * the one-CTA kernel always sums first to last).  The LayerNorm ones can
 * change the rounding of the row statistics and of dgamma / dbeta, within the
 * tolerances the tests state.
 *   FP8DL_DEBUG=1               print every launch and error message to stderr
 *                               (read once per process)
 *   FP8DL_GEMM_VARIANT=1sm|2sm  force the one-CTA or the CTA-pair FP8 GEMM
 *   FP8DL_GEMM_RASTER=m|n       group the GEMM tiles along rows (m) or columns (n)
 *   FP8DL_GEMM_GROUP=g          tiles per group (g > 0)
 *   FP8DL_GEMM_TILE_N=256|128   tile width of the plain pair GEMM (by default 128
 *                               only for a short GEMM with under two waves of
 *                               256-column tiles)
 *   FP8DL_GEMM_SNAKE=0          every GEMM tile sums K first to last
 *   FP8DL_LN_VARIANT=tiles      LayerNorm by the two-pass tile kernels
 *   FP8DL_LN_CLUSTERS=n         cap on the clusters of the LayerNorm cluster kernels
 *   FP8DL_PDL=0                 launch without programmatic dependent launch: every
 *                               kernel then starts only after the previous kernel of
 *                               its stream has finished (read once per process)
 * All but FP8DL_DEBUG and FP8DL_PDL are read at each call.
 *
 * Launch order.  The kernels of a short call (under 64 MB moved or 64 GFLOP)
 * are launched with the programmatic stream serialization attribute: such a
 * kernel may be scheduled while the previous kernel of the stream is still
 * running, does only its own set-up (shared-memory barriers, tensor-memory
 * allocation, descriptor prefetch), and waits for that kernel to complete
 * before its first access to global memory.  Every kernel makes that wait, so
 * stream order and results are those of ordinary launches. */

#ifdef __cplusplus
}
#endif
#endif /* FP8DL_H */
