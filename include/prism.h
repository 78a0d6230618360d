/*
 * prism.h -- C ABI of the batch-invariant W8A8 linear layer and the
 * candidate-restricted read-out (libprism.so, sm_103a).
 *
 * The operations follow "StartLux-Prism: Fast, exact inference for
 * StartLux-Decision models on NVIDIA GPUs" and its companion post
 * "把决策模型推理从 vLLM 换到 Prism":
 *   - activations are quantised per token after SmoothQuant smoothing
 *     (StartLux-Prism, section "Compute shared evidence once");
 *   - int8 products accumulate exactly in int32, split-K partial sums stay
 *     integers, and the result is scaled and added to the residual in a
 *     fixed rounding sequence (section "Bitwise consistency is not lossless
 *     quantization");
 *   - the output layer scores only each answer position's candidates and
 *     normalises within that set (post, sections 方案 and 实现要点), with a
 *     hard cap on the candidate count (section 复盘).
 *
 * Conventions for every entry point:
 *   - Ownership: the caller owns every buffer.  The library never allocates,
 *     frees or retains a pointer after the call returns.
 *   - Memory: every array argument is a DEVICE pointer on the current CUDA
 *     device (for example a torch tensor's data_ptr()).  Scalars are passed
 *     by value.  Strides ("ld*") are in elements and describe row-major
 *     matrices whose rows are contiguous.
 *   - Asynchrony: work is enqueued on `cuda_stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and the call returns without synchronising.
 *   - Errors: argument errors are detected on the host and returned before
 *     anything is enqueued.  PRISM_ERR_CUDA means the launch itself failed.
 *     Errors that only the device can see (bad candidate lists) are OR-ed
 *     into a caller-provided device error word; no kernel traps or asserts.
 *   - Determinism: every output row depends only on its own input row, the
 *     weights and the scales.  It is bit-identical for any batch size, batch
 *     composition, row order, split-K setting and internal tile choice.
 *   - Numerics (readings where the pages give no formula):
 *       quantiser  xs = x * inv_s (binary32 RN); amax = max |xs|;
 *                  q = clamp(rint_even(xs * RN(127/amax)), -127, 127);
 *                  a_scale = RN(amax / 127); rows with amax < 2^-120 give
 *                  q = 0, a_scale = 0.
 *       epilogue   y = bf16_rne(((float(acc) * a_scale[m]) * w_scale[n])
 *                               + residual[m,n]), one binary32 RN operation
 *                  per step, no fused multiply-add.
 *       read-out   logit = (float(acc) * a_scale[p]) * lm_scale[c] (binary32),
 *                  prob  = e_c / (e_1 + ... + e_n) summed in list order, with
 *                  e_c = exp(logit_c - max) from a Cody-Waite reduction and a
 *                  degree-7 Taylor polynomial in binary32 RN operations.
 */
#ifndef PRISM_H_
#define PRISM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PRISM_OK = 0,
  PRISM_ERR_INVALID_ARG = -1, /* NULL pointer, negative size, bad stride  */
  PRISM_ERR_ALIGNMENT = -2,   /* pointer or stride not 16-byte aligned,
                                 K not a multiple of 16                      */
  PRISM_ERR_UNSUPPORTED = -3, /* K above PRISM_MAX_K, split_k above
                                 PRISM_MAX_SPLIT_K, T above P * 64, ...      */
  PRISM_ERR_WORKSPACE = -4,   /* workspace missing or too small             */
  PRISM_ERR_CUDA = -5         /* a CUDA launch or runtime call failed       */
} prism_status;

/* Largest K for which every int32 accumulator is exact: K * 127 * 127 must
 * not exceed 2^31 - 1 (codes within +-127 on both sides).  With K a multiple
 * of 16 the usable maximum is 133136. */
#define PRISM_MAX_K 133144
/* Largest split-K factor accepted by prism_w8a8_linear. */
#define PRISM_MAX_SPLIT_K 64
/* Hard cap on candidates per answer position (post, section 复盘). */
#define PRISM_MAX_CANDIDATES 64
/* Largest hidden size accepted by the read-out (its quantised row is staged
 * on chip). */
#define PRISM_MAX_READOUT_K 65536

/* Bits OR-ed into the read-out's device error word. */
#define PRISM_DEV_ERR_OFFSETS   1u /* offsets outside [0, T] or decreasing    */
#define PRISM_DEV_ERR_COUNT     2u /* count outside [1, PRISM_MAX_CANDIDATES] */
#define PRISM_DEV_ERR_ID_RANGE  4u /* candidate id outside [0, V)             */
#define PRISM_DEV_ERR_DUPLICATE 8u /* the same id twice in one position       */
#define PRISM_DEV_ERR_ROW_RANGE 16u /* a row index outside the indexed matrix */

/*
 * prism_quant_act -- per-token activation quantisation with SmoothQuant
 * smoothing folded in (StartLux-Prism, "Compute shared evidence once").
 *
 *   x_bf16      [M, K] bf16, row stride ldx (ldx % 8 == 0, 16-byte aligned)
 *   inv_smooth  [K] float32 = 1/s_k, or NULL for no smoothing (16-byte aligned)
 *   q           [M, K] int8 out, row stride ldq (ldq % 16 == 0, 16-byte aligned)
 *   a_scale     [M] float32 out (4-byte aligned)
 *   M >= 0 (M == 0 enqueues nothing), 16 <= K <= PRISM_MAX_K, K % 16 == 0.
 * Inputs must be finite and x * inv_s must not overflow.
 */
int prism_quant_act(const void *x_bf16, int64_t ldx, const float *inv_smooth,
                    int64_t M, int64_t K, int8_t *q, int64_t ldq,
                    float *a_scale, void *cuda_stream);

/*
 * prism_quant_act_rows -- prism_quant_act on selected rows of x: output row i
 * (q row i, a_scale[i]) is the quantisation of x row rows[i].  For the last
 * layer restricted to the positions needed for answers (StartLux-Prism,
 * "Compute shared evidence once"): every step is per token, so the results
 * are the full layer's rows at those positions, bit for bit.
 *
 *   x_bf16, ldx, M_x  [M_x, K] bf16, all positions (alignment as prism_quant_act)
 *   rows, n_rows      [n_rows] int32 device indices into x, any order,
 *                     repeats allowed (4-byte aligned)
 *   inv_smooth, K, q, ldq, a_scale   as prism_quant_act, with n_rows rows out
 *   dev_error_word    device int32 or NULL: an index outside [0, M_x) ORs
 *                     in PRISM_DEV_ERR_ROW_RANGE and that row comes out as
 *                     q = 0, a_scale = NaN (so a linear on it gives NaN).
 *   n_rows == 0 enqueues nothing.
 */
int prism_quant_act_rows(const void *x_bf16, int64_t ldx, int64_t M_x,
                         const int32_t *rows, int64_t n_rows,
                         const float *inv_smooth, int64_t K, int8_t *q,
                         int64_t ldq, float *a_scale, int32_t *dev_error_word,
                         void *cuda_stream);

/*
 * Bytes of workspace prism_w8a8_linear needs for this shape and split-K
 * setting (split_k = 0 means the automatic schedule, as in the linear call:
 * arrival counters plus one int32 accumulator tile per tile it shares between
 * CTAs; about 4*M*N bytes plus counters for split_k > 1).  Returns 0
 * when no workspace is needed (split_k = 1, an automatic schedule of whole
 * tiles only, or a call of at most 8 rows, which needs no split).
 */
size_t prism_w8a8_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k);

/*
 * prism_w8a8_linear -- out = epilogue(q @ w^T) with exact int32 accumulation
 * (StartLux-Prism, "Bitwise consistency is not lossless quantization").
 *
 *   q, ldq         [M, K] int8 activations (prism_quant_act's output)
 *   a_scale        [M] float32 per-token scales
 *   w, ldw         [N, K] int8 weights, K contiguous (nn.Linear layout),
 *                  codes in [-127, 127] like the activations' (the range
 *                  prism_smooth_requant produces).  PRISM_MAX_K is the bound
 *                  for that range; a code of -128 keeps the sums exact only
 *                  while K * 127 * 128 < 2^31 (K <= 132096 in steps of 16).
 *   w_scale        [N] float32 per-output-channel scales
 *   residual, ldr  [M, N] bf16 or NULL; may be the same buffer as out
 *   out, ldo       [M, N] bf16 output
 *   acc_out        [M, N] int32 dense (stride N) copy of the accumulator, or
 *                  NULL (a debugging aid; costs 4*M*N bytes of writes)
 *   split_k        0 = automatic: a balanced schedule that gives every SM the
 *                  same number of K stages -- whole tiles first, then the K
 *                  ranges of the remaining tiles shared between CTAs, whose
 *                  int32 partial sums are added (integer reductions) into the
 *                  tile's accumulator, read back by the last CTA to finish
 *                  the tile.  1..PRISM_MAX_SPLIT_K: every tile's
 *                  K range cut into split_k equal pieces, partial sums added
 *                  as integers.  The result does not depend on split_k.
 *   workspace      device memory of at least
 *                  prism_w8a8_workspace_bytes(M, N, K, split_k) bytes, 256-byte
 *                  aligned, ZEROED by the caller before its first use.  Every
 *                  call leaves it zeroed again, so one zeroing serves all later
 *                  calls.  Calls sharing a workspace must not overlap in time
 *                  (use one stream, or one workspace per stream).  May be NULL
 *                  when the required size is 0.
 * Alignment: q, w 16-byte aligned with ldq, ldw % 16 == 0 and K % 16 == 0;
 * residual and out need only bf16 (2-byte) alignment and any ldr, ldo >= N
 * (even strides on 4-byte-aligned bases take a faster paired store).
 * M == 0 or N == 0 enqueues nothing.
 */
int prism_w8a8_linear(const int8_t *q, int64_t ldq, const float *a_scale,
                      const int8_t *w, int64_t ldw, const float *w_scale,
                      const void *residual_bf16, int64_t ldr, void *out_bf16,
                      int64_t ldo, int32_t *acc_out, int64_t M, int64_t N,
                      int64_t K, int split_k, void *workspace,
                      size_t workspace_bytes, void *cuda_stream);

/*
 * prism_w8a8_linear_rows -- prism_w8a8_linear whose residual row for output
 * row m is residual row residual_rows[m]: the residual add of a layer
 * restricted to answer positions, reading the full hidden state's rows
 * (StartLux-Prism, "Compute shared evidence once").  Output row m equals row
 * residual_rows[m] of the full layer's output when q row m is that
 * position's quantised input.
 *
 *   residual_bf16, ldr, M_res  [M_res, N] bf16, required (not NULL)
 *   residual_rows              [M] int32 device indices (4-byte aligned)
 *   dev_error_word             device int32 or NULL: an index outside
 *                              [0, M_res) ORs in PRISM_DEV_ERR_ROW_RANGE and
 *                              that output row becomes NaN (bf16 0x7fc0)
 *   out must not overlap the residual (output rows may be other tiles'
 *   residual rows).  Every other argument, the workspace rules and the
 *   alignment rules are those of prism_w8a8_linear.
 */
int prism_w8a8_linear_rows(const int8_t *q, int64_t ldq, const float *a_scale,
                           const int8_t *w, int64_t ldw, const float *w_scale,
                           const void *residual_bf16, int64_t ldr, int64_t M_res,
                           const int32_t *residual_rows, void *out_bf16,
                           int64_t ldo, int32_t *acc_out, int64_t M, int64_t N,
                           int64_t K, int split_k, void *workspace,
                           size_t workspace_bytes, int32_t *dev_error_word,
                           void *cuda_stream);

/*
 * Tensor-parallel building blocks (StartLux-Prism, "Bitwise consistency is
 * not lossless quantization": with tensor parallelism the int32 partial sums
 * are combined before scaling, so a layer gives the same bits on any number
 * of GPUs).  A row-parallel layer whose rank r holds columns [k_r, k_r+1) of
 * the activations and of the weight runs
 *     prism_act_amax       on its activation shard        -> amax[M]
 *     MAX all-reduce of amax across the ranks (exact)
 *     prism_quant_act_amax on its shard with that amax    -> q, a_scale
 *     prism_w8a8_gemm_s32  on its shard                   -> acc[M, N] int32
 *     SUM all-reduce of acc across the ranks (exact: integers)
 *     prism_w8a8_epilogue  on the sum                     -> out[M, N]
 * and every rank ends with the one-device layer's output, bit for bit.  The
 * collectives are the caller's (NCCL or any other integer/float reduction).
 */

/* amax[m] = max_k |x[m, k] * inv_smooth[k]| (binary32, exact max): the first
 * half of prism_quant_act.  Arguments and alignment as prism_quant_act;
 * amax [M] float32 out, 4-byte aligned.  M == 0 enqueues nothing. */
int prism_act_amax(const void *x_bf16, int64_t ldx, const float *inv_smooth,
                   int64_t M, int64_t K, float *amax, void *cuda_stream);

/* The second half of prism_quant_act: q and a_scale of each row from the
 * given amax[m] (rows below 2^-120 give q = 0, a_scale = 0), the codes
 * rint_even(x * inv_s * RN(127 / amax)) clamped to +-127.  With amax the
 * maximum over a row's shards, each rank's codes are the full row's codes
 * for its columns.  Arguments and alignment as prism_quant_act. */
int prism_quant_act_amax(const void *x_bf16, int64_t ldx, const float *inv_smooth,
                         const float *amax, int64_t M, int64_t K, int8_t *q,
                         int64_t ldq, float *a_scale, void *cuda_stream);

/* acc[M, N] = q @ w^T exactly in int32 (dense, row stride N, 4-byte aligned;
 * 16-byte aligned and N % 4 == 0 takes vector stores), no scaling: a rank's
 * partial sums.  q, w, split_k, workspace and alignment as prism_w8a8_linear. */
int prism_w8a8_gemm_s32(const int8_t *q, int64_t ldq, const int8_t *w,
                        int64_t ldw, int32_t *acc, int64_t M, int64_t N,
                        int64_t K, int split_k, void *workspace,
                        size_t workspace_bytes, void *cuda_stream);

/* out[m, n] = bf16_rne(((float(acc[m, n]) * a_scale[m]) * w_scale[n])
 *                      [+ residual[m, n]]) -- the linear's epilogue, one
 * binary32 RN operation per step, on given int32 accumulators [M, N] (row
 * stride ldc >= N).  residual may be NULL or the same buffer as out.
 * Alignment: acc, a_scale, w_scale 4 bytes, out and residual 2 bytes (16
 * bytes with ldc % 4 == 0 and ldo, ldr % 8 == 0 take vector accesses). */
int prism_w8a8_epilogue(const int32_t *acc, int64_t ldc, const float *a_scale,
                        const float *w_scale, const void *residual_bf16,
                        int64_t ldr, void *out_bf16, int64_t ldo, int64_t M,
                        int64_t N, void *cuda_stream);

/*
 * W4A8 on 4-bit weights (StartLux-Prism, "Compute shared evidence once":
 * Q4_K_M files and a W4A8 run).  The weight is symmetric per output channel:
 * codes in [-8, 7] (a load-time requantisation gives [-7, 7]) with one
 * float32 scale per channel, packed two per byte -- byte j of a row holds
 * code 2j in its low nibble and code 2j+1 in its high nibble (4-bit two's
 * complement).  The result is the W8A8 linear's on the unpacked codes, bit
 * for bit: the same exact int32 contraction and epilogue.
 *
 *   w4, ldw4   [N, K/2] packed bytes, row stride ldw4 >= K/2 bytes
 *              (ldw4 % 16 == 0, 16-byte aligned); K % 32 == 0
 *   every other argument as prism_w8a8_linear, except the workspace:
 *   workspace  at least prism_w4a8_workspace_bytes(M, N, K, split_k) bytes,
 *              256-byte aligned.  Calls of at most 8 rows stream the packed
 *              codes directly and need none; larger calls unpack the codes
 *              into its first 256-aligned N*K bytes (rewritten every call)
 *              and give the rest to the W8A8 kernel, whose part must be
 *              zero at the first call (zero the whole buffer once).
 */
size_t prism_w4a8_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k);

int prism_w4a8_linear(const int8_t *q, int64_t ldq, const float *a_scale,
                      const uint8_t *w4, int64_t ldw4, const float *w_scale,
                      const void *residual_bf16, int64_t ldr, void *out_bf16,
                      int64_t ldo, int32_t *acc_out, int64_t M, int64_t N,
                      int64_t K, int split_k, void *workspace,
                      size_t workspace_bytes, void *cuda_stream);

/* Packed 4-bit codes [N, K/2] -> int8 codes [N, K] (for callers that keep
 * an unpacked copy for prism_w8a8_linear).  K % 32 == 0; ldw4, ldw % 16 == 0;
 * both 16-byte aligned. */
int prism_unpack_w4(const uint8_t *w4, int64_t ldw4, int64_t N, int64_t K,
                    int8_t *w, int64_t ldw, void *cuda_stream);

/*
 * The linear with its codes held as binary16 values.  sm_103a's tensor cores
 * have no integer MMA; their f16 MMA is exact on int8 codes (every code is
 * exact in binary16, every product exact in the fp32 accumulator, and the
 * kernel drains the accumulator into int32 every 1024 K, below 2^24).  Held
 * as binary16 in memory, the codes go from global memory to the MMA by TMA
 * alone, without the shared-memory widening pass of prism_w8a8_linear: the
 * faster route for compute-bound calls (hundreds of token rows and more), at
 * twice the operand bytes.  The results are prism_w8a8_linear's, bit for bit
 * (StartLux-Prism, "Bitwise consistency is not lossless quantization").
 *
 * prism_quant_act_f16 -- prism_quant_act writing each code as a binary16
 * value (exact integers in [-127, 127]).
 *   qh, ldqh   [M, K] binary16 out (ldqh % 8 == 0, 16-byte aligned)
 *   every other argument and rule as prism_quant_act.
 */
int prism_quant_act_f16(const void *x_bf16, int64_t ldx, const float *inv_smooth,
                        int64_t M, int64_t K, uint16_t *qh, int64_t ldqh,
                        float *a_scale, void *cuda_stream);

/* int8 codes [rows, K] -> the same codes as binary16 [rows, K] (exact), the
 * weight operand of prism_w8a8_linear_f16; a load-time step.  K % 16 == 0,
 * ldw % 16 == 0, ldwh % 8 == 0, both 16-byte aligned, no overlap. */
int prism_codes_to_f16(const int8_t *w, int64_t ldw, int64_t rows, int64_t K,
                       uint16_t *wh, int64_t ldwh, void *cuda_stream);

/* Workspace bytes prism_w8a8_linear_f16 needs (split_k as in that call).
 * Its automatic schedule (split_k = 0) runs whole tiles in rounds and needs
 * none, unless the last round would leave most SMs idle: then the rounds with
 * the remainder tiles cut into equal K pieces side by side (or, for many
 * tiles of little K, the balanced schedule), whose arrival counters and
 * partial-sum slots this counts. */
size_t prism_w8a8_f16_workspace_bytes(int64_t M, int64_t N, int64_t K, int split_k);

/*
 * prism_w8a8_linear_f16 -- prism_w8a8_linear on binary16 codes:
 *   qh, ldq    [M, K] activation codes (prism_quant_act_f16), ldq % 8 == 0
 *   wh, ldw    [N, K] weight codes (prism_codes_to_f16), ldw % 8 == 0
 *   workspace  at least prism_w8a8_f16_workspace_bytes(M, N, K, split_k)
 *              bytes, 256-byte aligned, zeroed by the caller before its first
 *              use.  Every call leaves what must be zero at the next call
 *              zero again (the automatic schedule's arrival counters, split-K's
 *              accumulator); the automatic schedule's partial-sum slots are
 *              scratch whose contents never reach a result.  Calls sharing a
 *              workspace must not overlap in time.
 *   every other argument and the result as prism_w8a8_linear.
 * Codes must be integers in [-127, 127]; other binary16 values void the
 * exactness argument.
 */
int prism_w8a8_linear_f16(const uint16_t *qh, int64_t ldq, const float *a_scale,
                          const uint16_t *wh, int64_t ldw, const float *w_scale,
                          const void *residual_bf16, int64_t ldr, void *out_bf16,
                          int64_t ldo, int32_t *acc_out, int64_t M, int64_t N,
                          int64_t K, int split_k, void *workspace,
                          size_t workspace_bytes, void *cuda_stream);

/* Size of the fixed scratch array compiled into libprism.so for
 * prism_w8a8_linear_noalloc.  Every GPU that loads the library reserves it
 * until the process exits. */
#define PRISM_NOALLOC_SCRATCH_BYTES 8388608

/*
 * prism_w8a8_linear_noalloc -- prism_w8a8_linear without a workspace argument.
 * The pages describe no such call; it exists for callers that cannot provide
 * device scratch memory: a plugin host that hands the library only its own
 * input and output buffers, a latency-critical loop that must not call
 * cudaMalloc (which can synchronise the whole device), or a process whose
 * device memory budget is fixed up front.
 *
 * Arguments, layouts, alignment and results are exactly those of
 * prism_w8a8_linear (bit-identical outputs), minus workspace and
 * workspace_bytes.  Split-K scratch comes from a fixed array of
 * PRISM_NOALLOC_SCRATCH_BYTES inside the library; the call allocates nothing.
 *   - Explicit split_k > 1 on shapes whose scratch exceeds that size (about
 *     4*M*N bytes) returns PRISM_ERR_UNSUPPORTED and enqueues nothing.
 *   - split_k = 0 uses the balanced schedule when its partial tiles fit the
 *     array, else whole tiles only (same bits either way).
 *   - All calls on one device share the array.  Each call zeroes the part it
 *     uses on its own stream before computing, but calls that overlap on the
 *     GPU (other streams, unordered host threads) race on it: order them on
 *     one stream.
 *   - The first call on each device (with that device current) looks up the
 *     array's device address; make that first call before any stream capture.
 */
int prism_w8a8_linear_noalloc(const int8_t *q, int64_t ldq, const float *a_scale,
                              const int8_t *w, int64_t ldw, const float *w_scale,
                              const void *residual_bf16, int64_t ldr,
                              void *out_bf16, int64_t ldo, int32_t *acc_out,
                              int64_t M, int64_t N, int64_t K, int split_k,
                              void *cuda_stream);

/*
 * prism_smooth_requant -- load-time SmoothQuant requantisation of Q8_0
 * weights (StartLux-Prism, "Compute shared evidence once": the stored 8-bit
 * weights are requantised with the smoothing factors folded in).  Per output
 * row n and input channel k, in binary32 with one rounding per step:
 *     v        = (d[n, k/32] * q[n, k]) * s[k]      (the first product is exact)
 *     amax     = max_k |v|
 *     w[n, k]  = round-half-even(v * (127 / amax))  (always within +-127)
 *     w_scale[n] = amax / 127
 * and a row whose amax is below 2^-120 becomes zeros with scale 0.
 *
 *   q, ldq        [N, K] int8 Q8_0 codes (ldq % 16 == 0, 16-byte aligned)
 *   d_f16, ldd    [N, K/32] binary16 block scales as raw bits (2-byte
 *                 aligned, ldd >= K/32)
 *   smooth        [K] float32 s_k (multiplies channel k; 16-byte aligned), or
 *                 NULL for s_k = 1
 *   w, ldw        [N, K] int8 out (ldw % 16 == 0, 16-byte aligned).  w may be
 *                 q itself (in place, ldw == ldq); any other overlap with an
 *                 input is not allowed.
 *   w_scale       [N] float32 out (4-byte aligned)
 *   N >= 0 (N == 0 enqueues nothing), 32 <= K <= PRISM_MAX_K, K % 32 == 0.
 * Every v must be finite.  The outputs feed prism_w8a8_linear as w, w_scale.
 */
int prism_smooth_requant(const int8_t *q, int64_t ldq, const uint16_t *d_f16,
                         int64_t ldd, const float *smooth, int64_t N, int64_t K,
                         int8_t *w, int64_t ldw, float *w_scale,
                         void *cuda_stream);

/*
 * prism_candidate_readout -- logits and probabilities for the candidate
 * tokens of each answer position only; the softmax runs over the candidates
 * (post "把决策模型推理从 vLLM 换到 Prism", sections 方案 and 实现要点: equal to
 * the full-vocabulary softmax renormalised on the candidates).
 *
 *   hidden_bf16, ldh  [P, K] bf16 final hidden states (ldh % 8 == 0)
 *   inv_smooth        [K] float32 or NULL
 *   lm_head, ldw      [V, K] int8 LM head (ldw % 16 == 0), lm_scale [V] float32
 *   cand_offsets      [P+1] int32 CSR offsets, cand_offsets[0] = 0,
 *                     cand_offsets[P] = T
 *   cand_ids          [T] int32 token ids, distinct within a position,
 *                     1..PRISM_MAX_CANDIDATES per position
 *   logits, probs     [T] float32 out, in CSR order
 *   dev_error_word    device int32: PRISM_DEV_ERR_* bits are OR-ed into it
 *                     for invalid positions, whose outputs are set to NaN.
 *                     The caller clears it.  May be NULL (errors then only
 *                     show as NaN outputs).
 *   workspace, workspace_bytes
 *                     device scratch of at least
 *                     prism_readout_workspace_bytes(P, T, K) bytes.  This
 *                     implementation needs none (each position is one CTA
 *                     whose cross-thread state stays in shared memory), so
 *                     the size query returns 0 and NULL / 0 are accepted;
 *                     a caller that always sizes and passes the workspace
 *                     stays correct if a later kernel needs scratch.
 *   P >= 0 (P == 0 enqueues nothing), T <= P * PRISM_MAX_CANDIDATES,
 *   16 <= K <= PRISM_MAX_READOUT_K, K % 16 == 0.
 */
int prism_candidate_readout(const void *hidden_bf16, int64_t ldh,
                            const float *inv_smooth, const int8_t *lm_head,
                            int64_t ldw, const float *lm_scale, int64_t V,
                            int64_t K, const int32_t *cand_offsets,
                            const int32_t *cand_ids, int64_t P, int64_t T,
                            float *logits, float *probs,
                            int32_t *dev_error_word, void *workspace,
                            size_t workspace_bytes, void *cuda_stream);

/*
 * The column-parallel read-out: the LM head split by vocabulary rows over
 * ranks, each holding rows [v0, v0 + V_shard) of the V-row head; the
 * candidate softmax needs only the candidates' logits, so the ranks exchange
 * T floats, not vocabulary-sized rows (post "把决策模型推理从 vLLM 换到 Prism",
 * sections 方案 and 实现要点).
 *
 * prism_candidate_logits -- prism_candidate_readout's logits for the
 * candidates this shard holds, and -0.0 for every other candidate:
 *   lm_head_shard, ldw   [V_shard, K] int8 rows v0 .. v0 + V_shard - 1 of the head
 *   lm_scale_shard       [V_shard] float32 their scales
 *   v0, V_shard, V       0 <= v0, v0 + V_shard <= V (the whole head's rows)
 *   every other argument as prism_candidate_readout (ids are whole-head ids,
 *   validated against V; an invalid position gets the error bits and NaN
 *   logits on every shard).
 * Since x + -0.0 == x for every binary32 x, the element-wise SUM of the
 * shards' logits (any order; one shard owns each candidate) is the one-device
 * read-out's logits bit for bit.
 *
 * prism_candidate_softmax -- the read-out's candidate softmax on those
 * combined logits:
 *   logits        [T] float32 in CSR order
 *   probs         [T] float32 out, bit for bit prism_candidate_readout's
 *   cand_offsets, P, T, dev_error_word as in prism_candidate_readout; a
 *   position with malformed offsets or a count outside [1, 64] gets the
 *   error bit and NaN probabilities, one with a NaN logit NaN probabilities.
 */
int prism_candidate_logits(const void *hidden_bf16, int64_t ldh,
                           const float *inv_smooth, const int8_t *lm_head_shard,
                           int64_t ldw, const float *lm_scale_shard, int64_t v0,
                           int64_t V_shard, int64_t V, int64_t K,
                           const int32_t *cand_offsets, const int32_t *cand_ids,
                           int64_t P, int64_t T, float *logits,
                           int32_t *dev_error_word, void *cuda_stream);
int prism_candidate_softmax(const float *logits, const int32_t *cand_offsets,
                            int64_t P, int64_t T, float *probs,
                            int32_t *dev_error_word, void *cuda_stream);

/* Bytes of workspace prism_candidate_readout needs for P positions, T
 * candidates and hidden size K: 0 for every shape in this implementation. */
size_t prism_readout_workspace_bytes(int64_t P, int64_t T, int64_t K);

/* Human-readable text for a prism_status value (static storage). */
const char *prism_status_string(int status);

/* Library version as major * 10000 + minor * 100 + patch. */
int prism_version(void);

/* The cudaError_t code behind the calling thread's most recent
 * PRISM_ERR_CUDA (0 if none), then cleared; its text is copied into buf
 * (NUL-terminated, truncated to buf_bytes) when buf is not NULL. */
int prism_last_cuda_error(char *buf, size_t buf_bytes);

/*
 * Which contraction kernel prism_w8a8_linear would launch for this shape:
 * 0 = none (empty); 1 = warp-level mma.sync s8 kernel; 2 = tcgen05 kernel,
 * tokens on the 128-row MMA side; 3 = tcgen05 kernel, output channels on the
 * 128-row side and tokens on the N side; 4 = weight-streaming dp4a kernel
 * (calls of at most 2 token rows); 5 = weight-streaming mma.sync kernel
 * (calls of 3 to 16 token rows: decode steps, answer rows).  Kinds 2-5 are
 * the default.  The environment variable PRISM_LINEAR_PATH overrides the
 * choice (diagnostics; results are bit-identical on every kernel): "mma" the
 * mma.sync s8 kernel, "tc" tcgen05 for every shape, "gemv" the dp4a kernel
 * for calls of up to 8 rows, "stream" the mma.sync weight stream for calls of
 * up to 16 rows.
 */
int prism_w8a8_kernel_kind(int64_t M, int64_t N, int64_t K);

/* The split-K factor an automatic (split_k = 0) call would use: 0 for the
 * tensor-core kernel's balanced schedule (K ranges of varying length, see
 * prism_w8a8_linear), else the uniform factor of the mma.sync kernel. */
int prism_w8a8_auto_split(int64_t M, int64_t N, int64_t K);

/* Device error bits (PRISM_DEVSTATUS_*) raised by kernels since the last
 * query, then cleared.  Synchronous: waits for all work on the device.
 * A nonzero value means some output of that period is invalid. */
#define PRISM_DEVSTATUS_WAIT_TIMEOUT 1u /* a bounded on-chip wait expired */
int prism_device_status(uint32_t *flags);

/*
 * Diagnostics for the bounded on-chip waits of the tensor-core kernels
 * (prism_w8a8_linear's, prism_w8a8_linear_f16's) on the current device.
 * limit_ns > 0 arms a test mode for the calls that follow: every pipeline
 * wait is limited to limit_ns, and each CTA withholds its first
 * chunk-complete signal, so the wait for it cannot complete and expires.
 * The kernel then raises PRISM_DEVSTATUS_WAIT_TIMEOUT, lets every copy it
 * started land and every MMA it issued complete, releases its tensor memory
 * and returns.  limit_ns = 0 disarms the mode (the default: a 2 s limit,
 * every signal sent).  The outputs of any call that raised the bit are
 * invalid, and a workspace it used must be zeroed again before its next use.
 */
int prism_debug_wait_expiry(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* PRISM_H_ */
