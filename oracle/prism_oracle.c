/*
 * prism_oracle.c -- plain, slow, obviously correct CPU definition of the
 * batch-invariant W8A8 linear layer and the candidate-restricted read-out of
 * "StartLux-Prism: Fast, exact inference for StartLux-Decision models on
 * NVIDIA GPUs".
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the parity oracle: only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * The product path never calls it, and it shares no code, header, table or
 * constant with the CUDA library; both sides were written independently from
 * the same definitions.
 *
 * Build: any C99 compiler, with floating-point contraction OFF
 * (-ffp-contract=off) and without fast-math, so every float operation below
 * is one IEEE-754 binary32 round-to-nearest-even operation, in program order.
 * OpenMP (optional) only splits independent rows across threads.
 *
 * Sources (page, section):
 *  [P1-evidence]  StartLux-Prism (English), "Compute shared evidence once":
 *                 Q8_0 weights requantised with SmoothQuant at startup
 *                 (oracle_smooth_requant),
 *                 activations quantised per token for W8A8 execution; the
 *                 last layer restricted to the positions needed for answers.
 *  [P1-bitwise]   same page, "Bitwise consistency is not lossless
 *                 quantization": int8 products accumulate exactly in int32,
 *                 then are scaled and added to the residual in a fixed
 *                 rounding sequence; split-K partial sums stay integers;
 *                 scaling, addition and read-out paths are fixed.
 *  [P4-plan]      "把决策模型推理从 vLLM 换到 Prism", section 方案: scores only
 *                 for valid candidates, normalised within the candidate set,
 *                 mathematically equal to full-vocabulary scoring followed by
 *                 renormalisation; INT8 tensor cores with INT32 accumulation.
 *  [P4-impl]      same page, section 实现要点: the candidate-softmax identity
 *                 (full softmax gathered on the candidates and renormalised
 *                 equals the softmax of the candidate logits).
 *  [P4-review]    same page, section 复盘: a hard cap on the candidate count.
 *
 * Where the pages leave a step open, the reading used here is stated at the
 * function (quantiser rounding and scale form, epilogue order, read-out
 * precision, exp).  Parity pins for every function live in the test suite.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MAX_K 133144        /* largest K with K * 127 * 127 <= 2^31 - 1 */
#define ORACLE_MAX_CANDIDATES 64   /* hard cap per answer position [P4-review] */

#define ORACLE_ERR_ROW_RANGE 16u   /* a row index outside the indexed matrix */

/* ---------------------------------------------------------------- bf16 --- */

/* bfloat16 is the top half of a binary32: widening is exact. */
static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even (finite inputs;
 * a NaN becomes the canonical quiet NaN). */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)0x7fc0u;
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

int oracle_max_k(void) { return ORACLE_MAX_K; }
int oracle_max_candidates(void) { return ORACLE_MAX_CANDIDATES; }

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------- per-token quantiser --- */
/*
 * [P1-evidence]: activations are quantised per token; SmoothQuant moves
 * outlier magnitude from activations into weights through a per-input-channel
 * factor s_k, so the activation seen by the quantiser is x_k / s_k.  The hot
 * path receives inv_s[k] = 1/s_k (a model parameter) and multiplies.
 *
 * Reading (the pages give no formula): symmetric, no zero point, 127 levels
 * each side, round half to even, multiply by 127/amax rather than divide by
 * the scale:
 *     xs_k     = x_k * inv_s_k                     (binary32 RN)
 *     amax     = max_k |xs_k|
 *     inv_a    = 127 / amax                        (binary32 RN)
 *     q_k      = clamp(rint(xs_k * inv_a), -127, 127)
 *     a_scale  = amax / 127                        (binary32 RN)
 * A row whose amax is below 2^-120 (all zeros, or so tiny that 127/amax
 * would overflow) quantises to q = 0 with a_scale = 0.
 */
/* The two halves of the quantiser.  oracle_act_amax: amax_m = max_k
 * |x_mk * inv_s_k| (binary32, exact max).  oracle_quant_act_amax: the codes and
 * scale of each row from a given amax_m, which for one device is the row's
 * own; a tensor-parallel layer whose ranks hold K-shards of the row passes
 * the maximum over the ranks' amax, so every rank uses the scale of the
 * whole row ([P1-bitwise]: the same bits on any number of GPUs). */
void oracle_act_amax(const uint16_t *x, int64_t ldx, const float *inv_s,
                     int64_t M, int64_t K, float *amax)
{
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        const uint16_t *xr = x + m * ldx;
        float am = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float xs = bf16_to_float(xr[k]);
            if (inv_s) xs = xs * inv_s[k];
            float a = fabsf(xs);
            if (a > am) am = a;
        }
        amax[m] = am;
    }
}

void oracle_quant_act_amax(const uint16_t *x, int64_t ldx, const float *inv_s,
                           const float *amax, int64_t M, int64_t K, int8_t *q,
                           int64_t ldq, float *a_scale)
{
    const float tiny = ldexpf(1.0f, -120);
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        const uint16_t *xr = x + m * ldx;
        int8_t *qr = q + m * ldq;
        const float am = amax[m];
        if (!(am >= tiny)) {
            for (int64_t k = 0; k < K; ++k) qr[k] = 0;
            a_scale[m] = 0.0f;
            continue;
        }
        float inv_a = 127.0f / am;
        for (int64_t k = 0; k < K; ++k) {
            float xs = bf16_to_float(xr[k]);
            if (inv_s) xs = xs * inv_s[k];
            float t = rintf(xs * inv_a);       /* default mode: ties to even */
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            qr[k] = (int8_t)t;
        }
        a_scale[m] = am / 127.0f;
    }
}

void oracle_quant_act(const uint16_t *x, int64_t ldx, const float *inv_s,
                      int64_t M, int64_t K, int8_t *q, int64_t ldq,
                      float *a_scale)
{
    /* a_scale first holds the row maxima, then the scales (row by row, each
     * amax is read before its scale overwrites it) */
    oracle_act_amax(x, ldx, inv_s, M, K, a_scale);
    oracle_quant_act_amax(x, ldx, inv_s, a_scale, M, K, q, ldq, a_scale);
}

/* ------------------------------------ SmoothQuant startup requantisation --- */
/*
 * [P1-evidence]: the stored Q8_0 weights are requantised with SmoothQuant at
 * startup.  Q8_0 keeps each weight row in blocks of 32 int8 values that share
 * one binary16 scale d.  SmoothQuant moves activation outliers into the
 * weights: input channel k of every weight row is multiplied by s_k while the
 * activations are divided by it (oracle_quant_act receives 1/s_k).  The
 * result is requantised per output channel into the int8 weights and binary32
 * per-channel scales that the W8A8 linear consumes.
 *
 * Reading (the pages name the steps only):
 *     v_nk       = (d_n(k/32) * q_nk) * s_k         d*q is exact in binary32 (an
 *                                                   11-bit significand times a 7-bit
 *                                                   integer); one RN for the product with s_k
 *     amax_n     = max_k |v_nk|
 *     inv_n      = 127 / amax_n                     (binary32 RN)
 *     w_nk       = clamp(rint(v_nk * inv_n), -127, 127)
 *     w_scale_n  = amax_n / 127                     (binary32 RN)
 * the rounding and scale form of the activation quantiser; a row whose amax is
 * below 2^-120 requantises to zeros with scale 0.  s == NULL means s_k = 1.
 * d is given as binary16 bit patterns, [N, K/32] with row stride ldd; K is a
 * multiple of 32.  Inputs must keep every v finite.
 */

/* binary16 -> binary32, exact (normals, subnormals, zeros, infinities; a NaN
 * stays a NaN). */
static float f16_to_float(uint16_t h)
{
    const uint32_t sign = (uint32_t)(h >> 15) << 31;
    const uint32_t e = (h >> 10) & 0x1fu;
    const uint32_t m = h & 0x3ffu;
    float f;
    if (e == 0) {
        f = ldexpf((float)m, -24);                 /* subnormal or zero: m * 2^-24, exact */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        u |= sign;
        memcpy(&f, &u, sizeof f);
        return f;
    }
    uint32_t u;
    if (e == 31)
        u = sign | 0x7f800000u | (m << 13);        /* infinity or NaN */
    else
        u = sign | ((e - 15u + 127u) << 23) | (m << 13);
    memcpy(&f, &u, sizeof f);
    return f;
}

void oracle_f16_to_float(const uint16_t *h, int64_t n, float *f)
{
    for (int64_t i = 0; i < n; ++i)
        f[i] = f16_to_float(h[i]);
}

void oracle_smooth_requant(const int8_t *q, int64_t ldq, const uint16_t *d, int64_t ldd,
                           const float *s, int64_t N, int64_t K, int8_t *w, int64_t ldw,
                           float *w_scale)
{
    const float tiny = ldexpf(1.0f, -120);
    int64_t n;
#pragma omp parallel for schedule(static)
    for (n = 0; n < N; ++n) {
        const int8_t *qr = q + n * ldq;
        const uint16_t *dr = d + n * ldd;
        int8_t *wr = w + n * ldw;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = f16_to_float(dr[k / 32]) * (float)qr[k];
            if (s) v = v * s[k];
            float a = fabsf(v);
            if (a > amax) amax = a;
        }
        if (!(amax >= tiny)) {
            for (int64_t k = 0; k < K; ++k) wr[k] = 0;
            w_scale[n] = 0.0f;
            continue;
        }
        float inv = 127.0f / amax;
        for (int64_t k = 0; k < K; ++k) {
            float v = f16_to_float(dr[k / 32]) * (float)qr[k];
            if (s) v = v * s[k];
            float t = rintf(v * inv);            /* default mode: ties to even */
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            wr[k] = (int8_t)t;
        }
        w_scale[n] = amax / 127.0f;
    }
}

/* ------------------------------------------- exact integer contraction --- */
/*
 * [P1-bitwise], [P4-plan]: acc[m,n] = sum_k q[m,k] * w[n,k], exact.  The sum
 * is formed in int64 and must fit int32 (guaranteed for K <= ORACLE_MAX_K).
 * Returns 0, or -1 if some sum does not fit (never for valid inputs).
 */
int oracle_gemm_s32(const int8_t *q, int64_t ldq, const int8_t *w, int64_t ldw,
                    int64_t M, int64_t N, int64_t K, int32_t *acc, int64_t ldc)
{
    int bad = 0;
    int64_t m;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (m = 0; m < M; ++m) {
        const int8_t *qr = q + m * ldq;
        for (int64_t n = 0; n < N; ++n) {
            const int8_t *wr = w + n * ldw;
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k)
                s += (int64_t)qr[k] * (int64_t)wr[k];
            if (s > INT32_MAX || s < INT32_MIN) bad = 1;
            acc[m * ldc + n] = (int32_t)s;
        }
    }
    return bad ? -1 : 0;
}

/*
 * [P1-bitwise]: split-K partial sums remain integers.  The K range is cut into
 * S contiguous pieces of ceil(K/S) columns; each piece's partial is an int32
 * and the partials are added as int32 in piece order.  Integer addition is
 * exact, so this must equal oracle_gemm_s32 for every S (an invariant the
 * tests check).
 */
int oracle_gemm_s32_splitk(const int8_t *q, int64_t ldq, const int8_t *w,
                           int64_t ldw, int64_t M, int64_t N, int64_t K,
                           int S, int32_t *acc, int64_t ldc)
{
    if (S < 1) return -1;
    int64_t piece = (K + S - 1) / S;
    int bad = 0;
    int64_t m;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (m = 0; m < M; ++m) {
        const int8_t *qr = q + m * ldq;
        for (int64_t n = 0; n < N; ++n) {
            const int8_t *wr = w + n * ldw;
            int64_t total = 0;
            for (int s = 0; s < S; ++s) {
                int64_t k0 = (int64_t)s * piece, k1 = k0 + piece;
                if (k1 > K) k1 = K;
                int32_t part = 0;
                for (int64_t k = k0; k < k1; ++k)
                    part += (int32_t)qr[k] * (int32_t)wr[k];
                total += part;
            }
            if (total > INT32_MAX || total < INT32_MIN) bad = 1;
            acc[m * ldc + n] = (int32_t)total;
        }
    }
    return bad ? -1 : 0;
}

/* -------------------------------------------- fixed-order epilogue ------- */
/*
 * [P1-bitwise]: after exact int32 accumulation the result is scaled and added
 * to the residual "with a fixed rounding sequence".  Reading of that sequence
 * (each step one binary32 RN operation, no fused multiply-add, no bias):
 *     t = float(acc)              (int32 -> binary32, RN)
 *     t = t * a_scale[m]
 *     t = t * w_scale[n]
 *     t = t + float(residual)     (only when a residual is given)
 *     y = bf16_rne(t)
 */
void oracle_epilogue(const int32_t *acc, int64_t ldc, const float *a_scale,
                     const float *w_scale, const uint16_t *residual,
                     int64_t ldr, int64_t M, int64_t N, uint16_t *out,
                     int64_t ldo)
{
    int64_t m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            float t = (float)acc[m * ldc + n];
            t = t * a_scale[m];
            t = t * w_scale[n];
            if (residual) t = t + bf16_to_float(residual[m * ldr + n]);
            out[m * ldo + n] = float_to_bf16_rne(t);
        }
    }
}

/* One whole W8A8 linear call: contraction then epilogue.  acc_out (may be
 * NULL) receives the int32 accumulator, row stride N. */
int oracle_w8a8_linear(const int8_t *q, int64_t ldq, const float *a_scale,
                       const int8_t *w, int64_t ldw, const float *w_scale,
                       const uint16_t *residual, int64_t ldr, int64_t M,
                       int64_t N, int64_t K, uint16_t *out, int64_t ldo,
                       int32_t *acc_out)
{
    int32_t *acc = acc_out;
    int rc = oracle_gemm_s32(q, ldq, w, ldw, M, N, K, acc, N);
    if (rc) return rc;
    oracle_epilogue(acc, N, a_scale, w_scale, residual, ldr, M, N, out, ldo);
    return 0;
}

/* ------------------------------------------------------------ W4A8 --- */
/*
 * [P1-shared] names Q4_K_M weights loaded directly and a W4A8 run; the pages
 * give no arithmetic.  Reading: 4-bit weights are symmetric per output
 * channel, codes in [-7, 7] with one binary32 scale per channel (the form a
 * load-time requantisation leaves, as for Q8_0), packed two per byte: byte j
 * of a row holds code 2j in its low nibble and code 2j+1 in its high nibble,
 * each a 4-bit two's complement number.  W4A8 is then the W8A8 linear on the
 * unpacked codes: the same exact int32 contraction and epilogue.
 */
void oracle_unpack_w4(const uint8_t *w4, int64_t ldw4, int64_t N, int64_t K,
                      int8_t *w, int64_t ldw)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const unsigned b = w4[n * ldw4 + k / 2];
            const unsigned nib = (k % 2 == 0) ? (b & 0xfu) : (b >> 4);
            w[n * ldw + k] = (int8_t)(nib < 8 ? (int)nib : (int)nib - 16);
        }
}

int oracle_w4a8_linear(const int8_t *q, int64_t ldq, const float *a_scale,
                       const uint8_t *w4, int64_t ldw4, const float *w_scale,
                       const uint16_t *residual, int64_t ldr, int64_t M,
                       int64_t N, int64_t K, uint16_t *out, int64_t ldo,
                       int32_t *acc_out, int8_t *w_scratch)
{
    /* w_scratch: N * K bytes for the unpacked codes */
    oracle_unpack_w4(w4, ldw4, N, K, w_scratch, K);
    return oracle_w8a8_linear(q, ldq, a_scale, w_scratch, K, w_scale, residual, ldr,
                              M, N, K, out, ldo, acc_out);
}

/* ------------------------------------- restriction to answer positions --- */
/*
 * [P1-shared]: in the last layer only the positions needed for answers are
 * computed.  Every step of the layer is per token, so the restricted layer is
 * the full layer's rows at those positions; these two functions state it by
 * running the full definitions above on the selected rows.
 *
 * oracle_quant_act_rows: q row i, a_scale[i] = the quantisation of x row
 * rows[i] (x has M_x rows).  An index outside [0, M_x) gives a zero q row,
 * a NaN scale, and ORACLE_ERR_ROW_RANGE in the returned error bits.
 */
uint32_t oracle_quant_act_rows(const uint16_t *x, int64_t ldx, int64_t M_x,
                               const int32_t *rows, int64_t n_rows,
                               const float *inv_s, int64_t K, int8_t *q,
                               int64_t ldq, float *a_scale)
{
    uint32_t err = 0;
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t r = rows[i];
        if (r < 0 || r >= M_x) {
            memset(q + i * ldq, 0, (size_t)K);
            a_scale[i] = NAN;
            err |= ORACLE_ERR_ROW_RANGE;
            continue;
        }
        oracle_quant_act(x + r * ldx, ldx, inv_s, 1, K, q + i * ldq, ldq, a_scale + i);
    }
    return err;
}

/*
 * oracle_w8a8_linear_rows: oracle_w8a8_linear whose residual row for output
 * row m is residual row res_rows[m] (the residual has M_res rows).  An index
 * outside [0, M_res) makes output row m NaN (bf16 0x7fc0) and sets
 * ORACLE_ERR_ROW_RANGE in *err.  Returns what oracle_w8a8_linear returns.
 */
int oracle_w8a8_linear_rows(const int8_t *q, int64_t ldq, const float *a_scale,
                            const int8_t *w, int64_t ldw, const float *w_scale,
                            const uint16_t *residual, int64_t ldr, int64_t M_res,
                            const int32_t *res_rows, int64_t M, int64_t N,
                            int64_t K, uint16_t *out, int64_t ldo,
                            int32_t *acc_out, uint32_t *err)
{
    int rc = oracle_gemm_s32(q, ldq, w, ldw, M, N, K, acc_out, N);
    if (rc) return rc;
    for (int64_t m = 0; m < M; ++m) {
        const int64_t r = res_rows[m];
        if (r < 0 || r >= M_res) {
            for (int64_t n = 0; n < N; ++n) out[m * ldo + n] = 0x7fc0u;
            *err |= ORACLE_ERR_ROW_RANGE;
            continue;
        }
        oracle_epilogue(acc_out + m * N, N, a_scale + m, w_scale, residual + r * ldr, ldr, 1, N,
                        out + m * ldo, ldo);
    }
    return 0;
}

/* ------------------------------------------------------------- exp ------- */
/*
 * Exponential used by the candidate softmax, for x <= 0.  Reading: the pages
 * say the read-out path is fixed but name no exp; a function both sides can
 * evaluate bit for bit is needed, so it is defined here by a published method
 * and evaluated with explicit binary32 RN operations:
 *   Cody-Waite argument reduction (W. J. Cody, W. Waite, "Software Manual for
 *   the Elementary Functions", 1980): x = n ln2 + r with n = rint(x log2 e);
 *   ln2 is split as LN2_HI + LN2_LO where LN2_HI = 355/512 (nine significant
 *   bits, so n * LN2_HI is exact for |n| < 2^15) and LN2_LO = RN(ln2 - 355/512);
 *   r = (x - n*LN2_HI) - n*LN2_LO.
 *   e^r from its Taylor series truncated after r^7/7! (|r| < 0.35, truncation
 *   error below 1e-8 relative), Horner form, coefficients RN(1/k!).
 *   Result = p * 2^n, 2^n built in the exponent field; n < -126 gives 0.
 */
float oracle_exp(float x)
{
    const float LOG2E = 0x1.715476p+0f;        /* RN(1/ln 2)          */
    const float LN2_HI = 0x1.63p-1f;           /* 355/512             */
    const float LN2_LO = -0x1.bd0106p-13f;     /* RN(ln 2 - 355/512)  */
    const float C2 = 0x1p-1f;                  /* 1/2!                */
    const float C3 = 0x1.555556p-3f;           /* RN(1/3!)            */
    const float C4 = 0x1.555556p-5f;           /* RN(1/4!)            */
    const float C5 = 0x1.111112p-7f;           /* RN(1/5!)            */
    const float C6 = 0x1.6c16c2p-10f;          /* RN(1/6!)            */
    const float C7 = 0x1.a01a02p-13f;          /* RN(1/7!)            */
    if (x != x) return x;
    if (x > 0.0f) x = 0.0f;                    /* domain is x <= 0    */
    float n = rintf(x * LOG2E);
    if (n < -126.0f) return 0.0f;
    float r = x - n * LN2_HI;
    r = r - n * LN2_LO;
    float p = C7;
    p = p * r + C6;
    p = p * r + C5;
    p = p * r + C4;
    p = p * r + C3;
    p = p * r + C2;
    p = p * r + 1.0f;
    p = p * r + 1.0f;
    uint32_t bits = (uint32_t)((int)n + 127) << 23;
    float two_n;
    memcpy(&two_n, &bits, sizeof two_n);
    return p * two_n;
}

void oracle_exp_batch(const float *x, int64_t n, float *y)
{
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_exp(x[i]);
}

/* ------------------------------------------- candidate read-out ---------- */
/*
 * [P1-evidence], [P4-plan], [P4-impl]: the output layer scores only the valid
 * candidates of each answer position and normalises within that set.
 *   1. The hidden row h_p is quantised exactly like any activation row
 *      (oracle_quant_act, optional smoothing).
 *   2. For each candidate id c: acc = sum_k q_p[k] * W[c,k]  (exact int32).
 *   3. logit = (float(acc) * a_scale[p]) * lm_scale[c]   (binary32 RN; the
 *      logit is kept in binary32, not rounded to bf16 -- reading).
 *   4. mx = max logit; e_c = oracle_exp(logit_c - mx); s = sum of e_c in the
 *      caller's candidate order; prob_c = e_c / s.
 * Candidate lists are CSR: cand_offsets[P+1], cand_ids[T].  Returns 0; or a
 * negative code without touching that position's outputs' validity rules:
 * -1 offsets malformed, -2 count outside [1, 64], -3 id outside [0, V),
 * -4 duplicate id within a position.  Invalid positions get NaN outputs.
 */
int oracle_candidate_readout(const uint16_t *h, int64_t ldh, const float *inv_s,
                             const int8_t *lm_head, int64_t ldw,
                             const float *lm_scale, int64_t V, int64_t K,
                             const int32_t *cand_offsets,
                             const int32_t *cand_ids, int64_t P, int64_t T,
                             float *logits, float *probs)
{
    const float qnan = nanf("");
    int status = 0;
    if (cand_offsets[0] != 0 || cand_offsets[P] != T) return -1;
    int64_t p;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : status)
    for (p = 0; p < P; ++p) {
        int64_t b = cand_offsets[p], e = cand_offsets[p + 1];
        int64_t cnt = e - b;
        int err = 0;
        if (b < 0 || e > T || cnt < 0) err = -1;
        else if (cnt < 1 || cnt > ORACLE_MAX_CANDIDATES) err = -2;
        else {
            for (int64_t i = b; i < e && !err; ++i) {
                if (cand_ids[i] < 0 || cand_ids[i] >= V) err = -3;
                for (int64_t j = b; j < i && !err; ++j)
                    if (cand_ids[j] == cand_ids[i]) err = -4;
            }
        }
        if (err) {
            if (b >= 0 && e <= T)
                for (int64_t i = b; i < e; ++i) logits[i] = probs[i] = qnan;
            if (err < status) status = err;
            continue;
        }
        int8_t qrow[ORACLE_MAX_K];
        float a_scale;
        oracle_quant_act(h + p * ldh, ldh, inv_s, 1, K, qrow, K, &a_scale);
        float e_val[ORACLE_MAX_CANDIDATES];
        float mx = -INFINITY;
        for (int64_t i = b; i < e; ++i) {
            const int8_t *wr = lm_head + (int64_t)cand_ids[i] * ldw;
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)qrow[k] * (int64_t)wr[k];
            float t = (float)(int32_t)s;
            t = t * a_scale;
            t = t * lm_scale[cand_ids[i]];
            logits[i] = t;
            if (t > mx) mx = t;
        }
        float sum = 0.0f;
        for (int64_t i = b; i < e; ++i) {
            e_val[i - b] = oracle_exp(logits[i] - mx);
            sum = sum + e_val[i - b];
        }
        for (int64_t i = b; i < e; ++i) probs[i] = e_val[i - b] / sum;
    }
    return status;
}

/*
 * Column-parallel read-out (the LM head split by vocabulary rows; a reading
 * of [P4-plan]: the candidate softmax needs only the candidates' logits).
 *
 * oracle_candidate_logits_shard: the logits of oracle_candidate_readout for
 * the candidates whose id lies in [v0, v0 + Vs), from the shard's rows
 * (lm_shard row id - v0, lm_scale_shard[id - v0]); -0.0 for every other
 * candidate of a valid position.  Validation and return codes as
 * oracle_candidate_readout (ids checked against the whole head's V);
 * invalid positions get NaN logits.
 */
int oracle_candidate_logits_shard(const uint16_t *h, int64_t ldh, const float *inv_s,
                                  const int8_t *lm_shard, int64_t ldw,
                                  const float *lm_scale_shard, int64_t v0, int64_t Vs,
                                  int64_t V, int64_t K, const int32_t *cand_offsets,
                                  const int32_t *cand_ids, int64_t P, int64_t T,
                                  float *logits)
{
    const float qnan = nanf("");
    int status = 0;
    if (cand_offsets[0] != 0 || cand_offsets[P] != T) return -1;
    for (int64_t p = 0; p < P; ++p) {
        int64_t b = cand_offsets[p], e = cand_offsets[p + 1];
        int64_t cnt = e - b;
        int err = 0;
        if (b < 0 || e > T || cnt < 0) err = -1;
        else if (cnt < 1 || cnt > ORACLE_MAX_CANDIDATES) err = -2;
        else {
            for (int64_t i = b; i < e && !err; ++i) {
                if (cand_ids[i] < 0 || cand_ids[i] >= V) err = -3;
                for (int64_t j = b; j < i && !err; ++j)
                    if (cand_ids[j] == cand_ids[i]) err = -4;
            }
        }
        if (err) {
            if (b >= 0 && e <= T)
                for (int64_t i = b; i < e; ++i) logits[i] = qnan;
            if (err < status) status = err;
            continue;
        }
        int8_t qrow[ORACLE_MAX_K];
        float a_scale;
        oracle_quant_act(h + p * ldh, ldh, inv_s, 1, K, qrow, K, &a_scale);
        for (int64_t i = b; i < e; ++i) {
            const int64_t id = cand_ids[i];
            if (id < v0 || id >= v0 + Vs) {
                logits[i] = -0.0f;
                continue;
            }
            const int8_t *wr = lm_shard + (id - v0) * ldw;
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)qrow[k] * (int64_t)wr[k];
            float t = (float)(int32_t)s;
            t = t * a_scale;
            t = t * lm_scale_shard[id - v0];
            logits[i] = t;
        }
    }
    return status;
}

/*
 * oracle_candidate_softmax: step 4 of oracle_candidate_readout on given
 * logits -- mx = max logit; e_c = oracle_exp(logit_c - mx); s = sum of e_c
 * in list order; prob_c = e_c / s.  Returns -1 / -2 for malformed offsets or
 * a count outside [1, 64] (NaN probabilities); a position with a NaN logit
 * gets NaN probabilities (its error was reported where the logits were made).
 */
int oracle_candidate_softmax(const float *logits, const int32_t *cand_offsets, int64_t P,
                             int64_t T, float *probs)
{
    const float qnan = nanf("");
    int status = 0;
    if (cand_offsets[0] != 0 || cand_offsets[P] != T) return -1;
    for (int64_t p = 0; p < P; ++p) {
        int64_t b = cand_offsets[p], e = cand_offsets[p + 1];
        int64_t cnt = e - b;
        int err = 0;
        if (b < 0 || e > T || cnt < 0) err = -1;
        else if (cnt < 1 || cnt > ORACLE_MAX_CANDIDATES) err = -2;
        int has_nan = 0;
        if (!err)
            for (int64_t i = b; i < e; ++i) has_nan |= logits[i] != logits[i];
        if (err || has_nan) {
            if (b >= 0 && e <= T)
                for (int64_t i = b; i < e; ++i) probs[i] = qnan;
            if (err < status) status = err;
            continue;
        }
        float mx = -INFINITY;
        for (int64_t i = b; i < e; ++i)
            if (logits[i] > mx) mx = logits[i];
        float e_val[ORACLE_MAX_CANDIDATES];
        float sum = 0.0f;
        for (int64_t i = b; i < e; ++i) {
            e_val[i - b] = oracle_exp(logits[i] - mx);
            sum = sum + e_val[i - b];
        }
        for (int64_t i = b; i < e; ++i) probs[i] = e_val[i - b] / sum;
    }
    return status;
}

/* ------------------------------------------------ bf16 helpers, exported -- */
void oracle_bf16_to_float(const uint16_t *h, int64_t n, float *f)
{
    for (int64_t i = 0; i < n; ++i) f[i] = bf16_to_float(h[i]);
}

void oracle_float_to_bf16(const float *f, int64_t n, uint16_t *h)
{
    for (int64_t i = 0; i < n; ++i) h[i] = float_to_bf16_rne(f[i]);
}
