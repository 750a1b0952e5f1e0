/*
 * fp8_oracle.c -- plain, slow, obviously correct CPU oracle for the FP8
 * delayed-scaling linear layer and its mixed-precision master step.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the CPU
 * baseline leg of the benchmark are the only users of this file's library.
 * It includes no header and calls no function of the CUDA library, and the
 * CUDA library includes and links nothing from here.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        [-fopenmp] (OpenMP only splits independent rows / elements across
 *        threads; it never reorders a sum).
 *
 * Pages cited (title -- site):
 *   [TE-FP8]  "Transformer Engine으로 FP8 사용하기" -- coniverse.tistory.com
 *   [MP]      "LLM) Mixed-Precision 개념 및 학습 방법 알아보기"
 *             -- data-newbie.tistory.com
 *   [PT-FP8]  "Các kiểu dữ liệu FP8 gốc của PyTorch ..." (PyTorch native FP8
 *             data types) -- hotroai.com
 *   [H100-Q]  "Как работает FP8 quantization на H100 (Transformer Engine)?"
 *             -- aivaro.ru
 *
 * Every function here is pinned by a CPU test against something other than
 * itself (the pages' printed values, torch's float8 casts, brute force,
 * exact rational arithmetic, closed forms); none is "parity unpinned".
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_E4M3 = 0, ORC_E5M2 = 1 };
enum { ORC_AMAX_MAX = 0, ORC_AMAX_MOST_RECENT = 1 };

/* ------------------------------------------------------------------------ */
/* Formats ([TE-FP8] "Introduction to FP8"; [PT-FP8] finfo table;           */
/* [H100-Q] section 1): E4M3 = 1 sign, 4 exponent (bias 7), 3 mantissa bits,*/
/* largest finite 448, no infinities, NaN = S.1111.111. E5M2 = 1 sign,      */
/* 5 exponent (bias 15), 2 mantissa bits, IEEE-style Inf/NaN at exponent 31,*/
/* largest finite 57344.                                                     */
/* ------------------------------------------------------------------------ */

static int fmt_mbits(int fmt) { return fmt == ORC_E4M3 ? 3 : 2; }
static int fmt_bias(int fmt) { return fmt == ORC_E4M3 ? 7 : 15; }
/* floor(log2(largest finite)) */
static int fmt_emax(int fmt) { return fmt == ORC_E4M3 ? 8 : 15; }
static uint8_t fmt_maxcode(int fmt) { return fmt == ORC_E4M3 ? 0x7E : 0x7B; }

int orc_version(void) { return 1; }

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

double orc_fmt_max(int fmt) { return fmt == ORC_E4M3 ? 448.0 : 57344.0; }

/* Decoder: the value a code stands for, written out from the bit fields. */
double orc_decode(int fmt, uint8_t c)
{
    const int s = c >> 7;
    double v;
    if (fmt == ORC_E4M3) {
        const int e = (c >> 3) & 0xF, m = c & 0x7;
        if (e == 0xF && m == 0x7)
            return NAN;
        if (e == 0)
            v = ldexp((double)m / 8.0, -6);           /* subnormal */
        else
            v = ldexp(1.0 + (double)m / 8.0, e - 7);  /* normal */
    } else {
        const int e = (c >> 2) & 0x1F, m = c & 0x3;
        if (e == 0x1F)
            return m == 0 ? (s ? -INFINITY : INFINITY) : NAN;
        if (e == 0)
            v = ldexp((double)m / 4.0, -14);
        else
            v = ldexp(1.0 + (double)m / 4.0, e - 15);
    }
    return s ? -v : v;
}

/*
 * Encoder: round-to-nearest-even of the exact binary value of an fp32 input,
 * computed with integer arithmetic on its bits, saturating at the largest
 * finite value.
 *   - |x| above the largest finite value (Inf included) -> +-largest finite
 *     (the cast "saturates"; [TE-FP8] "Introduction to FP8" gives the ranges);
 *   - NaN -> 0x7F (positive NaN code of both formats);
 *   - -0 -> 0x80; values below half the smallest subnormal -> signed zero;
 *   - gradual underflow into the subnormals (finfo lists a smallest *normal*
 *     value, [PT-FP8] finfo table, so the codes below it are subnormals).
 */
uint8_t orc_encode(int fmt, float x)
{
    uint32_t b;
    memcpy(&b, &x, sizeof b);
    const uint8_t sign = (b >> 31) ? 0x80 : 0x00;
    const uint32_t a = b & 0x7FFFFFFFu;
    const int mb = fmt_mbits(fmt), bias = fmt_bias(fmt);
    const int emin = 1 - bias; /* exponent of the smallest normal */

    if (a > 0x7F800000u)
        return 0x7F;                         /* NaN */
    if (a == 0x7F800000u)
        return sign | fmt_maxcode(fmt);      /* +-Inf saturates */
    if (a == 0)
        return sign;                         /* +-0 */

    /* |x| = M * 2^E with an integer significand M */
    const uint32_t ef = a >> 23;
    uint64_t M;
    int E;
    if (ef == 0) {
        M = a & 0x7FFFFFu;
        E = -149;
    } else {
        M = (a & 0x7FFFFFu) | 0x800000u;
        E = (int)ef - 150;
    }
    const int lead = E + (63 - __builtin_clzll(M)); /* floor(log2 |x|) */
    if (lead > fmt_emax(fmt))
        return sign | fmt_maxcode(fmt);      /* at least 2^(emax+1): saturate */

    /* q = exponent of one unit in the last place of the target at |x| */
    int q = (lead > emin ? lead : emin) - mb;
    const int sh = q - E;
    uint64_t n;
    if (sh <= 0) {
        n = M << (-sh);
    } else if (sh >= 40) {
        n = 0; /* M < 2^24 is below half a unit */
    } else {
        const uint64_t rem = M & ((1ull << sh) - 1ull);
        const uint64_t half = 1ull << (sh - 1);
        n = M >> sh;
        if (rem > half || (rem == half && (n & 1ull)))
            n += 1; /* round half to even */
    }
    if (n == 0)
        return sign;
    if (n == (1ull << (mb + 1))) { /* rounding carried into the next binade */
        n >>= 1;
        q += 1;
    }
    int efield, mfield;
    if (n < (1ull << mb)) { /* subnormal: only when q == emin - mb */
        efield = 0;
        mfield = (int)n;
    } else {
        efield = q + mb + bias;
        mfield = (int)(n - (1ull << mb));
    }
    if (fmt == ORC_E4M3) {
        if (efield > 15 || (efield == 15 && mfield == 7))
            return sign | fmt_maxcode(fmt);
    } else {
        if (efield >= 31)
            return sign | fmt_maxcode(fmt);
    }
    return (uint8_t)(sign | (efield << mb) | mfield);
}

static float bf16_to_f32(uint16_t h)
{
    const uint32_t b = (uint32_t)h << 16; /* bf16 is the top half of fp32 */
    float f;
    memcpy(&f, &b, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* Cast under a scale ([H100-Q] section 3, steps 2-3; [TE-FP8] "Scaling     */
/* factor 선택 전략"): q[i] = encode(fl32(x[i] * scale)). The product is one */
/* IEEE fp32 multiply; bf16 inputs widen to fp32 exactly first.             */
/* ------------------------------------------------------------------------ */

void orc_cast_f32(const float *x, int64_t n, float scale, int fmt, uint8_t *q)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) {
        const float p = x[i] * scale;
        q[i] = orc_encode(fmt, p);
    }
}

void orc_cast_bf16(const uint16_t *x, int64_t n, float scale, int fmt, uint8_t *q)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) {
        const float p = bf16_to_f32(x[i]) * scale;
        q[i] = orc_encode(fmt, p);
    }
}

/* The transposed copy: qt[c * rows + r] = q[r * cols + c]. */
void orc_transpose_u8(const uint8_t *q, int64_t rows, int64_t cols, uint8_t *qt)
{
    int64_t c;
#pragma omp parallel for schedule(static)
    for (c = 0; c < cols; ++c)
        for (int64_t r = 0; r < rows; ++r)
            qt[c * rows + r] = q[r * cols + c];
}

/* amax = max |x[i]| over the unscaled input, starting at +0; a NaN element */
/* never wins a comparison and so is ignored ([TE-FP8] "Scaling factor 선택  */
/* 전략"; [H100-Q] section 3, step 2).                                       */
float orc_amax_f32(const float *x, int64_t n)
{
    float m = 0.0f;
    int64_t i;
#pragma omp parallel for reduction(max : m) schedule(static)
    for (i = 0; i < n; ++i) {
        const float a = fabsf(x[i]);
        if (a > m)
            m = a;
    }
    return m;
}

float orc_amax_bf16(const uint16_t *x, int64_t n)
{
    float m = 0.0f;
    int64_t i;
#pragma omp parallel for reduction(max : m) schedule(static)
    for (i = 0; i < n; ++i) {
        const float a = fabsf(bf16_to_f32(x[i]));
        if (a > m)
            m = a;
    }
    return m;
}

/* ------------------------------------------------------------------------ */
/* Delayed scaling ([TE-FP8] "Scaling factor 선택 전략" and the              */
/* DelayedScaling recipe under "FP8 사용방안(recipe)"; [H100-Q] section 10). */
/* One update of one tensor's bookkeeping, in this order:                   */
/*   1. roll the history one place (newest at index 0) and insert cur_amax; */
/*   2. a = max over the history (algo "max") or the newest entry           */
/*      ("most_recent");                                                    */
/*   3. if a is positive and finite: s = fl32(fmt_max / a) * 2^-margin,      */
/*      rounded once to fp32; the scale takes s when s is finite and > 0;    */
/*      otherwise the scale keeps its value;                                 */
/*   4. scale_inv = fl32(1 / scale); cur_amax = 0.                           */
/* ------------------------------------------------------------------------ */

void orc_scale_update(float *hist, int32_t L, float *scale, float *scale_inv, float *cur_amax,
                      int fmt, int algo, int32_t margin)
{
    for (int32_t j = L - 1; j >= 1; --j)
        hist[j] = hist[j - 1];
    if (L >= 1)
        hist[0] = *cur_amax;

    float a;
    if (algo == ORC_AMAX_MAX) {
        a = 0.0f;
        for (int32_t j = 0; j < L; ++j)
            if (hist[j] > a)
                a = hist[j];
    } else {
        a = (L >= 1) ? hist[0] : *cur_amax;
    }

    if (a > 0.0f && isfinite(a)) {
        const float s = (float)orc_fmt_max(fmt) / a;      /* one fp32 division */
        const double t = (double)s * ldexp(1.0, -margin); /* exact in fp64 */
        const float s2 = (float)t;                        /* one rounding */
        if (isfinite(s2) && s2 > 0.0f)
            *scale = s2;
    }
    *scale_inv = 1.0f / *scale;
    *cur_amax = 0.0f;
}

/* ------------------------------------------------------------------------ */
/* GEMM reference. The FP8 linear computes products of FP8 operands and     */
/* accumulates them in high precision ([MP] "Accumulation into FP32"), then */
/* divides out the two scales ([H100-Q] section 3, step 4) and adds the     */
/* bias ([PT-FP8] the torch._scaled_mm listing takes a bias):               */
/*   ref[i, j] = (sum_k dec(A[i, k]) * dec(B[j, k])) * sinv_a * sinv_b       */
/*               + bias[j]                                                  */
/* with A (rows_a x kc) and B (rows_b x kc) both contiguous along k. The sum */
/* is a plain loop in fp64. Every FP8 x FP8 product is exact in fp64, and   */
/* for E4M3 x E4M3 the whole sum is exact up to kc = 2^14 (the products span */
/* 2^-18 .. 2^18). abs_out, when given, receives                            */
/* sum_k |dec(A[i,k]) dec(B[j,k])| * sinv_a * sinv_b, the scale of the       */
/* accumulation error a correct kernel may make.                            */
/* Only the rows listed in row_idx (or all rows when row_idx is NULL) are   */
/* computed; out has n_rows x rows_b entries.                               */
/* ------------------------------------------------------------------------ */

void orc_gemm_ref(const uint8_t *A, int fmt_a, const uint8_t *B, int fmt_b, int64_t rows_a,
                  int64_t rows_b, int64_t kc, const int64_t *row_idx, int64_t n_rows, double sinv_a,
                  double sinv_b, const double *bias, double *out, double *abs_out)
{
    (void)rows_a;
    double lut_a[256], lut_b[256];
    for (int c = 0; c < 256; ++c) {
        lut_a[c] = orc_decode(fmt_a, (uint8_t)c);
        lut_b[c] = orc_decode(fmt_b, (uint8_t)c);
    }
    /* decode B once into fp64 */
    double *bd = (double *)malloc((size_t)(rows_b * kc > 0 ? rows_b * kc : 1) * sizeof(double));
    if (!bd)
        return;
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < rows_b * kc; ++t)
        bd[t] = lut_b[B[t]];

    int64_t ii;
#pragma omp parallel for schedule(dynamic, 1)
    for (ii = 0; ii < n_rows; ++ii) {
        const int64_t i = row_idx ? row_idx[ii] : ii;
        double *ad = (double *)malloc((size_t)(kc > 0 ? kc : 1) * sizeof(double));
        if (!ad)
            continue;
        for (int64_t k = 0; k < kc; ++k)
            ad[k] = lut_a[A[i * kc + k]];
        for (int64_t j = 0; j < rows_b; ++j) {
            const double *bj = bd + j * kc;
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < kc; ++k) {
                const double p = ad[k] * bj[k];
                s += p;
                sa += fabs(p);
            }
            out[ii * rows_b + j] = s * sinv_a * sinv_b + (bias ? bias[j] : 0.0);
            if (abs_out)
                abs_out[ii * rows_b + j] = sa * sinv_a * sinv_b;
        }
        free(ad);
    }
    free(bd);
}

/* ------------------------------------------------------------------------ */
/* Mixed-precision master step ([MP] "FP32 Master Copy of Weights",         */
/* "Mixed-Precision Training Iteration" steps 5 and 7, and the dynamic      */
/* loss-scale procedure that skips a step on Inf/NaN and grows S after a    */
/* run of clean steps; [H100-Q] section 7, FP32 master weights with FP8     */
/* copies).                                                                 */
/*   pass 1: found_inf = any gradient is Inf or NaN.                        */
/*   found_inf: S = S * backoff, growth = 0, nothing else changes.          */
/*   otherwise, per element (all fp32, fused multiply-adds correctly        */
/*   rounded as C's fmaf):                                                  */
/*       u = fp32(g) * fl32(1 / S)            -- unscale                    */
/*       v = fmaf(mu, v, u)                   -- momentum                   */
/*       w = fmaf(-lr, v, w)                  -- FP32 master update         */
/*       w8 = encode_E4M3(fl32(w * scale_w))  -- FP8 copy for the next step */
/*       cur_amax_w = max(cur_amax_w, |w|)                                  */
/*     then growth += 1 and, when growth reaches growth_interval,           */
/*     S = S * growth_factor and growth = 0.                                */
/* ------------------------------------------------------------------------ */

void orc_master_step(const uint16_t *g, int64_t n, float *w, float *v, uint8_t *w8, float scale_w,
                     float *cur_amax_w, float *S, int32_t *growth, int32_t *found_inf, float lr,
                     float mu, float backoff, float growth_factor, int32_t growth_interval)
{
    int found = 0;
    int64_t i;
#pragma omp parallel for reduction(| : found) schedule(static)
    for (i = 0; i < n; ++i)
        if ((g[i] & 0x7F80u) == 0x7F80u) /* exponent all ones: Inf or NaN */
            found |= 1;
    *found_inf = found;
    if (found) {
        *S = *S * backoff;
        *growth = 0;
        return;
    }
    const float inv_s = 1.0f / *S;
    const float neg_lr = -lr;
    float am = *cur_amax_w;
#pragma omp parallel for reduction(max : am) schedule(static)
    for (i = 0; i < n; ++i) {
        const float u = bf16_to_f32(g[i]) * inv_s;
        const float vn = fmaf(mu, v[i], u);
        const float wn = fmaf(neg_lr, vn, w[i]);
        v[i] = vn;
        w[i] = wn;
        w8[i] = orc_encode(ORC_E4M3, wn * scale_w);
        const float a = fabsf(wn);
        if (a > am)
            am = a;
    }
    *cur_amax_w = am;
    *growth += 1;
    if (*growth >= growth_interval) {
        *S = *S * growth_factor;
        *growth = 0;
    }
}

/* ------------------------------------------------------------------------ */
/* Bias gradient of the linear layer y = x W^T + b (the te.Linear example   */
/* with bias=True under [TE-FP8] "FP8 사용방안(recipe)", backward under      */
/* "Backward Pass 처리"): db[c] = sum_r dy[r, c], a plain fp64 column sum of */
/* the unscaled gradient; abs_out[c] = sum_r |dy[r, c]| bounds the rounding  */
/* error of any fp32 summation order. dy is fp32 (is_bf16 = 0) or bf16 bits. */
/* ------------------------------------------------------------------------ */

void orc_dbias(const void *dy, int is_bf16, int64_t rows, int64_t cols, double *out, double *abs_out)
{
    int64_t c;
#pragma omp parallel for schedule(static)
    for (c = 0; c < cols; ++c) {
        double s = 0.0, a = 0.0;
        for (int64_t r = 0; r < rows; ++r) {
            const double v = is_bf16 ? (double)bf16_to_f32(((const uint16_t *)dy)[r * cols + c])
                                     : (double)((const float *)dy)[r * cols + c];
            s += v;
            a += fabs(v);
        }
        out[c] = s;
        if (abs_out)
            abs_out[c] = a;
    }
}

/* ------------------------------------------------------------------------ */
/* Adam master step. The PyTorch-native FP8 page trains its model with      */
/* torch.optim.Adam ([PT-FP8], the float8_experimental training loop); the  */
/* mixed-precision frame is the SGD step's ([MP]: unscale by 1/S, skip on   */
/* Inf/NaN and lower S, FP32 master, low-precision copy). The update, each  */
/* operation one correctly rounded fp32 operation in this order:            */
/*   u   = fp32(g) * fl32(1 / S)                                            */
/*   b1t = fl32(b1p * beta1),  b2t = fl32(b2p * beta2)  (beta^t; b1p, b2p   */
/*         hold beta^(t-1), start at 1, advance on clean steps only)        */
/*   m   = fmaf(beta1, m, fl32(1 - beta1) * u)                              */
/*   v   = fmaf(beta2, v, fl32(1 - beta2) * fl32(u * u))                    */
/*   mh  = m / fl32(1 - b1t),  vh = v / fl32(1 - b2t)                       */
/*   w   = fmaf(-lr, mh / (sqrtf(vh) + eps), w)                             */
/*   w8  = encode_E4M3(fl32(w * scale_w)); cur_amax_w = max(.., |w|)        */
/* then, on a clean step, b1p = b1t, b2p = b2t and the loss-scale update.   */
/* ------------------------------------------------------------------------ */

void orc_adam_step(const uint16_t *g, int64_t n, float *w, float *m, float *v, uint8_t *w8, float scale_w,
                   float *cur_amax_w, float *S, int32_t *growth, int32_t *found_inf, float *b1p, float *b2p,
                   float lr, float beta1, float beta2, float eps, float backoff, float growth_factor,
                   int32_t growth_interval)
{
    int found = 0;
    int64_t i;
#pragma omp parallel for reduction(| : found) schedule(static)
    for (i = 0; i < n; ++i)
        if ((g[i] & 0x7F80u) == 0x7F80u)
            found |= 1;
    *found_inf = found;
    if (found) {
        *S = *S * backoff;
        *growth = 0;
        return;
    }
    const float inv_s = 1.0f / *S;
    const float b1t = *b1p * beta1, b2t = *b2p * beta2;
    const float c1 = 1.0f - beta1, c2 = 1.0f - beta2;
    const float bc1 = 1.0f - b1t, bc2 = 1.0f - b2t;
    const float neg_lr = -lr;
    float am = *cur_amax_w;
#pragma omp parallel for reduction(max : am) schedule(static)
    for (i = 0; i < n; ++i) {
        const float u = bf16_to_f32(g[i]) * inv_s;
        const float mn = fmaf(beta1, m[i], c1 * u);
        const float uu = u * u;
        const float vn = fmaf(beta2, v[i], c2 * uu);
        const float mh = mn / bc1;
        const float vh = vn / bc2;
        const float den = sqrtf(vh) + eps;
        const float wn = fmaf(neg_lr, mh / den, w[i]);
        m[i] = mn;
        v[i] = vn;
        w[i] = wn;
        w8[i] = orc_encode(ORC_E4M3, wn * scale_w);
        const float a = fabsf(wn);
        if (a > am)
            am = a;
    }
    *cur_amax_w = am;
    *b1p = b1t;
    *b2p = b2t;
    *growth += 1;
    if (*growth >= growth_interval) {
        *S = *S * growth_factor;
        *growth = 0;
    }
}
