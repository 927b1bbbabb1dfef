/*
 * fp8_oracle.c -- CPU oracle for the FP8 delayed-scaling linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * GPU path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or constant generator with the CUDA library, and it includes nothing from
 * it.
 *
 * Sources (the three web pages this method is described on):
 *  [P1] "NVIDIA Transformer Engine and FP8 mixed precision: implementation
 *       guide" (ai-tool-zukan.com) -- section "What are Transformer Engine and
 *       FP8 mixed precision" (E4M3 = 4 exponent / 3 mantissa bits for the
 *       forward pass, E5M2 = 5 / 2 for the backward pass; dynamic scaling
 *       watches each tensor's range) and section "Dynamic scaling and the FP8
 *       recipe" (DelayedScaling: margin, fp8_format, amax_history_len;
 *       Format.HYBRID = E4M3 forward, E5M2 backward).
 *  [P2] "FP8 quantization with NVIDIA TensorRT" (ai.warp-studio.com) -- section
 *       on the FP8 workflow (Q/DQ nodes, Absolute-Max calibration).
 *  [P3] "Mixed-precision training" wiki note (notes.yuuk.io) -- "Definition"
 *       table: FP8 E4M3 (S1E4M3) max 448, relative error ~1e-1; FP8 E5M2
 *       (S1E5M2) max 57,344, relative error ~2e-1, same range as FP16; and the
 *       "per-tensor scaling is the key" bullet (delayed or just-in-time
 *       scaling), "extension to FP8" bullet (only the GEMMs run in FP8, with
 *       higher-precision accumulation).
 *
 * Readings taken where the pages are silent (each one is listed in the design
 * notes of the repository):
 *  - The E4M3 variant is the one whose largest finite value is 448: exponent
 *    field 15 holds finite values, only S.1111.111 is NaN, no infinities.  An
 *    IEEE-style E4M3 would stop at 240, which contradicts the 448 of [P3].
 *    E5M2 is IEEE-style (bias 15, infinities and NaNs at exponent 31), which
 *    gives 57,344 and "the same range as FP16".
 *  - Scaled cast: v = fl32(x * s) (one IEEE binary32 multiply), then v is
 *    rounded to the nearest FP8 value with ties to the even code; |v| beyond
 *    the largest finite value (and +-inf) saturates to +-max; NaN stays NaN;
 *    the sign of zero is kept.
 *  - amax = max |x| over the tensor, NaN entries skipped, result exact.
 *  - Scale update (the formula of the delayed-scaling recipe):
 *    history <- [amax, history[0 .. L-2]];  m = max(history);
 *    if 0 < m < inf:  s = fl32(fl32(fmax / m) * 2^-margin), +inf clamped to
 *    FLT_MAX, s_inv = fl32(1 / s);  otherwise s and s_inv stay as they were.
 *  - GEMM: operands decoded exactly, products and sums exact (integer path)
 *    or in double (sampled path); dequant epilogue
 *    y = bf16_rne(fl32(fl32(acc) * fl32(sa_inv * sb_inv))).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#if !defined(FLT_EVAL_METHOD) || FLT_EVAL_METHOD != 0
#error "the oracle needs float expressions evaluated in binary32 (FLT_EVAL_METHOD == 0)"
#endif

#define OR_E4M3 0
#define OR_E5M2 1

/* ------------------------------------------------------------------------ */
/* BF16 (S1E8M7, [P3] Definition table): the top 16 bits of a binary32.      */
/* ------------------------------------------------------------------------ */

float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 value to the nearest BF16 value, ties to an even last
 * mantissa bit; NaN stays a (quiet) NaN.  The 16 dropped bits are compared
 * with the halfway pattern 0x8000 directly. */
uint16_t or_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t drop = u & 0xffffu;
    if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u)))
        keep += 1u; /* may carry into the exponent: that is the next binade (or inf) */
    return (uint16_t)keep;
}

/* ------------------------------------------------------------------------ */
/* FP8 decode from the bit fields ([P1] format section, [P3] Definition).    */
/* ------------------------------------------------------------------------ */

double or_fp8_decode(uint8_t code, int fmt)
{
    int s = code >> 7;
    double v;
    if (fmt == OR_E4M3) {
        int e = (code >> 3) & 0xf, m = code & 7;
        if (e == 15 && m == 7)
            return NAN;
        if (e == 0)
            v = ldexp((double)m, -9);             /* m/8 * 2^(1-7) */
        else
            v = ldexp(1.0 + m / 8.0, e - 7);
    } else {
        int e = (code >> 2) & 0x1f, m = code & 3;
        if (e == 31)
            return m == 0 ? (s ? -INFINITY : INFINITY) : NAN;
        if (e == 0)
            v = ldexp((double)m, -16);            /* m/4 * 2^(1-15) */
        else
            v = ldexp(1.0 + m / 4.0, e - 15);
    }
    return s ? -v : v;
}

/* Largest finite code (sign bit clear) and its value. */
static int max_code(int fmt) { return fmt == OR_E4M3 ? 0x7e : 0x7b; }

double or_fp8_max(int fmt) { return or_fp8_decode((uint8_t)max_code(fmt), fmt); }

/* ------------------------------------------------------------------------ */
/* FP8 encode of a binary32 value: nearest representable value, ties to the */
/* even code, saturating.  Non-negative finite codes 0..max_code are in      */
/* increasing order of value, so a binary search finds the two neighbours.  */
/* ------------------------------------------------------------------------ */

uint8_t or_fp8_encode_f32(float v, int fmt)
{
    if (isnan(v))
        return 0x7f; /* a NaN code of either format; compared as a class */
    int neg = signbit(v) ? 1 : 0;
    double a = fabs((double)v);
    int top = max_code(fmt);
    int code;
    if (a >= or_fp8_decode((uint8_t)top, fmt)) {
        code = top;                                   /* saturate (also +-inf) */
    } else {
        int lo = 0, hi = top;                         /* value(lo) <= a < value(hi) */
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (or_fp8_decode((uint8_t)mid, fmt) <= a)
                lo = mid;
            else
                hi = mid;
        }
        double vlo = or_fp8_decode((uint8_t)lo, fmt);
        double vhi = or_fp8_decode((uint8_t)hi, fmt);
        double twice = 2.0 * a, mid = vlo + vhi;      /* both exact in double */
        if (twice < mid)
            code = lo;
        else if (twice > mid)
            code = hi;
        else
            code = (lo % 2 == 0) ? lo : hi;           /* tie: even code */
    }
    return (uint8_t)((neg << 7) | code);
}

void or_fp8_encode_f32_array(const float *v, int64_t n, int fmt, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_fp8_encode_f32(v[i], fmt);
}

/* ------------------------------------------------------------------------ */
/* amax: max |x| over a BF16 tensor ([P1] dynamic scaling; [P2] Absolute-    */
/* Max).  NaN entries never compare greater, so they are skipped.           */
/* ------------------------------------------------------------------------ */

float or_amax_bf16(const uint16_t *x, int64_t n)
{
    float m = 0.0f;
#pragma omp parallel for reduction(max : m) schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(or_bf16_to_f32(x[i]));
        if (a > m)
            m = a;
    }
    return m;
}

/* ------------------------------------------------------------------------ */
/* Scaled cast with transposed copy: out[r][c] = enc(fl32(x[r][c] * s)) and  */
/* out_t[c][r] = out[r][c] ([P2] Q node; the transpose lets every GEMM take  */
/* both operands contiguous along the contracted dimension).                 */
/* ------------------------------------------------------------------------ */

void or_quantize(const uint16_t *x, int64_t rows, int64_t cols, float scale, int fmt,
                 uint8_t *out, uint8_t *out_t)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            float v = or_bf16_to_f32(x[r * cols + c]) * scale; /* binary32 multiply */
            uint8_t q = or_fp8_encode_f32(v, fmt);
            if (out)
                out[r * cols + c] = q;
            if (out_t)
                out_t[c * rows + r] = q;
        }
    }
}

/* The same scaled cast of an fp32 tensor, in element order, and its amax   */
/* (the Q node applied to binary32 values; amax as for BF16, NaN skipped).   */
void or_quantize_f32(const float *x, int64_t n, float scale, int fmt, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_fp8_encode_f32(x[i] * scale, fmt); /* binary32 multiply */
}

float or_amax_f32(const float *x, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > m) /* false for NaN */
            m = a;
    }
    return m;
}

/* ------------------------------------------------------------------------ */
/* Delayed-scaling update of one tensor's state ([P1] DelayedScaling:        */
/* margin, amax_history_len; the scale formula above).                       */
/* ------------------------------------------------------------------------ */

void or_history_update(float *hist, int32_t L, float amax, float *scale, float *scale_inv,
                       int fmt, int32_t margin)
{
    for (int32_t i = L - 1; i > 0; --i)
        hist[i] = hist[i - 1];
    hist[0] = amax;
    float m = 0.0f;
    for (int32_t i = 0; i < L; ++i)
        if (hist[i] > m)
            m = hist[i];
    if (m > 0.0f && isfinite(m)) {
        float fmax = (float)or_fp8_max(fmt);
        float q = fmax / m;                           /* binary32 divide */
        float s = (float)ldexp((double)q, -margin);   /* exact, then one rounding */
        if (isinf(s))
            s = FLT_MAX;
        *scale = s;
        *scale_inv = 1.0f / s;                        /* binary32 divide */
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM on FP8 operands, both stored with the contracted index contiguous:   */
/* acc[i][j] = sum_k A[i][k] * B[j][k]  ([P3] "extension to FP8": FP8        */
/* operands, higher-precision accumulation).                                 */
/* ------------------------------------------------------------------------ */

/* Double accumulation over output rows [row0, row0 + nrows).  Every product
 * of two FP8 values is exact in double; only the running sum rounds. */
void or_gemm_tn_f64(const uint8_t *A, int fa, const uint8_t *B, int fb, int64_t M, int64_t N,
                    int64_t K, int64_t row0, int64_t nrows, double *acc)
{
    (void)M;
    double ta[256], tb[256];
    for (int c = 0; c < 256; ++c) {
        ta[c] = or_fp8_decode((uint8_t)c, fa);
        tb[c] = or_fp8_decode((uint8_t)c, fb);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const uint8_t *a = A + (row0 + i) * K;
        for (int64_t j = 0; j < N; ++j) {
            const uint8_t *b = B + j * K;
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k)
                s += ta[a[k]] * tb[b[k]];
            acc[i * N + j] = s;
        }
    }
}

/* Exact accumulation.  In units of 2^-16 every E4M3 value is an integer of
 * magnitude <= 448 * 2^16 and every E5M2 value one of magnitude
 * <= 57344 * 2^16 < 2^32, so a product is an integer (units 2^-32) below
 * 2^64 and a sum over K <= 2^32 terms fits a signed 128-bit integer.  The
 * exact sum is returned rounded once to double.  Non-finite codes are not
 * allowed here (returns -1). */
int or_gemm_tn_exact(const uint8_t *A, int fa, const uint8_t *B, int fb, int64_t M, int64_t N,
                     int64_t K, double *acc)
{
    int64_t ia[256], ib[256];
    for (int c = 0; c < 256; ++c) {
        double da = or_fp8_decode((uint8_t)c, fa), db = or_fp8_decode((uint8_t)c, fb);
        ia[c] = isfinite(da) ? (int64_t)ldexp(da, 16) : INT64_MIN;
        ib[c] = isfinite(db) ? (int64_t)ldexp(db, 16) : INT64_MIN;
    }
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            __int128 s = 0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t x = ia[A[i * K + k]], y = ib[B[j * K + k]];
                if (x == INT64_MIN || y == INT64_MIN)
                    return -1;
                s += (__int128)x * (__int128)y;
            }
            acc[i * N + j] = ldexp((double)s, -32);
        }
    }
    return 0;
}

/* Dequant epilogue: y = bf16_rne(fl32(fl32(acc) * fl32(sa_inv * sb_inv))). */
void or_epilogue(const double *acc, int64_t n, float sa_inv, float sb_inv, uint16_t *y)
{
    float sab = sa_inv * sb_inv;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float a = (float)acc[i];
        y[i] = or_f32_to_bf16(a * sab);
    }
}

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* LayerNorm (the te.LayerNorm drop-in of the implementation guide, section  */
/* "Basic structure of FP8 training code"), in double:                       */
/*   mean_r = sum_c x[r][c] / C,  var_r = sum_c (x[r][c] - mean_r)^2 / C,    */
/*   rstd_r = 1 / sqrt(var_r + eps),                                         */
/*   y[r][c] = (x[r][c] - mean_r) * rstd_r * gamma[c] + beta[c].             */
/* ------------------------------------------------------------------------ */

void or_layernorm(const uint16_t *x, const uint16_t *gamma, const uint16_t *beta, int64_t rows,
                  int64_t cols, double eps, double *y, double *mean, double *rstd)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * cols;
        double s = 0.0;
        for (int64_t c = 0; c < cols; ++c)
            s += (double)or_bf16_to_f32(xr[c]);
        double mu = s / (double)cols;
        double v = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            double d = (double)or_bf16_to_f32(xr[c]) - mu;
            v += d * d;
        }
        v /= (double)cols;
        double rs = 1.0 / sqrt(v + eps);
        mean[r] = mu;
        rstd[r] = rs;
        for (int64_t c = 0; c < cols; ++c)
            y[r * cols + c] = ((double)or_bf16_to_f32(xr[c]) - mu) * rs *
                              (double)or_bf16_to_f32(gamma[c]) + (double)or_bf16_to_f32(beta[c]);
    }
}

/* ------------------------------------------------------------------------ */
/* FP16 (S1E5M10, [P3] Definition table: max 65,504): encode by nearest      */
/* value with ties to the even code, saturating at +-65504 (the same reading */
/* as the FP8 casts); decode from the fields.                                 */
/* ------------------------------------------------------------------------ */

float or_f16_decode(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 31)
        return m ? NAN : (s ? -INFINITY : INFINITY);
    v = e == 0 ? ldexp((double)m, -24) : ldexp(1.0 + m / 1024.0, e - 15);
    return (float)(s ? -v : v);
}

uint16_t or_f16_encode(float f)
{
    if (isnan(f))
        return 0x7e00;
    int neg = signbit(f) ? 1 : 0;
    double a = fabs((double)f);
    int top = 0x7bff, code;
    if (a >= (double)or_f16_decode((uint16_t)top)) {
        code = top;
    } else {
        int lo = 0, hi = top;
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if ((double)or_f16_decode((uint16_t)mid) <= a)
                lo = mid;
            else
                hi = mid;
        }
        double vlo = or_f16_decode((uint16_t)lo), vhi = or_f16_decode((uint16_t)hi);
        if (2.0 * a < vlo + vhi)
            code = lo;
        else if (2.0 * a > vlo + vhi)
            code = hi;
        else
            code = (lo % 2 == 0) ? lo : hi;
    }
    return (uint16_t)((neg << 15) | code);
}

/* ------------------------------------------------------------------------ */
/* One Adam step with decoupled optimizer-state precision ([P3] bullet       */
/* "precision decoupling": first moment FP8, second moment FP16, master      */
/* weights FP16 with tensor scaling).  All arithmetic in binary32, one       */
/* rounding per operation, in this order (Adam with bias correction, the     */
/* textbook form: m_hat = m / (1 - b1^t), v_hat = v / (1 - b2^t); AdamW's    */
/* decoupled weight decay):                                                  */
/*   m  = b1*m + (1-b1)*g,   v = b2*v + (1-b2)*(g*g)                         */
/*   u  = (m / bc1) / (sqrt(v / bc2) + eps)                                   */
/*   w  = w - lr*(u + wd*w)                                                   */
/* with m decoded from its E4M3 codes times m_sinv and w from its FP16 codes */
/* times w_sinv.  Just-in-time per-tensor scaling of the new states:         */
/* amax over all elements first, then the scale formula with a history of    */
/* one (fmax 448 for m, 65504 for w), then the encodes.  Outputs: new m      */
/* codes, v (FP16), w codes (FP16), the model's BF16 weight, the two amaxes  */
/* and the new scales / inverses (kept when an amax is 0 or not finite).     */
/* ------------------------------------------------------------------------ */

static void adam_elem(float g, float m, float v, float w, float lr, float b1, float b2, float eps,
                      float wd, float bc1, float bc2, float *mo, float *vo, float *wo)
{
    m = b1 * m + (1.0f - b1) * g;
    v = b2 * v + (1.0f - b2) * (g * g);
    float u = (m / bc1) / (sqrtf(v / bc2) + eps);
    w = w - lr * (u + wd * w);
    *mo = m;
    *vo = v;
    *wo = w;
}

void or_adam_step(const uint16_t *grad, int64_t n, uint8_t *m1, float *m1_scale,
                  float *m1_scale_inv, uint16_t *m2, uint16_t *w16, float *w_scale,
                  float *w_scale_inv, uint16_t *w_bf16, float *amax, float lr, float b1, float b2,
                  float eps, float wd, float bc1, float bc2, int32_t margin)
{
    float am_m = 0.0f, am_w = 0.0f;
    const float msi = *m1_scale_inv, wsi = *w_scale_inv;
    for (int64_t i = 0; i < n; ++i) {
        float mo, vo, wo;
        adam_elem(or_bf16_to_f32(grad[i]), (float)or_fp8_decode(m1[i], OR_E4M3) * msi,
                  or_f16_decode(m2[i]), or_f16_decode(w16[i]) * wsi, lr, b1, b2, eps, wd, bc1,
                  bc2, &mo, &vo, &wo);
        if (fabsf(mo) > am_m)
            am_m = fabsf(mo);
        if (fabsf(wo) > am_w)
            am_w = fabsf(wo);
    }
    amax[0] = am_m;
    amax[1] = am_w;
    /* the new scales: the update formula applied to a one-entry history */
    float hm[1] = {0.0f}, hw[1] = {0.0f};
    float sm = *m1_scale, smi = *m1_scale_inv, sw = *w_scale, swi = *w_scale_inv;
    or_history_update(hm, 1, am_m, &sm, &smi, OR_E4M3, margin);
    /* FP16's largest finite value replaces the FP8 one for the weights */
    if (am_w > 0.0f && isfinite(am_w)) {
        float q = 65504.0f / am_w;
        float s = (float)ldexp((double)q, -margin);
        if (isinf(s))
            s = FLT_MAX;
        sw = s;
        swi = 1.0f / s;
    }
    for (int64_t i = 0; i < n; ++i) {
        float mo, vo, wo;
        adam_elem(or_bf16_to_f32(grad[i]), (float)or_fp8_decode(m1[i], OR_E4M3) * msi,
                  or_f16_decode(m2[i]), or_f16_decode(w16[i]) * wsi, lr, b1, b2, eps, wd, bc1,
                  bc2, &mo, &vo, &wo);
        m1[i] = or_fp8_encode_f32(mo * sm, OR_E4M3);
        m2[i] = or_f16_encode(vo);
        w16[i] = or_f16_encode(wo * sw);
        w_bf16[i] = or_f32_to_bf16(wo);
    }
    *m1_scale = sm;
    *m1_scale_inv = smi;
    *w_scale = sw;
    *w_scale_inv = swi;
}

/* Initial decoupled-precision Adam state of a BF16 weight tensor w (same     */
/* bullet): zero moments (first-moment scale and inverse 1), and the master  */
/* weights in FP16 under the just-in-time tensor scale of w itself: the      */
/* recipe formula on a one-entry history with FP16's largest finite value,   */
/*   s_w = fl32(fl32(65504 / amax(w)) * 2^-margin), s_w = 1 when amax(w) is   */
/*   0 or not finite;  w16[i] = enc_f16(fl32(w[i] * s_w)).                   */
/* amax[0] = 0 (the first moment), amax[1] = amax(w).                        */

void or_adam_init(const uint16_t *w, int64_t n, int32_t margin, uint8_t *m1, float *m1_scale,
                  float *m1_scale_inv, uint16_t *m2, uint16_t *w16, float *w_scale,
                  float *w_scale_inv, float *amax)
{
    float am = or_amax_bf16(w, n);
    float s = 1.0f;
    if (am > 0.0f && isfinite(am)) {
        float q = 65504.0f / am;                      /* binary32 divide */
        s = (float)ldexp((double)q, -margin);         /* exact, then one rounding */
        if (isinf(s))
            s = FLT_MAX;
    }
    for (int64_t i = 0; i < n; ++i) {
        m1[i] = 0;
        m2[i] = 0;
        w16[i] = or_f16_encode(or_bf16_to_f32(w[i]) * s); /* binary32 multiply */
    }
    *m1_scale = 1.0f;
    *m1_scale_inv = 1.0f;
    *w_scale = s;
    *w_scale_inv = 1.0f / s;                          /* binary32 divide */
    amax[0] = 0.0f;
    amax[1] = am;
}

/* ------------------------------------------------------------------------ */
/* Sum of FP8 tensors sharing one scale ([P3] bullet "per-tensor scaling is  */
/* the key": FP8 all-reduce with one scalar shared by all ranks,             */
/* s'_g = min(s'_1, ..., s'_N)).  q holds nranks parts of n codes each;      */
/*   out[i] = bf16_rne( sum_r dec(q[r][i]) * fl32(1 / scale) ),              */
/* the sum and the product exact, rounded once to BF16 (round to nearest,    */
/* ties to even; overflow to +-inf; gradual underflow, a nonzero value that   */
/* rounds to zero keeps its sign; an exact zero is +0).  Non-finite parts    */
/* follow IEEE arithmetic: a NaN code, or +inf and -inf together, give NaN;  */
/* one kind of infinity gives that infinity times fl32(1 / scale) (NaN when  */
/* that factor is 0 or NaN); a finite sum times a non-finite factor is that  */
/* factor's product with the sum's sign (NaN for a zero sum or a NaN factor). */
/* ------------------------------------------------------------------------ */

/* Every finite FP8 value is an integer number of quanta: 2^-9 for E4M3, 2^-16 */
/* for E5M2 (the smallest subnormal of each format).                           */
static int quantum_exp(int fmt) { return fmt == OR_E4M3 ? -9 : -16; }

/* The nearest BF16 of the exact value (neg ? -1 : 1) * P * 2^e, P >= 0.       */
static uint16_t bf16_of_exact(int neg, unsigned __int128 P, int e)
{
    if (P == 0)
        return 0x0000;                                 /* an exact zero: +0 */
    int nb = 0;                                        /* bit length of P */
    for (unsigned __int128 t = P; t != 0; t >>= 1)
        ++nb;
    int lead = nb - 1 + e;                             /* 2^lead <= value < 2^(lead+1) */
    int u = lead - 7;                                  /* BF16 keeps 8 significant bits */
    if (u < -133)
        u = -133;                                      /* the subnormal quantum 2^-133 */
    int shift = u - e;                                 /* value = P * 2^e = (P >> shift) * 2^u + rest */
    unsigned __int128 M;
    if (shift <= 0) {
        M = P << (-shift);                             /* exact: fewer than 9 bits */
    } else {
        M = P >> shift;
        unsigned __int128 rest = P - (M << shift);
        unsigned __int128 half = (unsigned __int128)1 << (shift - 1);
        if (rest > half || (rest == half && (M & 1)))
            M += 1;                                    /* may reach 2^8: still exact below */
    }
    double mag = ldexp((double)M, u);                  /* exact: M <= 256 */
    float f = mag >= 0x1p128 ? INFINITY : (float)mag;  /* exact when finite */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)((bits >> 16) | (neg ? 0x8000u : 0u));
}

void or_dequant_sum(const uint8_t *q, int32_t nranks, int64_t n, int fmt, float scale,
                    uint16_t *out)
{
    const float sinv = 1.0f / scale;                   /* binary32 divide */
    int se;
    const float sm = frexpf(sinv, &se);                /* sinv = sm * 2^se, 0.5 <= |sm| < 1 */
    const int64_t sig = (int64_t)ldexpf(fabsf(sm), 24); /* 24-bit integer significand */
    const int sneg = sinv < 0.0f;
    const int g = quantum_exp(fmt);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        int64_t acc = 0;                               /* exact: < 2^16 parts of < 2^32 quanta */
        int nan = 0, pinf = 0, ninf = 0;
        for (int32_t r = 0; r < nranks; ++r) {
            double v = or_fp8_decode(q[(int64_t)r * n + i], fmt);
            if (isnan(v))
                nan = 1;
            else if (v == INFINITY)
                pinf = 1;
            else if (v == -INFINITY)
                ninf = 1;
            else
                acc += (int64_t)ldexp(v, -g);          /* exact integer count of quanta */
        }
        float res;
        if (nan || (pinf && ninf)) {
            res = NAN;
        } else if (pinf || ninf) {
            res = (pinf ? INFINITY : -INFINITY) * sinv; /* IEEE: NaN when sinv is 0 or NaN */
        } else if (isnan(sinv) || isinf(sinv)) {
            res = (float)acc * sinv;                   /* exact sign; 0 * inf = NaN */
        } else {
            int neg = (acc < 0) != sneg;
            unsigned __int128 P = (unsigned __int128)(acc < 0 ? -acc : acc) *
                                  (unsigned __int128)sig;
            out[i] = bf16_of_exact(acc != 0 && sig != 0 ? neg : 0, P, g + se - 24);
            continue;
        }
        out[i] = or_f32_to_bf16(res);
    }
}
