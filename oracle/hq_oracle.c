/*
 * hq_oracle.c -- the plain, slow CPU oracle for the quantized-weight matvec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA
 * library; it is written from the definitions on the pages:
 *
 *   [NST]  "One Native Stack for Private, Continuously-Learning AI",
 *          section "The Unified Quant Core" (the Q8_0 = symmetric 34 B / 32 and
 *          Q4_0 = symmetric 18 B / 32 block formats, taken from ggml) and
 *          section "The Central Efficiency Thesis", Lemma "QLoRA over the
 *          unified core is exact" (y_i = sum_j What_ij x_j with What the CPU
 *          dequantization of the stored bytes, accumulated in f32 per block).
 *   [EPS]  "Economical Serving and the hanzo.ai Platform", subsection
 *          "One Quant-Agnostic Core, Not a Kernel-per-Quant Zoo" (one core
 *          reused for decode and for every routed MoE expert).
 *   [ZEN]  "Blue -- porting zen-nano (Qwen3-0.6B) to deterministic on-chain
 *          inference", section "Quantization recipe (validated)" (per-output-
 *          channel symmetric int8 weights, s_w[o] = max|W[o,:]|/127,
 *          Wq = round(W/s_w) in [-127,127]; requant by gemmlowp's
 *          SaturatingRoundingDoublingHighMul then RoundingDivideByPOT to int8,
 *          all integer), section "Gaps vs the current toy engine", item 3,
 *          and section "Architecture" (the feed-forward is SwiGLU(gate, up,
 *          down)).
 *   [NST]  also section "Ported Versus Novel": every format, Q4_K included, is
 *          taken verbatim from ggml.  Q4_K is therefore ggml's super-block of
 *          256 weights in 144 bytes: fp16 d, fp16 dmin, 12 bytes packing eight
 *          6-bit sub-block scales and eight 6-bit sub-block mins, then 128
 *          bytes of 4-bit quants; w = d * sc_j * q - dmin * m_j for sub-block j.
 *   [EPS]  also paragraph "MoE is the cheapest-per-quality tier" (a sparsely
 *          gated mixture: the output is the gate-weighted sum of the chosen
 *          experts' outputs).
 *
 * Readings taken where the pages are silent: fp16 scale rounded to nearest-even from an fp32 d; q = round(w/d)
 * with round-half-away-from-zero in fp32; Q4_0 nibble n = min(15, floor(w/d +
 * 8.5)) with d = (signed absmax)/-8 and ggml's nibble order (byte j holds
 * element j low, element j+16 high); all-zero blocks give d = 0 (Q4_0: -0.0,
 * n = 8); int8 output saturates to [-128,127]; shift[o] is a right shift in
 * [0,31].
 *
 * Float matvecs accumulate in f64 and also return T = sum_j |w_deq * x_j| for
 * the tolerance |y - y_ref| <= 1e-3 * T + 1e-5.  The int8 path is exact.
 * Build with -ffp-contract=off: no fused multiply-add may change a result.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define HQO_QK 32             /* weights per block (both formats)          */
#define HQO_Q8_0_BYTES 34     /* 2 B fp16 scale + 32 x int8                */
#define HQO_Q4_0_BYTES 18     /* 2 B fp16 scale + 16 B of nibbles          */
#define HQO_QK_K 256          /* Q4_K: weights per super-block              */
#define HQO_Q4_K_BYTES 144    /* 2 B d + 2 B dmin + 12 B scales/mins + 128 B nibbles */

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 <-> binary32, written from the format definition:       */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.                  */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

float hqo_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);             /* subnormal: m * 2^-24     */
    } else if (e == 31) {
        if (m) return bits_f32(0x7fc00000u | ((uint32_t)sign << 31));
        v = INFINITY;
    } else {
        v = ldexp(1024.0 + (double)m, e - 25); /* (1 + m/1024) * 2^(e-15) */
    }
    return (float)(sign ? -v : v);
}

/* Round a float to the nearest binary16, ties to even.  Overflow -> inf. */
uint16_t hqo_float_to_half_rne(float f)
{
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    /* largest finite half is 65504; values >= 65520 round up to infinity */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    int e;
    (void)frexp(a, &e);                        /* a = f * 2^e, f in [0.5,1) */
    int exp_h = e - 1;                         /* a in [2^exp_h, 2^(exp_h+1)) */
    if (exp_h < -14) exp_h = -14;              /* subnormal range spacing   */
    double ulp = ldexp(1.0, exp_h - 10);       /* spacing of halves there   */
    double k = a / ulp;                        /* exact: power-of-two scale */
    double kf = floor(k);
    double rem = k - kf;
    uint32_t ki = (uint32_t)kf;
    if (rem > 0.5 || (rem == 0.5 && (ki & 1u))) ki += 1;
    /* ki is the integer multiple of ulp; build the bit pattern */
    uint32_t bits;
    if (exp_h == -14 && ki < 1024u) {
        bits = ki;                             /* subnormal (or rounds to min normal at 1024) */
    } else {
        if (ki >= 2048u) { ki >>= 1; exp_h += 1; }   /* carried into next binade */
        if (exp_h > 15) return (uint16_t)(sign | 0x7c00u);
        bits = ((uint32_t)(exp_h + 15) << 10) | (ki - 1024u);
    }
    return (uint16_t)(sign | bits);
}

/* ------------------------------------------------------------------------ */
/* Quantizers (the data-preparation step, done once on the host).            */
/* ------------------------------------------------------------------------ */

static int32_t clamp_i32(int32_t v, int32_t lo, int32_t hi)
{
    return v < lo ? lo : (v > hi ? hi : v);
}

/* Q8_0: per block of 32 along a row, d = max|w| / 127 (fp32), stored as fp16
 * (RNE); q_j = round(w_j / d) (fp32 division, half away from zero), clamped
 * to [-127,127].  Block = { fp16 d little-endian, int8 q[32] }. */
void hqo_quantize_q8_0(const float *W, int64_t rows, int64_t cols, uint8_t *out)
{
    int64_t nb = cols / HQO_QK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *w = W + r * cols + b * HQO_QK;
            uint8_t *blk = out + (r * nb + b) * HQO_Q8_0_BYTES;
            float amax = 0.0f;
            for (int j = 0; j < HQO_QK; ++j) {
                float a = fabsf(w[j]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            uint16_t dh = hqo_float_to_half_rne(d);
            blk[0] = (uint8_t)(dh & 0xff);
            blk[1] = (uint8_t)(dh >> 8);
            for (int j = 0; j < HQO_QK; ++j) {
                int32_t q = 0;
                if (d != 0.0f) {
                    float t = w[j] / d;
                    q = clamp_i32((int32_t)roundf(t), -127, 127);
                }
                blk[2 + j] = (uint8_t)(int8_t)q;
            }
        }
    }
}

/* Q4_0: per block, m = the element of largest |w| (first on ties), keeping
 * its sign; d = m / -8 (fp32), stored fp16 (RNE); n_j = min(15, floor(w_j/d
 * + 8.5)) (the absmax element maps to n = 0).  Byte j (0..15) holds element j
 * in its low nibble and element j+16 in its high nibble.  d == 0: all n = 8. */
void hqo_quantize_q4_0(const float *W, int64_t rows, int64_t cols, uint8_t *out)
{
    int64_t nb = cols / HQO_QK;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const float *w = W + r * cols + b * HQO_QK;
            uint8_t *blk = out + (r * nb + b) * HQO_Q4_0_BYTES;
            float amax = 0.0f, m = 0.0f;
            for (int j = 0; j < HQO_QK; ++j) {
                float a = fabsf(w[j]);
                if (a > amax) { amax = a; m = w[j]; }
            }
            float d = m / -8.0f;
            uint16_t dh = hqo_float_to_half_rne(d);
            blk[0] = (uint8_t)(dh & 0xff);
            blk[1] = (uint8_t)(dh >> 8);
            int n[HQO_QK];
            for (int j = 0; j < HQO_QK; ++j) {
                if (d != 0.0f) {
                    float t = w[j] / d + 8.5f;
                    int32_t v = (int32_t)floorf(t);
                    n[j] = clamp_i32(v, 0, 15);
                } else {
                    n[j] = 8;
                }
            }
            for (int j = 0; j < 16; ++j)
                blk[2 + j] = (uint8_t)((n[j] & 0x0f) | ((n[j + 16] & 0x0f) << 4));
        }
    }
}

/* Q4_K sub-block j (0..7) of a super-block: its 6-bit scale and 6-bit min
 * from the 12 packed bytes.  Sub-blocks 0..3 keep both in the low 6 bits of
 * bytes j and j+4; sub-blocks 4..7 keep their low 4 bits in the two nibbles of
 * byte j+4 (scale low, min high) and their top 2 bits in the top 2 bits of
 * bytes j-4 (scale) and j (min). */
static void q4k_scale_min(const uint8_t *s12, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = s12[j] & 63;
        *m = s12[j + 4] & 63;
    } else {
        *sc = (s12[j + 4] & 0x0f) | ((s12[j - 4] >> 6) << 4);
        *m = (s12[j + 4] >> 4) | ((s12[j] >> 6) << 4);
    }
}

/* Element e (0..255) of a Q4_K super-block: sub-block j = e / 32 reads the
 * quant bytes of group j / 2 (32 bytes); an even sub-block takes the low
 * nibbles of that group, an odd one the high nibbles. */
static int q4k_quant(const uint8_t *blk, int e)
{
    int j = e / 32, l = e % 32;
    uint8_t b = blk[16 + 32 * (j / 2) + l];
    return (j & 1) ? (b >> 4) : (b & 0x0f);
}

/* Q4_K encoder (the pages print none; this is a plain min/max reading of the
 * format).  Per sub-block of 32: mn = min(0, min w), mx = max w, scale =
 * (mx - mn) / 15 and min = -mn (fp32).  d = max scale / 63 and dmin = max min
 * / 63 (fp32; the maxima are taken from +0 upwards), stored fp16 (RNE).  sc_j = min(63, round(scale_j * (63 / max
 * scale))), m_j likewise with the mins (0 when the maximum is 0).  Then, with
 * the stored fp16 values, a = d * sc_j and b = dmin * m_j (fp32, exact), q =
 * clamp(round((w + b) / a), 0, 15) (fp32, half away from zero), q = 0 when
 * a == 0.  Rows are cols / 256 super-blocks, no padding. */
void hqo_quantize_q4_k(const float *W, int64_t rows, int64_t cols, uint8_t *out)
{
    int64_t nsb = cols / HQO_QK_K;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const float *w = W + r * cols + sb * HQO_QK_K;
            uint8_t *blk = out + (r * nsb + sb) * HQO_Q4_K_BYTES;
            float scale[8], minv[8], max_scale = 0.0f, max_min = 0.0f;
            for (int j = 0; j < 8; ++j) {
                float mn = w[32 * j], mx = w[32 * j];
                for (int l = 1; l < 32; ++l) {
                    if (w[32 * j + l] < mn) mn = w[32 * j + l];
                    if (w[32 * j + l] > mx) mx = w[32 * j + l];
                }
                if (mn > 0.0f) mn = 0.0f;
                scale[j] = (mx - mn) / 15.0f;
                minv[j] = -mn;
                if (scale[j] > max_scale) max_scale = scale[j];
                if (minv[j] > max_min) max_min = minv[j];
            }
            uint16_t dh = hqo_float_to_half_rne(max_scale / 63.0f);
            uint16_t mh = hqo_float_to_half_rne(max_min / 63.0f);
            float inv_s = max_scale > 0.0f ? 63.0f / max_scale : 0.0f;
            float inv_m = max_min > 0.0f ? 63.0f / max_min : 0.0f;
            int sc[8], mq[8];
            for (int j = 0; j < 8; ++j) {
                sc[j] = clamp_i32((int32_t)roundf(scale[j] * inv_s), 0, 63);
                mq[j] = clamp_i32((int32_t)roundf(minv[j] * inv_m), 0, 63);
            }
            blk[0] = (uint8_t)(dh & 0xff);
            blk[1] = (uint8_t)(dh >> 8);
            blk[2] = (uint8_t)(mh & 0xff);
            blk[3] = (uint8_t)(mh >> 8);
            for (int j = 0; j < 4; ++j) {
                blk[4 + j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 4) << 6));
                blk[8 + j] = (uint8_t)(mq[j] | ((mq[j + 4] >> 4) << 6));
                blk[12 + j] = (uint8_t)((sc[j + 4] & 0x0f) | ((mq[j + 4] & 0x0f) << 4));
            }
            float dq = hqo_half_to_float(dh), mqf = hqo_half_to_float(mh);
            int q[HQO_QK_K];
            for (int j = 0; j < 8; ++j) {
                float a = dq * (float)sc[j], b = mqf * (float)mq[j];
                for (int l = 0; l < 32; ++l) {
                    int32_t v = 0;
                    if (a > 0.0f) {
                        float t = (w[32 * j + l] + b) / a;
                        v = clamp_i32((int32_t)roundf(t), 0, 15);
                    }
                    q[32 * j + l] = v;
                }
            }
            for (int g = 0; g < 4; ++g)
                for (int l = 0; l < 32; ++l)
                    blk[16 + 32 * g + l] = (uint8_t)(q[64 * g + l] | (q[64 * g + 32 + l] << 4));
        }
    }
}

/* Per-output-channel symmetric int8 ([ZEN] "Quantization recipe"):
 * s[o] = max|W[o,:]| / 127 (fp32); Wq[o,j] = round(W[o,j] / s[o]) (fp32,
 * half away from zero) clamped to [-127,127]; s[o] == 0 gives 0.  With
 * rows = 1 this is the static per-tensor activation quantizer as well. */
void hqo_quantize_i8_rows(const float *W, int64_t rows, int64_t cols,
                          int8_t *Wq, float *scale)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *w = W + r * cols;
        float amax = 0.0f;
        for (int64_t j = 0; j < cols; ++j) {
            float a = fabsf(w[j]);
            if (a > amax) amax = a;
        }
        float s = amax / 127.0f;
        scale[r] = s;
        for (int64_t j = 0; j < cols; ++j) {
            int32_t q = 0;
            if (s != 0.0f) q = clamp_i32((int32_t)roundf(w[j] / s), -127, 127);
            Wq[r * cols + j] = (int8_t)q;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Dequantization: the stored bytes define the weights (DEQ_cpu of [NST]).   */
/* ------------------------------------------------------------------------ */

static uint16_t load_u16le(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

void hqo_dequant_q8_0(const uint8_t *bytes, int64_t rows, int64_t cols, double *Wd)
{
    int64_t nb = cols / HQO_QK;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = bytes + (r * nb + b) * HQO_Q8_0_BYTES;
            double d = (double)hqo_half_to_float(load_u16le(blk));
            for (int j = 0; j < HQO_QK; ++j)
                Wd[r * cols + b * HQO_QK + j] = d * (double)(int8_t)blk[2 + j];
        }
}

void hqo_dequant_q4_0(const uint8_t *bytes, int64_t rows, int64_t cols, double *Wd)
{
    int64_t nb = cols / HQO_QK;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const uint8_t *blk = bytes + (r * nb + b) * HQO_Q4_0_BYTES;
            double d = (double)hqo_half_to_float(load_u16le(blk));
            for (int j = 0; j < 16; ++j) {
                int lo = blk[2 + j] & 0x0f;
                int hi = blk[2 + j] >> 4;
                Wd[r * cols + b * HQO_QK + j] = d * (double)(lo - 8);
                Wd[r * cols + b * HQO_QK + j + 16] = d * (double)(hi - 8);
            }
        }
}

/* Q4_K: w = d * sc_j * q - dmin * m_j (f64, exact for the stored values). */
static double q4k_weight(const uint8_t *blk, int e)
{
    int sc, m;
    q4k_scale_min(blk + 4, e / 32, &sc, &m);
    double d = (double)hqo_half_to_float(load_u16le(blk));
    double dmin = (double)hqo_half_to_float(load_u16le(blk + 2));
    return d * (double)sc * (double)q4k_quant(blk, e) - dmin * (double)m;
}

void hqo_dequant_q4_k(const uint8_t *bytes, int64_t rows, int64_t cols, double *Wd)
{
    int64_t nsb = cols / HQO_QK_K;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t sb = 0; sb < nsb; ++sb) {
            const uint8_t *blk = bytes + (r * nsb + sb) * HQO_Q4_K_BYTES;
            for (int e = 0; e < HQO_QK_K; ++e)
                Wd[r * cols + sb * HQO_QK_K + e] = q4k_weight(blk, e);
        }
}

/* ------------------------------------------------------------------------ */
/* Float matvecs: y[v][i] = sum_j w_deq[i][j] * x[v][j], in f64, plus        */
/* T[v][i] = sum_j |w_deq[i][j] * x[v][j]|.  x is [n_vec][cols], y and T are */
/* [n_vec][rows].  One row is dequantized at a time, from the stored bytes.  */
/* ------------------------------------------------------------------------ */

static void matvec_rows(int fmt, const uint8_t *bytes, const float *x,
                        int64_t row_lo, int64_t row_hi, int64_t rows, int64_t cols,
                        int n_vec, double *y, double *T)
{
    if (fmt == 'K') {                          /* Q4_K super-blocks */
        int64_t nsb = cols / HQO_QK_K;
        for (int64_t i = row_lo; i < row_hi; ++i)
            for (int v = 0; v < n_vec; ++v) {
                double acc = 0.0, aabs = 0.0;
                for (int64_t sb = 0; sb < nsb; ++sb) {
                    const uint8_t *blk = bytes + (i * nsb + sb) * HQO_Q4_K_BYTES;
                    for (int e = 0; e < HQO_QK_K; ++e) {
                        double p = q4k_weight(blk, e) * (double)x[(int64_t)v * cols + sb * HQO_QK_K + e];
                        acc += p;
                        aabs += fabs(p);
                    }
                }
                y[(int64_t)v * rows + i] = acc;
                if (T) T[(int64_t)v * rows + i] = aabs;
            }
        return;
    }
    int64_t nb = cols / HQO_QK;
    int64_t bpb = fmt == 8 ? HQO_Q8_0_BYTES : HQO_Q4_0_BYTES;
    for (int64_t i = row_lo; i < row_hi; ++i) {
        for (int v = 0; v < n_vec; ++v) {
            double acc = 0.0, aabs = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                const uint8_t *blk = bytes + (i * nb + b) * bpb;
                double d = (double)hqo_half_to_float(load_u16le(blk));
                for (int j = 0; j < HQO_QK; ++j) {
                    int q;
                    if (fmt == 8) q = (int8_t)blk[2 + j];
                    else q = (j < 16 ? (blk[2 + j] & 0x0f) : (blk[2 + j - 16] >> 4)) - 8;
                    double w = d * (double)q;
                    double p = w * (double)x[(int64_t)v * cols + b * HQO_QK + j];
                    acc += p;
                    aabs += fabs(p);
                }
            }
            y[(int64_t)v * rows + i] = acc;
            if (T) T[(int64_t)v * rows + i] = aabs;
        }
    }
}

void hqo_matvec_q8_0(const uint8_t *W, const float *x, int64_t rows, int64_t cols,
                     int n_vec, double *y, double *T)
{
    matvec_rows(8, W, x, 0, rows, rows, cols, n_vec, y, T);
}

void hqo_matvec_q4_0(const uint8_t *W, const float *x, int64_t rows, int64_t cols,
                     int n_vec, double *y, double *T)
{
    matvec_rows(4, W, x, 0, rows, rows, cols, n_vec, y, T);
}

void hqo_matvec_q4_k(const uint8_t *W, const float *x, int64_t rows, int64_t cols,
                     int n_vec, double *y, double *T)
{
    matvec_rows('K', W, x, 0, rows, rows, cols, n_vec, y, T);
}

/* Rows [row_lo, row_hi) only, for sampled checks at full size (fmt 8: Q8_0,
 * 4: Q4_0, 'K': Q4_K). */
void hqo_matvec_rows(int fmt, const uint8_t *W, const float *x, int64_t row_lo,
                     int64_t row_hi, int64_t rows, int64_t cols, int n_vec,
                     double *y, double *T)
{
    matvec_rows(fmt, W, x, row_lo, row_hi, rows, cols, n_vec, y, T);
}

/* ------------------------------------------------------------------------ */
/* MoE ([NST] "The Unified Quant Core"; [EPS]): every routed expert is the   */
/* same matvec on that expert's matrix.  For token t and slot k,             */
/* y[t][k] = W_bank[ids[t][k]] . x(t,k), x(t,k) = x[t] (shared) or x[t][k].   */
/* No router weighting.  ids outside [0, n_experts) make the call fail (-1). */
/* ------------------------------------------------------------------------ */

int hqo_moe_matvec_q8_0(const uint8_t *bank, const int32_t *ids, const float *x,
                        int x_per_slot, int64_t n_experts, int n_active,
                        int64_t rows, int64_t cols, int n_vec, double *y, double *T)
{
    int64_t mat_bytes = rows * (cols / HQO_QK) * HQO_Q8_0_BYTES;
    for (int t = 0; t < n_vec; ++t)
        for (int k = 0; k < n_active; ++k) {
            int32_t e = ids[t * n_active + k];
            if (e < 0 || e >= n_experts) return -1;
            const float *xv = x + (x_per_slot ? ((int64_t)t * n_active + k) : (int64_t)t) * cols;
            double *yv = y + ((int64_t)t * n_active + k) * rows;
            double *Tv = T ? T + ((int64_t)t * n_active + k) * rows : 0;
            matvec_rows(8, bank + (int64_t)e * mat_bytes, xv, 0, rows, rows, cols, 1, yv, Tv);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Integer path ([ZEN] "Quantization recipe"): gemmlowp fixed point.         */
/* ------------------------------------------------------------------------ */

/* SaturatingRoundingDoublingHighMul: the high 32 bits of 2*a*b, rounded to
 * nearest with ties toward +infinity; the one overflowing case
 * a = b = INT32_MIN saturates to INT32_MAX. */
int32_t hqo_srdhm(int32_t a, int32_t b)
{
    if (a == INT32_MIN && b == INT32_MIN) return INT32_MAX;
    int64_t ab = (int64_t)a * (int64_t)b;
    int64_t nudge = ab >= 0 ? ((int64_t)1 << 30) : (1 - ((int64_t)1 << 30));
    return (int32_t)((ab + nudge) / ((int64_t)1 << 31));   /* C division truncates */
}

/* RoundingDivideByPOT: x / 2^e rounded to nearest, ties away from zero. */
int32_t hqo_rdivbypot(int32_t x, int e)
{
    int64_t mask = ((int64_t)1 << e) - 1;
    int64_t rem = (int64_t)x & mask;
    int64_t thr = (mask >> 1) + (x < 0 ? 1 : 0);
    int64_t q = (int64_t)x >> e;                            /* arithmetic shift */
    return (int32_t)(q + (rem > thr ? 1 : 0));
}

int8_t hqo_requant(int32_t acc, int32_t mult, int32_t shift)
{
    int32_t r = hqo_rdivbypot(hqo_srdhm(acc, mult), shift);
    return (int8_t)clamp_i32(r, -128, 127);
}

/* y[v][o] = requant( sum_j Wq[o][j] * xq[v][j] ); the int32 accumulator is
 * also returned in acc (if non-null).  Sums are taken in int64 and must fit
 * int32 (they do for |w|,|x| <= 127 and cols < 133,000); -1 otherwise. */
int hqo_matvec_i8_requant(const int8_t *Wq, const int8_t *xq, const int32_t *mult,
                          const int32_t *shift, int64_t rows, int64_t cols,
                          int n_vec, int8_t *y, int32_t *acc)
{
    for (int v = 0; v < n_vec; ++v)
        for (int64_t o = 0; o < rows; ++o) {
            int64_t s = 0;
            for (int64_t j = 0; j < cols; ++j)
                s += (int64_t)Wq[o * cols + j] * (int64_t)xq[(int64_t)v * cols + j];
            if (s > INT32_MAX || s < INT32_MIN) return -1;
            if (acc) acc[(int64_t)v * rows + o] = (int32_t)s;
            y[(int64_t)v * rows + o] = hqo_requant((int32_t)s, mult[o], shift[o]);
        }
    return 0;
}

void hqo_requant_array(const int32_t *acc, const int32_t *mult, const int32_t *shift,
                       int64_t n, int64_t rows, int8_t *y)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = hqo_requant(acc[i], mult[i % rows], shift[i % rows]);
}

/* Real multiplier M in (0, 1) -> (mult, shift) with M ~= mult * 2^-31 * 2^-shift:
 * M = f * 2^-shift with f in [0.5, 1); mult = round(f * 2^31) (half away from
 * zero); if that reaches 2^31 then mult = 2^30 and shift -= 1.  Returns -1 if
 * M is not in (0,1) or the shift would exceed 31. */
int hqo_requant_params(const double *M, int64_t n, int32_t *mult, int32_t *shift)
{
    for (int64_t i = 0; i < n; ++i) {
        double m = M[i];
        if (!(m > 0.0 && m < 1.0)) return -1;
        int e;
        double f = frexp(m, &e);          /* m = f * 2^e, f in [0.5,1), e <= 0 */
        int s = -e;
        long long q = llround(ldexp(f, 31));
        if (q == (1LL << 31)) { q = 1LL << 30; s -= 1; }
        if (s > 31 || s < 0) return -1;
        mult[i] = (int32_t)q;
        shift[i] = s;
    }
    return 0;
}

/* ---------------------------------------------------------------- QLoRA adapter term
 * [NST] section "The Central Efficiency Thesis", Lemma "QLoRA over the unified
 * core is exact": y_i = sum_j What_ij x_j + (alpha/r) (B_A (A x))_i, with
 * A in R^{r x d_in} and B_A in R^{d_out x r} stored in bf16.  The oracle
 * returns the adapter term alone (the base term is the matvec above), in f64:
 *   u_k       = sum_j A[k][j] * x[v][j]
 *   delta[v][i] = scale * sum_k B[i][k] * u_k          (scale = alpha / r)
 * and T[v][i] = |scale| * sum_k |B[i][k]| * sum_j |A[k][j] * x[v][j]|, the
 * magnitude the float tolerance is taken against. */

/* bf16 is the upper half of an fp32 bit pattern. */
float hqo_bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int hqo_lora_delta(const uint16_t *A, const uint16_t *B, const float *x, double scale,
                   int64_t rank, int64_t rows, int64_t cols, int64_t n_vec,
                   double *delta, double *T)
{
    /* any rank >= 1: u = A x and its magnitudes live in heap buffers of rank
       entries; returns -1 (and writes nothing) if rank < 1 or they cannot be
       allocated, 0 otherwise */
    if (rank < 1) return -1;
    double *u = (double *)malloc((size_t)rank * sizeof(double));
    double *ua = (double *)malloc((size_t)rank * sizeof(double));
    if (!u || !ua) { free(u); free(ua); return -1; }
    for (int64_t v = 0; v < n_vec; ++v) {
        /* the bracket (A x) first, as the Lemma writes it */
        for (int64_t k = 0; k < rank; ++k) {
            u[k] = 0.0;
            ua[k] = 0.0;
            for (int64_t j = 0; j < cols; ++j) {
                double p = (double)hqo_bf16_to_float(A[k * cols + j]) * (double)x[v * cols + j];
                u[k] += p;
                ua[k] += fabs(p);
            }
        }
        /* then B_A applied to it, and the scale */
        for (int64_t i = 0; i < rows; ++i) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < rank; ++k) {
                double b = (double)hqo_bf16_to_float(B[i * rank + k]);
                acc += b * u[k];
                mag += fabs(b) * ua[k];
            }
            delta[v * rows + i] = scale * acc;
            T[v * rows + i] = fabs(scale) * mag;
        }
    }
    free(u);
    free(ua);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* MoE epilogues.                                                            */
/*                                                                           */
/* SwiGLU ([ZEN] "Architecture": every layer's feed-forward is               */
/* SwiGLU(gate, up, down)).  Reading: the gate is swish-1, silu(z) =         */
/* z * sigmoid(z) = z / (1 + e^-z), as in the GLU-variant definition of      */
/* SwiGLU; the hidden value is h_i = silu(gate_i) * up_i.  Reading of the     */
/* layout: an expert's gate and up matrices are stored as one matrix with    */
/* their rows interleaved, row 2i = gate row i and row 2i+1 = up row i, so a */
/* matvec output y gives h_i = silu(y[2i]) * y[2i+1].                        */
/* ------------------------------------------------------------------------ */

double hqo_silu(double z)
{
    return z / (1.0 + exp(-z));
}

void hqo_swiglu_pairs(const double *y, int64_t n_pairs, double *h)
{
    for (int64_t i = 0; i < n_pairs; ++i) {
        double gate = y[2 * i], up = y[2 * i + 1];
        h[i] = hqo_silu(gate) * up;
    }
}

/* Router-weighted sum over the slots ([EPS] "MoE is the cheapest-per-      */
/* quality tier": a sparsely gated mixture reads only its chosen experts;    */
/* the layer's output is the gate-weighted sum of those experts' outputs).   */
/* w[t][k] is the router's weight for token t's slot k (an input: the router */
/* itself is not on the path).  out[t][i] = sum_k w[t][k] * y[t][k][i], k in */
/* slot order, and Tout = sum_k |w[t][k]| * T[t][k][i], the magnitude the    */
/* float tolerance is taken against.                                         */
void hqo_moe_combine(const double *y, const double *T, const float *w, int n_vec, int n_active,
                     int64_t rows, double *out, double *Tout)
{
    for (int t = 0; t < n_vec; ++t)
        for (int64_t i = 0; i < rows; ++i) {
            double acc = 0.0, mag = 0.0;
            for (int k = 0; k < n_active; ++k) {
                double wk = (double)w[t * n_active + k];
                int64_t at = ((int64_t)t * n_active + k) * rows + i;
                acc += wk * y[at];
                if (T) mag += fabs(wk) * T[at];
            }
            out[(int64_t)t * rows + i] = acc;
            if (Tout) Tout[(int64_t)t * rows + i] = mag;
        }
}

int hqo_version(void) { return 1; }
