/*
 * q8_oracle.c -- plain, slow, scalar CPU oracle for the Q8_0 quantized
 * projection.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  The CUDA library never links,
 * includes or calls it, and it shares no code, header or table with that
 * library.
 *
 * Build: any C11 compiler with -O2 -ffp-contract=off (no fast-math), so that
 * every float expression below rounds exactly as written (a*b+c is never
 * contracted into an FMA).  OpenMP, when enabled, only splits the independent
 * output rows n across threads; the arithmetic of each output is unchanged.
 *
 * Sources.  The pages describing the method are the rustdoc pages of
 * logicaffeine_compile:
 *   [lane]   codegen_cuda::lane, module description ("CudaKnobs": the three
 *            activation numerics, fuse_quant) and "Modules: kernels" (an
 *            activation quantized in a producer's epilogue);
 *   [author] model::author, module description (weights recorded as
 *            <var>.q / <var>.s: Q8_0 quants and block scales) and
 *            "Functions: decode_head" (final norm, LM head, arg-max);
 *   [stream] spatial::streamed, "A weight moves as it is stored" (int8
 *            values and block scales folded inside the product).
 * The pages state none of the formulas; where they are silent the readings
 * below are the ones listed with the design notes (block of 32, symmetric
 * +-127 codes, fp16 weight scales, f32 activation scales, round half away
 * from zero, the 14-bit hi/lo split, RMSNorm with an f64 sum of squares).
 *
 * Every function here is pinned by tests that do not call it twice: numpy's
 * binary16 conversion, brute-force dequantise-then-dense products, Python
 * exact rationals, closed-form special cases and hand-worked examples.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 32

int orc_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- binary16 */

/* IEEE binary16 value of the bit pattern h (exact in float). */
float orc_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* zero or subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/1024) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/*
 * Round a float to binary16, nearest-even, by the definition: find the
 * binary16 quantum at |f|'s binade, divide (exact: a power of two), round the
 * quotient to an integer with ties to even, multiply back, then encode.
 */
uint16_t orc_f32_to_f16(float f) {
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00);
    if (a == 0.0) return sign;
    if (isinf(f)) return (uint16_t)(sign | 0x7c00);
    int e;
    frexp(a, &e);                /* a in [2^(e-1), 2^e) */
    int eb = e - 1;              /* binade exponent */
    double quantum = (eb >= -14) ? ldexp(1.0, eb - 10) : ldexp(1.0, -24);
    double r = a / quantum;      /* exact */
    double fl = floor(r);
    double frac = r - fl;        /* exact */
    double n;
    if (frac > 0.5)
        n = fl + 1.0;
    else if (frac < 0.5)
        n = fl;
    else
        n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;   /* tie: to even */
    double v = n * quantum;      /* exact, may step into the next binade */
    if (v > 65504.0) return (uint16_t)(sign | 0x7c00);
    if (v < ldexp(1.0, -14)) {                         /* subnormal */
        return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -24)));
    }
    frexp(v, &e);
    eb = e - 1;
    int mant = (int)(v / ldexp(1.0, eb - 10)) - 1024;
    return (uint16_t)(sign | ((eb + 15) << 10) | mant);
}

static float clampf(float v, float lo, float hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

/* ---------------------------------------------------------- weight pack */

/*
 * Q8_0 pack [author: <var>.q / <var>.s].  Per row n and 32-value block b:
 *   amax = max |w|, d = amax / 127 (f32), s = binary16(d) (the stored scale),
 *   q = round_half_away(w / float(s)) clamped to [-127, 127]; q = 0 when s == 0.
 * Returns the number of blocks whose scale overflowed binary16 (then q = 0).
 */
int64_t orc_q8_pack(const float* w, int64_t N, int64_t K, int8_t* q, uint16_t* s) {
    int64_t nb = K / QK, overflow = 0;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* wb = w + n * K + b * QK;
            float amax = 0.0f;
            for (int i = 0; i < QK; ++i) {
                float a = fabsf(wb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            uint16_t sh = orc_f32_to_f16(d);
            float sf = orc_f16_to_f32(sh);
            if (isinf(sf)) overflow++;
            s[n * nb + b] = sh;
            for (int i = 0; i < QK; ++i) {
                float v = (sf == 0.0f) ? 0.0f : clampf(roundf(wb[i] / sf), -127.0f, 127.0f);
                if (isnan(v)) v = 0.0f;
                q[n * K + b * QK + i] = (int8_t)(int)v;
            }
        }
    }
    return overflow;
}

/* ------------------------------------------------- activation producers */

/*
 * RMSNorm producer [lane: kernels, "a residual added before a norm";
 * author: decode_head, "the final norm"].  Per row:
 *   ss = sum_k h_k^2 in f64 (k ascending), r = 1 / sqrt(ss / K + eps) in f64,
 *   rf = float(r), x_k = (h_k * rf) * g_k as two rounded f32 products.
 * g == NULL means a gain of one.  rf_out (nullable) receives r per row.
 */
void orc_rmsnorm(const float* h, const float* g, int64_t rows, int64_t K, float eps,
                 float* x, double* r_out) {
    for (int64_t m = 0; m < rows; ++m) {
        const float* hm = h + m * K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double hk = (double)hm[k];
            ss = ss + hk * hk;
        }
        double r = 1.0 / sqrt(ss / (double)K + (double)eps);
        float rf = (float)r;
        if (r_out) r_out[m] = r;
        for (int64_t k = 0; k < K; ++k) {
            float t = hm[k] * rf;
            x[m * K + k] = g ? t * g[k] : t;
        }
    }
}

/*
 * Residual added before the norm [lane: "Modules: kernels", a residual added
 * before a norm].  s = h + r per value, one f32 addition (the sum of two f32
 * values rounded once to f32); s is the RMSNorm's input and the updated
 * residual stream.
 */
void orc_residual_add(const float* h, const float* r, int64_t rows, int64_t K, float* s) {
    for (int64_t i = 0; i < rows * K; ++i) s[i] = h[i] + r[i];
}

/*
 * e^x in binary32, the one definition both sides of a SwiGLU parity check
 * compute (a decision of a quantised code rests on it).  Method: Cody and
 * Waite's argument reduction, x = k*ln2 + r with k = rint(x/ln2) and
 * |r| <= ln2/2, where ln2 is carried as a 16-bit head (so k*head is exact for
 * |k| <= 2^8) plus its binary32 remainder; then e^r by its Taylor series to
 * degree 7, 1 + r + r^2/2! + ... + r^7/7! (coefficients 1/i! rounded to
 * binary32), in Horner form with fused multiply-adds; then times 2^k in two
 * exact power-of-two steps.  Truncation error below r^8/8! < 6e-9 relative.
 *   1/ln2 -> 0x1.715476p+0, ln2 head 0x1.62e4p-1, remainder 0x1.7f7d1cp-20.
 */
float orc_exp_f32(float x) {
    if (x != x) return x;
    if (x > 88.75f) return INFINITY;
    if (x < -104.0f) return 0.0f;
    const float magic = 12582912.0f;   /* 1.5 * 2^23: rint by addition */
    const float t = fmaf(x, 0x1.715476p+0f, magic);
    const float kf = t - magic;
    const int k = (int)kf;
    float r = fmaf(-kf, 0x1.62e4p-1f, x);
    r = fmaf(-kf, 0x1.7f7d1cp-20f, r);
    float p = 0x1.a01a02p-13f;           /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);      /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);       /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);       /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);       /* 1/3! */
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    const int k1 = k >> 1, k2 = k - k1;   /* each in [-76, 64]: exact powers */
    return (p * ldexpf(1.0f, k1)) * ldexpf(1.0f, k2);
}

/*
 * The SwiGLU producer of the down projection [lane: "Modules: kernels", an
 * activation quantized in a producer's epilogue; the FFN whose gate and up
 * projections run as one fused matrix].  gu[m] holds the fused gate+up output
 * row: gate = gu[m][0..F), up = gu[m][F..2F).  x = silu(gate) * up with
 * silu(g) = g / (1 + e^-g), every step one binary32 rounding (e^-g by
 * orc_exp_f32, the division IEEE).
 */
void orc_swiglu(const float* gu, int64_t rows, int64_t F, float* x) {
    for (int64_t m = 0; m < rows; ++m) {
        const float* g = gu + m * 2 * F;
        const float* u = g + F;
        for (int64_t k = 0; k < F; ++k) {
            const float e = orc_exp_f32(-g[k]);
            const float silu = g[k] / (1.0f + e);
            x[m * F + k] = silu * u[k];
        }
    }
}

/*
 * The K/V slice of a fused QKV projection written into the row of a cache a
 * position names [lane: "Modules: kernels", a result written into the row of
 * a cache a position names].  y [rows][N] is the projection output; row m's
 * columns [kv_col, kv_col + D) are its K, [kv_col + D, kv_col + 2D) its V; the
 * caches are [rows][n_pos][D] (one per sequence) and row m's entries go to
 * cache row pos[m].  A position outside [0, n_pos) writes nothing and is
 * counted in the return value.
 */
int64_t orc_kv_write(const float* y, int64_t rows, int64_t N, const int32_t* pos, int64_t kv_col,
                     int64_t D, int64_t n_pos, float* k_cache, float* v_cache) {
    int64_t bad = 0;
    for (int64_t m = 0; m < rows; ++m) {
        if (pos[m] < 0 || pos[m] >= n_pos) {
            ++bad;
            continue;
        }
        for (int64_t d = 0; d < D; ++d) {
            k_cache[(m * n_pos + pos[m]) * D + d] = y[m * N + kv_col + d];
            v_cache[(m * n_pos + pos[m]) * D + d] = y[m * N + kv_col + D + d];
        }
    }
    return bad;
}

/*
 * Mode "one int8 word" [lane: CudaKnobs, llama.cpp's one int8 word].  Per row m
 * and block b: amax = max |x|, d = amax / 127 (f32, kept as f32),
 * q = round_half_away(x / d) clamped to [-127, 127]; q = 0 when d == 0.
 */
void orc_act_quant_i8(const float* x, int64_t rows, int64_t K, int8_t* xq, float* xd) {
    int64_t nb = K / QK;
    for (int64_t m = 0; m < rows; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* xb = x + m * K + b * QK;
            float amax = 0.0f;
            for (int i = 0; i < QK; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            xd[m * nb + b] = d;
            for (int i = 0; i < QK; ++i) {
                float v = (d == 0.0f) ? 0.0f : clampf(roundf(xb[i] / d), -127.0f, 127.0f);
                xq[m * K + b * QK + i] = (int8_t)(int)v;
            }
        }
    }
}

/*
 * Mode "two-word ~14-bit int8" [lane: CudaKnobs, the default numerics].  Per
 * row m and block b: d = amax / 8191 (f32), Q = round_half_away(x / d)
 * clamped to [-8191, 8191] (a signed 14-bit code), then split into two int8
 * words with Q = 128 * hi + lo:
 *   lo = ((Q + 64) mod 128) - 64   (Euclidean mod, lo in [-64, 63])
 *   hi = (Q - lo) / 128            (exact, hi in [-64, 64]).
 */
void orc_act_quant_i8x2(const float* x, int64_t rows, int64_t K, int8_t* xh, int8_t* xl,
                        float* xd) {
    int64_t nb = K / QK;
    for (int64_t m = 0; m < rows; ++m) {
        for (int64_t b = 0; b < nb; ++b) {
            const float* xb = x + m * K + b * QK;
            float amax = 0.0f;
            for (int i = 0; i < QK; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 8191.0f;
            xd[m * nb + b] = d;
            for (int i = 0; i < QK; ++i) {
                float v = (d == 0.0f) ? 0.0f : clampf(roundf(xb[i] / d), -8191.0f, 8191.0f);
                int Q = (int)v;
                int r = (Q + 64) % 128;
                if (r < 0) r += 128;
                int lo = r - 64;
                int hi = (Q - lo) / 128;
                xh[m * K + b * QK + i] = (int8_t)hi;
                xl[m * K + b * QK + i] = (int8_t)lo;
            }
        }
    }
}

/* ------------------------------------------------------ block dot products */

/*
 * Per-block int32 dots isum[m][n][b] = sum_{i<32} q[n][32b+i] * a[m][32b+i],
 * where a is the one-word code (xl == NULL) or the 14-bit code 128*hi + lo.
 * [stream: int8 values and block scales folded inside the product.]
 */
void orc_block_dots(const int8_t* q, const int8_t* xh, const int8_t* xl, int64_t N, int64_t K,
                    int64_t rows, int32_t* isum) {
    int64_t nb = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < rows; ++m) {
            for (int64_t b = 0; b < nb; ++b) {
                int32_t acc = 0;
                for (int i = 0; i < QK; ++i) {
                    int64_t k = b * QK + i;
                    int32_t a = xl ? 128 * (int32_t)xh[m * K + k] + (int32_t)xl[m * K + k]
                                   : (int32_t)xh[m * K + k];
                    acc += (int32_t)q[n * K + k] * a;
                }
                isum[(m * N + n) * nb + b] = acc;
            }
        }
    }
}

/*
 * Quantized projection, one-word or two-word mode [lane: CudaKnobs].
 *   y[m][n] = sum_b float(isum[m][n][b]) * (float(S[n][b]) * xd[m][b])
 * in f32, b ascending; the scale product is rounded first, then the product
 * with the block dot, then the sum.  norm[m][n] (nullable) receives the f64
 * sum of |float(isum)| * |S * xd|, the scale of the float tolerance.
 */
void orc_proj_q(const int8_t* q, const uint16_t* s, const int8_t* xh, const int8_t* xl,
                const float* xd, int64_t N, int64_t K, int64_t rows, float* y, double* norm) {
    int64_t nb = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < rows; ++m) {
            float acc = 0.0f;
            double nrm = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                int32_t isum = 0;
                for (int i = 0; i < QK; ++i) {
                    int64_t k = b * QK + i;
                    int32_t a = xl ? 128 * (int32_t)xh[m * K + k] + (int32_t)xl[m * K + k]
                                   : (int32_t)xh[m * K + k];
                    isum += (int32_t)q[n * K + k] * a;
                }
                float sw = orc_f16_to_f32(s[n * nb + b]);
                float sc = sw * xd[m * nb + b];
                float t = (float)isum * sc;
                acc = acc + t;
                nrm += fabs((double)(float)isum) * fabs((double)sw * (double)xd[m * nb + b]);
            }
            y[m * N + n] = acc;
            if (norm) norm[m * N + n] = nrm;
        }
    }
}

/*
 * Quantized projection, f32 activations with f64 sums [lane: CudaKnobs].
 *   y[m][n] = sum_k double(float(S[n][k/32]) * float(q[n][k])) * double(x[m][k])
 * accumulated in f64, k ascending.  The weight product is exact in f32
 * (11 x 7 bits) and its product with x exact in f64 (18 x 24 bits), so only
 * the sum rounds.  norm (nullable) is the f64 sum of the absolute terms.
 */
void orc_proj_f64(const int8_t* q, const uint16_t* s, const float* x, int64_t N, int64_t K,
                  int64_t rows, double* y, double* norm) {
    int64_t nb = K / QK;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t m = 0; m < rows; ++m) {
            double acc = 0.0, nrm = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                float wk = orc_f16_to_f32(s[n * nb + k / QK]) * (float)q[n * K + k];
                double t = (double)wk * (double)x[m * K + k];
                acc = acc + t;
                nrm = nrm + fabs(t);
            }
            y[m * N + n] = acc;
            if (norm) norm[m * N + n] = nrm;
        }
    }
}

/* ------------------------------------------------------------------ arg-max */

/*
 * Arg-max of each logit row [author: decode_head / decode_step, "the step
 * ends with the arg-max of the logits"]: the smallest n holding the maximum
 * (equal values, including -0 and +0, keep the earlier index).  A NaN logit
 * is no candidate (a Q8_0 block whose binary16 scale overflowed carries an
 * infinite scale, and 0 * inf is NaN); a row of NaN only gives index 0 and the
 * value NaN.  A row of -inf gives index 0 and -inf.
 */
void orc_argmax_f32(const float* logits, int64_t rows, int64_t N, int32_t* tok, float* best) {
    for (int64_t m = 0; m < rows; ++m) {
        int64_t bi = -1;
        float bv = 0.0f;
        for (int64_t n = 0; n < N; ++n) {
            float v = logits[m * N + n];
            if (isnan(v)) continue;
            if (bi < 0 || v > bv) {
                bv = v;
                bi = n;
            }
        }
        if (bi < 0) {
            bi = 0;
            bv = NAN;
        }
        tok[m] = (int32_t)bi;
        if (best) best[m] = bv;
    }
}

void orc_argmax_f64(const double* logits, int64_t rows, int64_t N, int32_t* tok, double* best) {
    for (int64_t m = 0; m < rows; ++m) {
        int64_t bi = -1;
        double bv = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            double v = logits[m * N + n];
            if (isnan(v)) continue;
            if (bi < 0 || v > bv) {
                bv = v;
                bi = n;
            }
        }
        if (bi < 0) {
            bi = 0;
            bv = NAN;
        }
        tok[m] = (int32_t)bi;
        if (best) best[m] = bv;
    }
}

/* ------------------------------------------------- RMSNorm near-tie report */

/*
 * Whether the f64 RMS scale r of a row lies within rel * r of an f32 rounding
 * boundary (the midpoint of two neighbouring binary32 values), where another
 * correct evaluation of r -- another summation order of sum h^2, or an
 * evaluation accurate to rel -- may round to the other f32 neighbour, so
 * rf = float(r), and with it the row's codes, may differ from the oracle's
 * [lane: CudaKnobs fuse_quant; the producer's norm].  Used to classify a
 * mismatch of quantised codes, never to accept one silently.
 */
int orc_near_tie(double r, double rel) {
    if (!(r > 0.0) || isinf(r)) return 0;
    float f = (float)r;
    if ((double)f == r) return 0;
    float other = r > (double)f ? nextafterf(f, INFINITY) : nextafterf(f, -INFINITY);
    double mid = ((double)f + (double)other) * 0.5;   /* exact: 25 significant bits */
    return fabs(r - mid) <= rel * r;
}
