/*
 * Sparse MLA decode oracle -- plain, slow, obviously correct CPU code.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg call this file. The decode library never links, includes
 * or calls it, and it shares no code with the library.
 *
 * What it computes (the "attn_sparse" page, module docstring, paragraphs
 * "Per CTA", "Precision" and "Rows of count 0"; the SparseDcpDecode kernel
 * and its merge method), read with ONE split and the whole row as ONE chunk,
 * so that the P anchor is the maximum over all of the row's keys:
 *
 *   for row b, head h, with n = clamp(counts[b], 0, W) and keys
 *   j_i = indices[b, i], i < n:
 *     S_i  = sum_{c<576} dec(q8[b,h,c]) * dec(kv8[j_i,c])      exact (fp64),
 *            then rounded once to fp32                         ("FP32 logits")
 *     s_i  = fp32(lambda * S_i),  lambda = fp32(sm*q_s*k_s*log2 e)
 *     m    = max_i s_i
 *     P_i  = fp32(2^(fp32(s_i - fp32(m - log2 448))))          exact exp2
 *     P8_i = E4M3 round-to-nearest-even, saturating at +-448
 *     T    = sum_i P_i                 (unquantized P, accumulated in fp64)
 *     A_c  = sum_i P8_i * dec(kv8[j_i, c]),  c < 512          (exact, fp64)
 *     out  = BF16_RNE(k_s * A_c / T)
 *     lse  = ln 2 * (m - log2 448 + log2 T)                   (natural log)
 *   n == 0: out = 0, lse = -inf.
 *
 * The fp32 roundings of S, s, the anchor bias and the exp2 argument follow the
 * kernel's own arithmetic, which the page fixes to Float32; every sum is
 * carried in fp64, where the sums of E4M3 products are exact.
 *
 * Mode SMO_MODE_UNQUANT skips the E4M3 rounding of P (P8_i = P_i): the fp64
 * reference the E4M3 error bound is measured against.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define SMO_ROW 576
#define SMO_LATENT 512
#define SMO_E4M3_MAX 448.0

enum { SMO_MODE_RECIPE = 0, SMO_MODE_UNQUANT = 1 };

/* ---- E4M3 (OCP FP8, the "fn" variant: no infinities, S.1111.111 is NaN) ---- */

/* Value of an E4M3 code: sign bit 7, exponent bits 6..3 with bias 7, mantissa
 * bits 2..0; exponent 0 holds the subnormals m/8 * 2^-6. */
double smo_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* E4M3 of x, rounded to the nearest code (ties to the even code) and
 * saturated to +-448 ("E4M3 (satfinite, RN)", the page's
 * store_fp8_pair_shared). A linear search over the 127 non-negative finite
 * codes. */
uint8_t smo_e4m3_encode(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= SMO_E4M3_MAX) return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(smo_e4m3_decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best_d = d;
            best = c;
        }
    }
    return (uint8_t)(sign | best);
}

/* bfloat16 bits of x rounded to nearest even: 8 significant bits, the
 * exponent range of fp32 (subnormal quantum 2^-133), overflow to infinity. */
uint16_t smo_bf16_rne(double x) {
    if (isnan(x)) return 0x7FC0;
    double a = fabs(x);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else if (a < ldexp(1.0, -126)) {
        r = ldexp(nearbyint(ldexp(a, 133)), -133);
    } else {
        int e;
        double f = frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
        r = ldexp(nearbyint(ldexp(f, 8)), e - 8);
    }
    float rf = (r >= ldexp(1.0, 128)) ? INFINITY : (float)r; /* exact */
    if (signbit(x)) rf = -rf;
    uint32_t bits;
    memcpy(&bits, &rf, 4);
    return (uint16_t)(bits >> 16);
}

/* The base-2 logit scale: sm_scale * q_scale * k_scale * log2(e), the
 * page's scale_log2 (run_sparse passes it precomputed), evaluated in fp64
 * and rounded once to fp32. */
float smo_scale_log2(float sm_scale, float q_scale, float k_scale) {
    double v = (double)sm_scale * (double)q_scale * (double)k_scale;
    return (float)(v * 1.4426950408889634073599246810019);
}

static float f32(double x) { return (float)x; }

/* Exact logit S of (row b, head h) against cache row j, in fp64: each
 * E4M3 x E4M3 product has at most 8 significant bits and the 576-term sum
 * stays far inside fp64's 53 bits. */
static double logit_exact(const uint8_t* q_bh, const uint8_t* kv_row, const double* dec) {
    double s = 0.0;
    for (int c = 0; c < SMO_ROW; ++c) s += dec[q_bh[c]] * dec[kv_row[c]];
    return s;
}

/* The same with the query given by its values (qv[c]: the value the query
 * column stands for, already exact in fp64). */
static double logit_exact_v(const double* qv, const uint8_t* kv_row, const double* dec) {
    double s = 0.0;
    for (int c = 0; c < SMO_ROW; ++c) s += qv[c] * dec[kv_row[c]];
    return s;
}

/* ---- BF16 query split into E4M3 hi + lo (the mla_attn page: "q_split", the
 * bf16 Q rows to "E4M3 hi, lo of q 2^k"; "fp8_split4", x ~ hi + lo) ----------
 * Reading: one power-of-two scale 2^k per (row, head), the largest k with
 * amax * 2^k <= 448 (amax = max |q| over the 576 columns; k = 0 when amax is
 * 0; k clamped to [-32, 32]); hi = E4M3(q 2^k), lo = E4M3(q 2^k - hi), both
 * round-to-nearest-even and saturating. q 2^k and q 2^k - hi are exact in
 * fp64 (and fp32). The logit is then sum (hi + lo) kv, and the query scale
 * 2^-k goes into lambda: lambda_h = fp32(sm * 2^-k * k_s * log2 e). */
static double bf16_value(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
}

int smo_q_split_exponent(double amax) {
    if (!(amax > 0.0)) return 0;
    int e = 0;
    const double m = frexp(amax, &e); /* amax = m 2^e, m in [0.5, 1) */
    /* amax 2^k <= 448 = 0.875 * 2^9  <=>  m 2^(e + k) <= 0.875 2^9 */
    int k = (m <= 0.875) ? 9 - e : 8 - e;
    if (k < -32) k = -32;
    if (k > 32) k = 32;
    return k;
}

/* Splits one 576-column bf16 query row; returns k. */
int smo_q_split(const uint16_t* q_row, uint8_t* hi, uint8_t* lo) {
    double amax = 0.0;
    for (int c = 0; c < SMO_ROW; ++c) {
        const double a = fabs(bf16_value(q_row[c]));
        if (a > amax) amax = a;
    }
    const int k = smo_q_split_exponent(amax);
    for (int c = 0; c < SMO_ROW; ++c) {
        const double x = ldexp(bf16_value(q_row[c]), k);
        hi[c] = smo_e4m3_encode(x);
        lo[c] = smo_e4m3_encode(x - smo_e4m3_decode(hi[c]));
    }
    return k;
}

static int32_t clamp_count(int32_t c, int32_t W) {
    if (c < 0) return 0;
    if (c > W) return W;
    return c;
}

/* Per-key intermediate values of one (row, head): the exact logit S, the
 * scaled fp32 logit s, the unquantized fp32 P and its E4M3 code. Returns n.
 * Used by the tests to check single steps of the recipe. */
int32_t smo_row_head_terms(const uint8_t* q, const uint8_t* kv, int64_t N,
                           const int32_t* indices, int32_t W, const int32_t* counts,
                           int32_t H, int32_t b, int32_t h,
                           float sm_scale, float q_scale, float k_scale,
                           double* S_out, float* s_out, float* P_out, uint8_t* P8_out,
                           float* m_out) {
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = smo_e4m3_decode((uint8_t)c);
    const float lam = smo_scale_log2(sm_scale, q_scale, k_scale);
    const float log2_448 = f32(log2(SMO_E4M3_MAX));
    const int32_t n = clamp_count(counts[b], W);
    const uint8_t* qbh = q + ((int64_t)b * H + h) * SMO_ROW;
    float m = -INFINITY;
    for (int32_t i = 0; i < n; ++i) {
        int64_t j = indices[(int64_t)b * W + i];
        if (j < 0 || j >= N) return -1;
        double S = logit_exact(qbh, kv + j * SMO_ROW, dec);
        float s = f32((double)lam * (double)f32(S));
        if (S_out) S_out[i] = S;
        if (s_out) s_out[i] = s;
        if (s > m) m = s;
    }
    float bias = f32((double)m - (double)log2_448);
    for (int32_t i = 0; i < n && (P_out || P8_out); ++i) {
        int64_t j = indices[(int64_t)b * W + i];
        float s = f32((double)lam * (double)f32(logit_exact(qbh, kv + j * SMO_ROW, dec)));
        float P = f32(exp2((double)f32((double)s - (double)bias)));
        if (P_out) P_out[i] = P;
        if (P8_out) P8_out[i] = smo_e4m3_encode(P);
    }
    if (m_out) *m_out = m;
    return n;
}

/* One (row, head): the query as values qv[576], its lambda, the row's n
 * keys. Writes 512 outputs and the LSE; returns 1 if an index lies outside
 * [0, N). */
static int decode_bh(const double* qv, float lam, const uint8_t* kv, int64_t N,
                     const int32_t* row_idx, int32_t n, float k_scale, int mode,
                     const double* dec, uint16_t* o16, double* o64, double* lse_out) {
    const float log2_448 = f32(log2(SMO_E4M3_MAX));
    /* Rows of count 0 write zeros and LSE -inf ("Rows of count 0"). */
    if (n == 0) {
        for (int c = 0; c < SMO_LATENT; ++c) {
            o16[c] = 0;
            if (o64) o64[c] = 0.0;
        }
        *lse_out = -INFINITY;
        return 0;
    }

    float* s = (float*)malloc(sizeof(float) * (size_t)n);
    double* A = (double*)calloc(SMO_LATENT, sizeof(double));
    int row_bad = 0;

    /* Logits: FP8 x FP8 over all 576 columns, FP32 result, scaled to base 2
     * ("s * scale_log2"). */
    float m = -INFINITY;
    for (int32_t i = 0; i < n; ++i) {
        int64_t j = row_idx[i];
        if (j < 0 || j >= N) {
            row_bad = 1;
            s[i] = -INFINITY;
            continue;
        }
        double S = logit_exact_v(qv, kv + j * SMO_ROW, dec);
        s[i] = f32((double)lam * (double)f32(S));
        if (s[i] > m) m = s[i];
    }

    /* P at 448 of the row maximum, E4M3 (RN, satfinite); the sum T of the
     * unquantized P; A = P8 x V over the 512 latent columns. */
    const float bias = f32((double)m - (double)log2_448);
    double T = 0.0;
    for (int32_t i = 0; i < n && !row_bad; ++i) {
        int64_t j = row_idx[i];
        float P = f32(exp2((double)f32((double)s[i] - (double)bias)));
        T += (double)P;
        double P8 = (mode == SMO_MODE_UNQUANT) ? (double)P : dec[smo_e4m3_encode(P)];
        const uint8_t* v = kv + j * SMO_ROW;
        for (int c = 0; c < SMO_LATENT; ++c) A[c] += P8 * dec[v[c]];
    }

    /* Output BF16(k_scale * A / T) and LSE = ln2 * (m - log2 448 + log2 T) (the
     * merge: "BF16(sum * k_scale / total)", "max + log2(total / 448)", natural
     * log for the plain output). */
    for (int c = 0; c < SMO_LATENT; ++c) {
        double o = row_bad ? NAN : (double)k_scale * A[c] / T;
        o16[c] = smo_bf16_rne(o);
        if (o64) o64[c] = o;
    }
    *lse_out = row_bad ? NAN
                       : 0.69314718055994530941723212145818 *
                             ((double)m - log2(SMO_E4M3_MAX) + log2(T));
    free(s);
    free(A);
    return row_bad;
}

/* The whole decode. out_bf16 [B,H,512] (bf16 bits), out_f64 [B,H,512]
 * (k_s*A/T before the BF16 rounding; may be NULL), lse [B,H] (natural log).
 * Returns 0, or -1 if an index of a valid entry lies outside [0, N). */
int smo_sparse_mla_decode(const uint8_t* q, const uint8_t* kv, int64_t N,
                          const int32_t* indices, int32_t W, const int32_t* counts,
                          int32_t B, int32_t H,
                          float sm_scale, float q_scale, float k_scale,
                          int mode, int nthreads,
                          uint16_t* out_bf16, double* out_f64, double* lse) {
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = smo_e4m3_decode((uint8_t)c);
    const float lam = smo_scale_log2(sm_scale, q_scale, k_scale);
    int bad = 0;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        const int32_t b = (int32_t)(bh / H);
        const uint8_t* qbh = q + bh * SMO_ROW;
        double qv[SMO_ROW];
        for (int c = 0; c < SMO_ROW; ++c) qv[c] = dec[qbh[c]];
        bad |= decode_bh(qv, lam, kv, N, indices + (int64_t)b * W, clamp_count(counts[b], W),
                         k_scale, mode, dec, out_bf16 + bh * SMO_LATENT,
                         out_f64 ? out_f64 + bh * SMO_LATENT : NULL, lse + bh);
    }
    return bad ? -1 : 0;
}

/* The decode with a BF16 query [B,H,576] (bf16 bits), each (row, head) split
 * into E4M3 hi + lo at its own power-of-two scale (smo_q_split): the logit is
 * sum (hi + lo) kv and lambda_h = fp32(sm * 2^-k * k_s * log2 e); everything
 * after the logits as smo_sparse_mla_decode. k_out [B,H] (may be NULL)
 * receives each split's exponent. */
int smo_sparse_mla_decode_bf16q(const uint16_t* q, const uint8_t* kv, int64_t N,
                                const int32_t* indices, int32_t W, const int32_t* counts,
                                int32_t B, int32_t H, float sm_scale, float k_scale,
                                int mode, int nthreads,
                                uint16_t* out_bf16, double* out_f64, double* lse,
                                int32_t* k_out) {
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = smo_e4m3_decode((uint8_t)c);
    int bad = 0;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        const int32_t b = (int32_t)(bh / H);
        uint8_t hi[SMO_ROW], lo[SMO_ROW];
        const int k = smo_q_split(q + bh * SMO_ROW, hi, lo);
        if (k_out) k_out[bh] = k;
        double qv[SMO_ROW];
        for (int c = 0; c < SMO_ROW; ++c) qv[c] = dec[hi[c]] + dec[lo[c]];
        const float lam = smo_scale_log2(sm_scale, (float)ldexp(1.0, -k), k_scale);
        bad |= decode_bh(qv, lam, kv, N, indices + (int64_t)b * W, clamp_count(counts[b], W),
                         k_scale, mode, dec, out_bf16 + bh * SMO_LATENT,
                         out_f64 ? out_f64 + bh * SMO_LATENT : NULL, lse + bh);
    }
    return bad ? -1 : 0;
}

/* Threads OpenMP would use for nthreads <= 0 (1 without OpenMP). */
int smo_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
