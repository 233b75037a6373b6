/*
 * oracle.c -- plain, slow CPU oracle for single-query (decode-step) attention
 * against an f16 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Source of the method: "Developing Apple Metal Kernels in Rust - A Deep Dive
 * Through Attention", section "The MSL, briefly":
 *   - kernel attention_qk_f16: score[h,pos] = (sum_i Q[h,i] * K_cache[pos,h,i])
 *     * (1/sqrt(head_dim)), replaced by -infinity when pos > current_pos, stored
 *     as half into scores[h*seq_len + pos];
 *   - kernel attention_pv_f16: per head, global max over the scores, global sum
 *     of exp(score - max), then out[h,d] = sum_i exp(score_i - max)/sum * V[i,h,d],
 *     stored as half.
 * Layouts (same section, argument comments): Q [n_heads, head_dim],
 * K_cache / V_cache [seq_len, n_heads, head_dim], scores [n_heads, seq_len],
 * output [n_heads, head_dim].  Element (pos, head, i) of the cache sits at
 * (pos*n_heads + head)*head_dim + i.
 *
 * Readings taken where the page is silent:
 *   - a leading batch dimension: Q [B,H,D], caches [B,S,H,D], out [B,H,D],
 *     one current_pos per sequence, sequences independent;
 *   - current_pos >= seq_len masks nothing (the page's test "pos > current_pos"
 *     then never fires), so the live length is L = min(cp, S-1) + 1;
 *   - the fused result is the exact masked softmax attention; this oracle
 *     evaluates it in fp64 on the f16 inputs decoded exactly, and does not round
 *     the scores to f16 (that round trip belongs to the page's two-dispatch
 *     design, reproduced separately below for the split calls).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (see build.py).
 * -ffp-contract=off matters for the page-precision emulator: the page writes a
 * multiply then an add, each rounded to fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- IEEE 754 binary16 <-> wider types, from the format's definition ---- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), e - 25); /* (1 + frac/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Round a float to binary16, round-to-nearest, ties to even.  Every step below
 * is exact in double except rint(), which rounds to an integer with ties to even
 * under the default rounding mode. */
uint16_t oracle_f32_to_f16_rne(float f) {
    double x = (double)f;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: the unit is 2^-24 */
        double q = rint(a * ldexp(1.0, 24));
        return (uint16_t)(sign | (uint16_t)q); /* q == 1024 is the smallest normal */
    }
    int ex;
    (void)frexp(a, &ex); /* a = m * 2^ex with m in [0.5, 1) */
    int E = ex - 1;      /* a in [2^E, 2^(E+1)) */
    double q = rint(a * ldexp(1.0, 10 - E)); /* in [1024, 2048] */
    if (q == 2048.0) {
        q = 1024.0;
        E += 1;
    }
    if (E + 15 >= 31) return (uint16_t)(sign | 0x7c00); /* overflow to infinity */
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024.0));
}

static int64_t live_length(uint32_t cp, int64_t S) {
    /* positions 0..cp are unmasked; cp >= S masks nothing */
    return ((int64_t)cp >= S - 1 ? S - 1 : (int64_t)cp) + 1;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Fused decode attention, fp64.  For each sequence b and head h:
 *   L      = min(cp_b, S-1) + 1
 *   s_p    = (sum_i Q[b,h,i] K[b,p,h,i]) / sqrt(D)          for p < L
 *   M      = max_p s_p
 *   w_p    = exp(s_p - M) / sum_{q<L} exp(s_q - M)
 *   out[d] = sum_{p<L} w_p V[b,p,h,d]
 * Positions p >= L get weight exactly zero (the page's -infinity score), so they
 * are not read at all.  Two plain passes over the live positions.
 */
void oracle_decode_f64(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                       int64_t B, int64_t H, int64_t D, int64_t S,
                       const uint32_t *current_pos, double *out, int nthreads) {
    set_threads(nthreads);
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < B * H; ++bh) {
            const int64_t b = bh / H, h = bh % H;
            const int64_t L = live_length(current_pos[b], S);
            const uint16_t *q = Q + (b * H + h) * D;
            double M = -INFINITY;
            for (int64_t p = 0; p < L; ++p) {
                const uint16_t *k = K + ((b * S + p) * H + h) * D;
                double dot = 0.0;
                for (int64_t i = 0; i < D; ++i)
                    dot += oracle_f16_to_f64(q[i]) * oracle_f16_to_f64(k[i]);
                s[p] = dot * inv_sqrt_d;
                if (s[p] > M) M = s[p];
            }
            double den = 0.0;
            for (int64_t p = 0; p < L; ++p) {
                s[p] = exp(s[p] - M);
                den += s[p];
            }
            double *o = out + (b * H + h) * D;
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t p = 0; p < L; ++p) {
                const uint16_t *v = V + ((b * S + p) * H + h) * D;
                const double w = s[p] / den;
                for (int64_t d = 0; d < D; ++d) o[d] += w * oracle_f16_to_f64(v[d]);
            }
        }
        free(s);
    }
}

/*
 * Decode attention over a paged KV cache, fp64.  The cache holds pages of
 * page_size positions: K_pages / V_pages [num_pages, page_size, H, D].  Position
 * p of sequence b lives in page table[b * max_pages + p / page_size] at row
 * p % page_size, so the logical cache of sequence b is
 *   K[b, p, h, :] = K_pages[table[b, p / page_size], p % page_size, h, :]
 * with capacity S = page_size * max_pages.  Everything else is the fused
 * computation above (same live length, scores, softmax and weighted sum).
 * Page indices outside [0, num_pages) are not read: the affected sequence's
 * output is set to NaN, which no valid result equals.
 */
void oracle_decode_paged_f64(const uint16_t *Q, const uint16_t *K_pages,
                             const uint16_t *V_pages, int64_t B, int64_t H, int64_t D,
                             int64_t page_size, int64_t max_pages, const int32_t *table,
                             int64_t num_pages, const uint32_t *current_pos, double *out,
                             int nthreads) {
    set_threads(nthreads);
    const int64_t S = page_size * max_pages;
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < B * H; ++bh) {
            const int64_t b = bh / H, h = bh % H;
            const int64_t L = live_length(current_pos[b], S);
            const uint16_t *q = Q + (b * H + h) * D;
            double *o = out + (b * H + h) * D;
            int bad = 0;
            for (int64_t p = 0; p < L; ++p) {
                const int64_t pg = table[b * max_pages + p / page_size];
                if (pg < 0 || pg >= num_pages) bad = 1;
            }
            if (bad) {
                for (int64_t d = 0; d < D; ++d) o[d] = NAN;
                continue;
            }
            double M = -INFINITY;
            for (int64_t p = 0; p < L; ++p) {
                const int64_t pg = table[b * max_pages + p / page_size];
                const uint16_t *k = K_pages + ((pg * page_size + p % page_size) * H + h) * D;
                double dot = 0.0;
                for (int64_t i = 0; i < D; ++i)
                    dot += oracle_f16_to_f64(q[i]) * oracle_f16_to_f64(k[i]);
                s[p] = dot * inv_sqrt_d;
                if (s[p] > M) M = s[p];
            }
            double den = 0.0;
            for (int64_t p = 0; p < L; ++p) {
                s[p] = exp(s[p] - M);
                den += s[p];
            }
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t p = 0; p < L; ++p) {
                const int64_t pg = table[b * max_pages + p / page_size];
                const uint16_t *v = V_pages + ((pg * page_size + p % page_size) * H + h) * D;
                const double w = s[p] / den;
                for (int64_t d = 0; d < D; ++d) o[d] += w * oracle_f16_to_f64(v[d]);
            }
        }
        free(s);
    }
}

/*
 * The QK step in fp64: scores[b,h,p] = (Q[b,h,:] . K[b,p,h,:]) / sqrt(D) for
 * p <= cp_b, exactly -infinity for p > cp_b (kernel attention_qk_f16).  All S
 * positions are produced, like the page's [n_heads, seq_len] scores buffer.
 */
void oracle_qk_f64(const uint16_t *Q, const uint16_t *K, int64_t B, int64_t H,
                   int64_t D, int64_t S, const uint32_t *current_pos,
                   double *scores, int nthreads) {
    set_threads(nthreads);
    const double inv_sqrt_d = 1.0 / sqrt((double)D);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const int64_t b = bh / H, h = bh % H;
        const uint16_t *q = Q + (b * H + h) * D;
        double *row = scores + (b * H + h) * S;
        for (int64_t p = 0; p < S; ++p) {
            if ((uint64_t)p > (uint64_t)current_pos[b]) {
                row[p] = -INFINITY;
                continue;
            }
            const uint16_t *k = K + ((b * S + p) * H + h) * D;
            double dot = 0.0;
            for (int64_t i = 0; i < D; ++i)
                dot += oracle_f16_to_f64(q[i]) * oracle_f16_to_f64(k[i]);
            row[p] = dot * inv_sqrt_d;
        }
    }
}

/*
 * The PV step in fp64 on given f16 scores (kernel attention_pv_f16): softmax
 * over all S scores of a row (masked entries are -infinity and get weight 0),
 * then out[b,h,d] = sum_{p<S} w_p V[b,p,h,d].  As on the page, every position is
 * multiplied in, so a non-finite V at a zero-weight position propagates.
 */
void oracle_pv_f64(const uint16_t *scores, const uint16_t *V, int64_t B,
                   int64_t H, int64_t D, int64_t S, double *out, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel
    {
        double *w = (double *)malloc(sizeof(double) * (size_t)S);
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < B * H; ++bh) {
            const int64_t b = bh / H, h = bh % H;
            const uint16_t *row = scores + (b * H + h) * S;
            double M = -INFINITY;
            for (int64_t p = 0; p < S; ++p) {
                const double s = oracle_f16_to_f64(row[p]);
                if (s > M) M = s;
            }
            double den = 0.0;
            for (int64_t p = 0; p < S; ++p) {
                w[p] = exp(oracle_f16_to_f64(row[p]) - M);
                den += w[p];
            }
            double *o = out + (b * H + h) * D;
            for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t p = 0; p < S; ++p) {
                const uint16_t *v = V + ((b * S + p) * H + h) * D;
                const double wp = w[p] / den;
                for (int64_t d = 0; d < D; ++d) o[d] += wp * oracle_f16_to_f64(v[d]);
            }
        }
        free(w);
    }
}

/*
 * The QK step at the page's own precision, for the split-call cross-check:
 *   scale = 1.0f / sqrt(float(head_dim))                     (fp32)
 *   score = 0.0f; for i in index order: score += float(q_i) * float(k_i)
 *                                      (fp32 multiply, then fp32 add)
 *   score *= scale                                           (fp32)
 *   score = -infinity if pos > current_pos
 *   scores[b,h,pos] = half(score)                            (round to nearest even)
 * Output is binary16 bit patterns [B,H,S].
 */
void oracle_qk_pages_f16(const uint16_t *Q, const uint16_t *K, int64_t B,
                         int64_t H, int64_t D, int64_t S,
                         const uint32_t *current_pos, uint16_t *scores,
                         int nthreads) {
    set_threads(nthreads);
    const float scale = 1.0f / sqrtf((float)D);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < B * H; ++bh) {
        const int64_t b = bh / H, h = bh % H;
        const uint16_t *q = Q + (b * H + h) * D;
        uint16_t *row = scores + (b * H + h) * S;
        for (int64_t p = 0; p < S; ++p) {
            const uint16_t *k = K + ((b * S + p) * H + h) * D;
            float score = 0.0f;
            for (int64_t i = 0; i < D; ++i) {
                volatile float prod = (float)oracle_f16_to_f64(q[i]) *
                                      (float)oracle_f16_to_f64(k[i]);
                score = score + prod;
            }
            score = score * scale;
            if ((uint64_t)p > (uint64_t)current_pos[b]) score = -INFINITY;
            row[p] = oracle_f32_to_f16_rne(score);
        }
    }
}

/*
 * Row softmax over the last dimension, fp64 (the fm_softmax operation of
 * Foundry's docs/metal.md: x [rows, cols] -> out [rows, cols]): per row
 *   out[r, c] = exp(x[r, c] - max_c x[r, c]) / sum_c exp(x[r, c] - max_c x[r, c]).
 * -infinity entries get weight 0; a row that is all -infinity (or holds a NaN)
 * gives NaN, as the definition does.
 */
void oracle_softmax_f64(const float *x, int64_t rows, int64_t cols, double *out,
                        int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * cols;
        double *o = out + r * cols;
        double M = -INFINITY;
        int has_nan = 0;
        for (int64_t c = 0; c < cols; ++c) {
            if (isnan(xr[c])) has_nan = 1;
            if ((double)xr[c] > M) M = (double)xr[c];
        }
        double den = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            o[c] = exp((double)xr[c] - M);
            den += o[c];
        }
        for (int64_t c = 0; c < cols; ++c) o[c] = has_nan ? NAN : o[c] / den;
    }
}

/*
 * Rotary position embedding of one token per sequence, fp64 ("Tutorial 16:
 * Writing Custom Metal Kernels", section 5, FastRoPE: vectors split into pairs,
 * a 2D rotation of each pair by an angle set by the position, the position
 * offset given per batch entry).  For sequence b at position pos_b and pair i
 * (i < rope_dims / 2), theta_i = base^(-2 i / rope_dims) and a = pos_b * theta_i:
 *   non-traditional (default): the pair is (x[i], x[i + rope_dims/2]);
 *   traditional:               the pair is (x[2i], x[2i + 1]);
 *   (u, w) -> (u cos a - w sin a, u sin a + w cos a).
 * Channels from rope_dims on are copied unchanged.
 * x [B, H, D] f16 -> out [B, H, D] fp64.
 */
void oracle_rope_f64(const uint16_t *x, int64_t B, int64_t H, int64_t D, int64_t rope_dims,
                     double base, int traditional, const uint32_t *position, double *out) {
    const int64_t half = rope_dims / 2;
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t h = 0; h < H; ++h) {
            const uint16_t *xv = x + (b * H + h) * D;
            double *o = out + (b * H + h) * D;
            for (int64_t d = 0; d < D; ++d) o[d] = oracle_f16_to_f64(xv[d]);
            for (int64_t i = 0; i < half; ++i) {
                const double theta = pow(base, -2.0 * (double)i / (double)rope_dims);
                const double a = (double)position[b] * theta;
                const int64_t i0 = traditional ? 2 * i : i;
                const int64_t i1 = traditional ? 2 * i + 1 : i + half;
                const double u = oracle_f16_to_f64(xv[i0]), w = oracle_f16_to_f64(xv[i1]);
                o[i0] = u * cos(a) - w * sin(a);
                o[i1] = u * sin(a) + w * cos(a);
            }
        }
    }
}

/* Vectorised helpers for the tests that pin the conversions themselves. */
void oracle_f16_to_f64_array(const uint16_t *in, double *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f64(in[i]);
}

void oracle_f32_to_f16_array(const float *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16_rne(in[i]);
}
