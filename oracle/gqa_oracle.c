/*
 * Reference oracle for the fused GQA decode-attention step -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is a plain, slow, deliberately unoptimised CPU statement of what one decode
 * step computes.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the library under test never calls it and shares no code with it.
 *
 * Arithmetic: IEEE binary64 throughout, over inputs that are bf16 bit patterns widened
 * exactly to double.  The only roundings to bf16 are the ones the operation defines
 * (the rotated q and k rows, which are bf16 tensors like every activation on the path).
 *
 * What is computed, and where it is stated:
 *   - QK RMSNorm then RoPE on the new token, folded into one step
 *     ("Qwen3-14B Optimization", section 2.1 Shape 4 and section 3.3 on folding the
 *      QK-norm reciprocal into RoPE; the lo/hi RoPE halves there fix the half-split
 *      pairing (i, i + d/2)).
 *   - k stored post-RoPE, v stored raw, at the new token's slot before attention reads
 *     the cache ("ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)", section 0.5.1
 *     preconditions P2-P4; "Qwen3-14B Optimization", section 2.1 "Then: buy it": the
 *     paged block-slot-head-dim cache layout).
 *   - Attention: softmax(q K^T / sqrt(d)) V for every query head h against KV head
 *     floor(h / G) (ADR-0060, section 0 reference dimensions and section 3).  The
 *     brute-force form below is the plain definition; the streaming form follows the
 *     per-tile recurrence of ADR-0060 section 3 and the log-sum-exp merge of section 4,
 *     so that the two can be checked against each other.
 *
 *   - The 4-bit KV cache ("Qwen3-14B Optimization", section 2.3): Lloyd-Max codebook
 *     indices packed two per byte, dequantized by gather, renormalize, scale, unrotate.
 *   - Chunked causal prefill: the same per-token prologue for a block of T new tokens,
 *     then causal attention of each of them over the cache (ADR-0060 section 5.4); a
 *     blocked form follows that section's past / partial / future tile classes.
 *
 * Parity pins (the tests that tie this file to the pages and to mathematics, not to
 * itself) live in tests/test_oracle_pins.py, tests/test_oracle_prefill_pins.py and
 * tests/test_oracle_q4_pins.py.
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ bf16 <-> double */

double oracle_bf16_to_double(uint16_t bits) {
    uint32_t w = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even (IEEE 754 roundTiesToEven),
 * in one step from binary64 (no intermediate binary32 rounding).  bf16 carries 8
 * significant bits, so the spacing of representable values at magnitude
 * [2^(e-1), 2^e) is 2^(e-8); below the normal range the spacing stays at 2^-133. */
uint16_t oracle_round_bf16(double z) {
    if (isnan(z)) return (uint16_t)0x7fc0;
    uint16_t sign = signbit(z) ? (uint16_t)0x8000 : (uint16_t)0;
    double a = fabs(z);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7f80);
    int e;
    (void)frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int qexp = e - 8;
    if (qexp < -133) qexp = -133;
    double n = rint(ldexp(a, -qexp));   /* default rounding mode: nearest, ties to even */
    double v = ldexp(n, qexp);
    if (v > 0x1.fep127) return (uint16_t)(sign | 0x7f80);
    float f = (float)v;                 /* exact: v has at most 8 significant bits */
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    return (uint16_t)(sign | (uint16_t)(w >> 16));
}

/* ------------------------------------------------------------------ QK-norm, RoPE */

/* RMSNorm of one head vector: y_i = x_i * r * w_i with r = 1 / sqrt(mean(x^2) + eps).
 * w == NULL means no norm (y = x). */
void oracle_rmsnorm(const double *x, const double *w, int d, double eps, double *y) {
    if (!w) {
        for (int i = 0; i < d; ++i) y[i] = x[i];
        return;
    }
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)d + eps);
    for (int i = 0; i < d; ++i) y[i] = x[i] * r * w[i];
}

/* Rotary embedding at integer position pos, half-split pairing (i, i + d/2):
 *   phi_i = pos * theta^(-2i/d)
 *   z_i       = y_i cos phi_i - y_{i+d/2} sin phi_i
 *   z_{i+d/2} = y_{i+d/2} cos phi_i + y_i sin phi_i                                     */
void oracle_rope(const double *y, int d, long long pos, double theta, double *z) {
    int half = d / 2;
    for (int i = 0; i < half; ++i) {
        double inv_freq = pow(theta, -2.0 * (double)i / (double)d);
        double phi = (double)pos * inv_freq;
        double c = cos(phi), s = sin(phi);
        z[i] = y[i] * c - y[i + half] * s;
        z[i + half] = y[i + half] * c + y[i] * s;
    }
}

/* ------------------------------------------------------------------ cache addressing */

/* Cache row that holds token t of sequence b.
 *   paged (page_table != NULL): [num_blocks, block_size, H_kv, d];
 *       row = page_table[b][t / block_size] * block_size + t % block_size
 *   contiguous (page_table == NULL): [B, max_seq, H_kv, d]; row = b * max_seq + t        */
static long long cache_row(const int32_t *page_table, int max_blocks, int block_size,
                           int max_seq, int b, int t) {
    if (page_table) {
        long long page = page_table[(long long)b * max_blocks + t / block_size];
        return page * block_size + t % block_size;
    }
    return (long long)b * max_seq + t;
}

typedef struct {
    int B, Hq, Hkv, d;
    int block_size;      /* tokens per page when paged */
    int max_seq;         /* per-sequence capacity in tokens */
    long long num_rows;  /* rows in the cache pool (num_blocks * block_size, or B * max_seq) */
} oracle_geom_t;

/* ------------------------------------------------------------------ prologue */

/* One decode step's prologue.  For every sequence b with new-token position p = positions[b]:
 *   q_rot[b, h]          = bf16(RoPE_p(RMSNorm(q_new[b, h], q_norm_w)))
 *   k_cache[slot(b, p)]  = bf16(RoPE_p(RMSNorm(k_new[b, kv], k_norm_w)))
 *   v_cache[slot(b, p)]  = v_new[b, kv]        (bit copy)
 * Returns 0, or a positive code when an index is out of range (nothing is written for
 * that sequence): 1 = position outside [0, seq_len), 2 = seq_len outside [1, max_seq],
 * 3 = page id outside the pool.                                                           */
int oracle_prologue(const oracle_geom_t *g,
                    const uint16_t *q_new, const uint16_t *k_new, const uint16_t *v_new,
                    uint16_t *k_cache, uint16_t *v_cache,
                    const int32_t *page_table, const int32_t *seq_lens, const int32_t *positions,
                    const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                    double rope_theta, double eps, uint16_t *q_rot) {
    const int d = g->d;
    int status = 0;
    int max_blocks = g->block_size > 0 ? (g->max_seq + g->block_size - 1) / g->block_size : 0;
    double *x = malloc(sizeof(double) * d), *y = malloc(sizeof(double) * d);
    double *z = malloc(sizeof(double) * d);
    double *qw = malloc(sizeof(double) * d), *kw = malloc(sizeof(double) * d);
    for (int i = 0; i < d; ++i) {
        qw[i] = q_norm_w ? oracle_bf16_to_double(q_norm_w[i]) : 1.0;
        kw[i] = k_norm_w ? oracle_bf16_to_double(k_norm_w[i]) : 1.0;
    }
    for (int b = 0; b < g->B; ++b) {
        int L = seq_lens[b], p = positions[b];
        if (L < 1 || L > g->max_seq) { status = 2; continue; }
        if (p < 0 || p >= L) { status = 1; continue; }
        long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, p);
        if (row < 0 || row >= g->num_rows) { status = 3; continue; }
        for (int h = 0; h < g->Hq; ++h) {
            const uint16_t *src = q_new + ((long long)b * g->Hq + h) * d;
            for (int i = 0; i < d; ++i) x[i] = oracle_bf16_to_double(src[i]);
            oracle_rmsnorm(x, q_norm_w ? qw : NULL, d, eps, y);
            oracle_rope(y, d, p, rope_theta, z);
            uint16_t *dst = q_rot + ((long long)b * g->Hq + h) * d;
            for (int i = 0; i < d; ++i) dst[i] = oracle_round_bf16(z[i]);
        }
        for (int kv = 0; kv < g->Hkv; ++kv) {
            const uint16_t *src = k_new + ((long long)b * g->Hkv + kv) * d;
            for (int i = 0; i < d; ++i) x[i] = oracle_bf16_to_double(src[i]);
            oracle_rmsnorm(x, k_norm_w ? kw : NULL, d, eps, y);
            oracle_rope(y, d, p, rope_theta, z);
            uint16_t *kdst = k_cache + (row * g->Hkv + kv) * d;
            uint16_t *vdst = v_cache + (row * g->Hkv + kv) * d;
            const uint16_t *vsrc = v_new + ((long long)b * g->Hkv + kv) * d;
            for (int i = 0; i < d; ++i) {
                kdst[i] = oracle_round_bf16(z[i]);
                vdst[i] = vsrc[i];
            }
        }
    }
    free(x); free(y); free(z); free(qw); free(kw);
    return status;
}

/* ------------------------------------------------------------------ attention */

/* Brute-force attention for one (b, h): the full score vector, max-subtracted softmax,
 * weighted sum of V.  out has d doubles.                                                 */
static void attend_one(const oracle_geom_t *g, const uint16_t *q_rot,
                       const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *page_table, int max_blocks, int L, int b, int h,
                       double *scores, double *out) {
    const int d = g->d, G = g->Hq / g->Hkv, kv = h / G;
    const double scale = 1.0 / sqrt((double)d);
    const uint16_t *q = q_rot + ((long long)b * g->Hq + h) * d;
    double m = -INFINITY;
    for (int t = 0; t < L; ++t) {
        long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t);
        const uint16_t *k = k_cache + (row * g->Hkv + kv) * d;
        double s = 0.0;
        for (int i = 0; i < d; ++i) s += oracle_bf16_to_double(q[i]) * oracle_bf16_to_double(k[i]);
        scores[t] = s * scale;
        if (scores[t] > m) m = scores[t];
    }
    double l = 0.0;
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    for (int t = 0; t < L; ++t) {
        double w = exp(scores[t] - m);
        l += w;
        long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t);
        const uint16_t *v = v_cache + (row * g->Hkv + kv) * d;
        for (int i = 0; i < d; ++i) out[i] += w * oracle_bf16_to_double(v[i]);
    }
    for (int i = 0; i < d; ++i) out[i] /= l;
}

/* out[b, h, :] for every (b, h) -- or, when pairs != NULL, for the n_pairs listed
 * (b, h) pairs only, written to out[k, :] in list order.  Returns the thread count used. */
int oracle_attention(const oracle_geom_t *g, const uint16_t *q_rot,
                     const uint16_t *k_cache, const uint16_t *v_cache,
                     const int32_t *page_table, const int32_t *seq_lens,
                     const int32_t *pairs, int n_pairs, double *out) {
    int max_blocks = g->block_size > 0 ? (g->max_seq + g->block_size - 1) / g->block_size : 0;
    long long n = pairs ? n_pairs : (long long)g->B * g->Hq;
    int threads = 1;
#pragma omp parallel
    {
#ifdef _OPENMP
#pragma omp single
        threads = omp_get_num_threads();
#endif
        double *scores = malloc(sizeof(double) * (size_t)(g->max_seq > 0 ? g->max_seq : 1));
#pragma omp for schedule(dynamic, 1)
        for (long long k = 0; k < n; ++k) {
            int b = pairs ? pairs[2 * k] : (int)(k / g->Hq);
            int h = pairs ? pairs[2 * k + 1] : (int)(k % g->Hq);
            attend_one(g, q_rot, k_cache, v_cache, page_table, max_blocks, seq_lens[b], b, h,
                       scores, out + k * g->d);
        }
        free(scores);
    }
    return threads;
}

/* Streaming form for one (b, h), used only to check the brute-force form: the token
 * range [0, L) is cut at split_bounds (n_splits + 1 ascending token indices, first 0,
 * last L; empty splits allowed).  Each split runs the per-tile online-softmax recurrence
 * over tiles of `tile` tokens, seeded m = -inf, l = 0, O = 0:
 *     m' = max(m, max_t s_t);  P_t = exp(s_t - m');  c = exp(m - m')
 *     l  = l * c + sum_t P_t;  O = O * c + sum_t P_t V_t;  m = m'
 * and the splits' unnormalised partials are folded left to right with the log-sum-exp
 * merge  m = max(m_a, m_b); l = l_a e^(m_a - m) + l_b e^(m_b - m);
 *        O = O_a e^(m_a - m) + O_b e^(m_b - m),  then normalised once: out = O / l.
 * A split with no tokens keeps m = -inf, l = 0 and is skipped by the merge.            */
void oracle_attention_streaming(const oracle_geom_t *g, const uint16_t *q_rot,
                                const uint16_t *k_cache, const uint16_t *v_cache,
                                const int32_t *page_table, int L, int b, int h, int tile,
                                const int32_t *split_bounds, int n_splits, double *out) {
    const int d = g->d, G = g->Hq / g->Hkv, kv = h / G;
    const double scale = 1.0 / sqrt((double)d);
    int max_blocks = g->block_size > 0 ? (g->max_seq + g->block_size - 1) / g->block_size : 0;
    const uint16_t *q = q_rot + ((long long)b * g->Hq + h) * d;
    double *O = malloc(sizeof(double) * d), *Oacc = malloc(sizeof(double) * d);
    double *s = malloc(sizeof(double) * (size_t)tile);
    double m_acc = -INFINITY, l_acc = 0.0;
    for (int i = 0; i < d; ++i) Oacc[i] = 0.0;
    for (int sp = 0; sp < n_splits; ++sp) {
        int lo = split_bounds[sp], hi = split_bounds[sp + 1];
        double m = -INFINITY, l = 0.0;
        for (int i = 0; i < d; ++i) O[i] = 0.0;
        for (int t0 = lo; t0 < hi; t0 += tile) {
            int n = hi - t0 < tile ? hi - t0 : tile;
            double mt = -INFINITY;
            for (int j = 0; j < n; ++j) {
                long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t0 + j);
                const uint16_t *k = k_cache + (row * g->Hkv + kv) * d;
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += oracle_bf16_to_double(q[i]) * oracle_bf16_to_double(k[i]);
                s[j] = acc * scale;
                if (s[j] > mt) mt = s[j];
            }
            double m_new = m > mt ? m : mt;
            double c = exp(m - m_new);          /* m = -inf on the first tile: c = 0 */
            l *= c;
            for (int i = 0; i < d; ++i) O[i] *= c;
            for (int j = 0; j < n; ++j) {
                double P = exp(s[j] - m_new);
                l += P;
                long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t0 + j);
                const uint16_t *v = v_cache + (row * g->Hkv + kv) * d;
                for (int i = 0; i < d; ++i) O[i] += P * oracle_bf16_to_double(v[i]);
            }
            m = m_new;
        }
        if (l == 0.0) continue;                 /* empty split */
        if (l_acc == 0.0) {
            m_acc = m; l_acc = l;
            for (int i = 0; i < d; ++i) Oacc[i] = O[i];
            continue;
        }
        double mm = m_acc > m ? m_acc : m;
        double sa = exp(m_acc - mm), sb = exp(m - mm);
        l_acc = l_acc * sa + l * sb;
        for (int i = 0; i < d; ++i) Oacc[i] = Oacc[i] * sa + O[i] * sb;
        m_acc = mm;
    }
    for (int i = 0; i < d; ++i) out[i] = Oacc[i] / l_acc;
    free(O); free(Oacc); free(s);
}

/* ------------------------------------------------------------------ chunked prefill */

/* Chunked causal prefill ("ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)",
 * section 5.4 PREFILL, no SP: the prompt is resident in the cache and the query is a
 * block of T tokens).  Sequence b receives T new tokens at positions s_b .. s_b + T - 1,
 * s_b = q_start[b]; its cache already holds positions [0, s_b).  Token i of the chunk
 * (position p = s_b + i) goes through the same per-token prologue as a decode step:
 *   q_rot[b, i, h]      = bf16(RoPE_p(RMSNorm(q_new[b, i, h])))
 *   k_cache[slot(b, p)] = bf16(RoPE_p(RMSNorm(k_new[b, i, kv])))
 *   v_cache[slot(b, p)] = v_new[b, i, kv]                          (bit copy)
 * Tensors: q_new, q_rot [B, T, H_q, d]; k_new, v_new [B, T, H_kv, d].
 * Returns 0, or a positive code (nothing written for that sequence): 1 = q_start < 0,
 * 2 = s_b + T > max_seq, 3 = a page id outside the pool.                               */
int oracle_prefill_prologue(const oracle_geom_t *g, int T,
                            const uint16_t *q_new, const uint16_t *k_new, const uint16_t *v_new,
                            uint16_t *k_cache, uint16_t *v_cache, const int32_t *page_table,
                            const int32_t *q_start, const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                            double rope_theta, double eps, uint16_t *q_rot) {
    const int d = g->d;
    int status = 0;
    int max_blocks = g->block_size > 0 ? (g->max_seq + g->block_size - 1) / g->block_size : 0;
    double *x = malloc(sizeof(double) * d), *y = malloc(sizeof(double) * d);
    double *z = malloc(sizeof(double) * d);
    double *qw = malloc(sizeof(double) * d), *kw = malloc(sizeof(double) * d);
    for (int i = 0; i < d; ++i) {
        qw[i] = q_norm_w ? oracle_bf16_to_double(q_norm_w[i]) : 1.0;
        kw[i] = k_norm_w ? oracle_bf16_to_double(k_norm_w[i]) : 1.0;
    }
    for (int b = 0; b < g->B; ++b) {
        int s = q_start[b];
        if (s < 0) { status = 1; continue; }
        if ((long long)s + T > g->max_seq) { status = 2; continue; }
        int bad_page = 0;
        for (int i = 0; i < T && !bad_page; ++i) {
            long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, s + i);
            if (row < 0 || row >= g->num_rows) bad_page = 1;
        }
        if (bad_page) { status = 3; continue; }
        for (int i = 0; i < T; ++i) {
            const int p = s + i;
            const long long tok = (long long)b * T + i;
            for (int h = 0; h < g->Hq; ++h) {
                const uint16_t *src = q_new + (tok * g->Hq + h) * d;
                for (int e = 0; e < d; ++e) x[e] = oracle_bf16_to_double(src[e]);
                oracle_rmsnorm(x, q_norm_w ? qw : NULL, d, eps, y);
                oracle_rope(y, d, p, rope_theta, z);
                uint16_t *dst = q_rot + (tok * g->Hq + h) * d;
                for (int e = 0; e < d; ++e) dst[e] = oracle_round_bf16(z[e]);
            }
            long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, p);
            for (int kv = 0; kv < g->Hkv; ++kv) {
                const uint16_t *src = k_new + (tok * g->Hkv + kv) * d;
                for (int e = 0; e < d; ++e) x[e] = oracle_bf16_to_double(src[e]);
                oracle_rmsnorm(x, k_norm_w ? kw : NULL, d, eps, y);
                oracle_rope(y, d, p, rope_theta, z);
                uint16_t *kdst = k_cache + (row * g->Hkv + kv) * d;
                uint16_t *vdst = v_cache + (row * g->Hkv + kv) * d;
                const uint16_t *vsrc = v_new + (tok * g->Hkv + kv) * d;
                for (int e = 0; e < d; ++e) {
                    kdst[e] = oracle_round_bf16(z[e]);
                    vdst[e] = vsrc[e];
                }
            }
        }
    }
    free(x); free(y); free(z); free(qw); free(kw);
    return status;
}

/* Causal attention of the chunk, brute force: for chunk token i of sequence b (position
 * p = q_start[b] + i) and query head h (KV head floor(h / G)),
 *     out[b, i, h] = sum_{t <= p} softmax_t(q_rot[b, i, h] . K_t / sqrt(d)) V_t
 * over the cache after the prologue -- every earlier token and the token itself, none
 * after it (zeros for a sequence whose chunk is out of range).  out is [B, T, H_q, d]; or, when triples != NULL, one d-vector per listed
 * (b, i, h) in list order.  Returns the thread count used.                              */
int oracle_prefill_attention(const oracle_geom_t *g, int T, const uint16_t *q_rot,
                             const uint16_t *k_cache, const uint16_t *v_cache,
                             const int32_t *page_table, const int32_t *q_start,
                             const int32_t *triples, int n_triples, double *out) {
    int max_blocks = g->block_size > 0 ? (g->max_seq + g->block_size - 1) / g->block_size : 0;
    long long n = triples ? n_triples : (long long)g->B * T * g->Hq;
    int threads = 1;
#pragma omp parallel
    {
#ifdef _OPENMP
#pragma omp single
        threads = omp_get_num_threads();
#endif
        double *scores = malloc(sizeof(double) * (size_t)(g->max_seq > 0 ? g->max_seq : 1));
#pragma omp for schedule(dynamic, 1)
        for (long long k = 0; k < n; ++k) {
            int b, i, h;
            if (triples) {
                b = triples[3 * k]; i = triples[3 * k + 1]; h = triples[3 * k + 2];
            } else {
                b = (int)(k / ((long long)T * g->Hq));
                i = (int)((k / g->Hq) % T);
                h = (int)(k % g->Hq);
            }
            double *o = out + k * g->d;
            if (q_start[b] < 0 || (long long)q_start[b] + T > g->max_seq) {  /* chunk out of range */
                for (int e = 0; e < g->d; ++e) o[e] = 0.0;
                continue;
            }
            const int L = q_start[b] + i + 1;
            const int G = g->Hq / g->Hkv, kv = h / G;
            const double scale = 1.0 / sqrt((double)g->d);
            const uint16_t *q = q_rot + (((long long)b * T + i) * g->Hq + h) * g->d;
            double m = -INFINITY;
            for (int t = 0; t < L; ++t) {
                long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t);
                const uint16_t *kr = k_cache + (row * g->Hkv + kv) * g->d;
                double acc = 0.0;
                for (int e = 0; e < g->d; ++e) acc += oracle_bf16_to_double(q[e]) * oracle_bf16_to_double(kr[e]);
                scores[t] = acc * scale;
                if (scores[t] > m) m = scores[t];
            }
            double l = 0.0;
            for (int e = 0; e < g->d; ++e) o[e] = 0.0;
            for (int t = 0; t < L; ++t) {
                double w = exp(scores[t] - m);
                l += w;
                long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t);
                const uint16_t *vr = v_cache + (row * g->Hkv + kv) * g->d;
                for (int e = 0; e < g->d; ++e) o[e] += w * oracle_bf16_to_double(vr[e]);
            }
            for (int e = 0; e < g->d; ++e) o[e] /= l;
        }
        free(scores);
    }
    return threads;
}

/* Blocked form for one (b, h), used only to check the brute-force form: the chunk's
 * queries are cut into blocks of qb tokens and the keys into tiles of kt tokens, and
 * each (query block [qs, qe), key tile [ks, ke)) pair, in absolute positions, is one of
 * the three classes of ADR-0060 section 5.4:
 *     ke <= qs  -> all past:   no mask;
 *     ks >= qe  -> all future: skipped;
 *     otherwise -> partial:    the triangular additive mask (0 where key <= query,
 *                              -inf after it) is added to the tile's scores.
 * Each query row runs the online-softmax recurrence of section 3 over the tiles it does
 * not skip (seeded m = -inf, l = 0, O = 0; a row whose tile is all masked leaves its
 * state unchanged), normalised once at the end.  out is [T, d].                         */
void oracle_prefill_blocked(const oracle_geom_t *g, int T, const uint16_t *q_rot,
                            const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *page_table, const int32_t *q_start, int b, int h,
                            int qb, int kt, double *out) {
    const int d = g->d, G = g->Hq / g->Hkv, kv = h / G;
    const double scale = 1.0 / sqrt((double)d);
    int max_blocks = g->block_size > 0 ? (g->max_seq + g->block_size - 1) / g->block_size : 0;
    const int s0 = q_start[b];
    if (s0 < 0 || (long long)s0 + T > g->max_seq) {  /* chunk out of range: zeros */
        for (long long e = 0; e < (long long)T * d; ++e) out[e] = 0.0;
        return;
    }
    double *S = malloc(sizeof(double) * (size_t)qb * kt);
    double *m = malloc(sizeof(double) * qb), *l = malloc(sizeof(double) * qb);
    for (int i0 = 0; i0 < T; i0 += qb) {
        const int nq = T - i0 < qb ? T - i0 : qb;
        const int qs = s0 + i0, qe = qs + nq;
        for (int r = 0; r < nq; ++r) {
            m[r] = -INFINITY; l[r] = 0.0;
            for (int e = 0; e < d; ++e) out[(long long)(i0 + r) * d + e] = 0.0;
        }
        for (int ks = 0; ks < qe; ks += kt) {      /* tiles with ks >= qe: all future, skipped */
            const int ke = ks + kt;
            const int partial = !(ke <= qs);
            for (int r = 0; r < nq; ++r) {
                const uint16_t *q = q_rot + (((long long)b * T + i0 + r) * g->Hq + h) * d;
                for (int c = 0; c < kt; ++c) {
                    const int t = ks + c;
                    double mask = 0.0;
                    if (partial && t > qs + r) mask = -INFINITY;
                    if (mask == -INFINITY) { S[r * kt + c] = -INFINITY; continue; }
                    long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t);
                    const uint16_t *kr = k_cache + (row * g->Hkv + kv) * d;
                    double acc = 0.0;
                    for (int e = 0; e < d; ++e) acc += oracle_bf16_to_double(q[e]) * oracle_bf16_to_double(kr[e]);
                    S[r * kt + c] = acc * scale + mask;
                }
            }
            for (int r = 0; r < nq; ++r) {
                double mt = -INFINITY;
                for (int c = 0; c < kt; ++c) if (S[r * kt + c] > mt) mt = S[r * kt + c];
                if (mt == -INFINITY) continue;          /* every key of this tile masked */
                const double m_new = m[r] > mt ? m[r] : mt;
                const double corr = exp(m[r] - m_new);  /* 0 on the row's first tile */
                double *o = out + (long long)(i0 + r) * d;
                l[r] *= corr;
                for (int e = 0; e < d; ++e) o[e] *= corr;
                for (int c = 0; c < kt; ++c) {
                    if (S[r * kt + c] == -INFINITY) continue;
                    const double P = exp(S[r * kt + c] - m_new);
                    l[r] += P;
                    long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, ks + c);
                    const uint16_t *vr = v_cache + (row * g->Hkv + kv) * d;
                    for (int e = 0; e < d; ++e) o[e] += P * oracle_bf16_to_double(vr[e]);
                }
                m[r] = m_new;
            }
        }
        for (int r = 0; r < nq; ++r)
            for (int e = 0; e < d; ++e) out[(long long)(i0 + r) * d + e] /= l[r];
    }
    free(S); free(m); free(l);
}

/* ------------------------------------------------------------------ 4-bit KV cache */

/* The quantized KV cache of "Qwen3-14B Optimization", section 2.3 (TurboQuant): each
 * cache row (one token, one KV head, d = 128) is stored as 4-bit Lloyd-Max codebook
 * indices, two per byte -- byte c holds idx[c + 64] * 16 + idx[c] -- and dequantized by
 * gather -> renormalize -> scale -> unrotate.  The pages give neither the codebook, the
 * rotation nor the scale format; the readings here (and in the library):
 *   codebook  the 16 reconstruction levels of the Lloyd-Max quantizer of a standard
 *             normal variable (Lloyd's algorithm; Max 1960), as bf16 values (an input);
 *   rotation  R = H D / sqrt(d): the Sylvester-ordered Walsh-Hadamard matrix times a
 *             diagonal of +-1 signs (an input), orthogonal;
 *   quantize  s = ||x||, t = sqrt(d) R x / s, idx_i = the nearest level to t_i (the lower
 *             index on a tie);
 *   scale     one per row: sigma = s / ||c[idx]||, so that the dequantized row is
 *             x^ = sigma R^T c[idx]  (gather c[idx], renormalize to unit length, scale by
 *             s, unrotate).  A zero row has s = 0 and dequantizes to zero.            */

/* Lloyd's algorithm for the `levels`-level quantizer of N(0,1): thresholds at the
 * midpoints of adjacent levels, each level the conditional mean of its cell,
 *   E[X | a < X < b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a)),
 * iterated from uniformly spaced levels until nothing moves.  Writes levels[levels]
 * (ascending) and thresholds[levels - 1]; returns the iterations used.                 */
static double std_pdf(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
static double std_cdf(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

int oracle_lloyd_max(int levels, double *lv, double *thr) {
    for (int j = 0; j < levels; ++j) lv[j] = -3.0 + 6.0 * (j + 0.5) / levels;
    int it;
    for (it = 0; it < 100000; ++it) {
        for (int j = 0; j + 1 < levels; ++j) thr[j] = 0.5 * (lv[j] + lv[j + 1]);
        double moved = 0.0;
        for (int j = 0; j < levels; ++j) {
            double a = j == 0 ? -INFINITY : thr[j - 1], b = j + 1 == levels ? INFINITY : thr[j];
            double pa = isinf(a) ? 0.0 : std_pdf(a), pb = isinf(b) ? 0.0 : std_pdf(b);
            double mass = (isinf(b) ? 1.0 : std_cdf(b)) - (isinf(a) ? 0.0 : std_cdf(a));
            double c = (pa - pb) / mass;
            moved = fmax(moved, fabs(c - lv[j]));
            lv[j] = c;
        }
        if (moved < 1e-15) break;
    }
    for (int j = 0; j + 1 < levels; ++j) thr[j] = 0.5 * (lv[j] + lv[j + 1]);
    return it;
}

/* y = R x = H (D x) / sqrt(d) and x = R^T y = D H y / sqrt(d), H the Sylvester Hadamard
 * matrix (H[i][j] = (-1)^popcount(i & j)), written out as the plain matrix product.  */
static int popcount_i(int v) { int c = 0; while (v) { c += v & 1; v >>= 1; } return c; }

void oracle_rotate(const double *x, const int8_t *signs, int d, double *y) {
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < d; ++j) acc += ((popcount_i(i & j) & 1) ? -1.0 : 1.0) * signs[j] * x[j];
        y[i] = acc / sqrt((double)d);
    }
}

void oracle_unrotate(const double *y, const int8_t *signs, int d, double *x) {
    for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += ((popcount_i(i & j) & 1) ? -1.0 : 1.0) * y[i];
        x[j] = signs[j] * acc / sqrt((double)d);
    }
}

/* Quantize one row x[d] (d = 128): packed[d / 2] bytes and *sigma.                      */
void oracle_q4_quantize(const double *x, const int8_t *signs, const uint16_t *codebook_bf16, int d,
                        uint8_t *packed, double *sigma) {
    double c[16], y[256];
    int idx[256];
    for (int j = 0; j < 16; ++j) c[j] = oracle_bf16_to_double(codebook_bf16[j]);
    double s = 0.0;
    for (int i = 0; i < d; ++i) s += x[i] * x[i];
    s = sqrt(s);
    oracle_rotate(x, signs, d, y);
    double cn = 0.0;
    for (int i = 0; i < d; ++i) {
        double t = s > 0.0 ? sqrt((double)d) * y[i] / s : 0.0;
        int best = 0;
        for (int j = 1; j < 16; ++j)
            if (fabs(t - c[j]) < fabs(t - c[best])) best = j;
        idx[i] = best;
        cn += c[best] * c[best];
    }
    for (int b = 0; b < d / 2; ++b) packed[b] = (uint8_t)(idx[b + d / 2] * 16 + idx[b]);
    *sigma = s > 0.0 ? s / sqrt(cn) : 0.0;
}

/* The dequantized row x^ = sigma R^T c[idx] of a packed row.                            */
void oracle_q4_dequantize(const uint8_t *packed, double sigma, const int8_t *signs,
                          const uint16_t *codebook_bf16, int d, double *x) {
    double y[256];
    for (int i = 0; i < d; ++i) {
        int idx = i < d / 2 ? packed[i] % 16 : packed[i - d / 2] / 16;
        y[i] = sigma * oracle_bf16_to_double(codebook_bf16[idx]);
    }
    oracle_unrotate(y, signs, d, x);
}

/* Attention over a 4-bit cache, brute force per (b, h): scores q_rot[b, h] . x^_t / sqrt(d)
 * over the dequantized rows x^_t = sigma_t R^T c[idx_t], t < seq_lens[b], then the softmax
 * weights applied to the dequantized value rows.  Sequences with ok[b] == 0 (or ok NULL
 * meaning all valid) give zeros.  out [B, H_q, d], or the listed (b, h) pairs in order. */
void oracle_q4_attention(const oracle_geom_t *g, const uint16_t *q_rot, const uint8_t *k_idx, const uint8_t *v_idx,
                         const float *k_scale, const float *v_scale, const int32_t *page_table,
                         const int32_t *seq_lens, const int *ok, const int8_t *signs, const uint16_t *codebook,
                         const int32_t *pairs, int n_pairs, double *out) {
    const int d = g->d, half = d / 2;
    int max_blocks = g->block_size > 0 ? (g->max_seq + g->block_size - 1) / g->block_size : 0;
    long long n = pairs ? n_pairs : (long long)g->B * g->Hq;
#pragma omp parallel
    {
        double *kr = malloc(sizeof(double) * d), *vr = malloc(sizeof(double) * d);
        double *sc = malloc(sizeof(double) * (size_t)(g->max_seq > 0 ? g->max_seq : 1));
#pragma omp for schedule(dynamic, 1)
        for (long long k = 0; k < n; ++k) {
            int b = pairs ? pairs[2 * k] : (int)(k / g->Hq), h = pairs ? pairs[2 * k + 1] : (int)(k % g->Hq);
            double *o = out + k * d;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            if (ok && !ok[b]) continue;
            const int G = g->Hq / g->Hkv, kv = h / G, L = seq_lens[b];
            const uint16_t *q = q_rot + ((long long)b * g->Hq + h) * d;
            double m = -INFINITY;
            for (int t = 0; t < L; ++t) {
                long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t);
                oracle_q4_dequantize(k_idx + (row * g->Hkv + kv) * half, (double)k_scale[row * g->Hkv + kv], signs,
                                     codebook, d, kr);
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += oracle_bf16_to_double(q[i]) * kr[i];
                sc[t] = acc / sqrt((double)d);
                if (sc[t] > m) m = sc[t];
            }
            double l = 0.0;
            for (int t = 0; t < L; ++t) {
                long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, t);
                oracle_q4_dequantize(v_idx + (row * g->Hkv + kv) * half, (double)v_scale[row * g->Hkv + kv], signs,
                                     codebook, d, vr);
                double w = exp(sc[t] - m);
                l += w;
                for (int i = 0; i < d; ++i) o[i] += w * vr[i];
            }
            for (int i = 0; i < d; ++i) o[i] /= l;
        }
        free(kr); free(vr); free(sc);
    }
}

/* One decode step over a 4-bit cache.  As oracle_prologue + oracle_attention, except that
 * the new token's k row (the exact RoPE(RMSNorm(k_new)) value) and v row (v_new) are
 * quantized into k_idx/v_idx [rows, H_kv, d/2] and k_scale/v_scale [rows, H_kv] (fp32),
 * and attention reads the dequantized rows x^ of the cache.  Brute force per (b, h); out
 * [B, H_q, d] (or the listed (b, h) pairs).  Returns the status of the prologue.        */
int oracle_q4_decode_step(const oracle_geom_t *g,
                          const uint16_t *q_new, const uint16_t *k_new, const uint16_t *v_new,
                          uint8_t *k_idx, uint8_t *v_idx, float *k_scale, float *v_scale,
                          const int32_t *page_table, const int32_t *seq_lens, const int32_t *positions,
                          const uint16_t *q_norm_w, const uint16_t *k_norm_w, double rope_theta, double eps,
                          const int8_t *signs, const uint16_t *codebook,
                          const int32_t *pairs, int n_pairs, uint16_t *q_rot, double *out) {
    const int d = g->d, half = d / 2;
    int status = 0;
    int max_blocks = g->block_size > 0 ? (g->max_seq + g->block_size - 1) / g->block_size : 0;
    double *x = malloc(sizeof(double) * d), *y = malloc(sizeof(double) * d), *z = malloc(sizeof(double) * d);
    double *qw = malloc(sizeof(double) * d), *kw = malloc(sizeof(double) * d);
    for (int i = 0; i < d; ++i) {
        qw[i] = q_norm_w ? oracle_bf16_to_double(q_norm_w[i]) : 1.0;
        kw[i] = k_norm_w ? oracle_bf16_to_double(k_norm_w[i]) : 1.0;
    }
    int *ok = calloc((size_t)g->B, sizeof(int));
    for (int b = 0; b < g->B; ++b) {
        int L = seq_lens[b], p = positions[b];
        if (L < 1 || L > g->max_seq) { status = 2; continue; }
        if (p < 0 || p >= L) { status = 1; continue; }
        long long row = cache_row(page_table, max_blocks, g->block_size, g->max_seq, b, p);
        if (row < 0 || row >= g->num_rows) { status = 3; continue; }
        ok[b] = 1;
        for (int h = 0; h < g->Hq; ++h) {
            const uint16_t *src = q_new + ((long long)b * g->Hq + h) * d;
            for (int i = 0; i < d; ++i) x[i] = oracle_bf16_to_double(src[i]);
            oracle_rmsnorm(x, q_norm_w ? qw : NULL, d, eps, y);
            oracle_rope(y, d, p, rope_theta, z);
            for (int i = 0; i < d; ++i) q_rot[((long long)b * g->Hq + h) * d + i] = oracle_round_bf16(z[i]);
        }
        for (int kv = 0; kv < g->Hkv; ++kv) {
            const uint16_t *src = k_new + ((long long)b * g->Hkv + kv) * d;
            for (int i = 0; i < d; ++i) x[i] = oracle_bf16_to_double(src[i]);
            oracle_rmsnorm(x, k_norm_w ? kw : NULL, d, eps, y);
            oracle_rope(y, d, p, rope_theta, z);
            double sg;
            oracle_q4_quantize(z, signs, codebook, d, k_idx + (row * g->Hkv + kv) * half, &sg);
            k_scale[row * g->Hkv + kv] = (float)sg;
            const uint16_t *vs = v_new + ((long long)b * g->Hkv + kv) * d;
            for (int i = 0; i < d; ++i) x[i] = oracle_bf16_to_double(vs[i]);
            oracle_q4_quantize(x, signs, codebook, d, v_idx + (row * g->Hkv + kv) * half, &sg);
            v_scale[row * g->Hkv + kv] = (float)sg;
        }
    }
    oracle_q4_attention(g, q_rot, k_idx, v_idx, k_scale, v_scale, page_table, seq_lens, ok, signs, codebook,
                        pairs, n_pairs, out);
    free(x); free(y); free(z); free(qw); free(kw); free(ok);
    return status;
}

/* ------------------------------------------------------------------ threads */

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
