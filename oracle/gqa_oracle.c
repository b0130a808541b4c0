/*
 * gqa_oracle.c -- fp64 CPU oracle for causal grouped-query attention with RoPE.
 *
 * TEST INFRASTRUCTURE.  This file exists to check the CUDA path.  Only the test
 * suite, the package smoke check and the benchmark's CPU-baseline leg load it; the
 * product path never calls it.  It shares no source, header, table or helper with the
 * CUDA library, and it includes nothing from it.
 *
 * Every function is the plain definition written out in double precision, in the order
 * the pages give it: frequencies -> rotation -> scores -> mask -> softmax -> weighted
 * sum.  No tiling, no online softmax, no fusion.  Rotating every key once before the
 * scores is the definition itself (the scores use the rotated K').
 *
 * Sources, by page and section:
 *   [PL3] imoz.jp, "PLaMo 3アーキテクチャ徹底解析":
 *         §4.2  GQA: consecutive query heads share one KV head, g(h) = floor(h / G);
 *         §4.4  the cache holds K before RoPE; K positions 0..S-1 and Q positions
 *               S-T..S-1 are generated inside attention; the local cache keeps the last
 *               W-1 tokens and re-numbers positions from 0;
 *         §4.5  A = softmax_s(Q'K'^T * scale + M), O = A V; no softcap, no dropout;
 *         §5.1  causal: key j visible from query i iff j <= i; local window also needs
 *               i - j < W (self plus the previous W-1 tokens);
 *         §6.1  split-half pairs (j, j + d/2), omega_j = theta^(-2j/d);
 *         §6.3  YaRN: boundaries j_low/j_high (not rounded), alpha_j = clip(...),
 *               omega~_j = omega_j [(1 - alpha_j) + alpha_j / s]; amplitude 1 + 0.1 ln s
 *               multiplies both cos and sin;
 *         §6.4  p-RoPE: pairs at or above the rotated fraction get frequency 0 (identity),
 *               the exponent's denominator stays the full head dimension;
 *         §3.2, §4.3  RMSNorm with an effective gain (offset + weight), per head for
 *               q_norm / k_norm (offset 1, eps 1e-6); V is not normalised.
 *         §5.2, §8  Gemma 4's global layers share one projection for K and V
 *               (attention_k_eq_v): with Z its output, K = RoPE(N_{gamma_k}(Z)) and
 *               V = N_1(Z), the gain-free RMSNorm.
 *   [LLA] disassemble-channel.com LLaMA tutorial, GQA section: g(i) = floor(i n_kv / h),
 *         the same grouping written with the KV-head count.
 *
 * Planted-mistake builds: compiling with -DORC_PLANT=<n> injects one deliberate error
 * (see orc_plant below).  The test suite builds such variants to show that its pins
 * catch each kind of mistake.  The default build plants nothing.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORC_PLANT
#define ORC_PLANT 0
#endif

#define ORC_PI 3.14159265358979323846

int orc_plant(void) { return ORC_PLANT; }

/* bfloat16 bits -> value: the top 16 bits of an IEEE binary32. */
static double bf16_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double orc_bf16_to_double(uint16_t h) { return bf16_to_f64(h); }

/* [PL3 §6.3] amplitude correction applied to both cos and sin. */
double orc_yarn_amp(double s) { return 1.0 + 0.1 * log(s); }

/* [PL3 §6.3] interpolation boundary for one beta: (d/2) ln(L0 / (2 pi beta)) / ln(base).
 * For d = 128 the page writes the factor d/2 as 64. */
double orc_yarn_boundary(int d, double base, double L0, double beta) {
    return (d / 2.0) * log(L0 / (2.0 * ORC_PI * beta)) / log(base);
}

/* Per-pair angular frequencies omega_j, j = 0 .. d/2-1.
 *   [PL3 §6.1] omega_j = base^(-2j/d)
 *   [PL3 §6.3] if yarn_s != 1: omega_j *= (1 - alpha_j) + alpha_j / yarn_s
 *   [PL3 §6.4] if rotate_fraction < 1: omega_j = 0 for j >= rotate_fraction * d/2
 * Returns 0, or -1 on a bad argument. */
int orc_inv_freq(double *w, int d, double base, double yarn_s, double L0,
                 double beta_fast, double beta_slow, double rotate_fraction) {
    if (!w || d <= 0 || (d % 2) != 0 || !(base > 1.0) || !(yarn_s >= 1.0) ||
        !(rotate_fraction > 0.0 && rotate_fraction <= 1.0))
        return -1;
    const int half = d / 2;
    const int yarn = (yarn_s != 1.0);
    double jl = 0.0, jh = 1.0;
    if (yarn) {
        jl = orc_yarn_boundary(d, base, L0, beta_fast);
        jh = orc_yarn_boundary(d, base, L0, beta_slow);
    }
    int n_rot = half;
    if (rotate_fraction < 1.0) n_rot = (int)floor(rotate_fraction * half + 0.5);
    for (int j = 0; j < half; ++j) {
#if ORC_PLANT == 5
        double om = pow(base, -2.0 * j / half);      /* planted: wrong exponent denominator */
#else
        double om = pow(base, -2.0 * j / d);
#endif
        if (yarn) {
            double a = (j - jl) / (jh - jl);
            if (a < 0.0) a = 0.0;
            if (a > 1.0) a = 1.0;
#if ORC_PLANT == 6
            om = om * (a + (1.0 - a) / yarn_s);      /* planted: interpolation reversed */
#else
            om = om * ((1.0 - a) + a / yarn_s);
#endif
        }
        if (j >= n_rot) om = 0.0;
        w[j] = om;
    }
    return 0;
}

/* [PL3 §6.1, §6.3] rotate one head vector in place at position pos:
 *   a' = a c - b s,  b' = a s + b c,  (a, b) = (x_j, x_{j+d/2}),
 *   c = amp cos(pos omega_j), s = amp sin(pos omega_j). */
void orc_rope_rotate(double *x, int d, double pos, const double *w, double amp) {
    const int half = d / 2;
    for (int j = 0; j < half; ++j) {
        const double ang = pos * w[j];
        const double c = amp * cos(ang), s = amp * sin(ang);
        const double a = x[j], b = x[j + half];
#if ORC_PLANT == 1
        x[j] = a * c + b * s;                         /* planted: sign flip */
        x[j + half] = -a * s + b * c;
#else
        x[j] = a * c - b * s;
        x[j + half] = a * s + b * c;
#endif
    }
}

/* [PL3 §3.2, §4.3] RMSNorm of `rows` vectors of n values (bf16 bits), in double:
 *   N(x) = gamma (*) x / sqrt((1/n) sum_r x_r^2 + eps)
 * gamma is the effective gain, offset plus stored weight (q_norm and k_norm: offset 1,
 * n = head dim, eps = 1e-6, one gain shared by every head); gamma == NULL means no gain
 * (all ones, the gain-free norm Gemma 4 puts on V).  No mean is subtracted. */
void orc_rms_norm(const uint16_t *x, long rows, int n, const double *gamma, double eps,
                  double *out) {
    for (long i = 0; i < rows; ++i) {
        const uint16_t *xr = x + (size_t)i * n;
        double ss = 0.0;
        for (int r = 0; r < n; ++r) {
            const double v = bf16_to_f64(xr[r]);
            ss += v * v;
        }
#if ORC_PLANT == 8
        const double inv = 1.0 / sqrt(ss + eps);       /* planted: sum, not mean */
#else
        const double inv = 1.0 / sqrt(ss / n + eps);
#endif
        for (int r = 0; r < n; ++r)
            out[(size_t)i * n + r] = (gamma ? gamma[r] : 1.0) * bf16_to_f64(xr[r]) * inv;
    }
}

/* [PL3 §5.1] may the query at position qpos see the key at kpos? window <= 0: causal. */
static int orc_allowed(long qpos, long kpos, int window) {
    if (kpos > qpos) return 0;
#if ORC_PLANT == 2
    if (window > 0 && qpos - kpos > window) return 0; /* planted: window one too wide */
#else
    if (window > 0 && qpos - kpos >= window) return 0;
#endif
    return 1;
}

int orc_allowed_pub(long qpos, long kpos, int window) { return orc_allowed(qpos, kpos, window); }

/* [PL3 §4.2, §4.5] KV head of query head h: consecutive groups of G = Hq/Hkv heads. */
static int orc_kv_head(int h, int Hq, int Hkv) {
#if ORC_PLANT == 3
    return h % Hkv;                                   /* planted: interleaved groups */
#else
    return h / (Hq / Hkv);
#endif
}

int orc_kv_head_pub(int h, int Hq, int Hkv) { return orc_kv_head(h, Hq, Hkv); }

/* [PL3 §4.5, §5.1] one query row: scores of the rotated query qr against the rotated
 * keys Kr [S, d], the mask, the softmax over the visible keys and the weighted sum of
 * V [S, d].  z [S] and ok [S] are scratch; lse and wrow (the weights, [S]) are nullable. */
static void orc_attend_row(const double *qr, const double *Kr, const double *Vd, long S,
                           int d, long qpos, int window, double scale, double *z, char *ok,
                           double *orow, double *lse, double *wrow) {
    double m = -INFINITY;
    for (long s = 0; s < S; ++s) {
        ok[s] = (char)orc_allowed(qpos, s, window);
        if (!ok[s]) { z[s] = -INFINITY; continue; }
        const double *kr = Kr + (size_t)s * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += qr[c] * kr[c];
#if ORC_PLANT == 4
        z[s] = acc;                   /* planted: scale dropped */
#else
        z[s] = acc * scale;
#endif
        if (z[s] > m) m = z[s];
    }
    double l = 0.0;
    for (long s = 0; s < S; ++s) l += ok[s] ? exp(z[s] - m) : 0.0;
    for (int c = 0; c < d; ++c) orow[c] = 0.0;
    for (long s = 0; s < S; ++s) {
        if (!ok[s]) continue;
        const double a = exp(z[s] - m) / l;
        const double *vr = Vd + (size_t)s * d;
        for (int c = 0; c < d; ++c) orow[c] += a * vr[c];
    }
    if (lse) *lse = m + log(l);
    if (wrow)
        for (long s = 0; s < S; ++s) wrow[s] = ok[s] ? exp(z[s] - m) / l : 0.0;
}

/* The (b, h, t) of requested row r: from the rows array, or row-major (b, h, t) order. */
static void orc_row_coords(const int32_t *rows, long r, int Hq, int T, int *b, int *h, int *t) {
    if (rows) { *b = rows[3 * r]; *h = rows[3 * r + 1]; *t = rows[3 * r + 2]; }
    else { *b = (int)(r / ((long)Hq * T)); *h = (int)((r / T) % Hq); *t = (int)(r % T); }
}

/* How a layer turns its stored inputs into Q, K' and V (fp64), one vector at a time.
 *   plain  : Q, K, V as given (bf16 bits), K and Q then rotated ([PL3 §4.4]);
 *   shared : Gemma 4's global layers (attention_k_eq_v, [PL3 §8] and [PL3 §5.2]): one
 *            projection output Z per KV head gives both K = RoPE(N_{gamma_k}(Z)) and
 *            V = N_1(Z) (RMSNorm without a gain); the query is N_{gamma_q}(q), rotated. */
typedef struct {
    int shared;
    const double *q_gamma, *k_gamma;   /* shared only (NULL = gain 1) */
    double eps;
} orc_inputs;

static void orc_load_q(const orc_inputs *in, const uint16_t *src, int d, double *out) {
    if (in->shared) orc_rms_norm(src, 1, d, in->q_gamma, in->eps, out);
    else for (int c = 0; c < d; ++c) out[c] = bf16_to_f64(src[c]);
}

/* key s: kr = K (not yet rotated), vr = V, from the stored rows ks and vs */
static void orc_load_kv(const orc_inputs *in, const uint16_t *ks, const uint16_t *vs, int d,
                        double *kr, double *vr) {
    if (in->shared) {
        orc_rms_norm(ks, 1, d, in->k_gamma, in->eps, kr);
#if ORC_PLANT == 9
        orc_rms_norm(ks, 1, d, in->k_gamma, in->eps, vr);   /* planted: V keeps K's gain */
#else
        orc_rms_norm(ks, 1, d, NULL, in->eps, vr);
#endif
    } else {
        for (int r = 0; r < d; ++r) {
            kr[r] = bf16_to_f64(ks[r]);
            vr[r] = bf16_to_f64(vs[r]);
        }
    }
}

static int orc_attention_impl(const orc_inputs *in, const uint16_t *q, const uint16_t *k,
                              const uint16_t *v, int B, int T, int S, int Hq, int Hkv, int d,
                              int window, double scale, const double *w, double amp,
                              long pos_shift, const int32_t *rows, long nrows, double *o,
                              double *lse, double *weights, int nthreads) {
    if (!q || !k || !v || !w || !o || B <= 0 || T <= 0 || S <= 0 || T > S || Hq <= 0 ||
        Hkv <= 0 || (Hq % Hkv) != 0 || d <= 0 || (d % 2) != 0)
        return -1;
    const long total = rows ? nrows : (long)B * Hq * T;
    if (total <= 0) return 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    double *Kr = (double *)malloc(sizeof(double) * (size_t)S * d);
    double *Vd = (double *)malloc(sizeof(double) * (size_t)S * d);
    long *sel = (long *)malloc(sizeof(long) * (size_t)total);
    if (!Kr || !Vd || !sel) { free(Kr); free(Vd); free(sel); return -2; }

    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < Hkv; ++g) {
            /* the requested rows whose query head reads KV head g of batch b */
            long nsel = 0;
            for (long r = 0; r < total; ++r) {
                int rb, rh, rt;
                orc_row_coords(rows, r, Hq, T, &rb, &rh, &rt);
                if (rb == b && orc_kv_head(rh, Hq, Hkv) == g) sel[nsel++] = r;
            }
            if (nsel == 0) continue;
            const uint16_t *kb = k + ((size_t)b * Hkv + g) * (size_t)S * d;
            const uint16_t *vb = v + ((size_t)b * Hkv + g) * (size_t)S * d;
            /* K' = RoPE(K) at positions 0..S-1 ([PL3 §4.4]); V as the layer defines it. */
#pragma omp parallel for schedule(static)
            for (long s = 0; s < S; ++s) {
                double *kr = Kr + (size_t)s * d;
                orc_load_kv(in, kb + (size_t)s * d, vb + (size_t)s * d, d, kr,
                            Vd + (size_t)s * d);
                orc_rope_rotate(kr, d, (double)(s + pos_shift), w, amp);
            }
#pragma omp parallel
            {
                double *qr = (double *)malloc(sizeof(double) * (size_t)d);
                double *z = (double *)malloc(sizeof(double) * (size_t)S);
                char *ok = (char *)malloc((size_t)S);
#pragma omp for schedule(dynamic, 4)
                for (long i = 0; i < nsel; ++i) {
                    if (!qr || !z || !ok) continue;
                    const long r = sel[i];
                    int rb, rh, rt;
                    orc_row_coords(rows, r, Hq, T, &rb, &rh, &rt);
                    const long qpos = (long)(S - T) + rt;
                    orc_load_q(in, q + (((size_t)b * Hq + rh) * T + rt) * (size_t)d, d, qr);
                    orc_rope_rotate(qr, d, (double)(qpos + pos_shift), w, amp);
                    orc_attend_row(qr, Kr, Vd, S, d, qpos, window, scale, z, ok,
                                   o + (size_t)r * d, lse ? lse + r : NULL,
                                   weights ? weights + (size_t)r * S : NULL);
                }
                free(qr); free(z); free(ok);
            }
        }
    }
    free(Kr); free(Vd); free(sel);
    return 0;
}

/* Attention rows, fp64.
 *   q : [B, Hq, T, d] bf16 bits     k, v : [B, Hkv, S, d] bf16 bits (k before RoPE)
 *   Query t has position S - T + t, key s has position s ([PL3 §4.4]); pos_shift is
 *   added to every position before the rotation (the mask uses the differences only).
 *   rows : nrows triples (b, h, t), or NULL for all B*Hq*T rows in (b, h, t) order.
 *   o    : [nrows, d] outputs; lse: [nrows] natural-log sum of exp of the scaled
 *          scores (nullable); weights: [nrows, S] attention weights (nullable).
 * Returns 0, or -1 on a bad argument, -2 on allocation failure. */
int orc_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  int B, int T, int S, int Hq, int Hkv, int d, int window, double scale,
                  const double *w, double amp, long pos_shift,
                  const int32_t *rows, long nrows,
                  double *o, double *lse, double *weights, int nthreads) {
    const orc_inputs in = {0, NULL, NULL, 0.0};
    return orc_attention_impl(&in, q, k, v, B, T, S, Hq, Hkv, d, window, scale, w, amp,
                              pos_shift, rows, nrows, o, lse, weights, nthreads);
}

/* Attention of a layer whose K and V share one projection (Gemma 4 global layers,
 * attention_k_eq_v, [PL3 §5.2 and §8]), fp64:
 *   q : [B, Hq, T, d] bf16 bits, the query projection before its norm;
 *   z : [B, Hkv, S, d] bf16 bits, the shared projection output Z;
 *   Q' = RoPE(N_{q_gamma}(q)), K' = RoPE(N_{k_gamma}(Z)), V = N_1(Z) with
 *   N_gamma(x) = gamma (*) x / sqrt(mean(x^2) + eps) ([PL3 §3.2]; NULL gamma = gain 1).
 * Positions, mask, rows and outputs as orc_attention (pos_shift 0). */
int orc_attention_kv_shared(const uint16_t *q, const uint16_t *z, const double *q_gamma,
                            const double *k_gamma, double eps, int B, int T, int S, int Hq,
                            int Hkv, int d, int window, double scale, const double *w,
                            double amp, const int32_t *rows, long nrows, double *o,
                            double *lse, int nthreads) {
    const orc_inputs in = {1, q_gamma, k_gamma, eps};
    return orc_attention_impl(&in, q, z, z, B, T, S, Hq, Hkv, d, window, scale, w, amp, 0,
                              rows, nrows, o, lse, NULL, nthreads);
}

/* ---- cache index model ([PL3 §4.4]) ----------------------------------------------
 * Linear (global-layer) cache: `count` = tokens held; the new token goes to slot count
 *   (-1 if the cache is full); afterwards keys 0..count are the logical keys, at
 *   positions equal to their slots.
 * Ring (local-layer) cache of capacity cap = W: `count` = tokens ever appended; token
 *   number i lives in slot i mod cap; after the append the newest min(count+1, cap)
 *   tokens are retained (the W-1 kept plus the new one) and are re-numbered 0..R-1 in
 *   age order, the query taking position R-1. */
long orc_append_slot(int is_ring, long count_before, long cap) {
    if (cap <= 0 || count_before < 0) return -1;
    if (is_ring) return count_before % cap;
    return count_before < cap ? count_before : -1;
}

long orc_retained(int is_ring, long count_after, long cap) {
    if (is_ring) return count_after < cap ? count_after : cap;
    return count_after;
}

long orc_logical_slot(int is_ring, long count_after, long cap, long t) {
    if (!is_ring) return t;
    const long R = orc_retained(1, count_after, cap);
#if ORC_PLANT == 7
    return (count_after - R + t + 1) % cap;           /* planted: ring off by one */
#else
    return (count_after - R + t) % cap;
#endif
}

/* Gathers the R logical keys of sequence i after the append, in age order, from its
 * cache rows and the new row (placed where its slot appears): out [Hkv, R, d]. */
static void orc_gather_logical(const uint16_t *cache, const uint16_t *new_row, long cap,
                               int is_ring, long slot, long after, long R, int Hkv, int d,
                               uint16_t *out) {
    for (int g = 0; g < Hkv; ++g) {
        for (long t = 0; t < R; ++t) {
            const long sl = orc_logical_slot(is_ring, after, cap, t);
            const uint16_t *src = (sl == slot) ? new_row + (size_t)g * d
                                               : cache + ((size_t)g * cap + sl) * d;
            memcpy(out + ((size_t)g * R + t) * d, src, sizeof(uint16_t) * d);
        }
    }
}

static int orc_decode_impl(const orc_inputs *in, const uint16_t *q, const uint16_t *k_new,
                           const uint16_t *v_new, const uint16_t *const *k_cache,
                           const uint16_t *const *v_cache, const int64_t *cap,
                           const int64_t *count_before, const int32_t *is_ring,
                           const double *const *w, const double *amp, int nseq, int Hq,
                           int Hkv, int d, double scale, double *o, double *lse,
                           int64_t *slot_out, int64_t *count_out, int nthreads) {
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !cap || !count_before ||
        !is_ring || !w || !amp || !o || nseq <= 0 || Hq <= 0 || Hkv <= 0 ||
        (Hq % Hkv) != 0 || d <= 0)
        return -1;
    for (int i = 0; i < nseq; ++i) {
        const long c = cap[i];
        const long slot = orc_append_slot(is_ring[i], count_before[i], c);
        if (slot < 0) return -1;
        const long after = count_before[i] + 1;
        const long R = orc_retained(is_ring[i], after, c);
        uint16_t *kg = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)Hkv * R * d);
        uint16_t *vg = in->shared ? kg
                                  : (uint16_t *)malloc(sizeof(uint16_t) * (size_t)Hkv * R * d);
        if (!kg || !vg) { free(kg); if (vg != kg) free(vg); return -2; }
        orc_gather_logical(k_cache[i], k_new + (size_t)i * Hkv * d, c, is_ring[i], slot,
                           after, R, Hkv, d, kg);
        if (!in->shared)
            orc_gather_logical(v_cache[i], v_new + (size_t)i * Hkv * d, c, is_ring[i], slot,
                               after, R, Hkv, d, vg);
        const int window = is_ring[i] ? (int)c : 0;
        int rc = orc_attention_impl(in, q + (size_t)i * Hq * d, kg, vg, 1, 1, (int)R, Hq, Hkv,
                                    d, window, scale, w[i], amp[i], 0, NULL, 0,
                                    o + (size_t)i * Hq * d, lse ? lse + (size_t)i * Hq : NULL,
                                    NULL, nthreads);
        if (vg != kg) free(vg);
        free(kg);
        if (rc != 0) return rc;
        if (slot_out) slot_out[i] = slot;
        if (count_out) count_out[i] = after;
    }
    return 0;
}

/* One decode step over a batch: append each sequence's new K/V, then attend with its
 * one query over the logical keys.  Caches are read, never written: the appended token
 * is taken from k_new/v_new where its slot appears.
 *   q       : [nseq, Hq, d]        k_new, v_new : [nseq, Hkv, d]
 *   k_cache, v_cache : per sequence [Hkv, cap, d]  (slots as stored)
 *   w, amp  : per sequence frequencies [d/2] and amplitude
 *   o : [nseq, Hq, d], lse : [nseq, Hq] (nullable), slot_out / count_out (nullable).
 * Returns 0, -1 on a bad argument or a full linear cache, -2 on allocation failure. */
int orc_decode_step(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                    const uint16_t *const *k_cache, const uint16_t *const *v_cache,
                    const int64_t *cap, const int64_t *count_before, const int32_t *is_ring,
                    const double *const *w, const double *amp,
                    int nseq, int Hq, int Hkv, int d, double scale,
                    double *o, double *lse, int64_t *slot_out, int64_t *count_out,
                    int nthreads) {
    const orc_inputs in = {0, NULL, NULL, 0.0};
    return orc_decode_impl(&in, q, k_new, v_new, k_cache, v_cache, cap, count_before, is_ring,
                           w, amp, nseq, Hq, Hkv, d, scale, o, lse, slot_out, count_out,
                           nthreads);
}

/* One decode step of a layer whose K and V share one projection (attention_k_eq_v,
 * [PL3 §5.2 and §8]): the cache of sequence i holds the projection outputs Z of its past
 * tokens ([Hkv, cap, d], slots as stored), z_new [nseq, Hkv, d] the new token's, q
 * [nseq, Hq, d] its query before the norm.  Appends as orc_decode_step, then attends with
 * Q' = RoPE(N_{q_gamma}(q)), K' = RoPE(N_{k_gamma}(Z)), V = N_1(Z) over the logical keys. */
int orc_decode_step_kv_shared(const uint16_t *q, const uint16_t *z_new,
                              const uint16_t *const *z_cache, const int64_t *cap,
                              const int64_t *count_before, const int32_t *is_ring,
                              const double *const *w, const double *amp,
                              const double *q_gamma, const double *k_gamma, double eps,
                              int nseq, int Hq, int Hkv, int d, double scale, double *o,
                              double *lse, int64_t *slot_out, int64_t *count_out,
                              int nthreads) {
    const orc_inputs in = {1, q_gamma, k_gamma, eps};
    return orc_decode_impl(&in, q, z_new, z_new, z_cache, z_cache, cap, count_before, is_ring,
                           w, amp, nseq, Hq, Hkv, d, scale, o, lse, slot_out, count_out,
                           nthreads);
}
