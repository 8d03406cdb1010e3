/*
 * attn_oracle.c -- plain, slow, obviously correct CPU attention (TEST INFRASTRUCTURE).
 *
 * This file is the oracle the GPU path is checked against.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never does.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (attention.fkc.md, "attention_naive"): for every
 * (batch b, query head h, query row qi), with kv head g = h / (Hq / Hkv)
 * (the GQA broadcast of the page header), the full score row over all Sk keys
 * is materialised in float64:
 *
 *   s_j = scale * sum_d Q[b,h,qi,d] * K[b,g,j,d]
 *   s_j = c * tanh(s_j / c)                 if a softcap c is given
 *   s_j = s_j + slope[h] * (j - i)          if ALiBi slopes are given
 *   s_j = -inf                              if position j is not admissible
 *
 * where i = qpos0 + qi is the query row's position among the keys: qpos0 = 0
 * is the top-left alignment of position_admissible (row qi at position qi);
 * a decode row, the newest token of its sequence, sits at qpos0 = Sk - 1
 * ("gfx942 unified attention", section 4: bottom-right alignment, under which
 * a single non-causal query row is the causal one).
 *
 * admissible (attention.fkc.md, header: position_admissible):
 *   not (causal and j > i), not (left window and j + left < i),
 *   not (right window and j > i + right); plus an optional per-row inclusive
 *   key range [lo, hi] (row_bounds, [B, Sq, 2], indexed by the row qi) -- the
 *   reading used for rows "given a window that masks all keys".
 *
 * Then the stable softmax of section 2 of "gfx942 unified attention, from the
 * math up": M = max_j s_j, w_j = exp(s_j - M), L = sum_j w_j,
 * O[d] = sum_j w_j V[b,g,j,d] / L, lse = M + ln L.  A row with no finite score
 * is the all-zero row with lse = -inf (attention_naive, fully-masked rows).
 *
 * Inputs are read exactly as stored (bf16, f16 and f32 widen exactly to f64); scale,
 * slopes and softcap are the fp32 numbers the GPU receives, widened.
 *
 * A second entry, oracle_attn_tiled, walks the same problem the way
 * "attention_flash" and section 3 of "gfx942 unified attention" describe: query
 * tiles of BR rows, key tiles of BC columns, running max m, running
 * denominator l and running output o, rescaled by exp(m_old - m_new) at each
 * tile and divided by l at the end.  It exists only so the tests can check the
 * materialised oracle against the streaming recurrence.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 0, OR_F32 = 1, OR_F64 = 2, OR_F16 = 3 };

/* IEEE 754 binary16: sign, 5-bit exponent with bias 15, 10-bit fraction;
 * exponent 0 holds zeros and subnormals (2^-14 * f / 1024), exponent 31
 * infinities and NaNs.  Every value is exact in double. */
static double half_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)f, e - 25);
    return sign ? -v : v;
}

static double widen(int dtype, const void *base, int64_t i) {
    if (dtype == OR_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (dtype == OR_F16) return half_to_double(((const uint16_t *)base)[i]);
    if (dtype == OR_F32) return (double)((const float *)base)[i];
    return ((const double *)base)[i];
}

typedef struct {
    int dtype;
    const void *q, *k, *v;
    const float *slopes;
    const int32_t *row_bounds;
    int B, Hq, Hkv, Sq, Sk, D;
    double scale;
    int causal;
    long wl, wr;
    double softcap;
    long qpos0; /* position of query row 0 */
} problem;

/* position_admissible plus the optional per-row range. */
static int admissible(const problem *p, int b, int qi, int kj) {
    const long i = p->qpos0 + qi;
    if (p->causal && (long)kj > i) return 0;
    if (p->wl >= 0 && (long)kj + p->wl < i) return 0;
    if (p->wr >= 0 && (long)kj > i + p->wr) return 0;
    if (p->row_bounds) {
        const int32_t *rb = p->row_bounds + 2 * ((int64_t)b * p->Sq + qi);
        if (kj < rb[0] || kj > rb[1]) return 0;
    }
    return 1;
}

/* The score of (b, h, qi, kj) before masking: scale, then softcap, then ALiBi. */
static double score(const problem *p, int b, int h, int qi, int kj) {
    int g = h / (p->Hq / p->Hkv);
    int64_t qoff = (((int64_t)b * p->Hq + h) * p->Sq + qi) * p->D;
    int64_t koff = (((int64_t)b * p->Hkv + g) * p->Sk + kj) * p->D;
    double dot = 0.0;
    for (int d = 0; d < p->D; ++d)
        dot += widen(p->dtype, p->q, qoff + d) * widen(p->dtype, p->k, koff + d);
    double s = p->scale * dot;
    if (p->softcap > 0.0) s = p->softcap * tanh(s / p->softcap);
    if (p->slopes) s += (double)p->slopes[h] * (double)((long)kj - (p->qpos0 + qi));
    return s;
}

/* One materialised row: out[0..D), *lse. */
static void naive_row(const problem *p, int b, int h, int qi, double *srow, double *out, double *lse) {
    int g = h / (p->Hq / p->Hkv);
    double M = -INFINITY;
    for (int kj = 0; kj < p->Sk; ++kj) {
        srow[kj] = admissible(p, b, qi, kj) ? score(p, b, h, qi, kj) : -INFINITY;
        if (srow[kj] > M) M = srow[kj];
    }
    for (int d = 0; d < p->D; ++d) out[d] = 0.0;
    if (M == -INFINITY) {
        if (lse) *lse = -INFINITY;
        return;
    }
    double L = 0.0;
    for (int kj = 0; kj < p->Sk; ++kj) {
        if (srow[kj] == -INFINITY) continue;
        double w = exp(srow[kj] - M);
        L += w;
        int64_t voff = (((int64_t)b * p->Hkv + g) * p->Sk + kj) * p->D;
        for (int d = 0; d < p->D; ++d) out[d] += w * widen(p->dtype, p->v, voff + d);
    }
    for (int d = 0; d < p->D; ++d) out[d] /= L;
    if (lse) *lse = M + log(L);
}

static int check(const problem *p) {
    if (p->B <= 0 || p->Hq <= 0 || p->Hkv <= 0 || p->Sq <= 0 || p->Sk <= 0 || p->D <= 0) return -1;
    if (p->Hq % p->Hkv != 0) return -1;
    if (p->dtype < OR_BF16 || p->dtype > OR_F16) return -1;
    return 0;
}

/*
 * Materialised oracle.  rows == NULL computes every (b, h, qi) and writes
 * out[((b*Hq + h)*Sq + qi)*D + d]; otherwise it computes only the nrows flat
 * row indices rows[i] = (b*Hq + h)*Sq + qi and writes out[i*D + d].
 * lse (nullable) follows the same indexing without the D factor.  Query row
 * qi sits at position qpos0 + qi.
 */
int oracle_attn_rows(int dtype, const void *q, const void *k, const void *v,
                     const float *slopes, const int32_t *row_bounds,
                     int B, int Hq, int Hkv, int Sq, int Sk, int D,
                     double scale, int causal, long wl, long wr, double softcap,
                     long qpos0, const int64_t *rows, int64_t nrows, double *out, double *lse,
                     int nthreads) {
    problem p = {dtype, q, k, v, slopes, row_bounds, B, Hq, Hkv, Sq, Sk, D,
                 scale, causal, wl, wr, softcap, qpos0};
    if (check(&p)) return -1;
    int64_t total = rows ? nrows : (int64_t)B * Hq * Sq;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)Sk);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
        for (int64_t i = 0; i < total; ++i) {
            int64_t r = rows ? rows[i] : i;
            int qi = (int)(r % Sq);
            int h = (int)((r / Sq) % Hq);
            int b = (int)(r / ((int64_t)Sq * Hq));
            naive_row(&p, b, h, qi, srow, out + i * D, lse ? lse + i : NULL);
        }
        free(srow);
    }
    (void)nthreads;
    return 0;
}

/*
 * Tiled online-softmax oracle (attention_flash; section 3 of "gfx942 unified
 * attention").  Same arguments and output layout as the full-problem form of
 * oracle_attn_rows; BR query rows by BC keys per tile.
 */
int oracle_attn_tiled(int dtype, const void *q, const void *k, const void *v,
                      const float *slopes, const int32_t *row_bounds,
                      int B, int Hq, int Hkv, int Sq, int Sk, int D,
                      double scale, int causal, long wl, long wr, double softcap,
                      int BR, int BC, double *out, double *lse, int nthreads) {
    problem p = {dtype, q, k, v, slopes, row_bounds, B, Hq, Hkv, Sq, Sk, D,
                 scale, causal, wl, wr, softcap, 0};
    if (check(&p) || BR <= 0 || BC <= 0) return -1;
    int nqt = (Sq + BR - 1) / BR;
    int64_t units = (int64_t)B * Hq * nqt;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double *m = (double *)malloc(sizeof(double) * (size_t)BR);
        double *l = (double *)malloc(sizeof(double) * (size_t)BR);
        double *o = (double *)malloc(sizeof(double) * (size_t)BR * D);
        double *s = (double *)malloc(sizeof(double) * (size_t)BR * BC);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (int64_t u = 0; u < units; ++u) {
            int t = (int)(u % nqt);
            int h = (int)((u / nqt) % Hq);
            int b = (int)(u / ((int64_t)nqt * Hq));
            int g = h / (Hq / Hkv);
            int q0 = t * BR, nr = Sq - q0 < BR ? Sq - q0 : BR;
            for (int r = 0; r < nr; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.0;
                for (int d = 0; d < D; ++d) o[(size_t)r * D + d] = 0.0;
            }
            for (int k0 = 0; k0 < Sk; k0 += BC) {
                int nc = Sk - k0 < BC ? Sk - k0 : BC;
                for (int r = 0; r < nr; ++r) {
                    int qi = q0 + r;
                    double tile_max = -INFINITY;
                    for (int c = 0; c < nc; ++c) {
                        int kj = k0 + c;
                        double sc = admissible(&p, b, qi, kj) ? score(&p, b, h, qi, kj) : -INFINITY;
                        s[(size_t)r * BC + c] = sc;
                        if (sc > tile_max) tile_max = sc;
                    }
                    double m_new = m[r] > tile_max ? m[r] : tile_max;
                    if (m_new == -INFINITY) continue; /* nothing admissible yet */
                    double alpha = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
                    l[r] *= alpha;
                    for (int d = 0; d < D; ++d) o[(size_t)r * D + d] *= alpha;
                    for (int c = 0; c < nc; ++c) {
                        double sc = s[(size_t)r * BC + c];
                        if (sc == -INFINITY) continue;
                        double w = exp(sc - m_new);
                        l[r] += w;
                        int64_t voff = (((int64_t)b * Hkv + g) * Sk + k0 + c) * D;
                        for (int d = 0; d < D; ++d) o[(size_t)r * D + d] += w * widen(dtype, v, voff + d);
                    }
                    m[r] = m_new;
                }
            }
            for (int r = 0; r < nr; ++r) {
                int64_t row = ((int64_t)b * Hq + h) * Sq + q0 + r;
                for (int d = 0; d < D; ++d)
                    out[row * D + d] = l[r] > 0.0 ? o[(size_t)r * D + d] / l[r] : 0.0;
                if (lse) lse[row] = l[r] > 0.0 ? m[r] + log(l[r]) : -INFINITY;
            }
        }
        free(m);
        free(l);
        free(o);
        free(s);
    }
    (void)nthreads;
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
