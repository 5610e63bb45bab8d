/*
 * EntmaxKV oracle (fp64, plain C + OpenMP over heads).  TEST INFRASTRUCTURE
 * ONLY: see oracle.h for the method source, layouts and the readings taken
 * where the page is silent.  Every step below is the obvious loop; nothing is
 * blocked, fused or reordered beyond the definitions it cites.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <float.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

double oracle_widen(const void* base, int dtype, int64_t idx) {
    if (dtype == 0) return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* small helpers                                                             */
/* ------------------------------------------------------------------------ */

static int pages_of(const oracle_kv* kv, int b) {
    int n = kv->seq_lens[b];
    return (n + kv->page_size - 1) / kv->page_size;
}

static int valid_tokens(const oracle_kv* kv, int b, int p) {
    int rest = kv->seq_lens[b] - p * kv->page_size;
    return rest < kv->page_size ? rest : kv->page_size;
}

/* flat offset of element (block, kv head, token, coordinate) */
static int64_t kv_index(const oracle_kv* kv, int blk, int h, int t, int j) {
    return (((int64_t)blk * kv->num_kv_heads + h) * kv->page_size + t) * kv->head_dim + j;
}

static int64_t meta_index(const oracle_kv* kv, int blk, int h, int j) {
    return ((int64_t)blk * kv->num_kv_heads + h) * kv->head_dim + j;
}

static int head_at(const int32_t* heads, int i) { return heads ? heads[i] : i; }

static int head_count(const oracle_kv* kv, int num_q_heads, const int32_t* heads, int n_heads) {
    return heads ? n_heads : kv->batch * num_q_heads;
}

typedef struct { double v; int idx; } keyed;

/* descending value, then ascending index */
static int cmp_desc_then_idx(const void* a, const void* b) {
    const keyed* x = (const keyed*)a;
    const keyed* y = (const keyed*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

static int cmp_int(const void* a, const void* b) {
    int x = *(const int*)a, y = *(const int*)b;
    return (x > y) - (x < y);
}

static int cmp_double_desc(const void* a, const void* b) {
    double x = *(const double*)a, y = *(const double*)b;
    return (x < y) - (x > y);
}

/* ------------------------------------------------------------------------ */
/* [EntmaxKV §2.A] per-page metadata                                          */
/* ------------------------------------------------------------------------ */

int oracle_build_meta(const oracle_kv* kv, double* kmin, double* kmax,
                      double* mean, double* var) {
    if (!kv || kv->page_size <= 0 || kv->head_dim <= 0) return ORACLE_BAD_ARG;
    for (int b = 0; b < kv->batch; ++b) {
        int np = pages_of(kv, b);
#pragma omp parallel for schedule(static)
        for (int p = 0; p < np; ++p) {
            int blk = kv->page_table[(int64_t)b * kv->max_pages + p];
            int n = valid_tokens(kv, b, p);
            for (int h = 0; h < kv->num_kv_heads; ++h) {
                for (int j = 0; j < kv->head_dim; ++j) {
                    double lo = INFINITY, hi = -INFINITY, sum = 0.0;
                    for (int t = 0; t < n; ++t) {
                        double x = oracle_widen(kv->k_pool, kv->dtype, kv_index(kv, blk, h, t, j));
                        if (x < lo) lo = x;
                        if (x > hi) hi = x;
                        sum += x;
                    }
                    double mu = sum / n;
                    double ss = 0.0;  /* second pass: population variance */
                    for (int t = 0; t < n; ++t) {
                        double x = oracle_widen(kv->k_pool, kv->dtype, kv_index(kv, blk, h, t, j));
                        ss += (x - mu) * (x - mu);
                    }
                    int64_t o = meta_index(kv, blk, h, j);
                    if (kmin) kmin[o] = lo;
                    if (kmax) kmax[o] = hi;
                    if (mean) mean[o] = mu;
                    if (var) var[o] = ss / n;
                }
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* [EntmaxKV §2.A] bounding-box page bound                                   */
/* ------------------------------------------------------------------------ */

int oracle_score_bbox(const oracle_kv* kv, const float* q, int num_q_heads,
                      double scale, const double* kmin, const double* kmax,
                      const int32_t* heads, int n_heads, double* bound) {
    if (num_q_heads % kv->num_kv_heads) return ORACLE_BAD_ARG;
    int G = num_q_heads / kv->num_kv_heads;
    int nh = head_count(kv, num_q_heads, heads, n_heads);
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < nh; ++i) {
        int bh = head_at(heads, i);
        int b = bh / num_q_heads, h = bh % num_q_heads, kvh = h / G;
        const float* qv = q + (int64_t)bh * kv->head_dim;
        int np = pages_of(kv, b);
        for (int p = 0; p < np; ++p) {
            int blk = kv->page_table[(int64_t)b * kv->max_pages + p];
            double acc = 0.0;
            for (int j = 0; j < kv->head_dim; ++j) {
                int64_t o = meta_index(kv, blk, kvh, j);
                double a = (double)qv[j] * kmin[o];
                double c = (double)qv[j] * kmax[o];
                acc += a > c ? a : c;
            }
            bound[(int64_t)bh * kv->max_pages + p] = scale * acc;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* [EntmaxKV §2.B.1] top-k pages                                             */
/* ------------------------------------------------------------------------ */

int oracle_select_topk(const oracle_kv* kv, int num_q_heads, const double* bound,
                       int kp, const int32_t* heads, int n_heads,
                       int32_t* sel, int32_t* n_sel, double* kth, double* next) {
    if (kp < 0) return ORACLE_BAD_ARG;
    int nh = head_count(kv, num_q_heads, heads, n_heads);
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < nh; ++i) {
        int bh = head_at(heads, i);
        int b = bh / num_q_heads;
        int np = pages_of(kv, b);
        keyed* order = (keyed*)malloc(sizeof(keyed) * (np > 0 ? np : 1));
        for (int p = 0; p < np; ++p) {
            order[p].v = bound[(int64_t)bh * kv->max_pages + p];
            order[p].idx = p;
        }
        qsort(order, np, sizeof(keyed), cmp_desc_then_idx);
        int k = kp < np ? kp : np;
        int* chosen = (int*)malloc(sizeof(int) * (k > 0 ? k : 1));
        for (int r = 0; r < k; ++r) chosen[r] = order[r].idx;
        qsort(chosen, k, sizeof(int), cmp_int);
        for (int r = 0; r < k; ++r) sel[(int64_t)bh * kp + r] = chosen[r];
        n_sel[bh] = k;
        if (kth) kth[bh] = k > 0 ? order[k - 1].v : INFINITY;
        if (next) next[bh] = k < np ? order[k].v : -INFINITY;
        free(chosen);
        free(order);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* [EntmaxKV §2.A] Gaussian page statistics                                  */
/* ------------------------------------------------------------------------ */

int oracle_score_gauss(const oracle_kv* kv, const float* q, int num_q_heads,
                       double scale, const double* mean, const double* var,
                       const int32_t* heads, int n_heads, double* m, double* s) {
    if (num_q_heads % kv->num_kv_heads) return ORACLE_BAD_ARG;
    int G = num_q_heads / kv->num_kv_heads;
    int nh = head_count(kv, num_q_heads, heads, n_heads);
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < nh; ++i) {
        int bh = head_at(heads, i);
        int b = bh / num_q_heads, h = bh % num_q_heads, kvh = h / G;
        const float* qv = q + (int64_t)bh * kv->head_dim;
        int np = pages_of(kv, b);
        for (int p = 0; p < np; ++p) {
            int blk = kv->page_table[(int64_t)b * kv->max_pages + p];
            double mu = 0.0, v2 = 0.0;
            for (int j = 0; j < kv->head_dim; ++j) {
                int64_t o = meta_index(kv, blk, kvh, j);
                double qj = (double)qv[j];
                mu += qj * mean[o];
                v2 += qj * qj * var[o];
            }
            m[(int64_t)bh * kv->max_pages + p] = scale * mu;
            s[(int64_t)bh * kv->max_pages + p] = scale * sqrt(v2);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* [EntmaxKV §2.B.2] Gaussian-aware tau-hat selection                        */
/* ------------------------------------------------------------------------ */

/* E[(Y - tau)_+^e] for Y ~ N(mu, sigma^2), e = 2 (alpha = 1.5) or 1 (alpha = 2),
 * from the Gaussian partial moments with u = (mu - tau) / sigma:
 *   e = 2:  ((mu - tau)^2 + sigma^2) Phi(u) + (mu - tau) sigma phi(u)
 *   e = 1:  (mu - tau) Phi(u) + sigma phi(u)
 * sigma = 0 degenerates to (mu - tau)_+^e. */
static double gauss_partial_moment(double mu, double sigma, double tau, int e) {
    double a = mu - tau;
    if (!(sigma > 0.0)) {
        if (a <= 0.0) return 0.0;
        return e == 2 ? a * a : a;
    }
    double u = a / sigma;
    double Phi = 0.5 * erfc(-u / sqrt(2.0));
    double phi = exp(-0.5 * u * u) / sqrt(2.0 * M_PI);
    if (e == 2) return (a * a + sigma * sigma) * Phi + a * sigma * phi;
    return a * Phi + sigma * phi;
}

static int gauss_exponent(double alpha) {
    if (fabs(alpha - 1.5) < 1e-12) return 2;
    if (fabs(alpha - 2.0) < 1e-12) return 1;
    return 0;
}

double oracle_gauss_F(const double* m, const double* s, const int32_t* n, int np,
                      double alpha, double tau) {
    int e = gauss_exponent(alpha);
    if (!e) return NAN;
    double c = alpha - 1.0, acc = 0.0;
    for (int p = 0; p < np; ++p)
        acc += (double)n[p] * gauss_partial_moment(c * m[p], c * s[p], tau, e);
    return acc - 1.0;
}

static double estimated_max(double m, double s, int n) {
    /* reading: the expected-maximum scale of n Gaussian draws */
    return n > 1 ? m + sqrt(2.0 * log((double)n)) * s : m;
}

int oracle_select_gauss(const oracle_kv* kv, int num_q_heads, const double* m,
                        const double* s, double alpha, double delta, int cap,
                        const int32_t* heads, int n_heads, int32_t* sel,
                        int32_t* n_sel, double* tau_hat, double* zmax) {
    if (!gauss_exponent(alpha) || cap <= 0) return ORACLE_BAD_ARG;
    int nh = head_count(kv, num_q_heads, heads, n_heads);
    double c = alpha - 1.0;
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < nh; ++i) {
        int bh = head_at(heads, i);
        int b = bh / num_q_heads;
        int np = pages_of(kv, b);
        const double* mh = m + (int64_t)bh * kv->max_pages;
        const double* sh = s + (int64_t)bh * kv->max_pages;
        int32_t* cnt = (int32_t*)malloc(sizeof(int32_t) * np);
        keyed* est = (keyed*)malloc(sizeof(keyed) * np);
        double mu_max = -INFINITY, top = -INFINITY;
        for (int p = 0; p < np; ++p) {
            cnt[p] = valid_tokens(kv, b, p);
            est[p].v = estimated_max(mh[p], sh[p], cnt[p]);
            est[p].idx = p;
            if (zmax) zmax[(int64_t)bh * kv->max_pages + p] = est[p].v;
            if (c * mh[p] > mu_max) mu_max = c * mh[p];
            double t = c * mh[p] + 8.0 * c * sh[p];
            if (t > top) top = t;
        }
        /* F(mu_max - 1) >= 0 by Jensen (e >= 1); grow hi until F(hi) < 0. */
        double lo = mu_max - 1.0, hi = top + 1.0;
        while (oracle_gauss_F(mh, sh, cnt, np, alpha, hi) >= 0.0) hi += 2.0 * (hi - lo);
        for (int it = 0; it < 200; ++it) {
            double mid = 0.5 * (lo + hi);
            if (oracle_gauss_F(mh, sh, cnt, np, alpha, mid) >= 0.0) lo = mid; else hi = mid;
            double scale_t = fabs(mid) > 1.0 ? fabs(mid) : 1.0;
            if (hi - lo < 1e-14 * scale_t) break;
        }
        double th = 0.5 * (lo + hi);
        tau_hat[bh] = th;

        /* keep iff (alpha-1) zmax >= tau_hat - delta */
        qsort(est, np, sizeof(keyed), cmp_desc_then_idx);
        int pass = 0;
        for (int r = 0; r < np; ++r)
            if (c * est[r].v >= th - delta) ++pass;
        int k = pass;
        if (k > cap) k = cap;           /* cap by estimated-max rank */
        if (k == 0 && np > 0) k = 1;    /* at least the argmax page  */
        int* chosen = (int*)malloc(sizeof(int) * (k > 0 ? k : 1));
        for (int r = 0; r < k; ++r) chosen[r] = est[r].idx;
        qsort(chosen, k, sizeof(int), cmp_int);
        for (int r = 0; r < k; ++r) sel[(int64_t)bh * cap + r] = chosen[r];
        n_sel[bh] = k;
        free(chosen);
        free(est);
        free(cnt);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* alpha-entmax threshold (Peters, Niculae and Martins 2019)                 */
/* ------------------------------------------------------------------------ */

int oracle_entmax_tau(const double* zp, int n, double alpha, double* tau) {
    if (n <= 0) { *tau = INFINITY; return 0; }
    if (!(alpha > 1.0)) { *tau = NAN; return -1; }
    double* x = (double*)malloc(sizeof(double) * n);
    memcpy(x, zp, sizeof(double) * n);
    qsort(x, n, sizeof(double), cmp_double_desc);
    double top = x[0];
    for (int i = 0; i < n; ++i) x[i] -= top;   /* shift: x[0] = 0 */
    double t = NAN;
    int e = gauss_exponent(alpha);
    if (e == 1) {
        /* sparsemax: tau_k = (sum_{i<=k} x_(i) - 1) / k,
         * k* = max{k : x_(k) > tau_k} */
        double run = 0.0;
        int kstar = 1;
        double tk = -1.0;
        for (int k = 1; k <= n; ++k) {
            run += x[k - 1];
            double cand = (run - 1.0) / k;
            if (x[k - 1] > cand) { kstar = k; tk = cand; }
        }
        (void)kstar;
        t = tk;
    } else if (e == 2) {
        /* 1.5-entmax: on the top-k set, sum (x - tau)^2 = 1 gives
         * tau_k = M_k - sqrt((1 - ss_k) / k), M_k the mean and ss_k the
         * centred sum of squares; k* = max{k : 1 - ss_k >= 0, tau_k <= x_(k)} */
        double M = 0.0, ss = 0.0, tk = -1.0;
        for (int k = 1; k <= n; ++k) {
            double xv = x[k - 1];
            double d0 = xv - M;
            M += d0 / k;
            ss += d0 * (xv - M);
            if (ss <= 1.0) {
                double cand = M - sqrt((1.0 - ss) / k);
                if (cand <= xv) tk = cand;
            }
        }
        t = tk;
    } else {
        /* general alpha: bisection on f(tau) = sum (x - tau)_+^e - 1, which is
         * >= 0 at max - 1 and <= 0 at max - n^(1 - alpha) */
        double ex = 1.0 / (alpha - 1.0);
        double lo = -1.0, hi = -pow((double)n, 1.0 - alpha);
        for (int it = 0; it < 200 && hi - lo > 1e-16; ++it) {
            double mid = 0.5 * (lo + hi), f = -1.0;
            for (int i = 0; i < n; ++i)
                if (x[i] > mid) f += pow(x[i] - mid, ex);
            if (f >= 0.0) lo = mid; else hi = mid;
        }
        t = 0.5 * (lo + hi);
    }
    int support = 0;
    for (int i = 0; i < n; ++i) if (x[i] > t) ++support;
    *tau = t + top;
    free(x);
    return support;
}

int oracle_entmax_probs(const double* zp, int n, double alpha, double* p) {
    double tau;
    int k = oracle_entmax_tau(zp, n, alpha, &tau);
    double ex = 1.0 / (alpha - 1.0);
    for (int i = 0; i < n; ++i) {
        double a = zp[i] - tau;
        p[i] = a > 0.0 ? (ex == 1.0 ? a : (ex == 2.0 ? a * a : pow(a, ex))) : 0.0;
    }
    return k;
}

/* ------------------------------------------------------------------------ */
/* [EntmaxKV §2.C] sparse and full-cache alpha-entmax attention              */
/* ------------------------------------------------------------------------ */

/* z'_t = (alpha-1) * s * q.k_t for one token of block blk, kv head kvh */
static double shifted_score(const oracle_kv* kv, const float* qv, double scale,
                            double alpha, int blk, int kvh, int t) {
    double acc = 0.0;
    for (int j = 0; j < kv->head_dim; ++j)
        acc += (double)qv[j] * oracle_widen(kv->k_pool, kv->dtype, kv_index(kv, blk, kvh, t, j));
    return (alpha - 1.0) * (scale * acc);
}

static double weight(double zp, double tau, double alpha) {
    double a = zp - tau;
    if (!(a > 0.0)) return 0.0;
    double ex = 1.0 / (alpha - 1.0);
    if (ex == 1.0) return a;
    if (ex == 2.0) return a * a;
    return pow(a, ex);
}

int oracle_decode_sparse(const oracle_kv* kv, const float* q, int num_q_heads,
                         double scale, double alpha, const int32_t* sel,
                         const int32_t* n_sel, int cap, const int32_t* heads,
                         int n_heads, double* out, double* tau, int32_t* support,
                         double* psum) {
    if (num_q_heads % kv->num_kv_heads || !(alpha > 1.0)) return ORACLE_BAD_ARG;
    int G = num_q_heads / kv->num_kv_heads;
    int d = kv->head_dim, P = kv->page_size;
    int nh = head_count(kv, num_q_heads, heads, n_heads);
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(|:bad)
    for (int i = 0; i < nh; ++i) {
        int bh = head_at(heads, i);
        int b = bh / num_q_heads, h = bh % num_q_heads, kvh = h / G;
        const float* qv = q + (int64_t)bh * d;
        int np = pages_of(kv, b);
        int ns = n_sel[bh];
        double* zp = (double*)malloc(sizeof(double) * ((int64_t)(ns > 0 ? ns : 1) * P));
        int* tok_blk = (int*)malloc(sizeof(int) * ((int64_t)(ns > 0 ? ns : 1) * P));
        int* tok_t = (int*)malloc(sizeof(int) * ((int64_t)(ns > 0 ? ns : 1) * P));
        int n = 0;
        for (int r = 0; r < ns; ++r) {
            int p = sel[(int64_t)bh * cap + r];
            if (p < 0 || p >= np) { bad = 1; continue; }
            int blk = kv->page_table[(int64_t)b * kv->max_pages + p];
            int nt = valid_tokens(kv, b, p);
            for (int t = 0; t < nt; ++t) {
                zp[n] = shifted_score(kv, qv, scale, alpha, blk, kvh, t);
                tok_blk[n] = blk;
                tok_t[n] = t;
                ++n;
            }
        }
        double* o = out + (int64_t)bh * d;
        for (int j = 0; j < d; ++j) o[j] = 0.0;
        double t_ = INFINITY, ps = 0.0;
        int k = 0;
        if (n > 0) {
            k = oracle_entmax_tau(zp, n, alpha, &t_);
            for (int r = 0; r < n; ++r) {
                double w = weight(zp[r], t_, alpha);
                if (w == 0.0) continue;
                ps += w;
                for (int j = 0; j < d; ++j)
                    o[j] += w * oracle_widen(kv->v_pool, kv->dtype, kv_index(kv, tok_blk[r], kvh, tok_t[r], j));
            }
        }
        if (tau) tau[bh] = t_;
        if (support) support[bh] = k;
        if (psum) psum[bh] = ps;
        free(zp);
        free(tok_blk);
        free(tok_t);
    }
    return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* Softmax attention, the comparison method of [EntmaxKV] §1 and §4 (a softmax
 * whose dense tail is truncated to the kept pages).  Scores z = scale q.k over
 * the valid tokens of the selected pages, or of the whole sequence when full
 * is set; m = max z, out = sum_i e^(z_i - m) v_i / sum_i e^(z_i - m) and
 * lse = m + log sum_i e^(z_i - m).  With full set and a selection given,
 * outside = the full softmax's mass on tokens not in the kept pages. */
int oracle_decode_softmax(const oracle_kv* kv, const float* q, int num_q_heads,
                          double scale, const int32_t* sel, const int32_t* n_sel,
                          int cap, int full, const int32_t* heads, int n_heads,
                          double* out, double* lse, double* outside) {
    if (num_q_heads % kv->num_kv_heads || (!full && !sel)) return ORACLE_BAD_ARG;
    int G = num_q_heads / kv->num_kv_heads;
    int d = kv->head_dim;
    int nh = head_count(kv, num_q_heads, heads, n_heads);
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(|:bad)
    for (int i = 0; i < nh; ++i) {
        int bh = head_at(heads, i);
        int b = bh / num_q_heads, h = bh % num_q_heads, kvh = h / G;
        const float* qv = q + (int64_t)bh * d;
        int np = pages_of(kv, b);
        char* kept = (char*)calloc(np > 0 ? np : 1, 1);
        if (sel)
            for (int r = 0; r < n_sel[bh]; ++r) {
                int p = sel[(int64_t)bh * cap + r];
                if (p < 0 || p >= np) { bad = 1; continue; }
                kept[p] = 1;
            }
        /* every token attended to (all pages when full, else the kept ones) */
        int n = 0;
        for (int p = 0; p < np; ++p)
            if (full || kept[p]) n += valid_tokens(kv, b, p);
        double* z = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
        int* tb = (int*)malloc(sizeof(int) * (n > 0 ? n : 1));
        int* tt = (int*)malloc(sizeof(int) * (n > 0 ? n : 1));
        char* in = (char*)malloc(n > 0 ? n : 1);
        int k = 0;
        for (int p = 0; p < np; ++p) {
            if (!full && !kept[p]) continue;
            int blk = kv->page_table[(int64_t)b * kv->max_pages + p];
            for (int t = 0; t < valid_tokens(kv, b, p); ++t) {
                z[k] = shifted_score(kv, qv, scale, 2.0, blk, kvh, t);   /* (2-1) scale q.k */
                tb[k] = blk;
                tt[k] = t;
                in[k] = kept[p];
                ++k;
            }
        }
        double* o = out + (int64_t)bh * d;
        for (int j = 0; j < d; ++j) o[j] = 0.0;
        double m = -INFINITY, l = 0.0, lin = 0.0;
        for (int r = 0; r < n; ++r) m = z[r] > m ? z[r] : m;
        for (int r = 0; r < n; ++r) {
            double w = exp(z[r] - m);
            l += w;
            if (in[r]) lin += w;
            for (int j = 0; j < d; ++j)
                o[j] += w * oracle_widen(kv->v_pool, kv->dtype, kv_index(kv, tb[r], kvh, tt[r], j));
        }
        if (n > 0)
            for (int j = 0; j < d; ++j) o[j] /= l;
        if (lse) lse[bh] = n > 0 ? m + log(l) : -INFINITY;
        if (outside) outside[bh] = (full && sel && n > 0) ? (l - lin) / l : NAN;
        free(z); free(tb); free(tt); free(in); free(kept);
    }
    return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

int oracle_decode_full(const oracle_kv* kv, const float* q, int num_q_heads,
                       double scale, double alpha, const int32_t* sel,
                       const int32_t* n_sel, int cap, const int32_t* heads,
                       int n_heads, double* out, double* tau, int32_t* support,
                       double* delta, double* vnorm, int32_t* covered,
                       int32_t* support_pages) {
    if (num_q_heads % kv->num_kv_heads || !(alpha > 1.0)) return ORACLE_BAD_ARG;
    int G = num_q_heads / kv->num_kv_heads;
    int d = kv->head_dim;
    int nh = head_count(kv, num_q_heads, heads, n_heads);
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < nh; ++i) {
        int bh = head_at(heads, i);
        int b = bh / num_q_heads, h = bh % num_q_heads, kvh = h / G;
        const float* qv = q + (int64_t)bh * d;
        int np = pages_of(kv, b);
        int n = kv->seq_lens[b];
        double* zp = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
        char* kept = (char*)calloc(np > 0 ? np : 1, 1);
        if (sel)
            for (int r = 0; r < n_sel[bh]; ++r) {
                int p = sel[(int64_t)bh * cap + r];
                if (p >= 0 && p < np) kept[p] = 1;
            }
        int idx = 0;
        for (int p = 0; p < np; ++p) {
            int blk = kv->page_table[(int64_t)b * kv->max_pages + p];
            int nt = valid_tokens(kv, b, p);
            for (int t = 0; t < nt; ++t) zp[idx++] = shifted_score(kv, qv, scale, alpha, blk, kvh, t);
        }
        double t_ = INFINITY;
        int k = oracle_entmax_tau(zp, n, alpha, &t_);
        double* o = out + (int64_t)bh * d;
        for (int j = 0; j < d; ++j) o[j] = 0.0;
        double dl = 0.0, vmax = 0.0;
        int cov = 1, spages = 0;
        idx = 0;
        for (int p = 0; p < np; ++p) {
            int blk = kv->page_table[(int64_t)b * kv->max_pages + p];
            int nt = valid_tokens(kv, b, p);
            int page_has_support = 0;
            for (int t = 0; t < nt; ++t, ++idx) {
                double nv = 0.0;
                for (int j = 0; j < d; ++j) {
                    double v = oracle_widen(kv->v_pool, kv->dtype, kv_index(kv, blk, kvh, t, j));
                    nv += v * v;
                }
                nv = sqrt(nv);
                if (nv > vmax) vmax = nv;
                double w = weight(zp[idx], t_, alpha);
                if (w == 0.0) continue;
                page_has_support = 1;
                for (int j = 0; j < d; ++j)
                    o[j] += w * oracle_widen(kv->v_pool, kv->dtype, kv_index(kv, blk, kvh, t, j));
                if (!kept[p]) { dl += w; cov = 0; }
            }
            spages += page_has_support;
        }
        if (tau) tau[bh] = t_;
        if (support) support[bh] = k;
        if (delta) delta[bh] = sel ? dl : 0.0;
        if (vnorm) vnorm[bh] = vmax;
        if (covered) covered[bh] = sel ? cov : 1;
        if (support_pages) support_pages[bh] = spages;
        free(zp);
        free(kept);
    }
    return ORACLE_OK;
}
