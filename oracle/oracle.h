/*
 * EntmaxKV oracle: plain, slow, fp64 CPU implementation of support-aware sparse
 * alpha-entmax decode over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  It exists to check the CUDA library; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * Method source: the web page "Riepilogo Tecnico: EntmaxKV - Decodifica
 * Consapevole del Supporto per l'Attention Entmax" (cited below as [EntmaxKV]),
 *   §2    the paged pipeline with three components,
 *   §2.A  query-aware page scoring from per-page metadata (bounding box
 *         k_min/k_max; Gaussian first and second moments),
 *   §2.B  candidate selection (top-k pages by bound; Gaussian-aware tau-hat
 *         threshold with a safety margin Delta),
 *   §2.C  alpha-entmax attention over only the selected pages,
 *   §3    error bound ||o - o~|| <= 2 B delta and exact support recovery.
 * The alpha-entmax mapping itself is the standard one of Peters, Niculae and
 * Martins, "Sparse Sequence-to-Sequence Models" (ACL 2019):
 *   p_i = [(alpha-1) z_i - tau]_+^(1/(alpha-1)),  tau such that sum p = 1.
 *
 * Layouts (row-major):
 *   k_pool, v_pool  [num_blocks, Hkv, P, d]   fp32, or bf16 as uint16 bits
 *   page_table      int32 [B, max_pages]      logical page -> physical block
 *   seq_lens        int32 [B]
 *   q               fp32 [B, Hq, d]; query head h reads kv head h / (Hq/Hkv)
 *   per-page metadata (fp64 here) [num_blocks, Hkv, d]
 *   per-head page arrays          [B*Hq, max_pages]
 * A "head list" names flattened (b*Hq + h) indices to process; NULL = all.
 *
 * Readings of points the page leaves open are listed with each function.
 */
#ifndef ENTMAXKV_ORACLE_H
#define ENTMAXKV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    const void*    k_pool;
    const void*    v_pool;
    int            dtype;        /* 0 = fp32, 1 = bf16 bits */
    int            num_blocks;
    int            num_kv_heads;
    int            page_size;
    int            head_dim;
    const int32_t* page_table;
    int            max_pages;
    const int32_t* seq_lens;
    int            batch;
} oracle_kv;

void oracle_set_threads(int n);
int  oracle_get_threads(void);

/* Widen one stored K/V element to fp64 (bf16: bits << 16, exact). */
double oracle_widen(const void* base, int dtype, int64_t idx);

/* [EntmaxKV §2.A] per-page, per-coordinate k_min, k_max, mean and population
 * variance over the page's valid tokens.  Writes every block that a valid
 * logical page maps to; other entries are left untouched. */
int oracle_build_meta(const oracle_kv* kv, double* kmin, double* kmax,
                      double* mean, double* var);

/* [EntmaxKV §2.A] bounding-box bound U_p = s * sum_j max(q_j kmin_j, q_j kmax_j)
 * for every valid page; entries past a sequence's last page are untouched. */
int oracle_score_bbox(const oracle_kv* kv, const float* q, int num_q_heads,
                      double scale, const double* kmin, const double* kmax,
                      const int32_t* heads, int n_heads, double* bound);

/* [EntmaxKV §2.B.1] the min(kp, NP_b) pages with the largest bound, ties to the
 * lower logical page; sel is written in ascending page order.  kth = smallest
 * kept bound, next = largest bound not kept (-inf if every page is kept). */
int oracle_select_topk(const oracle_kv* kv, int num_q_heads, const double* bound,
                       int kp, const int32_t* heads, int n_heads,
                       int32_t* sel, int32_t* n_sel, double* kth, double* next);

/* [EntmaxKV §2.A] Gaussian page statistics of the score z = s q.k:
 * m_p = s q.mu_p,  s_p = s sqrt(sum_j q_j^2 var_pj). */
int oracle_score_gauss(const oracle_kv* kv, const float* q, int num_q_heads,
                       double scale, const double* mean, const double* var,
                       const int32_t* heads, int n_heads, double* m, double* s);

/* Approximate normalisation F(tau) = sum_p n_p E[((alpha-1)X_p - tau)_+^e] - 1,
 * X_p ~ N(m_p, s_p^2), e = 1/(alpha-1); alpha in {1.5, 2}. */
double oracle_gauss_F(const double* m, const double* s, const int32_t* n, int np,
                      double alpha, double tau);

/* [EntmaxKV §2.B.2] tau-hat from F = 0 by bisection; keep page p iff
 * (alpha-1) zmax_p >= tau_hat - delta, zmax_p = m_p + sqrt(2 ln n_p) s_p;
 * more than cap -> the cap pages with the largest zmax (ties: lower page);
 * none -> the argmax page.  sel ascending.  zmax (optional) receives zmax_p.
 * The page prints no formula for tau-hat or the estimated maximum, so these
 * are readings: parity unpinned against the page's own rule (the reading is
 * pinned to its definition by quadrature, root finding and the zero-variance
 * reduction in the tests). */
int oracle_select_gauss(const oracle_kv* kv, int num_q_heads, const double* m,
                        const double* s, double alpha, double delta, int cap,
                        const int32_t* heads, int n_heads, int32_t* sel,
                        int32_t* n_sel, double* tau_hat, double* zmax);

/* Exact alpha-entmax threshold of the shifted scores zp_i = (alpha-1) z_i:
 * sort-based closed forms for alpha = 2 and alpha = 1.5, bisection otherwise.
 * Returns the support size; n == 0 gives tau = +inf and 0. */
int oracle_entmax_tau(const double* zp, int n, double alpha, double* tau);

/* p_i = (zp_i - tau)_+^(1/(alpha-1)). */
int oracle_entmax_probs(const double* zp, int n, double alpha, double* p);

/* [EntmaxKV §2.C] alpha-entmax attention over the selected pages' valid tokens.
 * out = sum_i p_i v_i (fp64), tau in zp units, support = #{p_i > 0},
 * psum = sum_i p_i.  An empty selection gives out = 0, tau = +inf, support 0. */
int oracle_decode_sparse(const oracle_kv* kv, const float* q, int num_q_heads,
                         double scale, double alpha, const int32_t* sel,
                         const int32_t* n_sel, int cap, const int32_t* heads,
                         int n_heads, double* out, double* tau, int32_t* support,
                         double* psum);

/* Softmax attention over the selected pages' valid tokens (every valid token
 * when full): out = sum_i e^(z_i - m) v_i / sum_i e^(z_i - m), z = scale q.k,
 * lse = log sum_i e^(z_i).  full with sel: outside = the full softmax's mass
 * outside the kept pages (NaN otherwise).  No tokens: out = 0, lse = -inf. */
int oracle_decode_softmax(const oracle_kv* kv, const float* q, int num_q_heads,
                          double scale, const int32_t* sel, const int32_t* n_sel,
                          int cap, int full, const int32_t* heads, int n_heads,
                          double* out, double* lse, double* outside);

/* Full-cache alpha-entmax attention over every valid token, plus, when sel is
 * given, [EntmaxKV §3] quantities for that kept set: delta = full-cache mass of
 * tokens outside it, covered = (support within it).  vnorm = max_i ||v_i||_2;
 * support_pages = number of pages holding support tokens. */
int oracle_decode_full(const oracle_kv* kv, const float* q, int num_q_heads,
                       double scale, double alpha, const int32_t* sel,
                       const int32_t* n_sel, int cap, const int32_t* heads,
                       int n_heads, double* out, double* tau, int32_t* support,
                       double* delta, double* vnorm, int32_t* covered,
                       int32_t* support_pages);

#ifdef __cplusplus
}
#endif
#endif
