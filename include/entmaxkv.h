/*
 * entmaxkv.h - C ABI of the EntmaxKV sparse alpha-entmax decode library (sm_103a).
 *
 * The method: "Riepilogo Tecnico: EntmaxKV - Decodifica Consapevole del Supporto
 * per l'Attention Entmax" (cited as [EntmaxKV]).  Decode over a paged KV cache
 * runs four stages, each one entry point below:
 *   1. per-page key metadata, built on prefill/append       [EntmaxKV §2.A]
 *   2. query-aware page scoring from that metadata           [EntmaxKV §2.A]
 *   3. candidate page selection: top-k by bound, or the
 *      Gaussian-aware tau-hat threshold with margin Delta    [EntmaxKV §2.B]
 *   4. alpha-entmax attention over only the selected pages  [EntmaxKV §2.C]
 * alpha-entmax is p_i = [(alpha-1) z_i - tau]_+^(1/(alpha-1)) with tau such that
 * sum_i p_i = 1 (Peters, Niculae and Martins, ACL 2019); z_i = scale * q.k_i.
 * When the selected pages contain every token with p_i > 0 the result equals
 * full-cache attention [EntmaxKV §3].
 *
 * Conventions shared by every entry point
 * - Every pointer argument is a DEVICE pointer owned by the caller unless its
 *   comment says "host".  The library never allocates, frees or synchronises
 *   (except entmaxkv_read_device_status, which says so).
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Work is enqueued asynchronously on it.
 * - Arguments are checked on the host before any launch; a failed check returns
 *   a non-zero ekv_status and launches nothing.  Launch failures return
 *   EKV_CUDA_ERROR.  Malformed DEVICE data (a page-table entry outside
 *   [0, num_blocks), a selected page outside a sequence) is skipped by the
 *   kernels and recorded in a sticky per-device word read with
 *   entmaxkv_read_device_status.  Every wait inside a kernel (on an mbarrier
 *   that copies or other warps complete) is bounded by 2 s of %globaltimer; a
 *   wait that runs out stops the kernel's work, records a timeout in the same
 *   word and the kernel returns, so the context stays usable.
 * - Supported shapes: head_dim 64 or 128; page_size 16 or 32; num_q_heads a
 *   multiple of num_kv_heads with group size 1, 2, 4 or 8; K/V fp32 or bf16.
 * - Layouts (row-major, contiguous):
 *     k_pool, v_pool  [num_blocks, num_kv_heads, page_size, head_dim]
 *     page_table      int32 [batch, max_pages]: logical page -> physical block;
 *                     only entries below ceil(seq_lens[b] / page_size) are read
 *     seq_lens        int32 [batch], each in [0, max_pages * page_size]
 *     q               fp32 [batch, num_q_heads, head_dim]; query head h uses
 *                     kv head h / (num_q_heads / num_kv_heads)
 *     out             fp32 [batch, num_q_heads, head_dim]
 *     kmin, kmax      [num_blocks, num_kv_heads, head_dim] in the K dtype
 *     mean, var       fp32 [num_blocks, num_kv_heads, head_dim]
 * - No C++ exception crosses this boundary.
 */
#ifndef ENTMAXKV_H
#define ENTMAXKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EKV_OK = 0,
    EKV_INVALID_ARG = 1,          /* null pointer, bad size, alpha <= 1, ... */
    EKV_UNSUPPORTED = 2,          /* valid but outside the supported shapes  */
    EKV_WORKSPACE_TOO_SMALL = 3,
    EKV_CUDA_ERROR = 4,           /* a CUDA launch or query failed           */
    EKV_DEVICE_CHECK_FAILED = 5,  /* the kernels met malformed device data   */
    EKV_DEVICE_TIMEOUT = 6        /* a bounded wait inside a kernel gave up  */
} ekv_status;

typedef enum { EKV_F32 = 0, EKV_BF16 = 1 } ekv_dtype;

typedef enum {
    EKV_SELECT_TOPK = 0,   /* top-k pages by the bounding-box bound [EntmaxKV §2.B.1] */
    EKV_SELECT_GAUSS = 1,  /* Gaussian-aware tau-hat threshold      [EntmaxKV §2.B.2] */
    EKV_SELECT_TOPK_SHARED = 2  /* top-k shared by a kv head's query group: one page set
                                   per kv head, ranked by the group's largest bound */
} ekv_policy;

/* A paged KV cache.  All pointers are device pointers; the struct itself is
 * read on the host during the call only. */
typedef struct {
    const void*    k_pool;
    const void*    v_pool;
    int32_t        dtype;          /* ekv_dtype */
    int32_t        num_blocks;
    int32_t        num_kv_heads;
    int32_t        page_size;
    int32_t        head_dim;
    const int32_t* page_table;
    int32_t        max_pages;
    const int32_t* seq_lens;
    int32_t        batch;
} ekv_paged_kv;

/* Per-page key metadata [EntmaxKV §2.A]; device pointers, any may be NULL when
 * the corresponding statistic is not built or not read. */
typedef struct {
    void*  kmin;    /* per-coordinate minimum, K dtype (exact)   */
    void*  kmax;    /* per-coordinate maximum, K dtype (exact)   */
    float* mean;    /* per-coordinate mean over the valid tokens */
    float* var;     /* per-coordinate population variance        */
} ekv_page_meta;

/* Stage 1 [EntmaxKV §2.A, metadata "stored per page"]: for every sequence b and
 * logical page p in [first_page, min(first_page + num_pages, ceil(seq_lens[b] /
 * page_size))), compute the metadata of physical block page_table[b, p] for all
 * kv heads over the page's valid tokens (min(page_size, seq_lens[b] - p *
 * page_size)).  want_bbox writes kmin/kmax, want_gauss writes mean/var (the
 * chosen pointers must be non-NULL).  Call on prefill with first_page = 0 and
 * on append with the page(s) that changed. */
int entmaxkv_build_page_meta(const ekv_paged_kv* kv, int32_t first_page,
                             int32_t num_pages, const ekv_page_meta* meta,
                             int32_t want_bbox, int32_t want_gauss, void* stream);

/* Stage 2 [EntmaxKV §2.A]: query-aware page scores for every valid logical page.
 *   EKV_SELECT_TOPK:  page_scores fp32 [batch, num_q_heads, max_pages],
 *       U_p = scale * sum_j max(q_j kmin_j, q_j kmax_j) >= z for every token of
 *       page p (needs meta->kmin/kmax).
 *   EKV_SELECT_GAUSS: page_scores fp32 [batch, num_q_heads, max_pages, 2] holding
 *       (m_p, s_p) = (scale q.mean_p, scale sqrt(sum_j q_j^2 var_pj)), the mean
 *       and standard deviation of the page's scores under independent
 *       coordinates (needs meta->mean/var).
 *   EKV_SELECT_TOPK_SHARED: the same per-head bounds as EKV_SELECT_TOPK.
 * Entries past a sequence's last page are not written.  scale must be > 0. */
int entmaxkv_score_pages(const float* q, int32_t num_q_heads, float scale,
                         const ekv_paged_kv* kv, const ekv_page_meta* meta,
                         int32_t policy, float* page_scores, void* stream);

/* Stage 3 [EntmaxKV §2.B]: choose pages per (sequence, query head).
 *   cap_pages = budget_tokens / page_size (>= 1); sel int32 [batch,
 *   num_q_heads, cap_pages] receives page ids in ascending order, n_sel int32
 *   [batch, num_q_heads] their count.
 *   EKV_SELECT_TOPK: the min(cap_pages, NP_b) pages with the largest bound,
 *       ties to the lower page.  aux (nullable) fp32 [batch, num_q_heads, 2] =
 *       (smallest kept bound, largest bound not kept or -inf).
 *   EKV_SELECT_GAUSS (alpha 1.5 or 2 only): tau-hat solves
 *       sum_p n_p E[((alpha-1) X_p - tau)_+^(1/(alpha-1))] = 1 with
 *       X_p ~ N(m_p, s_p^2); page p is kept iff (alpha-1) zmax_p >= tau-hat -
 *       delta, zmax_p = m_p + sqrt(2 ln n_p) s_p; over cap_pages -> the
 *       cap_pages pages with the largest zmax (ties to the lower page); none ->
 *       the argmax page.  aux (nullable) = (tau-hat, pages passing the
 *       threshold before the cap).
 *   EKV_SELECT_TOPK_SHARED: one page set per (sequence, kv head), written to
 *       every query head of its group: the min(cap_pages, NP_b) pages with the
 *       largest S_p = max over the group's heads of U_p, ties to the lower
 *       page; aux = (smallest kept S_p, largest S_p not kept or -inf) for each
 *       head of the group.
 * workspace/ws_bytes are unused (pass NULL, 0). */
int entmaxkv_select(const float* page_scores, const ekv_paged_kv* kv,
                    int32_t num_q_heads, int32_t policy, int32_t budget_tokens,
                    float alpha, float delta, int32_t* sel, int32_t* n_sel,
                    float* aux, void* workspace, size_t ws_bytes, void* stream);

/* Stage 4 [EntmaxKV §2.C]: alpha-entmax attention over the selected pages.
 * For each (b, h): the valid tokens of pages sel[b, h, 0:n_sel[b, h]] (distinct
 * ids, any order, each < ceil(seq_lens[b] / page_size); duplicates count once)
 * are scored z = scale q.k, tau is the exact alpha-entmax threshold of
 * (alpha-1) z over them (a safeguarded Halley iteration for alpha 1.5 and 2,
 * bisection otherwise), and out = sum_i p_i v_i / sum_i p_i.  Each kv head's K
 * page is read once per step for its whole query group; only the V rows of
 * tokens with p_i > 0 are read.
 * out fp32 [batch, num_q_heads, head_dim]: device memory, or pinned host memory
 * mapped into the device's address space (the kernel then writes the result
 * there directly); any other pointer is EKV_INVALID_ARG.
 * tau_out (nullable) fp32 [batch, num_q_heads] in (alpha-1) z units; support_out
 * (nullable) int32 [batch, num_q_heads] = #{p_i > 0}.  An empty selection gives
 * out = 0, tau = +inf, support 0.  alpha > 1.  workspace: device scratch of at
 * least entmaxkv_workspace_size(...) bytes, 256-byte aligned, not shared with a
 * concurrent call. */
int entmaxkv_decode(const float* q, int32_t num_q_heads, float scale,
                    const ekv_paged_kv* kv, const int32_t* sel,
                    const int32_t* n_sel, int32_t cap_pages, float alpha,
                    float* out, float* tau_out, int32_t* support_out,
                    void* workspace, size_t ws_bytes, void* stream);

/* Stages 3 and 4 in one call [EntmaxKV §2.B, §2.C]: entmaxkv_select then
 * entmaxkv_decode on that selection, with the same results (sel, n_sel and aux
 * are written as entmaxkv_select writes them; out, tau_out and support_out as
 * entmaxkv_decode).  cap_pages = budget_tokens / page_size.  For the top-k
 * policies the selection kernel also builds, in the workspace, the union of
 * each kv head's selected pages that the decode reads (the G query heads of a
 * kv head select as one thread-block cluster), so the decode does not rebuild
 * it.  Arguments and checks as the two calls; workspace: at least
 * entmaxkv_workspace_size(..., cap_pages) bytes, 256-byte aligned, not shared
 * with a concurrent call. */
int entmaxkv_select_decode(const float* page_scores, const float* q, int32_t num_q_heads,
                           float scale, const ekv_paged_kv* kv, int32_t policy,
                           int32_t budget_tokens, float alpha, float delta, int32_t* sel,
                           int32_t* n_sel, float* aux, float* out, float* tau_out,
                           int32_t* support_out, void* workspace, size_t ws_bytes,
                           void* stream);

/* Full-cache alpha-entmax decode, the exact attention the sparse decode
 * approximates ([EntmaxKV] §1 and §3: sparse output equals it whenever the
 * kept pages hold its support).  For each (b, h): every valid token of
 * sequence b is scored z = scale q.k, tau is the exact alpha-entmax threshold of
 * (alpha-1) z over all of them (same solver as entmaxkv_decode) and out =
 * sum_i p_i v_i / sum_i p_i.  Each kv head's whole cache is read once for its
 * query group; only the V rows of tokens with p_i > 0 are read.
 * Arguments, outputs and errors as entmaxkv_decode without the selection;
 * workspace: at least entmaxkv_full_workspace_size(...) bytes, 256-byte
 * aligned, not shared with a concurrent call. */
int entmaxkv_decode_full(const float* q, int32_t num_q_heads, float scale,
                         const ekv_paged_kv* kv, float alpha, float* out,
                         float* tau_out, int32_t* support_out, void* workspace,
                         size_t ws_bytes, void* stream);

/* Host-only: bytes of workspace entmaxkv_decode_full needs for these sizes
 * (0 if the sizes are invalid). */
size_t entmaxkv_full_workspace_size(int32_t batch, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    int32_t page_size, int32_t max_pages);

/* Softmax attention over the selected pages: the comparison method of
 * [EntmaxKV] §1 and §4 (a softmax whose dense tail is truncated to the kept
 * pages), computed by the same plan and score kernels as entmaxkv_decode.
 * For each (b, h): z = scale q.k over the valid tokens of pages sel[b, h,
 * 0:n_sel[b, h]] (as entmaxkv_decode), out = sum_i e^(z_i - m) v_i /
 * sum_i e^(z_i - m) with m = max z, and lse_out (nullable) fp32 [batch,
 * num_q_heads] = log sum_i e^(z_i).  Every selected token has a positive weight,
 * so the V rows of all selected pages are read (each kv head's union once).
 * An empty selection gives out = 0, lse = -inf.  workspace: at least
 * entmaxkv_softmax_workspace_size(...) bytes, 256-byte aligned, not shared
 * with a concurrent call.  Errors as entmaxkv_decode. */
int entmaxkv_decode_softmax(const float* q, int32_t num_q_heads, float scale,
                            const ekv_paged_kv* kv, const int32_t* sel,
                            const int32_t* n_sel, int32_t cap_pages, float* out,
                            float* lse_out, void* workspace, size_t ws_bytes,
                            void* stream);

/* Full-cache softmax attention (every valid token): entmaxkv_decode_softmax
 * without a selection; workspace of entmaxkv_softmax_workspace_size(...,
 * cap_pages = max_pages) bytes. */
int entmaxkv_decode_softmax_full(const float* q, int32_t num_q_heads, float scale,
                                 const ekv_paged_kv* kv, float* out, float* lse_out,
                                 void* workspace, size_t ws_bytes, void* stream);

/* Host-only: bytes of workspace the softmax decodes need (0 if invalid). */
size_t entmaxkv_softmax_workspace_size(int32_t batch, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       int32_t page_size, int32_t max_pages,
                                       int32_t cap_pages);

/* Measurement aid [EntmaxKV §3]: after an entmaxkv_decode that used
 * `workspace` (same sizes), mass_out[b, h] (device fp32) = sum over the valid
 * tokens of the kept pages of ((alpha-1) z_i - tau[b, h])_+^(1/(alpha-1)), the
 * weight an alpha-entmax with threshold tau (device fp32 [batch, num_q_heads],
 * e.g. the full-cache tau_out of entmaxkv_decode_full) puts on the kept
 * tokens; 1 - mass_out is that distribution's mass outside the kept pages
 * (delta in the page's error bound).  Asynchronous on `stream`. */
int entmaxkv_kept_mass(void* workspace, int32_t batch, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                       int32_t max_pages, int32_t cap_pages, float alpha,
                       const float* tau, float* mass_out, void* stream);

/* Bytes of the scratch array built into the library for
 * entmaxkv_decode_noalloc. */
#define ENTMAXKV_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* Stage 4 without a caller-provided workspace.  The page has no counterpart of
 * this call; it exists for callers that cannot allocate device memory at the
 * point where they decode (code running inside an allocator callback, a plugin
 * that is handed only its input and output buffers, a server whose device
 * memory is fixed before it starts taking requests).  Same arguments, results
 * and checks as entmaxkv_decode, minus `workspace`/`ws_bytes`: the scratch is a
 * fixed array of ENTMAXKV_NOALLOC_SCRATCH_BYTES inside the library, one per
 * device that loads it, kept until the process exits.  It never allocates or
 * frees memory.
 * - Sizes whose workspace (entmaxkv_workspace_size) exceeds that array return
 *   EKV_WORKSPACE_TOO_SMALL and launch nothing.
 * - The first call on a device looks up the array's device address (with that
 *   device current) and caches it; make that first call before any stream
 *   capture.
 * - All calls on a device share the one array, which keeps whatever the last
 *   call left in it (each call re-initialises what it needs): calls whose work
 *   can overlap on the GPU (other streams, other host threads) race and must
 *   be serialised by the caller. */
int entmaxkv_decode_noalloc(const float* q, int32_t num_q_heads, float scale,
                            const ekv_paged_kv* kv, const int32_t* sel,
                            const int32_t* n_sel, int32_t cap_pages, float alpha,
                            float* out, float* tau_out, int32_t* support_out,
                            void* stream);

/* Host-only: bytes of workspace entmaxkv_decode needs for these sizes
 * (0 if the sizes are invalid). */
size_t entmaxkv_workspace_size(int32_t batch, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t page_size, int32_t max_pages,
                               int32_t cap_pages);

/* Host-only: a static string naming an ekv_status value. */
const char* entmaxkv_status_string(int32_t status);

/* Reads (and clears) the sticky device status word of the current device:
 * *status_out = EKV_DEVICE_TIMEOUT if a bounded wait gave up since the last
 * read (this takes precedence), else EKV_DEVICE_CHECK_FAILED if a kernel met
 * malformed device data, else EKV_OK.  Synchronises `stream`.  Returns
 * EKV_CUDA_ERROR if the copy fails. */
int entmaxkv_read_device_status(int32_t* status_out /* host */, void* stream);

/* Self-check of the bounded-wait give-up path (the page has no counterpart;
 * it is a health check for this library).  Launches one single-warp kernel on
 * `stream` that waits on an mbarrier whose phase can never complete, with a
 * limit of limit_us microseconds (1 .. 100000) instead of the kernels' 2 s.
 * The wait runs out, the kernel records a timeout exactly as the score, q.k
 * and softmax kernels do, and returns: the next entmaxkv_read_device_status
 * reports EKV_DEVICE_TIMEOUT.  No memory is copied and nothing waits on the
 * kernel.  Returns EKV_INVALID_ARG for a limit outside the range. */
int entmaxkv_check_wait_timeout(uint32_t limit_us, void* stream);

/* Input staging for a step whose query is in pinned host memory (not part of
 * the method): copies `bytes` from src to dst on `stream` with a kernel rather
 * than a copy engine, so a captured step has no copy-engine hand-off before its
 * first kernel; the score kernel that follows sets up while the copy runs and
 * reads q only after it.  src and dst must be device-accessible: device memory,
 * or host memory mapped into the device's address space (pinned, unified
 * addressing).  Returns EKV_INVALID_ARG for a null or inaccessible pointer;
 * bytes = 0 does nothing.  The caller keeps both buffers alive until the copy
 * has run. */
int entmaxkv_copy_in(void* dst, const void* src, size_t bytes, void* stream);

/* Measurement aid (not part of the method): record four caller-created
 * cudaEvent_t handles around the kernels of every later entmaxkv_decode call on
 * its stream: events[0] before the union plan, [1] before the score kernel,
 * [2] before the threshold-and-value kernel, [3] after it.  n_events = 0
 * (events may be NULL) turns it off.  Under stream capture the events become
 * external event-record nodes of the graph.  Process-wide, not thread-safe;
 * the events must outlive every decode call made while set. */
int entmaxkv_set_stage_events(void* const* events /* host array */, int32_t n_events);

/* Measurement aid: after an entmaxkv_decode that used `workspace` (same sizes),
 * copy per (sequence, kv head) unit the number of distinct pages whose K was
 * read (the union of the group's selections) and the number of distinct tokens
 * whose V row was read (tokens with p > 0 for some head of the group) into the
 * HOST arrays union_pages and v_rows (int32 [batch * num_kv_heads], either
 * nullable).  Writes a per-unit count field of the workspace (one small kernel)
 * and synchronises `stream`. */
int entmaxkv_decode_counts(void* workspace, int32_t batch, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                           int32_t max_pages, int32_t cap_pages, int32_t* union_pages,
                           int32_t* v_rows, void* stream);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t entmaxkv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* ENTMAXKV_H */
