// C ABI of the EntmaxKV decode library: host-side argument checks, workspace
// layout and dispatch to the kernel launchers.  Declarations and the contract
// of every entry point are in include/entmaxkv.h.
#include <cmath>
#include <cstdint>

#include "entmaxkv.h"
#include "internal.h"

namespace {

using ekv::KV;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_kv(const ekv_paged_kv* kv, bool need_k, bool need_v) {
    if (!kv) return EKV_INVALID_ARG;
    if (kv->dtype != EKV_F32 && kv->dtype != EKV_BF16) return EKV_INVALID_ARG;
    if (kv->num_blocks <= 0 || kv->num_kv_heads <= 0 || kv->page_size <= 0 ||
        kv->head_dim <= 0 || kv->max_pages <= 0 || kv->batch <= 0)
        return EKV_INVALID_ARG;
    if (!kv->page_table || !kv->seq_lens) return EKV_INVALID_ARG;
    if (need_k && !kv->k_pool) return EKV_INVALID_ARG;
    if (need_v && !kv->v_pool) return EKV_INVALID_ARG;
    if (need_k && !aligned16(kv->k_pool)) return EKV_INVALID_ARG;
    if (need_v && !aligned16(kv->v_pool)) return EKV_INVALID_ARG;
    if (kv->head_dim != 64 && kv->head_dim != 128) return EKV_UNSUPPORTED;
    if (kv->page_size != 16 && kv->page_size != 32) return EKV_UNSUPPORTED;
    if ((int64_t)kv->max_pages * kv->page_size > INT32_MAX) return EKV_UNSUPPORTED;
    return EKV_OK;
}

int check_heads(const ekv_paged_kv* kv, int32_t num_q_heads) {
    if (num_q_heads <= 0 || num_q_heads % kv->num_kv_heads) return EKV_INVALID_ARG;
    const int G = num_q_heads / kv->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return EKV_UNSUPPORTED;
    return EKV_OK;
}

KV to_kv(const ekv_paged_kv* kv) {
    return KV{kv->k_pool, kv->v_pool, kv->dtype, kv->num_blocks, kv->num_kv_heads, kv->page_size,
              kv->head_dim, kv->page_table, kv->max_pages, kv->seq_lens, kv->batch};
}

// The launchers report a shape outside what the kernels support with
// ekv::kShapeUnsupported; any other error came from CUDA itself.
int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return EKV_OK;
    if (e == ekv::kShapeUnsupported) return EKV_UNSUPPORTED;
    return EKV_CUDA_ERROR;
}

bool is_alpha(float a) { return std::isfinite(a) && a > 1.f; }

}  // namespace

extern "C" {

int32_t entmaxkv_version(void) { return 10000; }

const char* entmaxkv_status_string(int32_t s) {
    switch (s) {
        case EKV_OK: return "ok";
        case EKV_INVALID_ARG: return "invalid argument";
        case EKV_UNSUPPORTED: return "unsupported shape or option";
        case EKV_WORKSPACE_TOO_SMALL: return "workspace too small";
        case EKV_CUDA_ERROR: return "CUDA error";
        case EKV_DEVICE_CHECK_FAILED: return "malformed device data (page table or selection)";
        case EKV_DEVICE_TIMEOUT: return "a bounded wait inside a kernel gave up (device timeout)";
        default: return "unknown status";
    }
}

size_t entmaxkv_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t page_size, int32_t max_pages,
                               int32_t cap_pages) {
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
        head_dim <= 0 || page_size <= 0 || max_pages <= 0 || cap_pages <= 0)
        return 0;
    return ekv::decode_layout(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages,
                              cap_pages).total;
}

int entmaxkv_build_page_meta(const ekv_paged_kv* kv, int32_t first_page, int32_t num_pages,
                             const ekv_page_meta* meta, int32_t want_bbox, int32_t want_gauss,
                             void* stream) {
    int st = check_kv(kv, true, false);
    if (st) return st;
    if (!meta || first_page < 0 || num_pages < 0) return EKV_INVALID_ARG;
    if (!want_bbox && !want_gauss) return EKV_INVALID_ARG;
    if (want_bbox && (!meta->kmin || !meta->kmax)) return EKV_INVALID_ARG;
    if (want_gauss && (!meta->mean || !meta->var)) return EKV_INVALID_ARG;
    if (num_pages == 0 || first_page >= kv->max_pages) return EKV_OK;
    return from_cuda(ekv::launch_build_meta(to_kv(kv), first_page, num_pages, meta->kmin,
                                            meta->kmax, meta->mean, meta->var, want_bbox != 0,
                                            want_gauss != 0, static_cast<cudaStream_t>(stream)));
}

int entmaxkv_score_pages(const float* q, int32_t num_q_heads, float scale,
                         const ekv_paged_kv* kv, const ekv_page_meta* meta, int32_t policy,
                         float* page_scores, void* stream) {
    int st = check_kv(kv, false, false);
    if (st) return st;
    if ((st = check_heads(kv, num_q_heads))) return st;
    if (!q || !meta || !page_scores) return EKV_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return EKV_INVALID_ARG;
    if (policy == EKV_SELECT_TOPK || policy == EKV_SELECT_TOPK_SHARED) {
        if (!meta->kmin || !meta->kmax || !aligned16(meta->kmin) || !aligned16(meta->kmax))
            return EKV_INVALID_ARG;
        policy = EKV_SELECT_TOPK;          // the same per-head bounds
    } else if (policy == EKV_SELECT_GAUSS) {
        if (!meta->mean || !meta->var || !aligned16(meta->mean) || !aligned16(meta->var))
            return EKV_INVALID_ARG;
    } else {
        return EKV_INVALID_ARG;
    }
    return from_cuda(ekv::launch_score(q, num_q_heads, scale, to_kv(kv), meta->kmin, meta->kmax,
                                       meta->mean, meta->var, policy, page_scores,
                                       static_cast<cudaStream_t>(stream)));
}

int entmaxkv_select(const float* page_scores, const ekv_paged_kv* kv, int32_t num_q_heads,
                    int32_t policy, int32_t budget_tokens, float alpha, float delta,
                    int32_t* sel, int32_t* n_sel, float* aux, void* workspace, size_t ws_bytes,
                    void* stream) {
    (void)workspace;
    (void)ws_bytes;
    int st = check_kv(kv, false, false);
    if (st) return st;
    if ((st = check_heads(kv, num_q_heads))) return st;
    if (!page_scores || !sel || !n_sel) return EKV_INVALID_ARG;
    const int cap = budget_tokens / kv->page_size;
    if (budget_tokens <= 0 || cap < 1) return EKV_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (policy == EKV_SELECT_TOPK || policy == EKV_SELECT_TOPK_SHARED) {
        if (kv->max_pages > ekv::kMaxPagesTopk) return EKV_UNSUPPORTED;
        return from_cuda(ekv::launch_select_topk(page_scores, to_kv(kv), num_q_heads, cap, sel,
                                                 n_sel, aux, policy == EKV_SELECT_TOPK_SHARED, s));
    }
    if (policy == EKV_SELECT_GAUSS) {
        if (!is_alpha(alpha) || !std::isfinite(delta)) return EKV_INVALID_ARG;
        if (std::fabs(alpha - 1.5f) > 1e-6f && std::fabs(alpha - 2.f) > 1e-6f)
            return EKV_UNSUPPORTED;
        if (kv->max_pages > ekv::kMaxPagesGauss) return EKV_UNSUPPORTED;
        return from_cuda(ekv::launch_select_gauss(page_scores, to_kv(kv), num_q_heads, cap, alpha,
                                                  delta, sel, n_sel, aux, s));
    }
    return EKV_INVALID_ARG;
}

// Checks of a decode call's arguments; on success *L is its workspace layout.
// The device can read and write p: device or managed memory, or host memory
// mapped into the device's address space (pinned, unified addressing).
static bool device_accessible(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

static int check_decode(const float* q, int32_t num_q_heads, float scale, const ekv_paged_kv* kv,
                        const int32_t* sel, const int32_t* n_sel, int32_t cap_pages, float alpha,
                        const float* out, const void* workspace, size_t ws_bytes,
                        ekv::DecodeLayout* L) {
    int st = check_kv(kv, true, true);
    if (st) return st;
    if ((st = check_heads(kv, num_q_heads))) return st;
    if (!q || !sel || !n_sel || !out || !workspace) return EKV_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f) || !is_alpha(alpha)) return EKV_INVALID_ARG;
    if (cap_pages < 1) return EKV_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EKV_INVALID_ARG;
    if ((int64_t)kv->max_pages > ekv::kMaxPagesTopk) return EKV_UNSUPPORTED;
    if ((int64_t)kv->num_blocks * kv->num_kv_heads * kv->page_size > INT32_MAX) return EKV_UNSUPPORTED;
    *L = ekv::decode_layout(kv->batch, num_q_heads, kv->num_kv_heads, kv->head_dim,
                            kv->page_size, kv->max_pages, cap_pages);
    if (ws_bytes < L->total) return EKV_WORKSPACE_TOO_SMALL;
    if (!device_accessible(out)) return EKV_INVALID_ARG;   // last: one host query
    return EKV_OK;
}

static int decode_impl(const float* q, int32_t num_q_heads, float scale, const ekv_paged_kv* kv,
                       const int32_t* sel, const int32_t* n_sel, int32_t cap_pages, float alpha,
                       float* out, float* tau_out, int32_t* support_out, void* workspace,
                       size_t ws_bytes, void* stream) {
    ekv::DecodeLayout L;
    const int st = check_decode(q, num_q_heads, scale, kv, sel, n_sel, cap_pages, alpha, out,
                                workspace, ws_bytes, &L);
    if (st) return st;
    return from_cuda(ekv::launch_decode(q, num_q_heads, scale, to_kv(kv), sel, n_sel, cap_pages,
                                        alpha, out, tau_out, support_out, workspace, L,
                                        static_cast<cudaStream_t>(stream)));
}

int entmaxkv_decode(const float* q, int32_t num_q_heads, float scale, const ekv_paged_kv* kv,
                    const int32_t* sel, const int32_t* n_sel, int32_t cap_pages, float alpha,
                    float* out, float* tau_out, int32_t* support_out, void* workspace,
                    size_t ws_bytes, void* stream) {
    return decode_impl(q, num_q_heads, scale, kv, sel, n_sel, cap_pages, alpha, out, tau_out,
                       support_out, workspace, ws_bytes, stream);
}

int entmaxkv_select_decode(const float* page_scores, const float* q, int32_t num_q_heads,
                           float scale, const ekv_paged_kv* kv, int32_t policy,
                           int32_t budget_tokens, float alpha, float delta, int32_t* sel,
                           int32_t* n_sel, float* aux, float* out, float* tau_out,
                           int32_t* support_out, void* workspace, size_t ws_bytes,
                           void* stream) {
    if (!kv || !page_scores) return EKV_INVALID_ARG;
    if (budget_tokens <= 0 || kv->page_size <= 0 || budget_tokens / kv->page_size < 1)
        return EKV_INVALID_ARG;
    const int cap = budget_tokens / kv->page_size;
    ekv::DecodeLayout L;
    int st = check_decode(q, num_q_heads, scale, kv, sel, n_sel, cap, alpha, out, workspace,
                          ws_bytes, &L);
    if (st) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool planned = false;
    cudaError_t e;
    if (policy == EKV_SELECT_TOPK || policy == EKV_SELECT_TOPK_SHARED) {
        e = ekv::launch_select_topk(page_scores, to_kv(kv), num_q_heads, cap, sel, n_sel, aux,
                                    policy == EKV_SELECT_TOPK_SHARED, s, workspace, &L, &planned);
    } else if (policy == EKV_SELECT_GAUSS) {
        if (!std::isfinite(delta)) return EKV_INVALID_ARG;
        if (std::fabs(alpha - 1.5f) > 1e-6f && std::fabs(alpha - 2.f) > 1e-6f) return EKV_UNSUPPORTED;
        if (kv->max_pages > ekv::kMaxPagesGauss) return EKV_UNSUPPORTED;
        e = ekv::launch_select_gauss(page_scores, to_kv(kv), num_q_heads, cap, alpha, delta, sel,
                                     n_sel, aux, s);
    } else {
        return EKV_INVALID_ARG;
    }
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(ekv::launch_decode(q, num_q_heads, scale, to_kv(kv), sel, n_sel, cap, alpha,
                                        out, tau_out, support_out, workspace, L, s, planned));
}

size_t entmaxkv_full_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t page_size, int32_t max_pages) {
    return entmaxkv_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, page_size,
                                   max_pages, max_pages);
}

int entmaxkv_decode_full(const float* q, int32_t num_q_heads, float scale, const ekv_paged_kv* kv,
                         float alpha, float* out, float* tau_out, int32_t* support_out,
                         void* workspace, size_t ws_bytes, void* stream) {
    int st = check_kv(kv, true, true);
    if (st) return st;
    if ((st = check_heads(kv, num_q_heads))) return st;
    if (!q || !out || !workspace) return EKV_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f) || !is_alpha(alpha)) return EKV_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EKV_INVALID_ARG;
    if ((int64_t)kv->max_pages > ekv::kMaxPagesTopk) return EKV_UNSUPPORTED;
    if ((int64_t)kv->num_blocks * kv->num_kv_heads * kv->page_size > INT32_MAX) return EKV_UNSUPPORTED;
    const ekv::DecodeLayout L = ekv::decode_layout(kv->batch, num_q_heads, kv->num_kv_heads,
                                                   kv->head_dim, kv->page_size, kv->max_pages,
                                                   kv->max_pages);
    if (ws_bytes < L.total) return EKV_WORKSPACE_TOO_SMALL;
    return from_cuda(ekv::launch_decode_full(q, num_q_heads, scale, to_kv(kv), alpha, out, tau_out,
                                             support_out, workspace, L,
                                             static_cast<cudaStream_t>(stream)));
}

size_t entmaxkv_softmax_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t page_size, int32_t max_pages,
                                       int32_t cap_pages) {
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
        head_dim <= 0 || page_size <= 0 || max_pages <= 0 || cap_pages <= 0)
        return 0;
    return ekv::softmax_layout(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages,
                               cap_pages).total;
}

static int softmax_impl(const float* q, int32_t num_q_heads, float scale, const ekv_paged_kv* kv,
                        const int32_t* sel, const int32_t* n_sel, int32_t cap_pages, bool full,
                        float* out, float* lse_out, void* workspace, size_t ws_bytes,
                        void* stream) {
    int st = check_kv(kv, true, true);
    if (st) return st;
    if ((st = check_heads(kv, num_q_heads))) return st;
    if (!q || !out || !workspace || (!full && (!sel || !n_sel))) return EKV_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return EKV_INVALID_ARG;
    if (cap_pages < 1) return EKV_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return EKV_INVALID_ARG;
    if ((int64_t)kv->max_pages > ekv::kMaxPagesTopk) return EKV_UNSUPPORTED;
    if ((int64_t)kv->num_blocks * kv->num_kv_heads * kv->page_size > INT32_MAX) return EKV_UNSUPPORTED;
    const ekv::DecodeLayout L = ekv::softmax_layout(kv->batch, num_q_heads, kv->num_kv_heads,
                                                    kv->head_dim, kv->page_size, kv->max_pages,
                                                    cap_pages);
    if (ws_bytes < L.total) return EKV_WORKSPACE_TOO_SMALL;
    return from_cuda(ekv::launch_decode_softmax(q, num_q_heads, scale, to_kv(kv), sel, n_sel,
                                                cap_pages, full, out, lse_out, workspace, L,
                                                static_cast<cudaStream_t>(stream)));
}

int entmaxkv_decode_softmax(const float* q, int32_t num_q_heads, float scale,
                            const ekv_paged_kv* kv, const int32_t* sel, const int32_t* n_sel,
                            int32_t cap_pages, float* out, float* lse_out, void* workspace,
                            size_t ws_bytes, void* stream) {
    return softmax_impl(q, num_q_heads, scale, kv, sel, n_sel, cap_pages, false, out, lse_out,
                        workspace, ws_bytes, stream);
}

int entmaxkv_decode_softmax_full(const float* q, int32_t num_q_heads, float scale,
                                 const ekv_paged_kv* kv, float* out, float* lse_out,
                                 void* workspace, size_t ws_bytes, void* stream) {
    if (!kv) return EKV_INVALID_ARG;
    return softmax_impl(q, num_q_heads, scale, kv, nullptr, nullptr, kv->max_pages, true, out,
                        lse_out, workspace, ws_bytes, stream);
}

int entmaxkv_set_stage_events(void* const* events, int32_t n_events) {
    if (n_events != 0 && (n_events != 4 || !events)) return EKV_INVALID_ARG;
    ekv::set_decode_stage_events(reinterpret_cast<const cudaEvent_t*>(events), n_events);
    return EKV_OK;
}

int entmaxkv_decode_counts(void* workspace, int32_t batch, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                           int32_t max_pages, int32_t cap_pages, int32_t* union_pages,
                           int32_t* v_rows, void* stream) {
    if (!workspace || entmaxkv_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                              page_size, max_pages, cap_pages) == 0)
        return EKV_INVALID_ARG;
    const ekv::DecodeLayout L = ekv::decode_layout(batch, num_q_heads, num_kv_heads, head_dim,
                                                   page_size, max_pages, cap_pages);
    return from_cuda(ekv::read_decode_counts(workspace, L, union_pages, v_rows,
                                             static_cast<cudaStream_t>(stream)));
}

int entmaxkv_kept_mass(void* workspace, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t page_size, int32_t max_pages, int32_t cap_pages,
                       float alpha, const float* tau, float* mass_out, void* stream) {
    if (!workspace || !tau || !mass_out || !is_alpha(alpha)) return EKV_INVALID_ARG;
    if (entmaxkv_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages,
                                cap_pages) == 0)
        return EKV_INVALID_ARG;
    const ekv::DecodeLayout L = ekv::decode_layout(batch, num_q_heads, num_kv_heads, head_dim,
                                                   page_size, max_pages, cap_pages);
    return from_cuda(ekv::launch_kept_mass(num_q_heads, alpha, page_size, workspace, L, tau,
                                           mass_out, batch * num_q_heads,
                                           static_cast<cudaStream_t>(stream)));
}

int entmaxkv_read_device_status(int32_t* status_out, void* stream) {
    if (!status_out) return EKV_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int flag = 0;
    cudaError_t e = ekv::take_status_meta(&flag, s);
    if (e == cudaSuccess) e = ekv::take_status_score(&flag, s);
    if (e == cudaSuccess) e = ekv::take_status_select(&flag, s);
    if (e == cudaSuccess) e = ekv::take_status_decode(&flag, s);
    if (e == cudaSuccess) e = ekv::take_status_selfcheck(&flag, s);
    if (e != cudaSuccess) return EKV_CUDA_ERROR;
    *status_out = (flag & 2) ? EKV_DEVICE_TIMEOUT : (flag & 1) ? EKV_DEVICE_CHECK_FAILED : EKV_OK;
    return EKV_OK;
}

int entmaxkv_copy_in(void* dst, const void* src, size_t bytes, void* stream) {
    if (!dst || !src) return EKV_INVALID_ARG;
    if (bytes == 0) return EKV_OK;
    if (!device_accessible(dst) || !device_accessible(src)) return EKV_INVALID_ARG;
    return from_cuda(ekv::launch_copy_in(dst, src, bytes, static_cast<cudaStream_t>(stream)));
}

int entmaxkv_check_wait_timeout(uint32_t limit_us, void* stream) {
    if (limit_us == 0 || limit_us > 100000u) return EKV_INVALID_ARG;
    return from_cuda(ekv::launch_wait_timeout_check((uint64_t)limit_us * 1000u,
                                                    static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
