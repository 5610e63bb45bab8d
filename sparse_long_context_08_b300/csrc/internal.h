// Host-side interfaces between the C ABI (abi.cu) and the kernel translation
// units (meta.cu, score.cu, select.cu, decode.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ekv {

// A paged KV cache, already validated on the host (see entmaxkv.h for layouts).
struct KV {
    const void*    k;
    const void*    v;
    int            dtype;      // 0 fp32, 1 bf16
    int            nb;         // num_blocks
    int            hkv;        // num_kv_heads
    int            P;          // page_size
    int            D;          // head_dim
    const int32_t* pt;         // page_table [B, maxp]
    int            maxp;       // max_pages
    const int32_t* sl;         // seq_lens [B]
    int            B;          // batch
};

// Workspace of one decode call, carved from the caller's buffer.  U = B * Hkv
// units (sequence, kv head); a unit reads the union of its G heads' selected
// pages (at most Umax of them) once.  Scores are kept per unit in union order,
// [U][G][Umax * P], with -inf where a head did not select the page; the
// physical block of every union page is kept for the value stage.  vtok marks,
// per unit, the tokens whose V row was read (nvw words per unit).  When a
// head's selection (cap * P tokens) is larger than the threshold kernel keeps
// in shared memory, the candidates go to per-head global buffers of ccap =
// cap * P entries (cand_x, cand_pos; absent otherwise).
//
// The softmax decode adds partial-sum records (recs, nrec slots of G * (D + 1)
// floats): one slot per streaming warp plus one per unit.
//
// pmax [U][G][Umax] holds each head's largest z' on each union page (-inf
// where the head did not select it); plist [B * Hq][Umax] is the global page
// list of the large-selection threshold kernel (with cand_x / cand_pos).
struct DecodeLayout {
    int    U, G, Umax, nvw, ccap, nrec;
    size_t union_count, head_max, union_page, union_mask, union_blk, vtok, vrows;
    size_t z, pmax, tau, cand_x, cand_pos, plist, recs, total;
};
constexpr int kTpvSmemCand = 16384;      // candidates per head the shared-memory threshold kernel holds
constexpr int kPvMaxWarps = 4096;        // streaming-warp record slots of the softmax decode
DecodeLayout decode_layout(int B, int Hq, int Hkv, int D, int P, int max_pages, int cap,
                           bool candidates = true);
DecodeLayout softmax_layout(int B, int Hq, int Hkv, int D, int P, int max_pages, int cap);

cudaError_t launch_build_meta(const KV& kv, int first_page, int num_pages, void* kmin,
                              void* kmax, float* mean, float* var, bool bbox, bool gauss,
                              cudaStream_t s);
cudaError_t launch_score(const float* q, int Hq, float scale, const KV& kv, const void* kmin,
                         const void* kmax, const float* mean, const float* var, int policy,
                         float* out, cudaStream_t s);
// Top-k selection.  With plan_ws / plan_layout (a decode workspace and its
// layout) the selection may also write the decode's union plan into it; then
// *planned is set and the decode can skip its plan (launch_decode planned).
cudaError_t launch_select_topk(const float* bound, const KV& kv, int Hq, int kp, int32_t* sel,
                               int32_t* n_sel, float* aux, bool shared, cudaStream_t s,
                               void* plan_ws = nullptr, const DecodeLayout* plan_layout = nullptr,
                               bool* planned = nullptr);
cudaError_t launch_select_gauss(const float* ms, const KV& kv, int Hq, int cap, float alpha,
                                float delta, int32_t* sel, int32_t* n_sel, float* aux,
                                cudaStream_t s);
// planned: the union plan of this selection is already in the workspace (it
// was written by launch_select_topk), so the plan kernel is skipped.
cudaError_t launch_decode(const float* q, int Hq, float scale, const KV& kv, const int32_t* sel,
                          const int32_t* n_sel, int cap, float alpha, float* out, float* tau_out,
                          int32_t* support_out, void* ws, const DecodeLayout& L, cudaStream_t s,
                          bool planned = false);
// Softmax attention over the selected pages (full: every page), laid out by
// softmax_layout; lse_out (nullable) receives log sum_i e^(z_i).
cudaError_t launch_decode_softmax(const float* q, int Hq, float scale, const KV& kv,
                                  const int32_t* sel, const int32_t* n_sel, int cap, bool full,
                                  float* out, float* lse_out, void* ws, const DecodeLayout& L,
                                  cudaStream_t s);

// Full-cache decode: every valid token of every sequence, for all heads
// (workspace laid out by decode_layout(..., cap = max_pages)).
cudaError_t launch_decode_full(const float* q, int Hq, float scale, const KV& kv, float alpha,
                               float* out, float* tau_out, int32_t* support_out, void* ws,
                               const DecodeLayout& L, cudaStream_t s);

// Mass the alpha-entmax with per-head threshold tau puts on each head's kept
// tokens, from the scores a decode left in the workspace.
cudaError_t launch_kept_mass(int Hq, float alpha, int P, void* ws, const DecodeLayout& L,
                             const float* tau, float* mass, int BH, cudaStream_t s);

// Optional events recorded between the decode kernels (plan | qk | tpv):
// events[0] before plan, [1] before qk, [2] before tpv, [3] after tpv.
// n = 0 disables.  Process-wide; for measurement only.
void set_decode_stage_events(const cudaEvent_t* events, int n);

// Per-unit counters of the last decode that used this workspace: union pages
// whose K was read, and distinct tokens whose V row was read.
cudaError_t read_decode_counts(void* ws, const DecodeLayout& L, int32_t* union_pages,
                               int32_t* v_rows, cudaStream_t s);

// Returned by the launchers for a shape or size outside what the kernels
// support (reported as EKV_UNSUPPORTED); every other error is a CUDA failure.
constexpr cudaError_t kShapeUnsupported = cudaErrorNotSupported;

// Sticky device status words, one per translation unit: read, OR'd into
// *flag (bit 0 malformed data, bit 1 a bounded wait gave up), and cleared.
cudaError_t take_status_meta(int* flag, cudaStream_t s);
cudaError_t take_status_score(int* flag, cudaStream_t s);
cudaError_t take_status_select(int* flag, cudaStream_t s);
cudaError_t take_status_decode(int* flag, cudaStream_t s);
cudaError_t take_status_selfcheck(int* flag, cudaStream_t s);

// One kernel whose bounded wait on an mbarrier that never completes gives up
// after limit_ns and records the timeout bit (self-check of the give-up path).
cudaError_t launch_wait_timeout_check(uint64_t limit_ns, cudaStream_t s);

// Copies `bytes` from src to dst (both device-accessible) with a kernel that
// lets the next kernel of the stream start early (programmatic launch).
cudaError_t launch_copy_in(void* dst, const void* src, size_t bytes, cudaStream_t s);

// Limits of the selection kernels (pages held in shared memory per head).
constexpr int kMaxPagesTopk = 49152;
constexpr int kMaxPagesGauss = 12288;

}  // namespace ekv

// Per-TU definition of the status word and its host accessor.  Bit 0: the
// kernels met malformed device data (skipped); bit 1: a bounded wait gave up.
#define EKV_DEFINE_STATUS(NAME)                                                        \
    namespace ekv {                                                                    \
    static __device__ int g_status_word;                                               \
    __device__ __forceinline__ void flag_bad_data() { atomicOr(&g_status_word, 1); }  \
    __device__ __forceinline__ void flag_timeout() { atomicOr(&g_status_word, 2); }   \
    cudaError_t take_status_##NAME(int* flag, cudaStream_t s) {                        \
        int v = 0;                                                                     \
        cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status_word, sizeof(int), 0,   \
                                                  cudaMemcpyDeviceToHost, s);          \
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);                            \
        if (e != cudaSuccess) return e;                                                \
        if (v) {                                                                       \
            static const int zero = 0;                                                 \
            e = cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof(int), 0,          \
                                        cudaMemcpyHostToDevice, s);                    \
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);                        \
            *flag |= v;                                                                \
        }                                                                              \
        return e;                                                                      \
    }                                                                                  \
    }

// Compile-time dispatch over the supported (dtype, head_dim, group) shapes.
#define EKV_DISPATCH_D(D_, ...)                          \
    switch (D_) {                                        \
        case 64: { constexpr int kD = 64; __VA_ARGS__; } break;   \
        case 128: { constexpr int kD = 128; __VA_ARGS__; } break; \
        default: return ::ekv::kShapeUnsupported;        \
    }
#define EKV_DISPATCH_G(G_, ...)                          \
    switch (G_) {                                        \
        case 1: { constexpr int kG = 1; __VA_ARGS__; } break; \
        case 2: { constexpr int kG = 2; __VA_ARGS__; } break; \
        case 4: { constexpr int kG = 4; __VA_ARGS__; } break; \
        case 8: { constexpr int kG = 8; __VA_ARGS__; } break; \
        default: return ::ekv::kShapeUnsupported;        \
    }
#define EKV_DISPATCH_T(DT_, ...)                         \
    if ((DT_) == 1) { using T = ::ekv::bf16raw; __VA_ARGS__; } \
    else { using T = float; __VA_ARGS__; }
