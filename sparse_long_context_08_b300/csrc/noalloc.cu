// entmaxkv_decode_noalloc: the decode stage for callers that cannot allocate
// device memory (for example code running inside a custom allocator's callback,
// a plugin that is handed only input and output buffers by its host, or a
// process whose memory pool is fixed before serving starts).  The scratch that
// entmaxkv_decode takes from its caller lives here instead, in one fixed-size
// array in the library's own device image.
#include <cuda_runtime.h>

#include <mutex>

#include "entmaxkv.h"

namespace {

// One per device that loads the library; it stays allocated until the process
// exits.  Every call on a device shares it.
static __device__ __align__(256) unsigned char g_decode_scratch[ENTMAXKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EKV_CUDA_ERROR;
    if (dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!g_scratch_ptr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p)
                return EKV_CUDA_ERROR;
            g_scratch_ptr[dev] = p;
        }
        *out = g_scratch_ptr[dev];
        return EKV_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return EKV_CUDA_ERROR;
    *out = p;
    return EKV_OK;
}

}  // namespace

extern "C" int entmaxkv_decode_noalloc(const float* q, int32_t num_q_heads, float scale,
                                       const ekv_paged_kv* kv, const int32_t* sel,
                                       const int32_t* n_sel, int32_t cap_pages, float alpha,
                                       float* out, float* tau_out, int32_t* support_out,
                                       void* stream) {
    if (!kv) return EKV_INVALID_ARG;
    const size_t need = entmaxkv_workspace_size(kv->batch, num_q_heads, kv->num_kv_heads,
                                                kv->head_dim, kv->page_size, kv->max_pages,
                                                cap_pages);
    if (need == 0) return EKV_INVALID_ARG;
    if (need > (size_t)ENTMAXKV_NOALLOC_SCRATCH_BYTES) return EKV_WORKSPACE_TOO_SMALL;
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != EKV_OK) return st;
    // Nothing in the scratch has to start at zero: the decode's first kernel
    // resets the per-unit counters it uses, and every other entry is written
    // before it is read within the same call.
    return entmaxkv_decode(q, num_q_heads, scale, kv, sel, n_sel, cap_pages, alpha, out, tau_out,
                           support_out, scratch, (size_t)ENTMAXKV_NOALLOC_SCRATCH_BYTES, stream);
}
