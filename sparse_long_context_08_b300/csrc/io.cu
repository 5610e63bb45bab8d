// Input staging for a decode step whose query lives in pinned host memory: a
// kernel copy instead of a copy-engine transfer, so a captured step has no
// hand-off between the copy engine and the compute grids, and the score
// kernel (which reads q only after its dependency wait) sets up while the
// copy runs.  Not part of the method.
#include <algorithm>

#include "common.cuh"

namespace ekv {

constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
copy_in_kernel(unsigned char* __restrict__ dst, const unsigned char* __restrict__ src,
               size_t bytes, int vec) {
    pdl_trigger();                      // the next kernel may set up meanwhile
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (vec) {
        const size_t n = bytes / 16;
        for (size_t i = t; i < n; i += stride)
            reinterpret_cast<uint4*>(dst)[i] = __ldcv(reinterpret_cast<const uint4*>(src) + i);
    } else {
        for (size_t i = t; i < bytes; i += stride) dst[i] = src[i];
    }
}

cudaError_t launch_copy_in(void* dst, const void* src, size_t bytes, cudaStream_t s) {
    if (bytes == 0) return cudaSuccess;
    const int vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | bytes) &
                     15) == 0;
    const size_t items = vec ? bytes / 16 : bytes;
    const int grid = (int)std::min<size_t>(4 * 148, (items + kCopyThreads - 1) / kCopyThreads);
    return launch_kernel(copy_in_kernel, dim3(grid), dim3(kCopyThreads), 0, s,
                         static_cast<unsigned char*>(dst), static_cast<const unsigned char*>(src),
                         bytes, vec);
}

}  // namespace ekv
