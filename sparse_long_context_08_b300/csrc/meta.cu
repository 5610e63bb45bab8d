// Per-page key metadata builder [EntmaxKV §2.A: bounding box k_min/k_max and
// first/second moments, "stored per page"], run on prefill and append.
//
// One CTA per (logical page, sequence, kv head).  The page's P x D key tile is
// read with 16-byte vector loads: RC = D / (elements per 16 B) lanes cover a
// row, the remaining thread groups stride over tokens.  min/max are exact (they
// are stored values); mean and the population variance use two passes in fp32.
#include "common.cuh"

EKV_DEFINE_STATUS(meta)

namespace ekv {

constexpr int kMetaThreads = 256;

template <typename T, int D>
__global__ void __launch_bounds__(kMetaThreads)
build_meta_kernel(KV kv, int first_page, T* __restrict__ kmin, T* __restrict__ kmax,
                  float* __restrict__ mean, float* __restrict__ var, int want_bbox,
                  int want_gauss) {
    constexpr int EPC = Elem<T>::kPer16;
    constexpr int RC = D / EPC;                 // 16-byte chunks per key row
    constexpr int RG = kMetaThreads / RC;       // token groups
    __shared__ float s_a[RG][D];
    __shared__ float s_b[RG][D];
    __shared__ float s_c[RG][D];
    __shared__ float s_mean[D];

    const int p = first_page + blockIdx.x;
    const int b = blockIdx.y;
    const int h = blockIdx.z;
    const int len = kv.sl[b];
    const int np = min(kv.maxp, (len + kv.P - 1) / kv.P);
    if (p >= np) return;
    const int blk = kv.pt[(int64_t)b * kv.maxp + p];
    if (blk < 0 || blk >= kv.nb) {
        if (threadIdx.x == 0) flag_bad_data();
        return;
    }
    const int n = min(kv.P, len - p * kv.P);
    const int c = threadIdx.x % RC;
    const int rg = threadIdx.x / RC;
    const T* tile = static_cast<const T*>(kv.k) + ((int64_t)blk * kv.hkv + h) * kv.P * D;

    float mn[EPC], mx[EPC], sm[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) { mn[e] = INFINITY; mx[e] = -INFINITY; sm[e] = 0.f; }
    for (int t = rg; t < n; t += RG) {
        float x[EPC];
        Elem<T>::widen(ld_nc_v4(tile + (int64_t)t * D + c * EPC), x);
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
            mn[e] = fminf(mn[e], x[e]);
            mx[e] = fmaxf(mx[e], x[e]);
            sm[e] += x[e];
        }
    }
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
        s_a[rg][c * EPC + e] = sm[e];
        s_b[rg][c * EPC + e] = mn[e];
        s_c[rg][c * EPC + e] = mx[e];
    }
    __syncthreads();
    const int64_t o = ((int64_t)blk * kv.hkv + h) * D;
    for (int j = threadIdx.x; j < D; j += blockDim.x) {
        float s = 0.f, lo = INFINITY, hi = -INFINITY;
        for (int g = 0; g < RG; ++g) {
            s += s_a[g][j];
            lo = fminf(lo, s_b[g][j]);
            hi = fmaxf(hi, s_c[g][j]);
        }
        s_mean[j] = s / static_cast<float>(n);
        if (want_bbox) {
            Elem<T>::store(kmin, o + j, lo);
            Elem<T>::store(kmax, o + j, hi);
        }
    }
    if (!want_gauss) return;
    __syncthreads();
    float mu[EPC], ss[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) { mu[e] = s_mean[c * EPC + e]; ss[e] = 0.f; }
    for (int t = rg; t < n; t += RG) {
        float x[EPC];
        Elem<T>::widen(ld_nc_v4(tile + (int64_t)t * D + c * EPC), x);
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
            const float dlt = x[e] - mu[e];
            ss[e] = fmaf(dlt, dlt, ss[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < EPC; ++e) s_a[rg][c * EPC + e] = ss[e];
    __syncthreads();
    for (int j = threadIdx.x; j < D; j += blockDim.x) {
        float s = 0.f;
        for (int g = 0; g < RG; ++g) s += s_a[g][j];
        mean[o + j] = s_mean[j];
        var[o + j] = s / static_cast<float>(n);
    }
}

cudaError_t launch_build_meta(const KV& kv, int first_page, int num_pages, void* kmin,
                              void* kmax, float* mean, float* var, bool bbox, bool gauss,
                              cudaStream_t s) {
    const int pages = min(num_pages, kv.maxp - first_page);
    if (pages <= 0 || kv.B <= 0) return cudaSuccess;
    dim3 grid(pages, kv.B, kv.hkv);
    EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, {
        build_meta_kernel<T, kD><<<grid, kMetaThreads, 0, s>>>(
            kv, first_page, static_cast<T*>(kmin), static_cast<T*>(kmax), mean, var,
            bbox ? 1 : 0, gauss ? 1 : 0);
    }))
    return cudaGetLastError();
}

}  // namespace ekv
