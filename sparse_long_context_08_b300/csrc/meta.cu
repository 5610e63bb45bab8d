// Per-page key metadata builder [EntmaxKV §2.A: bounding box k_min/k_max and
// first/second moments, "stored per page"], run on prefill and append.
//
// A streaming kernel: the (sequence, logical page, kv head) pages of the call
// are flattened (sequence-major, the kv heads of one physical block
// adjacent, so consecutive pages are contiguous in HBM) and cut into one
// contiguous range per warp.  Every warp streams its pages through a private
// ring of 1-D bulk copies (one P x D page per copy, its own mbarriers, every
// wait bounded), resolving the physical blocks of 32 pages per page-table
// round trip.  Per page, lane l covers one 16-byte column chunk of every
// (32 / chunks-per-row)-th token; min, max and the sum come from one pass over
// the staged page, the population variance from a second pass around the
// exact fp32 mean, both over the page's valid tokens only.  min/max are
// stored values (exact in the K dtype).
#include <algorithm>

#include "common.cuh"

EKV_DEFINE_STATUS(meta)

namespace ekv {

constexpr int kMbWarps = 4;                  // warps per CTA (two CTAs per SM)
constexpr int kMbCtasPerSm = 2;
constexpr int kMbStageBytes = 24 * 1024;     // ring bytes per warp
constexpr int kMbMaxSeqs = 16384;

struct MbDesc { int blk, h, n; int64_t o; };   // block (-1: none), kv head, valid tokens, output row

// Page f of the call's flattened list: sequence by binary search over the
// per-sequence page-count prefix (s_pref[B + 1]), then its block and length.
__device__ __forceinline__ MbDesc mb_resolve(int f, int total, const int* s_pref, const KV& kv,
                                             int first_page) {
    MbDesc d{-1, 0, 0, 0};
    if (f >= total) return d;
    const int per = f / kv.hkv, h = f - per * kv.hkv;
    int lo = 0, hi = kv.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pref[mid] <= per) lo = mid; else hi = mid - 1;
    }
    const int p = first_page + (per - s_pref[lo]);
    int blk = __ldg(kv.pt + (int64_t)lo * kv.maxp + p);
    const int n = min(kv.P, __ldg(kv.sl + lo) - p * kv.P);
    if (blk < 0 || blk >= kv.nb) {
        flag_bad_data();
        blk = -1;
    }
    d.blk = blk;
    d.h = h;
    d.n = n;
    d.o = ((int64_t)max(blk, 0) * kv.hkv + h) * kv.D;
    return d;
}

template <typename T, int D>
__global__ void __launch_bounds__(kMbWarps * 32, kMbCtasPerSm)
build_meta_kernel(KV kv, int first_page, int num_pages, T* __restrict__ kmin,
                  T* __restrict__ kmax, float* __restrict__ mean, float* __restrict__ var,
                  int want_bbox, int want_gauss, int ns) {
    constexpr int EPC = Elem<T>::kPer16;           // elements per 16-byte chunk
    constexpr int CPR = D / EPC;                   // chunks per token row
    constexpr int RPP = 32 / CPR;                  // rows a warp pass covers
    static_assert(CPR <= 32 && 32 % CPR == 0, "row layout");
    extern __shared__ __align__(128) unsigned char s_mb[];
    __shared__ __align__(8) uint64_t s_bar[kMbWarps][8];
    __shared__ int red[40];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = kv.P;
    const uint32_t page_bytes = static_cast<uint32_t>(P * D * sizeof(T));
    unsigned char* ring = s_mb + (size_t)warp * ns * page_bytes;
    int* s_pref = reinterpret_cast<int*>(s_mb + (size_t)kMbWarps * ns * page_bytes);
    uint64_t* bar = s_bar[warp];
    {   // pages of the call per sequence: clamp(ceil(len / P) - first_page, 0, num_pages)
        const int B = kv.B;
        const int seg = (B + blockDim.x - 1) / blockDim.x;
        const int a0 = min(B, tid * seg), a1 = min(B, a0 + seg);
        auto cnt = [&](int x) {
            const int np = min(kv.maxp, (__ldg(kv.sl + x) + P - 1) / P);
            return max(0, min(np - first_page, num_pages));
        };
        int c = 0;
        for (int x = a0; x < a1; ++x) c += cnt(x);
        int tot;
        int run = block_exclusive_scan(c, red, &tot);
        for (int x = a0; x < a1; ++x) {
            s_pref[x] = run;
            run += cnt(x);
        }
        if (tid == 0) s_pref[B] = tot;
    }
    if (lane == 0) {
        for (int st = 0; st < ns; ++st) mbar_init(&bar[st], 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int total = s_pref[kv.B] * kv.hkv;
    const int64_t nwg = (int64_t)gridDim.x * kMbWarps;
    const int wg = blockIdx.x * kMbWarps + warp;
    const int f0 = (int)((int64_t)total * wg / nwg);
    const int f1 = (int)((int64_t)total * (wg + 1) / nwg);
    const int npg = f1 - f0;
    if (npg <= 0) return;
    const unsigned char* kbase = static_cast<const unsigned char*>(kv.k);
    const uint64_t evict_first = l2_evict_first_policy();

    // lanes hold the descriptors of pages [base, base + 32) of the range
    MbDesc cur = mb_resolve(f0 + lane, f1, s_pref, kv, first_page);
    MbDesc nxt{-1, 0, 0, 0};
    if (npg > 32) nxt = mb_resolve(f0 + 32 + lane, f1, s_pref, kv, first_page);
    int cur_base = 0;
    auto desc_of = [&](int k) -> MbDesc {
        if (k >= cur_base + 32) {
            cur = nxt;
            cur_base += 32;
            if (npg > cur_base + 32) nxt = mb_resolve(f0 + cur_base + 32 + lane, f1, s_pref, kv, first_page);
        }
        const int src = k - cur_base;
        return MbDesc{__shfl_sync(0xFFFFFFFFu, cur.blk, src), __shfl_sync(0xFFFFFFFFu, cur.h, src),
                      __shfl_sync(0xFFFFFFFFu, cur.n, src),
                      (int64_t)__shfl_sync(0xFFFFFFFFu, (long long)cur.o, src)};
    };
    auto issue = [&](int k, const MbDesc& d) {
        if (k >= npg || lane != 0) return;
        const int st = k % ns;
        if (d.blk >= 0) {
            mbar_arrive_expect_tx(&bar[st], page_bytes);
            bulk_g2s_hint(ring + (size_t)st * page_bytes,
                          kbase + ((int64_t)d.blk * kv.hkv + d.h) * page_bytes, page_bytes,
                          &bar[st], evict_first);
        } else {
            mbar_arrive(&bar[st]);
        }
    };
    MbDesc dq[8];
#pragma unroll
    for (int x = 0; x < 8; ++x)
        if (x < ns - 1 && x < npg) { dq[x] = desc_of(x); issue(x, dq[x]); }
    const int c = lane % CPR, r0 = lane / CPR;
    for (int k = 0; k < npg; ++k) {
        const int st = k % ns;
        if (k + ns - 1 < npg) {
            const MbDesc nd = desc_of(k + ns - 1);
            issue(k + ns - 1, nd);
            const int nst = (k + ns - 1) % ns;
#pragma unroll
            for (int x = 0; x < 8; ++x)
                if (x == nst) dq[x] = nd;
        }
        MbDesc d{};
#pragma unroll
        for (int x = 0; x < 8; ++x)
            if (x == st) d = dq[x];
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[st], (uint32_t)((k / ns) & 1)))) {
            if (lane == 0) {               // wait (bounded) for this warp's other copies
                flag_timeout();
                for (int j = 1; j < ns; ++j)
                    if (k + j < npg) mbar_wait(&bar[(k + j) % ns], (uint32_t)(((k + j) / ns) & 1));
            }
            return;
        }
        if (d.blk >= 0) {
            const T* pg = reinterpret_cast<const T*>(ring + (size_t)st * page_bytes);
            float mn[EPC], mx[EPC], sm[EPC];
#pragma unroll
            for (int e = 0; e < EPC; ++e) { mn[e] = INFINITY; mx[e] = -INFINITY; sm[e] = 0.f; }
            for (int t = r0; t < d.n; t += RPP) {
                float x[EPC];
                Elem<T>::widen(*reinterpret_cast<const uint4*>(pg + (size_t)t * D + c * EPC), x);
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    mn[e] = fminf(mn[e], x[e]);
                    mx[e] = fmaxf(mx[e], x[e]);
                    sm[e] += x[e];
                }
            }
#pragma unroll
            for (int o = CPR; o < 32; o <<= 1)
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    mn[e] = fminf(mn[e], __shfl_xor_sync(0xFFFFFFFFu, mn[e], o));
                    mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xFFFFFFFFu, mx[e], o));
                    sm[e] += __shfl_xor_sync(0xFFFFFFFFu, sm[e], o);
                }
            const float inv_n = 1.f / static_cast<float>(d.n);
            if (want_bbox && r0 == 0) {
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    Elem<T>::store(kmin, d.o + c * EPC + e, mn[e]);
                    Elem<T>::store(kmax, d.o + c * EPC + e, mx[e]);
                }
            }
            if (want_gauss) {
                float mu[EPC], ss[EPC];
#pragma unroll
                for (int e = 0; e < EPC; ++e) { mu[e] = sm[e] / static_cast<float>(d.n); ss[e] = 0.f; }
                for (int t = r0; t < d.n; t += RPP) {
                    float x[EPC];
                    Elem<T>::widen(*reinterpret_cast<const uint4*>(pg + (size_t)t * D + c * EPC), x);
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        const float dl = x[e] - mu[e];
                        ss[e] = fmaf(dl, dl, ss[e]);
                    }
                }
#pragma unroll
                for (int o = CPR; o < 32; o <<= 1)
#pragma unroll
                    for (int e = 0; e < EPC; ++e) ss[e] += __shfl_xor_sync(0xFFFFFFFFu, ss[e], o);
                if (r0 == 0) {
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        mean[d.o + c * EPC + e] = mu[e];
                        var[d.o + c * EPC + e] = ss[e] * inv_n;
                    }
                }
            }
        }
        __syncwarp();        // every lane is done with stage st before it is refilled
    }
}

static int sm_count_meta() {
    int dev = 0, v = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v;
}

template <typename T, int D>
static cudaError_t launch_build_meta_t(const KV& kv, int first_page, int num_pages, void* kmin,
                                       void* kmax, float* mean, float* var, bool bbox, bool gauss,
                                       cudaStream_t s) {
    if (kv.B > kMbMaxSeqs) return kShapeUnsupported;
    const int page_bytes = kv.P * D * (int)sizeof(T);
    // at least two stages per warp (fp32 pages of 32 x 128 take 32 KiB)
    const int ns = std::max(2, std::min(8, kMbStageBytes / page_bytes));
    const size_t smem = (size_t)kMbWarps * ns * page_bytes + (size_t)(kv.B + 1) * sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(build_meta_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(build_meta_kernel<T, D>, dim3(sm_count_meta() * kMbCtasPerSm),
                         dim3(kMbWarps * 32), smem, s, kv, first_page, num_pages,
                         static_cast<T*>(kmin), static_cast<T*>(kmax), mean, var, bbox ? 1 : 0,
                         gauss ? 1 : 0, ns);
}

cudaError_t launch_build_meta(const KV& kv, int first_page, int num_pages, void* kmin,
                              void* kmax, float* mean, float* var, bool bbox, bool gauss,
                              cudaStream_t s) {
    const int pages = min(num_pages, kv.maxp - first_page);
    if (pages <= 0 || kv.B <= 0) return cudaSuccess;
    EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, {
        return launch_build_meta_t<T, kD>(kv, first_page, pages, kmin, kmax, mean, var, bbox,
                                          gauss, s);
    }))
    return kShapeUnsupported;
}

}  // namespace ekv
