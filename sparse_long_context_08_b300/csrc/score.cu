// Query-aware page scoring [EntmaxKV §2.A].
//
//   bbox:  U_p = s * sum_j max(q_j kmin_j, q_j kmax_j)   (upper bound on s q.k)
//   gauss: m_p = s q.mean_p,  s_p = s sqrt(sum_j q_j^2 var_pj)
//
// HBM-bound streaming kernel.  The valid pages of all sequences, in
// (sequence, logical page) order, are cut into one contiguous range per CTA;
// the CTA stages the range's page-table entries in shared memory.  A warp owns
// one kv head (and a part of the range) at a time: LPR lanes per page row,
// each lane holding its DPL coordinates of the G query heads of that kv head
// in registers -- for the bound as max(q, 0) and min(q, 0), so that
// max(q kmin, q kmax) = max(q,0) kmax + min(q,0) kmin costs two FMAs and no
// compare -- and the row sums are reduced across lanes by a transposing
// butterfly.  Each lane prefetches its own slices of the next rows with
// cp.async into a private ring in shared memory (kScoreStages row pairs in
// flight per lane, with no register cost and no synchronisation between
// lanes: a lane only ever reads what it copied itself).
#include "common.cuh"

EKV_DEFINE_STATUS(score)

namespace ekv {

constexpr int kScoreWarps = 8;
constexpr int kScoreThreads = 32 * kScoreWarps;
constexpr int kScoreCtasPerSm = 2;
constexpr int kScoreStages = 8;                             // row pairs in flight per lane
constexpr int kScoreMaxSeqs = 16384;

// Sums a[0..C) over the 2*M lanes of an aligned lane group, handing lane lt
// the complete sum of value index lt / (2*M / C) (see qk in decode.cu).
template <int C, int M>
struct XRed {
    __device__ __forceinline__ static void run(float* a, int lt) {
        if constexpr (M >= 1) {
            if constexpr (C >= 2) {
                constexpr int H = C / 2;
                const bool up = (lt & M) != 0;
#pragma unroll
                for (int j = 0; j < H; ++j) {
                    const float send = up ? a[j] : a[j + H];
                    const float keep = up ? a[j + H] : a[j];
                    a[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, M);
                }
                XRed<H, M / 2>::run(a, lt);
            } else {
                a[0] += __shfl_xor_sync(0xFFFFFFFFu, a[0], M);
                XRed<1, M / 2>::run(a, lt);
            }
        }
    }
};

template <typename T, int D, int G, bool kGauss>
struct ScoreCfg {
    static constexpr int ES = sizeof(T);
    static constexpr int EPC = 16 / ES;                         // elements per 16 bytes
    static constexpr int DPL = (32 / G) < EPC ? (32 / G) : EPC; // coordinates per lane
    static constexpr int LPR = D / DPL;                         // lanes per row
    static constexpr int PPP = 32 / LPR;                        // pages per warp pass
    static constexpr int NV = kGauss ? 2 * G : G;               // sums per row
    static_assert(LPR <= 32 && NV <= LPR, "unsupported score shape");
};

// Asynchronous copy of one lane's DPL elements (8 or 16 bytes) into shared memory.
template <int BYTES>
__device__ __forceinline__ void cp_async_lane(void* dst, const void* src) {
    if constexpr (BYTES == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <typename T, int DPL>
__device__ __forceinline__ void widen_lane(const void* p, float* x) {
    if constexpr (DPL * sizeof(T) == 16) {
        Elem<T>::widen(*reinterpret_cast<const uint4*>(p), x);
    } else {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        if constexpr (sizeof(T) == 2) {
            x[0] = __uint_as_float(r.x << 16); x[1] = __uint_as_float(r.x & 0xFFFF0000u);
            x[2] = __uint_as_float(r.y << 16); x[3] = __uint_as_float(r.y & 0xFFFF0000u);
        } else {
            x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
        }
    }
}

template <typename T, int D, int G, bool kGauss>
__global__ void __launch_bounds__(kScoreThreads, kScoreCtasPerSm)
score_kernel(const float* __restrict__ q, int Hq, float scale, KV kv,
             const T* __restrict__ ma,      // bbox: kmin   gauss: mean
             const T* __restrict__ mb,      // bbox: kmax   gauss: var
             float* __restrict__ out, int nloc_max) {
    using C = ScoreCfg<T, D, G, kGauss>;
    constexpr int S = kScoreStages;
    constexpr int CB = C::DPL * sizeof(T);      // bytes a lane copies per row
    extern __shared__ __align__(16) unsigned char s_dyn[];
    // shared layout: rings [warps][S][2][32 lanes][CB] | sequence prefix [B + 1]
    // | page refs [nloc_max] | blocks [nloc_max]
    unsigned char* ring = s_dyn + (size_t)(threadIdx.x >> 5) * S * 2 * 32 * CB;
    int* sprefix = reinterpret_cast<int*>(s_dyn + (size_t)kScoreWarps * S * 2 * 32 * CB);
    int* sref = sprefix + kv.B + 1;             // (sequence << 17) | page
    int* sblk = sref + nloc_max;                // physical block, -1 if bad
    __shared__ int red[40];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    {
        const int B = kv.B;
        const int seg = (B + blockDim.x - 1) / blockDim.x;
        const int a0 = min(B, tid * seg), a1 = min(B, a0 + seg);
        int c = 0;
        for (int x = a0; x < a1; ++x) c += min(kv.maxp, (kv.sl[x] + kv.P - 1) / kv.P);
        int tot;
        int run = block_exclusive_scan(c, red, &tot);
        for (int x = a0; x < a1; ++x) {
            sprefix[x] = run;
            run += min(kv.maxp, (kv.sl[x] + kv.P - 1) / kv.P);
        }
        if (tid == 0) sprefix[B] = tot;
    }
    __syncthreads();
    const int total = sprefix[kv.B];
    const int f0 = (int)((int64_t)total * blockIdx.x / gridDim.x);
    const int f1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
    const int nloc = min(f1 - f0, nloc_max);
    for (int i = tid; i < nloc; i += blockDim.x) {
        const int f = f0 + i;
        int lo = 0, hi = kv.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sprefix[mid] <= f) lo = mid; else hi = mid - 1;
        }
        const int p = f - sprefix[lo];
        int blk = kv.pt[(int64_t)lo * kv.maxp + p];
        if (blk < 0 || blk >= kv.nb) {
            flag_bad_data();
            blk = -1;
        }
        sref[i] = (lo << 17) | p;
        sblk[i] = blk;
    }
    __syncthreads();
    if (nloc <= 0) return;

    const int Hkv = kv.hkv;
    const int parts = Hkv >= kScoreWarps ? 1 : kScoreWarps / Hkv;
    const int lt = lane % C::LPR;
    const int pl = lane / C::LPR;               // page of the item this lane reads
    constexpr int DUP = C::LPR / C::NV;
    unsigned char* mine = ring + (size_t)lane * CB;   // this lane's slot in every stage
    float qa[G][C::DPL], qb[G][C::DPL];         // bbox: max(q,0), min(q,0)   gauss: s q, s^2 q^2
    for (int col = warp; col < Hkv * parts; col += kScoreWarps) {
        const int kvh = col % Hkv, part = col / Hkv;
        const int c0 = nloc * part / parts, c1 = nloc * (part + 1) / parts;
        const int nit = (c1 - c0 + C::PPP - 1) / C::PPP;
        // item `it` covers pages c0 + it * PPP + [0, PPP); this lane reads one of them
        auto issue = [&](int it) {
            const int j = c0 + it * C::PPP + pl;
            const int blk = (it < nit && j < c1) ? sblk[j] : -1;
            if (blk >= 0) {
                const int64_t off = ((int64_t)blk * Hkv + kvh) * D + lt * C::DPL;
                unsigned char* st = mine + (size_t)(it % S) * 2 * 32 * CB;
                cp_async_lane<CB>(st, ma + off);
                cp_async_lane<CB>(st + 32 * CB, mb + off);
            }
            cp_async_commit();
        };
#pragma unroll
        for (int x = 0; x < S - 1; ++x) issue(x);
        int cur_b = -1;
        for (int it = 0; it < nit; ++it) {
            issue(it + S - 1);
            cp_async_wait<S - 1>();            // this lane's copies of item `it` have landed
            const int j = c0 + it * C::PPP + pl;
            const bool inr = j < c1;
            const int ref = inr ? sref[j] : -1;
            const bool live = inr && sblk[j] >= 0;
            const int b = ref >> 17;
            if (inr && b != cur_b) {
                cur_b = b;
                const float* qh = q + ((int64_t)b * Hq + kvh * G) * D + lt * C::DPL;
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < C::DPL; ++e) {
                        const float v = scale * __ldg(qh + h * D + e);
                        if constexpr (kGauss) { qa[h][e] = v; qb[h][e] = v * v; }
                        else { qa[h][e] = fmaxf(v, 0.f); qb[h][e] = fminf(v, 0.f); }
                    }
            }
            float acc[C::NV];
#pragma unroll
            for (int v = 0; v < C::NV; ++v) acc[v] = 0.f;
            if (live) {
                const unsigned char* st = mine + (size_t)(it % S) * 2 * 32 * CB;
                float xa[C::DPL], xb[C::DPL];
                widen_lane<T, C::DPL>(st, xa);
                widen_lane<T, C::DPL>(st + 32 * CB, xb);
                // paired FMAs over coordinate pairs: half the instructions,
                // two independent chains per sum
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < C::DPL; e += 2) {
                        const float2 ka = make_float2(xa[e], xa[e + 1]);
                        const float2 kb = make_float2(xb[e], xb[e + 1]);
                        if constexpr (kGauss) {
                            fma2(s0, make_float2(qa[h][e], qa[h][e + 1]), ka);
                            fma2(s1, make_float2(qb[h][e], qb[h][e + 1]), kb);
                        } else {
                            fma2(s0, make_float2(qa[h][e], qa[h][e + 1]), kb);
                            fma2(s0, make_float2(qb[h][e], qb[h][e + 1]), ka);
                        }
                    }
                    acc[h] = s0.x + s0.y;
                    if constexpr (kGauss) acc[G + h] = s1.x + s1.y;
                }
            }
            XRed<C::NV, C::LPR / 2>::run(acc, lt);
            if (inr && lt % DUP == 0) {
                const int vi = lt / DUP;
                const int h = vi % G;
                const int p = ref & ((1 << 17) - 1);
                const int64_t o = ((int64_t)b * Hq + kvh * G + h) * kv.maxp + p;
                if constexpr (kGauss) {
                    if (vi < G) out[2 * o] = live ? acc[0] : -INFINITY;
                    else out[2 * o + 1] = live ? sqrtf(fmaxf(acc[0], 0.f)) : 0.f;
                } else {
                    out[o] = live ? acc[0] : -INFINITY;
                }
            }
        }
        cp_async_wait<0>();
    }
}

static int sm_count_score() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
    int v = 148;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) cached[dev] = v;
    return v;
}

template <typename T, int D, int G, bool kGauss>
static cudaError_t launch_score_t(const float* q, int Hq, float scale, const KV& kv,
                                  const void* ma, const void* mb, float* out, cudaStream_t s) {
    if (kv.B > kScoreMaxSeqs || kv.maxp >= (1 << 17)) return cudaErrorInvalidValue;
    const int grid = sm_count_score() * kScoreCtasPerSm;
    const int64_t total_max = (int64_t)kv.B * kv.maxp;
    const int nloc_max = (int)((total_max + grid - 1) / grid) + 1;
    using C = ScoreCfg<T, D, G, kGauss>;
    const size_t ring_bytes = (size_t)kScoreWarps * kScoreStages * 2 * 32 * C::DPL * sizeof(T);
    const size_t smem = ring_bytes + (size_t)(kv.B + 1 + 2 * nloc_max) * sizeof(int);
    if (smem > 110 * 1024) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(score_kernel<T, D, G, kGauss>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(score_kernel<T, D, G, kGauss>, dim3(grid), dim3(kScoreThreads), smem, s, q, Hq,
                         scale, kv, static_cast<const T*>(ma), static_cast<const T*>(mb), out,
                         nloc_max);
}

cudaError_t launch_score(const float* q, int Hq, float scale, const KV& kv, const void* kmin,
                         const void* kmax, const float* mean, const float* var, int policy,
                         float* out, cudaStream_t s) {
    const int G = Hq / kv.hkv;
    if (policy == 1) {
        EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
            return launch_score_t<float, kD, kG, true>(q, Hq, scale, kv, mean, var, out, s);
        }))
    } else {
        EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
            return launch_score_t<T, kD, kG, false>(q, Hq, scale, kv, kmin, kmax, out, s);
        })))
    }
    return cudaErrorInvalidValue;
}

}  // namespace ekv
