// Query-aware page scoring [EntmaxKV §2.A].
//
//   bbox:  U_p = s * sum_j max(q_j kmin_j, q_j kmax_j)   (upper bound on s q.k)
//   gauss: m_p = s q.mean_p,  s_p = s sqrt(sum_j q_j^2 var_pj)
//
// HBM-bound streaming kernel.  One CTA covers `ppc` consecutive logical pages
// of one sequence and all kv heads: the metadata rows of one physical block
// (Hkv rows of D values) are contiguous, so each page costs a few contiguous
// KiB.  A row is read by LPR lanes with 16-byte loads; each lane keeps its
// slice of the G query heads of its kv head in registers (the GQA group
// shares every load), reduces over the LPR lanes with shuffles, and the CTA
// stages its [Hq, ppc] results in shared memory for one coalesced store.
#include "common.cuh"

EKV_DEFINE_STATUS(score)

namespace ekv {

constexpr int kScoreUnroll = 4;   // passes whose loads are issued together

template <typename T, int D, int G, bool kGauss>
__global__ void __launch_bounds__(512)
score_kernel(const float* __restrict__ q, int Hq, float scale, KV kv,
             const T* __restrict__ ma,      // bbox: kmin   gauss: mean
             const T* __restrict__ mb,      // bbox: kmax   gauss: var
             float* __restrict__ out, int ppc) {
    constexpr int EPC = Elem<T>::kPer16;
    constexpr int LPR = D / EPC;                 // lanes per metadata row
    constexpr int NOUT = kGauss ? 2 : 1;
    extern __shared__ float s_out[];             // [Hq][ppc][NOUT]

    const int Hkv = kv.hkv;
    const int rows_per_pass = blockDim.x / LPR;  // a multiple of Hkv
    const int ppp = rows_per_pass / Hkv;         // pages per pass
    const int lr = threadIdx.x % LPR;
    const int row = threadIdx.x / LPR;
    const int kvh = row % Hkv;
    const int pip = row / Hkv;
    const int b = blockIdx.y;
    const int p0 = blockIdx.x * ppc;
    const int len = kv.sl[b];
    const int np = min(kv.maxp, (len + kv.P - 1) / kv.P);
    if (p0 >= np) return;

    float qr[G][EPC];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < EPC; ++e)
            qr[h][e] = scale * q[((int64_t)b * Hq + kvh * G + h) * D + lr * EPC + e];

    const int32_t* pt = kv.pt + (int64_t)b * kv.maxp;
    for (int base = 0; base < ppc; base += ppp * kScoreUnroll) {
        uint4 ra[kScoreUnroll], rb[kScoreUnroll];
        bool ok[kScoreUnroll];
#pragma unroll
        for (int u = 0; u < kScoreUnroll; ++u) {
            const int pl = base + u * ppp + pip;
            const int p = p0 + pl;
            ok[u] = pl < ppc && p < np;
            int blk = ok[u] ? pt[p] : 0;
            if (ok[u] && (blk < 0 || blk >= kv.nb)) {
                ok[u] = false;
                if (lr == 0) flag_bad_data();
            }
            if (ok[u]) {
                const int64_t off = ((int64_t)blk * Hkv + kvh) * D + lr * EPC;
                ra[u] = ld_nc_v4(ma + off);
                rb[u] = ld_nc_v4(mb + off);
            }
        }
#pragma unroll
        for (int u = 0; u < kScoreUnroll; ++u) {
            const int pl = base + u * ppp + pip;
            if (pl >= ppc) continue;   // uniform across the CTA: ppc % ppp == 0
            float xa[EPC], xb[EPC];
            if (ok[u]) {
                Elem<T>::widen(ra[u], xa);
                Elem<T>::widen(rb[u], xb);
            } else {
#pragma unroll
                for (int e = 0; e < EPC; ++e) { xa[e] = 0.f; xb[e] = 0.f; }
            }
            float acc[G], acc2[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                acc[h] = 0.f;
                acc2[h] = 0.f;
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    if constexpr (kGauss) {
                        acc[h] = fmaf(qr[h][e], xa[e], acc[h]);
                        acc2[h] = fmaf(qr[h][e] * qr[h][e], xb[e], acc2[h]);
                    } else {
                        acc[h] = fmaf(qr[h][e], qr[h][e] >= 0.f ? xb[e] : xa[e], acc[h]);
                    }
                }
                acc[h] = group_sum<LPR>(acc[h]);
                if constexpr (kGauss) acc2[h] = group_sum<LPR>(acc2[h]);
            }
            float mine = 0.f, mine2 = 0.f;
#pragma unroll
            for (int h = 0; h < G; ++h)
                if (lr == h) { mine = acc[h]; mine2 = acc2[h]; }
            if (lr < G) {
                float* dst = s_out + ((int64_t)(kvh * G + lr) * ppc + pl) * NOUT;
                if constexpr (kGauss) {
                    dst[0] = ok[u] ? mine : -INFINITY;
                    dst[1] = ok[u] ? sqrtf(fmaxf(mine2, 0.f)) : 0.f;
                } else {
                    dst[0] = ok[u] ? mine : -INFINITY;
                }
            }
        }
    }
    __syncthreads();
    const int valid = min(ppc, np - p0);
    for (int i = threadIdx.x; i < Hq * ppc * NOUT; i += blockDim.x) {
        const int h = i / (ppc * NOUT);
        const int r = i - h * ppc * NOUT;
        if (r / NOUT < valid)
            out[((int64_t)b * Hq + h) * kv.maxp * NOUT + (int64_t)p0 * NOUT + r] = s_out[i];
    }
}

cudaError_t launch_score(const float* q, int Hq, float scale, const KV& kv, const void* kmin,
                         const void* kmax, const float* mean, const float* var, int policy,
                         float* out, cudaStream_t s) {
    const bool gauss = policy == 1;
    const int esz = gauss ? 4 : (kv.dtype == 1 ? 2 : 4);
    const int lpr = kv.D * esz / 16;
    const int row_threads = lpr * kv.hkv;
    if (row_threads > 512) return cudaErrorInvalidValue;
    const int threads = row_threads * max(1, 256 / row_threads);
    const int ppp = threads / row_threads;
    const int nout = gauss ? 2 : 1;
    // pages per CTA: enough CTAs for several waves, bounded by the staging buffer
    int sms = 148;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess)
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    const int64_t total_pages = (int64_t)kv.B * kv.maxp;
    int ppc = (int)((total_pages + (int64_t)sms * 6 - 1) / ((int64_t)sms * 6));
    const int smem_cap_pages = (48 * 1024) / (Hq * nout * 4);
    ppc = min(ppc, min(256, smem_cap_pages));
    ppc = max(ppp, (ppc / ppp) * ppp);
    if (ppc * Hq * nout * 4 > 48 * 1024) return cudaErrorInvalidValue;
    dim3 grid((kv.maxp + ppc - 1) / ppc, kv.B);
    const size_t smem = (size_t)ppc * Hq * nout * sizeof(float);
    const int G = Hq / kv.hkv;
    if (gauss) {
        EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
            score_kernel<float, kD, kG, true><<<grid, threads, smem, s>>>(
                q, Hq, scale, kv, mean, var, out, ppc);
        }))
    } else {
        EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
            score_kernel<T, kD, kG, false><<<grid, threads, smem, s>>>(
                q, Hq, scale, kv, static_cast<const T*>(kmin), static_cast<const T*>(kmax),
                out, ppc);
        })))
    }
    return cudaGetLastError();
}

}  // namespace ekv
