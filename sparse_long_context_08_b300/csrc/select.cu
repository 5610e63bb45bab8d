// Candidate page selection [EntmaxKV §2.B].
//
// Top-k (§2.B.1): one CTA per (sequence, query head) holds the head's page
// bounds as order-preserving uint32 keys in shared memory, finds the boundary
// with an MSB radix select that starts at the highest bit where the keys
// differ, then writes the selected pages in ascending order, ranked with warp
// ballots: ties at the k-th key go to the lower page ids.
//
// Gaussian tau-hat (§2.B.2): one CTA per (sequence, query head) solves
//   F(tau) = sum_p n_p E[((alpha-1) X_p - tau)_+^e] - 1 = 0,  X_p ~ N(m_p, s_p^2)
// with a safeguarded Newton iteration from tau = max_p (alpha-1) m_p - 1
// (F >= 0 there; F is convex and decreasing, so Newton climbs monotonically),
// keeps pages whose (alpha-1) * estimated max clears tau-hat - delta, and caps
// the kept set by estimated-max rank with the same radix select.
#include "common.cuh"
#include "mills_ratio.h"

EKV_DEFINE_STATUS(select)

namespace ekv {

constexpr int kSelThreads = 512;   // Gaussian select: two CTAs per SM (63 registers)

struct SelShared {
    int red[40];
    uint32_t ured[32];
    int digit, above;
};

// k-th largest key among keys[0..n) (1 <= k <= n) and how many entries equal
// to it are taken (the rest being strictly larger).  whist: [warps][256] ints.
__device__ void radix_kth(const uint32_t* keys, int n, int k, int* whist, int* hist,
                          SelShared& sh, uint32_t& kth, int& take_eq) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nw = blockDim.x >> 5;
    uint32_t prefix = 0, pmask = 0;
    int rem = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < nw * 256; i += blockDim.x) whist[i] = 0;
        __syncthreads();
        int* mine = whist + wid * 256;
        for (int i = tid; i < n; i += blockDim.x) {
            const uint32_t key = keys[i];
            if ((key & pmask) == prefix) atomicAdd(&mine[(key >> shift) & 255u], 1);
        }
        __syncthreads();
        for (int d = tid; d < 256; d += blockDim.x) {
            int s = 0;
            for (int w = 0; w < nw; ++w) s += whist[w * 256 + d];
            hist[d] = s;
        }
        __syncthreads();
        if (wid == 0) {
            int lsum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) lsum += hist[lane * 8 + j];
            // exclusive suffix sum over lanes (buckets above this lane's)
            int incl = lsum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_down_sync(0xFFFFFFFFu, incl, o);
                if (lane + o < 32) incl += v;
            }
            int acc = incl - lsum;
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                const int d = lane * 8 + j;
                const int c = hist[d];
                if (acc < rem && acc + c >= rem) { sh.digit = d; sh.above = acc; }
                acc += c;
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(sh.digit) << shift;
        pmask |= 255u << shift;
        rem -= sh.above;
        __syncthreads();
    }
    kth = prefix;
    take_eq = rem;
}

// Writes, in ascending index order, every i with keys[i] > kth plus the first
// take_eq indices with keys[i] == kth.  Returns the count; *next_key receives
// the largest key not taken (0 if all were taken).
__device__ int compact_topk(const uint32_t* keys, int n, uint32_t kth, int take_eq,
                            int32_t* dst, SelShared& sh, uint32_t* next_key) {
    const int tid = threadIdx.x;
    const int seg = (n + blockDim.x - 1) / blockDim.x;
    const int i0 = min(n, tid * seg), i1 = min(n, i0 + seg);
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += keys[i] == kth;
    int tot;
    int eq_rank = block_exclusive_scan(eq, sh.red, &tot);
    int cnt = 0;
    uint32_t best_out = 0;
    {
        int r = eq_rank;
        for (int i = i0; i < i1; ++i) {
            const uint32_t key = keys[i];
            bool take = key > kth;
            if (key == kth) { take = r < take_eq; ++r; }
            if (take) ++cnt; else best_out = max(best_out, key);
        }
    }
    int pos = block_exclusive_scan(cnt, sh.red, &tot);
    {
        int r = eq_rank;
        for (int i = i0; i < i1; ++i) {
            const uint32_t key = keys[i];
            bool take = key > kth;
            if (key == kth) { take = r < take_eq; ++r; }
            if (take) dst[pos++] = i;
        }
    }
    *next_key = block_max_u(best_out, sh.ured);
    return tot;
}

// Top-k by bound: one CTA per (sequence, query head), the head's bounds as
// order-preserving uint32 keys in shared memory.  The radix select starts at
// the highest bit where the smallest and largest keys differ (every key shares
// the bits above it, so no pass is wasted on them) and stops as soon as the
// boundary bin is taken whole.  Ties at the k-th key go to the lower pages.
constexpr int kTopkMaxThreads = 1024;

//
// Shared (gs > 0, the group size): one CTA per (sequence, kv head) ranks the
// pages by the largest bound over the group's gs query heads and gives every
// head of the group that one page set (one page set per kv head).
__global__ void __launch_bounds__(kTopkMaxThreads)
select_topk_kernel(const float* __restrict__ bound, KV kv, int Hq, int kp,
                   int32_t* __restrict__ sel, int32_t* __restrict__ n_sel,
                   float* __restrict__ aux, int gs) {
    extern __shared__ __align__(16) uint32_t keys[];   // [max_pages] keys, then [kp] selection
    __shared__ int hist[256];
    __shared__ uint32_t umin_red[32], umax_red[32];
    __shared__ int s_digit, s_above;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nt = blockDim.x, nwarps = nt >> 5;
    const int ng = gs > 0 ? gs : 1;       // heads that receive this CTA's selection
    const int bh = gs > 0 ? (blockIdx.x / kv.hkv) * Hq + (blockIdx.x % kv.hkv) * gs : blockIdx.x;
    const int b = bh / Hq;
    const int np = min(kv.maxp, (kv.sl[b] + kv.P - 1) / kv.P);
    const float* src = bound + (int64_t)bh * kv.maxp;
    int32_t* dst = sel + (int64_t)bh * kp;
    int32_t* s_sel = reinterpret_cast<int32_t*>(keys + kv.maxp);   // the row, written out coalesced
    const int k = min(kp, np);
    if (k <= 0) {
        if (tid < ng) {
            n_sel[bh + tid] = 0;
            if (aux) { aux[2 * (bh + tid)] = INFINITY; aux[2 * (bh + tid) + 1] = -INFINITY; }
        }
        return;
    }
    uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
    for (int base = 0; base < np; base += 16 * nt) {
        float v[16];                       // 16 coalesced loads in flight per thread
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = base + j * nt + tid;
            v[j] = i < np ? __ldcg(src + i) : 0.f;
        }
        for (int g = 1; g < ng; ++g) {     // shared: the group's largest bound
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = base + j * nt + tid;
                if (i < np) v[j] = fmaxf(v[j], __ldcg(src + (int64_t)g * kv.maxp + i));
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int i = base + j * nt + tid;
            if (i < np) {
                const uint32_t key = float_key(v[j]);
                keys[i] = key;
                kmn = min(kmn, key);
                kmx = max(kmx, key);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kmn = min(kmn, __shfl_xor_sync(0xFFFFFFFFu, kmn, o));
        kmx = max(kmx, __shfl_xor_sync(0xFFFFFFFFu, kmx, o));
    }
    if (lane == 0) { umin_red[wid] = kmn; umax_red[wid] = kmx; }
    for (int i = tid; i < 256; i += nt) hist[i] = 0;
    __syncthreads();
    kmn = lane < nwarps ? umin_red[lane] : 0xFFFFFFFFu;
    kmx = lane < nwarps ? umax_red[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kmn = min(kmn, __shfl_xor_sync(0xFFFFFFFFu, kmn, o));
        kmx = max(kmx, __shfl_xor_sync(0xFFFFFFFFu, kmx, o));
    }

    // B = {keys whose bits above `shift` equal `hi`}; everything above B is
    // taken, and `rem` more are taken from B.
    const uint32_t diff = kmn ^ kmx;
    int shift = diff ? 32 - __clz(diff) : 0;
    uint64_t hi = (uint64_t)kmx >> shift;
    int rem = k, nB = np;
    while (shift > 0 && nB != rem) {
        const int dbits = min(8, shift);
        shift -= dbits;
        const uint32_t dmask = (1u << dbits) - 1u;
        for (int i = tid; i < np; i += nt) {
            const uint32_t key = keys[i];
            if (((uint64_t)key >> (shift + dbits)) == hi) atomicAdd(&hist[(key >> shift) & dmask], 1);
        }
        __syncthreads();
        if (wid == 0) {
            int lsum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) lsum += hist[lane * 8 + j];
            int incl = lsum;       // inclusive suffix sum over lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_down_sync(0xFFFFFFFFu, incl, o);
                if (lane + o < 32) incl += v;
            }
            int acc = incl - lsum;
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                const int d = lane * 8 + j;
                const int c = hist[d];
                if (acc < rem && acc + c >= rem) { s_digit = d; s_above = acc; }
                acc += c;
            }
        }
        __syncthreads();
        const int d = s_digit;
        rem -= s_above;
        nB = hist[d];
        hi = (hi << dbits) | (uint64_t)d;
        __syncthreads();
        for (int i = tid; i < 256; i += nt) hist[i] = 0;
        __syncthreads();
    }
    const int takeB = rem;    // == nB when B is taken whole

    // compaction in page order: every warp walks a contiguous range of 32-key
    // chunks (consecutive shared-memory words, no bank conflicts) and ranks
    // keys with ballots; one prefix over the warp totals places the ranges
    __shared__ int s_wa[32], s_wb[32];
    const uint32_t below = (1u << lane) - 1u;
    const int nch = (np + 31) / 32;
    const int ch0 = nch * wid / nwarps, ch1 = nch * (wid + 1) / nwarps;
    int wa = 0, wb = 0;
    for (int c = ch0; c < ch1; ++c) {
        const int i = c * 32 + lane;
        const bool in = i < np;
        const uint64_t kh = in ? (uint64_t)keys[i] >> shift : 0u;
        wa += __popc(__ballot_sync(0xFFFFFFFFu, in && kh > hi));
        wb += __popc(__ballot_sync(0xFFFFFFFFu, in && kh == hi));
    }
    if (lane == 0) { s_wa[wid] = wa; s_wb[wid] = wb; }
    __syncthreads();
    int a = 0, r = 0;
    for (int w = 0; w < wid; ++w) { a += s_wa[w]; r += s_wb[w]; }
    uint32_t tmin = 0xFFFFFFFFu, nmax = 0u;
    bool any_out = false;
    for (int c = ch0; c < ch1; ++c) {
        const int i = c * 32 + lane;
        const bool in = i < np;
        const uint32_t key = in ? keys[i] : 0u;
        const uint64_t kh = (uint64_t)key >> shift;
        const uint32_t ma = __ballot_sync(0xFFFFFFFFu, in && kh > hi);
        const uint32_t mb = __ballot_sync(0xFFFFFFFFu, in && kh == hi);
        const int ra = a + __popc(ma & below);     // above keys before i
        const int rb = r + __popc(mb & below);     // boundary-bin keys before i
        bool take = false;
        if (in && kh > hi) {
            s_sel[ra + min(rb, takeB)] = i;
            take = true;
        } else if (in && kh == hi && rb < takeB) {
            s_sel[ra + rb] = i;
            take = true;
        }
        if (take) tmin = min(tmin, key);
        else if (in) { nmax = max(nmax, key); any_out = true; }
        a += __popc(ma);
        r += __popc(mb);
    }
    // smallest taken key (the k-th bound) and largest key left out; the
    // barrier also completes s_sel
    const int any = __syncthreads_or(any_out);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tmin = min(tmin, __shfl_xor_sync(0xFFFFFFFFu, tmin, o));
        nmax = max(nmax, __shfl_xor_sync(0xFFFFFFFFu, nmax, o));
    }
    if (lane == 0) { umin_red[wid] = tmin; umax_red[wid] = nmax; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < nwarps; ++w) {
            tmin = min(tmin, umin_red[w]);
            nmax = max(nmax, umax_red[w]);
        }
        for (int g = 0; g < ng; ++g) {
            n_sel[bh + g] = k;
            if (aux) {
                aux[2 * (bh + g)] = key_float(tmin);
                aux[2 * (bh + g) + 1] = any ? key_float(nmax) : -INFINITY;
            }
        }
    }
    // the row (and, shared, the group's other heads' copies) in whole sectors
    for (int x = tid; x < ng * k; x += nt) {
        const int g = x / k, r = x - g * k;
        dst[(int64_t)g * kp + r] = s_sel[r];
    }
}

// Phi(u) and phi(u) of the standard normal from one exponential: the tail
// Phi(-x) = phi(x) R(x), x = |u|, with R the Mills ratio in the rational form
// t P(t), t = 1 / (1 + x / 4) (coefficients fitted by gen_mills_ratio.py;
// fp32 relative error of R below 6e-7).  phi's argument -x^2 / 2 is taken
// with its rounding error (x^2 = x2 + x2e exactly), so phi keeps expf's
// accuracy for large x.
__device__ __forceinline__ float2 normal_cdf_pdf(float u) {
    const float x = fabsf(u);
    const float x2 = x * x;
    const float x2e = fmaf(x, x, -x2);
    const float phi = 0.398942280f * expf(-0.5f * x2) * fmaf(-0.5f, x2e, 1.f);
    const float t = __fdividef(1.f, fmaf(kMillsMap, x, 1.f));
    float p = kMillsP[kMillsDegree];
#pragma unroll
    for (int i = kMillsDegree - 1; i >= 0; --i) p = fmaf(p, t, kMillsP[i]);
    const float tail = phi * (t * p);
    return make_float2(u < 0.f ? tail : 1.f - tail, phi);
}

// E[(Y - tau)_+^e] and its derivative magnitude -dE/dtau for Y ~ N(mu, sig^2):
//   e = 2: E = (a^2 + sig^2) Phi(u) + a sig phi(u),   -dE = 2 (a Phi(u) + sig phi(u))
//   e = 1: E = a Phi(u) + sig phi(u),                  -dE = Phi(u)
// with a = mu - tau, u = a / sig; sig = 0 gives (a)_+^e.
// Also returns the second derivative d2E/dtau^2 (z): e = 2: 2 Phi(u);
// e = 1: phi(u) / sig (sig = 0: 2 [a > 0] and 0, the kinks aside).
template <int E>
__device__ __forceinline__ float3 gauss_moment(float mu, float sig, float tau) {
    const float a = mu - tau;
    if (!(sig > 0.f)) {
        const float ap = fmaxf(a, 0.f);
        return E == 2 ? make_float3(ap * ap, 2.f * ap, a > 0.f ? 2.f : 0.f)
                      : make_float3(ap, a > 0.f ? 1.f : 0.f, 0.f);
    }
    const float u = a / sig;
    const float2 cp = normal_cdf_pdf(u);
    const float Phi = cp.x, phi = cp.y;
    const float m1 = fmaf(a, Phi, sig * phi);
    if (E == 2)
        return make_float3(fmaf(fmaf(a, a, sig * sig), Phi, a * sig * phi), 2.f * m1, 2.f * Phi);
    return make_float3(m1, Phi, phi / sig);
}

template <int E>
__global__ void __launch_bounds__(kSelThreads, 2)
select_gauss_kernel(const float* __restrict__ ms, KV kv, int Hq, int cap, float alpha,
                    float delta, int32_t* __restrict__ sel, int32_t* __restrict__ n_sel,
                    float* __restrict__ aux) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ SelShared sh;
    __shared__ float4 fred[32];
    __shared__ float fmaxred[32];
    const int nw = blockDim.x >> 5;
    int* whist = reinterpret_cast<int*>(smem_raw);
    int* hist = whist + nw * 256;
    const int np_max = kv.maxp;
    float* s_mu = reinterpret_cast<float*>(hist + 256);
    float* s_sg = s_mu + np_max;
    float* s_n = s_sg + np_max;
    uint32_t* keys = reinterpret_cast<uint32_t*>(s_n + np_max);

    const int bh = blockIdx.x;
    const int b = bh / Hq;
    const int len = kv.sl[b];
    const int np = min(kv.maxp, (len + kv.P - 1) / kv.P);
    const float c = alpha - 1.f;
    const float* src = ms + (int64_t)bh * kv.maxp * 2;
    float mu_max = -INFINITY;
    for (int p = threadIdx.x; p < np; p += blockDim.x) {
        const float m = src[2 * p], s = src[2 * p + 1];
        const int n = min(kv.P, len - p * kv.P);
        const float zmax = n > 1 ? fmaf(sqrtf(2.f * logf(static_cast<float>(n))), s, m) : m;
        s_mu[p] = c * m;
        s_sg[p] = c * s;
        s_n[p] = static_cast<float>(n);
        keys[p] = float_key(zmax);
        mu_max = fmaxf(mu_max, c * m);
    }
    mu_max = block_max(mu_max, fmaxred);
    if (np <= 0) {
        if (threadIdx.x == 0) {
            n_sel[bh] = 0;
            if (aux) { aux[2 * bh] = INFINITY; aux[2 * bh + 1] = 0.f; }
        }
        return;
    }

    // safeguarded Halley iteration on the convex, decreasing F (F, its slope
    // -dF and curvature H come from the same pass over the pages).  mu_max - 1
    // is a lower bound of the root: the page holding mu_max alone gives
    // E[(X - mu_max + 1)_+^e] >= 1 by Jensen.  Starting at mu_max, where
    // the roots of these score distributions sit within a fraction of 1,
    // saves the climb from the bound.
    float lo = mu_max - 1.f, hi = INFINITY, tau = mu_max;
    for (int it = 0; it < 64; ++it) {
        float3 acc = make_float3(0.f, 0.f, 0.f);
        for (int p = threadIdx.x; p < np; p += blockDim.x) {
            const float3 v = gauss_moment<E>(s_mu[p], s_sg[p], tau);
            acc.x = fmaf(s_n[p], v.x, acc.x);
            acc.y = fmaf(s_n[p], v.y, acc.y);
            acc.z = fmaf(s_n[p], v.z, acc.z);
        }
        acc = block_sum3(acc, fred);
        const float F = acc.x - 1.f, dF = acc.y, H = acc.z;
        if (F == 0.f) break;                       // tau is the root
        if (F > 0.f) lo = tau; else hi = tau;
        // tau's resolution: 1e-7 relative, but never below two units in the
        // last place of tau (with a finer bound, a root just above a power of
        // two leaves tau stepping between neighbouring floats)
        const float at = fabsf(tau);
        const float ulp = __int_as_float(__float_as_int(at) & 0x7f800000) * 1.1920929e-7f;
        const float tol = fmaxf(1e-7f * fmaxf(1.f, at), 2.f * ulp);
        if (hi - lo <= tol) break;                 // bracketed to that resolution
        if (dF > 0.f) {
            // Halley's step; Newton's (never past the root from the left)
            // where the curvature term would turn it round
            const float den = 2.f * dF * dF - F * H;
            const float nxt = den > 0.f ? tau + 2.f * F * dF / den : tau + F / dF;
            if (fabsf(nxt - tau) <= tol) {         // converged (to fp32 resolution)
                if (nxt > lo && nxt < hi) tau = nxt;
                break;
            }
            if (nxt > lo && nxt < hi) { tau = nxt; continue; }
        }
        if (hi < INFINITY) {
            tau = 0.5f * (lo + hi);                // safeguard: bisect the bracket
        } else {
            tau = lo + fmaxf(1.f, 2.f * (lo - (mu_max - 1.f)));   // no upper end yet: expand
        }
    }
    const float tau_hat = tau;

    // threshold test; the uint32 key of a page that fails is 0 (below all)
    int pass = 0;
    for (int p = threadIdx.x; p < np; p += blockDim.x) {
        const float zmax = key_float(keys[p]);
        const bool ok = c * zmax >= tau_hat - delta;
        pass += ok;
        if (!ok) keys[p] = 0u;
    }
    pass = block_sum_i(pass, sh.red);
    int32_t* dst = sel + (int64_t)bh * cap;
    uint32_t kth = 1u;   // every passing page has a key >= 1
    int take_eq = 0;
    if (pass > cap) {
        radix_kth(keys, np, cap, whist, hist, sh, kth, take_eq);
    } else if (pass == 0) {
        // no page clears the threshold: keep the argmax estimated max (lowest id)
        for (int p = threadIdx.x; p < np; p += blockDim.x) {
            const int n = min(kv.P, len - p * kv.P);
            const float m = src[2 * p], s = src[2 * p + 1];
            keys[p] = float_key(n > 1 ? fmaf(sqrtf(2.f * logf(static_cast<float>(n))), s, m) : m);
        }
        radix_kth(keys, np, 1, whist, hist, sh, kth, take_eq);
    }
    uint32_t next_key;
    const int got = compact_topk(keys, np, kth, take_eq, dst, sh, &next_key);
    if (threadIdx.x == 0) {
        n_sel[bh] = got;
        if (aux) { aux[2 * bh] = tau_hat; aux[2 * bh + 1] = static_cast<float>(pass); }
    }
}

static int max_optin_smem() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 48 * 1024;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 48 * 1024;
    return v;
}

cudaError_t launch_select_topk(const float* bound, const KV& kv, int Hq, int kp, int32_t* sel,
                               int32_t* n_sel, float* aux, bool shared, cudaStream_t s) {
    // shared: one CTA per (sequence, kv head), G times fewer CTAs, so each
    // gets the most threads
    const int threads = shared ? 1024 : (kv.maxp <= 8192 ? 512 : 1024);
    const size_t smem = (size_t)kv.maxp * 4 + (size_t)kp * 4;
    if ((int)smem > max_optin_smem() - 4096) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int gs = shared ? Hq / kv.hkv : 0;
    return launch_kernel(select_topk_kernel, dim3(shared ? kv.B * kv.hkv : kv.B * Hq), dim3(threads),
                         smem, s, bound, kv, Hq, kp, sel, n_sel, aux, gs);
}

cudaError_t launch_select_gauss(const float* ms, const KV& kv, int Hq, int cap, float alpha,
                                float delta, int32_t* sel, int32_t* n_sel, float* aux,
                                cudaStream_t s) {
    const int threads = kSelThreads;
    const size_t smem = (size_t)(threads / 32) * 256 * 4 + 256 * 4 + (size_t)kv.maxp * 16;
    if ((int)smem > max_optin_smem() - 1024) return cudaErrorInvalidValue;
    const bool e2 = fabsf(alpha - 1.5f) < 1e-6f;
    cudaError_t e;
    if (e2) {
        e = cudaFuncSetAttribute(select_gauss_kernel<2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = launch_kernel(select_gauss_kernel<2>, dim3(kv.B * Hq), dim3(threads), smem, s, ms, kv,
                          Hq, cap, alpha, delta, sel, n_sel, aux);
        if (e != cudaSuccess) return e;
    } else {
        e = cudaFuncSetAttribute(select_gauss_kernel<1>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = launch_kernel(select_gauss_kernel<1>, dim3(kv.B * Hq), dim3(threads), smem, s, ms, kv,
                          Hq, cap, alpha, delta, sel, n_sel, aux);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace ekv
