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
#include <algorithm>

#include "common.cuh"
#include "mills_ratio.h"

EKV_DEFINE_STATUS(select)

#include "plan.cuh"

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

// ---------------------------------------------------------------------------
// Top-k by bound with register-resident keys (the default path).
//
// A CTA of kTkThreads threads holds up to kTkThreads * KPT keys, thread t the
// consecutive pages [t KPT, (t + 1) KPT) of its range, so the ascending page
// order of the output is the thread order.  The k-th largest key is found by
// an MSB radix select with 11-bit digits that starts at the highest bit where
// the range's keys differ and stops as soon as the boundary bin is taken whole
// (typically two passes over 4096 keys); ties at the k-th key go to the lower
// pages.  One packed block scan of (above, boundary-bin) counts places every
// taken page.
//
// Long sequences split their pages over a thread-block cluster of C <= 8
// CTAs: each CTA takes the top min(k, its pages) of its contiguous range and
// writes them, in page order, with their keys into the rank-0 CTA's shared
// memory (distributed shared memory); after one cluster barrier the rank-0
// CTA selects the k best of those candidates.  Every page of the global top k
// is in its range's top k (the order (bound desc, page asc) is total), so the
// result is the single-CTA one.
// ---------------------------------------------------------------------------
constexpr int kTkThreads = 512;
constexpr int kTkDigitBits = 11;
constexpr int kTkBins = 1 << kTkDigitBits;
constexpr int kTkMaxCluster = 8;

struct __align__(16) TkShared {
    int hist[2][kTkBins];            // one per radix pass, alternating (both zero between uses)
    int red[40];
    uint32_t umin[32], umax[32];
    int digit, above, nb;
    int cnt[kTkMaxCluster];          // rank-0 CTA: candidates each rank wrote
    uint32_t next[kTkMaxCluster];    // and the largest key each rank left out
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
                 ::: "memory");
}
// Split cluster barrier: arrive now, wait later (every CTA of the cluster has
// started once the wait returns, so its shared memory can be written).
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
// The same with release semantics: this thread's earlier shared-memory writes
// are visible to the cluster once the wait returns.
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// 32-bit store into the shared memory of CTA `rank` of this cluster, at the
// address `p` has in this CTA.
__device__ __forceinline__ void st_cluster_u32(const void* p, uint32_t rank, uint32_t v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}
// 32-bit OR into the shared memory of CTA `rank` (no value returned).
__device__ __forceinline__ void or_cluster_u32(const void* p, uint32_t rank, uint32_t v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(rank));
    asm volatile("red.shared::cluster.or.b32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// Block-wide min and max of one value per thread (every thread gets both).
__device__ __forceinline__ void tk_minmax(uint32_t& mn, uint32_t& mx, TkShared& sh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    __syncthreads();
    if (lane == 0) { sh.umin[wid] = mn; sh.umax[wid] = mx; }
    __syncthreads();
    mn = lane < nw ? sh.umin[lane] : 0xFFFFFFFFu;
    mx = lane < nw ? sh.umax[lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
}

// The boundary of the k largest among this block's valid keys (bit j of
// `valid` marks key[j]; 1 <= k <= the number of valid keys; kmn/kmx their
// extremes).  Key x is taken iff (x >> shift) > hi, or (x >> shift) == hi and
// fewer than takeB such keys precede it in key order.  Each radix pass costs
// two barriers: the histogram (alternating buffers, so the other one is
// cleared meanwhile), then warp 0 alone finds the boundary bin -- every lane
// sums its 64 consecutive bins, a suffix scan over the lanes picks the lane
// holding the boundary and the warp scans that lane's 64 bins.  Both
// histograms are zero on entry and are zero again before the next barrier
// the caller passes.
template <int KPT>
__device__ void tk_boundary(const uint32_t (&key)[KPT], uint32_t valid, int n, int k,
                            uint32_t kmn, uint32_t kmx, TkShared& sh, int& shift_out,
                            uint64_t& hi_out, int& takeB_out) {
    constexpr int BPL = kTkBins / 32;                   // bins per lane of warp 0
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const uint32_t diff = kmn ^ kmx;
    int shift = diff ? 32 - __clz(diff) : 0;
    uint64_t hi = (uint64_t)kmx >> shift;
    int rem = k, nB = n;
    int buf = 0;
    bool used = false;
    while (shift > 0 && nB != rem) {
        const int dbits = min(kTkDigitBits, shift);
        shift -= dbits;
        const uint32_t dmask = (1u << dbits) - 1u;
        int* hist = sh.hist[buf];
#pragma unroll
        for (int j = 0; j < KPT; ++j)
            if (((valid >> j) & 1u) && ((uint64_t)key[j] >> (shift + dbits)) == hi)
                atomicAdd(&hist[(key[j] >> shift) & dmask], 1);
        __syncthreads();
        if (wid == 0) {
            // lane's bins [lane BPL, +BPL) as 16-byte loads, rotated by the lane
            // (each quarter warp reads eight distinct bank groups)
            const int4* h4 = reinterpret_cast<const int4*>(hist + lane * BPL);
            int4 a4 = make_int4(0, 0, 0, 0);
#pragma unroll 4
            for (int i = 0; i < BPL / 4; ++i) {
                const int4 v4 = h4[(i + lane) & (BPL / 4 - 1)];
                a4.x += v4.x; a4.y += v4.y; a4.z += v4.z; a4.w += v4.w;
            }
            const int sum = (a4.x + a4.y) + (a4.z + a4.w);
            int incl = sum;                              // suffix sum over the lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_down_sync(0xFFFFFFFFu, incl, o);
                if (lane + o < 32) incl += v;
            }
            const int above_l = incl - sum;
            const uint32_t owner = __ballot_sync(0xFFFFFFFFu, above_l < rem && incl >= rem);
            const int L = __ffs(owner) - 1;              // exactly one lane
            const int base = __shfl_sync(0xFFFFFFFFu, above_l, L);
            // that lane's bins, two per lane, suffix-scanned
            const int b0 = L * BPL + 2 * lane;
            const int c0 = hist[b0], c1 = hist[b0 + 1];
            int pair = c0 + c1, pin = pair;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_down_sync(0xFFFFFFFFu, pin, o);
                if (lane + o < 32) pin += v;
            }
            int acc = base + pin - pair;                 // keys above this lane's two bins
            if (acc < rem && acc + c1 >= rem) { sh.digit = b0 + 1; sh.above = acc; sh.nb = c1; }
            acc += c1;
            if (acc < rem && acc + c0 >= rem) { sh.digit = b0; sh.above = acc; sh.nb = c0; }
        } else if (used) {
            // the other buffer, last read before the previous pass's second barrier
            int* other = sh.hist[buf ^ 1];
            for (int i = tid - 32; i < kTkBins; i += blockDim.x - 32) other[i] = 0;
        }
        __syncthreads();
        const int d = sh.digit;
        rem -= sh.above;
        nB = sh.nb;
        hi = (hi << dbits) | (uint64_t)d;
        buf ^= 1;
        used = true;
    }
    // leave both buffers zero: the last one (read before the barrier above)
    // and the other one if two or more passes ran
    if (used) {
        for (int i = tid; i < kTkBins; i += blockDim.x) sh.hist[buf ^ 1][i] = 0;
    }
    shift_out = shift;
    hi_out = hi;
    takeB_out = rem;
}

// Output positions of this thread's taken keys (in key order) given the
// boundary; calls f(j, pos) for each taken key j, then a barrier.  Also
// returns this thread's smallest taken and largest untaken valid key
// (0xFFFFFFFF / 0 if none): tk_minmax of them gives the block's.
template <int KPT, typename F>
__device__ __forceinline__ void tk_place(const uint32_t (&key)[KPT], uint32_t valid, int shift,
                                         uint64_t hi, int takeB, TkShared& sh, F&& f,
                                         uint32_t& tmin, uint32_t& nmax) {
    int a = 0, b = 0;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
        if ((valid >> j) & 1u) {
            const uint64_t kh = (uint64_t)key[j] >> shift;
            a += kh > hi;
            b += kh == hi;
        }
    int total;
    const int pre = block_exclusive_scan(a | (b << 16), sh.red, &total);
    int ra = pre & 0xFFFF, rb = pre >> 16;
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
        if ((valid >> j) & 1u) {
            const uint64_t kh = (uint64_t)key[j] >> shift;
            bool take = false;
            if (kh > hi) {
                f(j, ra + min(rb, takeB));
                ++ra;
                take = true;
            } else if (kh == hi) {
                if (rb < takeB) { f(j, ra + rb); take = true; }
                ++rb;
            }
            if (take) mn = min(mn, key[j]); else mx = max(mx, key[j]);
        }
    __syncthreads();
    tmin = mn;
    nmax = mx;
}

// gs = 0: one head per CTA (csize CTAs per head); gs > 0: one (sequence, kv
// head) per CTA group, keys = the largest bound of the group's gs query heads,
// result written to every head of the group.  Dynamic shared memory: [kp]
// ints (the output row), then, for csize > 1, the rank-0 candidate arrays
// [C][slot] keys and pages.
//
// PG > 0 (csize = 1, PG = the group size): the selection also builds the
// decode's union plan of each kv head (plan_from_bits) in the decode
// workspace `ws`.  Per-head selections run as a cluster of the group's PG
// CTAs: each ORs its pages into its bitmap in the rank-0 CTA's shared memory,
// and the rank-0 CTA, which copied its sequence's page-table row into shared
// memory at the start, builds the plan.  Shared selections set every head's
// bitmap from the CTA's own row.  Dynamic shared memory then also holds
// [PG][max_pages / 32] bitmap words and the [max_pages] page -> block map.
template <int KPT, int PG>
__global__ void __launch_bounds__(kTkThreads, 2)
select_topk_reg_kernel(const float* __restrict__ bound, KV kv, int Hq, int kp,
                       int32_t* __restrict__ sel, int32_t* __restrict__ n_sel,
                       float* __restrict__ aux, int gs, int csize, WS ws, DecodeLayout L) {
    extern __shared__ __align__(16) int32_t s_row[];
    __shared__ TkShared sh;
    const int tid = threadIdx.x;
    const int ng = gs > 0 ? gs : 1;
    const int unit = blockIdx.x / csize;
    const uint32_t rank = csize > 1 ? cluster_rank() : 0u;
    const int bh = gs > 0 ? (unit / kv.hkv) * Hq + (unit % kv.hkv) * gs : unit;
    const int b = bh / Hq;
    // the CTA's range is fixed by max_pages, so the bounds are loaded (in
    // bounds of the row) while the sequence length is still in flight; keys
    // past the sequence's pages are masked out below
    const int chunk = ((kv.maxp + csize - 1) / csize + 3) & ~3;    // a multiple of 4 pages
    const int p0 = (int)rank * chunk;
    const int span = max(0, min(kv.maxp - p0, chunk));
    const float* src = bound + (int64_t)bh * kv.maxp + p0;
    // plan mode: the unit, this CTA's head within it (its cluster rank), and
    // the rank-0 CTA's [PG][nwm] bitmaps and page -> block map (the sequence's
    // page-table row, an input of the step rather than the previous kernel's
    // output: copied in before the wait, checked where used)
    const int pu = gs > 0 ? unit : bh / (PG > 0 ? PG : 1);
    const uint32_t prank = (PG > 1 && gs == 0) ? cluster_rank() : 0u;
    const int nwm = (kv.maxp + 31) / 32;
    uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_row + kp);
    int* s_pblk = reinterpret_cast<int*>(
        (reinterpret_cast<uintptr_t>(s_bits + PG * nwm) + 15) & ~static_cast<uintptr_t>(15));
    if constexpr (PG > 0) {
        if (prank == 0) {
            const int32_t* pt = kv.pt + (int64_t)b * kv.maxp;
            const bool vec = (kv.maxp & 3) == 0 && (reinterpret_cast<uintptr_t>(kv.pt) & 15) == 0;
            if (vec) {
                for (int i = tid * 4; i < kv.maxp; i += kTkThreads * 4) cp_async16_zfill(s_pblk + i, pt + i, 16);
            } else {
                for (int i = tid; i < kv.maxp; i += kTkThreads) s_pblk[i] = __ldg(pt + i);
            }
            // cleared before the cluster barrier's arrive
            for (int i = tid; i < PG * nwm; i += kTkThreads) s_bits[i] = 0u;
        }
    }
    // the bound rows are still being written: only their lines' translation
    // and L2 placement are requested; the sequence length is an input
    {
        const int lines = (span + 31) / 32;
        for (int x = tid; x < ng * lines; x += kTkThreads) {
            const int g = x / lines;
            prefetch_l2_line(src + (int64_t)g * kv.maxp + (x - g * lines) * 32);
        }
    }
    const int seq_len = __ldg(kv.sl + b);
    pdl_wait();                         // the bounds are the previous kernel's output
    float v[KPT];
    {
        const bool vec = (kv.maxp & 3) == 0;
        for (int g = 0; g < ng; ++g) {
            const float* rs = src + (int64_t)g * kv.maxp;
#pragma unroll
            for (int j = 0; j < KPT; j += 4) {
                const int i = tid * KPT + j;
                float4 f;
                if (vec && i + 3 < span) {
                    f = __ldcg(reinterpret_cast<const float4*>(rs + i));
                } else {
                    f.x = i < span ? __ldcg(rs + i) : -INFINITY;
                    f.y = i + 1 < span ? __ldcg(rs + i + 1) : -INFINITY;
                    f.z = i + 2 < span ? __ldcg(rs + i + 2) : -INFINITY;
                    f.w = i + 3 < span ? __ldcg(rs + i + 3) : -INFINITY;
                }
                if (g == 0) {
                    v[j] = f.x; v[j + 1] = f.y; v[j + 2] = f.z; v[j + 3] = f.w;
                } else {       // shared: the group's largest bound
                    v[j] = fmaxf(v[j], f.x); v[j + 1] = fmaxf(v[j + 1], f.y);
                    v[j + 2] = fmaxf(v[j + 2], f.z); v[j + 3] = fmaxf(v[j + 3], f.w);
                }
            }
        }
    }
    const int np = min(kv.maxp, (seq_len + kv.P - 1) / kv.P);
    const int k = min(kp, np);
    if constexpr (PG > 0) {
        if (prank == 0) plan_reset_unit(Hq, PG, ws, L, kv, pu);
    }
    if (k <= 0) {                       // the same for every CTA of the cluster
        if (rank == 0 && tid < ng) {
            n_sel[bh + tid] = 0;
            if (aux) { aux[2 * (bh + tid)] = INFINITY; aux[2 * (bh + tid) + 1] = -INFINITY; }
        }
        if constexpr (PG > 0) {
            if (prank == 0) {
                if (tid == 0) ws.union_count[pu] = 0;             // an empty plan
                cp_async_wait_all();    // no copy into shared memory outlives the CTA
            }
        }
        return;
    }
    // waited for before the first remote store (plan mode: the bitmaps were
    // cleared before it)
    if (PG > 1 && gs == 0) cluster_arrive_release();
    else if (csize > 1) cluster_arrive_relaxed();
    const int n_loc = max(0, min(np - p0, chunk));
    for (int i = tid; i < 2 * kTkBins; i += kTkThreads) (&sh.hist[0][0])[i] = 0;

    // this thread's keys: pages p0 + [tid KPT, (tid + 1) KPT)
    uint32_t key[KPT];
    uint32_t valid = 0u;
    {
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
            key[j] = float_key(v[j]);
            if (tid * KPT + j < n_loc) valid |= 1u << j;
        }
    }
    uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
        if ((valid >> j) & 1u) { kmn = min(kmn, key[j]); kmx = max(kmx, key[j]); }
    tk_minmax(kmn, kmx, sh);

    const int k_loc = min(kp, n_loc);
    int shift, takeB;
    uint64_t hi;
    uint32_t tmin, nmax;
    if (csize == 1) {
        tk_boundary<KPT>(key, valid, n_loc, k_loc, kmn, kmx, sh, shift, hi, takeB);
        tk_place<KPT>(key, valid, shift, hi, takeB, sh,
                      [&](int j, int pos) { s_row[pos] = tid * KPT + j; }, tmin, nmax);
        // tk_place ends with a barrier: s_row is complete
        pdl_trigger();
        if constexpr (PG > 0) {
            if (gs > 0 || PG == 1) {
                // one row for every head of the group
                for (int r = tid; r < k; r += kTkThreads) {
                    const int p = s_row[r];
#pragma unroll
                    for (int g = 0; g < PG; ++g) atomicOr(&s_bits[g * nwm + (p >> 5)], 1u << (p & 31));
                }
                cp_async_wait_all();    // this thread's part of the page -> block map
                __syncthreads();
            } else {
                cluster_wait();         // every CTA of the cluster is running, bitmaps clear
                // the row into this head's bitmap in the rank-0 CTA
                for (int r = tid; r < k; r += kTkThreads) {
                    const int p = s_row[r];
                    or_cluster_u32(s_bits + prank * nwm + (p >> 5), 0u, 1u << (p & 31));
                }
                if (prank == 0) cp_async_wait_all();   // this thread's part of the map
                cluster_sync_all();     // the bitmaps are in the rank-0 CTA, its map complete
            }
        }
        for (int x = tid; x < ng * k; x += kTkThreads) {
            const int g = x / k, r = x - g * k;
            sel[(int64_t)(bh + g) * kp + r] = s_row[r];
        }
        if (tid < ng) n_sel[bh + tid] = k;
        if constexpr (PG > 0) {
            // nothing reads another CTA's memory past the cluster barrier
            if (prank == 0) plan_from_bits<PG>(kv, ws, L, pu, s_bits, nullptr, sh.red, s_pblk);
        }
        if (aux) {                      // off the critical path: the boundary keys
            tk_minmax(tmin, nmax, sh);
            if (tid < ng) {
                aux[2 * (bh + tid)] = key_float(tmin);
                aux[2 * (bh + tid) + 1] = k < np ? key_float(nmax) : -INFINITY;
            }
        }
        return;
    }

    // cluster: this range's top k_loc, in page order, to the rank-0 CTA
    const int slot = min(kp, chunk);
    uint32_t* c_key = reinterpret_cast<uint32_t*>(s_row + kp);
    int32_t* c_page = reinterpret_cast<int32_t*>(c_key + csize * slot);
    cluster_wait();                     // every CTA of the cluster is running
    if (n_loc > 0) {
        tk_boundary<KPT>(key, valid, n_loc, k_loc, kmn, kmx, sh, shift, hi, takeB);
        tk_place<KPT>(key, valid, shift, hi, takeB, sh,
                      [&](int j, int pos) {
                          st_cluster_u32(c_key + rank * slot + pos, 0u, key[j]);
                          st_cluster_u32(c_page + rank * slot + pos, 0u,
                                         static_cast<uint32_t>(p0 + tid * KPT + j));
                      }, tmin, nmax);
        tk_minmax(tmin, nmax, sh);
    } else {
        nmax = 0u;
    }
    if (tid == 0) {
        st_cluster_u32(&sh.cnt[rank], 0u, static_cast<uint32_t>(k_loc > 0 ? k_loc : 0));
        st_cluster_u32(&sh.next[rank], 0u, k_loc < n_loc ? nmax : 0u);
    }
    cluster_sync_all();                 // candidates visible in the rank-0 CTA
    pdl_trigger();
    if (rank != 0) return;              // nothing reads another CTA's memory past here

    // rank 0: the k best of the candidates; flat position x = r * slot + i
    // (i < cnt[r]) is ascending in page order
    uint32_t ck[KPT];
    uint32_t cvalid = 0u;
    int m = 0;
    uint32_t out_next = 0u;
    for (int r = 0; r < csize; ++r) { m += sh.cnt[r]; out_next = max(out_next, sh.next[r]); }
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const int x = tid * KPT + j;
        const int r = x / slot, i = x - r * slot;
        ck[j] = 0u;
        if (r < csize && i < sh.cnt[r]) { ck[j] = c_key[x]; cvalid |= 1u << j; }
    }
    kmn = 0xFFFFFFFFu;
    kmx = 0u;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
        if ((cvalid >> j) & 1u) { kmn = min(kmn, ck[j]); kmx = max(kmx, ck[j]); }
    tk_minmax(kmn, kmx, sh);
    tk_boundary<KPT>(ck, cvalid, m, k, kmn, kmx, sh, shift, hi, takeB);
    tk_place<KPT>(ck, cvalid, shift, hi, takeB, sh,
                  [&](int j, int pos) { s_row[pos] = c_page[tid * KPT + j]; }, tmin, nmax);
    tk_minmax(tmin, nmax, sh);
    for (int x = tid; x < ng * k; x += kTkThreads) {
        const int g = x / k, r = x - g * k;
        sel[(int64_t)(bh + g) * kp + r] = s_row[r];
    }
    if (tid < ng) {
        n_sel[bh + tid] = k;
        if (aux) {
            aux[2 * (bh + tid)] = key_float(tmin);
            aux[2 * (bh + tid) + 1] = k < np ? key_float(max(nmax, out_next)) : -INFINITY;
        }
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
__device__ __forceinline__ float3 gauss_moment(float mu, float sig, float isig, float tau) {
    const float a = mu - tau;
    if (!(sig > 0.f)) {
        const float ap = fmaxf(a, 0.f);
        return E == 2 ? make_float3(ap * ap, 2.f * ap, a > 0.f ? 2.f : 0.f)
                      : make_float3(ap, a > 0.f ? 1.f : 0.f, 0.f);
    }
    const float u = a * isig;
    const float2 cp = normal_cdf_pdf(u);
    const float Phi = cp.x, phi = cp.y;
    const float m1 = fmaf(a, Phi, sig * phi);
    if (E == 2)
        return make_float3(fmaf(fmaf(a, a, sig * sig), Phi, a * sig * phi), 2.f * m1, 2.f * Phi);
    return make_float3(m1, Phi, phi * isig);
}

template <int E, int KPT>
__global__ void __launch_bounds__(kSelThreads, 2)
select_gauss_kernel(const float* __restrict__ ms, KV kv, int Hq, int cap, float alpha,
                    float delta, int32_t* __restrict__ sel, int32_t* __restrict__ n_sel,
                    float* __restrict__ aux) {
    // shared layout: the top-k scratch (TkShared), then per page: scaled mean,
    // scaled std, its reciprocal, key
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ SelShared sh;
    __shared__ float4 fred[32];
    __shared__ float fmaxred[32];
    TkShared& tsh = *reinterpret_cast<TkShared*>(smem_raw);
    const int np_max = kv.maxp;
    float* s_mu = reinterpret_cast<float*>(smem_raw + sizeof(TkShared));
    float* s_sg = s_mu + np_max;
    float* s_isg = s_sg + np_max;
    uint32_t* keys = reinterpret_cast<uint32_t*>(s_isg + np_max);

    const int bh = blockIdx.x;
    const int b = bh / Hq;
    const int len = kv.sl[b];
    const int np = min(kv.maxp, (len + kv.P - 1) / kv.P);
    const float c = alpha - 1.f;
    const float* src = ms + (int64_t)bh * kv.maxp * 2;
    pdl_wait();                         // the page scores are the previous kernel's output
    float mu_max = -INFINITY;
    // every page's (m, s) in flight at once (KPT pages per thread, strided)
    float2 msv[KPT];
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const int p = j * kSelThreads + threadIdx.x;
        msv[j] = p < np ? __ldcg(reinterpret_cast<const float2*>(src) + p) : make_float2(0.f, 0.f);
    }
    const float zfull = sqrtf(2.f * logf(static_cast<float>(kv.P)));   // a full page's factor
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const int p = j * kSelThreads + threadIdx.x;
        if (p >= np) continue;
        const float m = msv[j].x, s = msv[j].y;
        const int n = min(kv.P, len - p * kv.P);
        const float zf = n == kv.P ? zfull : (n > 1 ? sqrtf(2.f * logf(static_cast<float>(n))) : 0.f);
        const float zmax = n > 1 ? fmaf(zf, s, m) : m;
        s_mu[p] = c * m;
        s_sg[p] = c * s;
        s_isg[p] = c * s > 0.f ? __frcp_rn(c * s) : 0.f;
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
            const float3 v = gauss_moment<E>(s_mu[p], s_sg[p], s_isg[p], tau);
            const float n = static_cast<float>(min(kv.P, len - p * kv.P));   // tokens of the page
            acc.x = fmaf(n, v.x, acc.x);
            acc.y = fmaf(n, v.y, acc.y);
            acc.z = fmaf(n, v.z, acc.z);
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
    pdl_trigger();                      // the decode's CTAs may take their places

    // threshold test; the uint32 key of a page that fails is 0 (below all)
    int pass = 0;
    for (int p = threadIdx.x; p < np; p += blockDim.x) {
        const float zmax = key_float(keys[p]);
        const bool ok = c * zmax >= tau_hat - delta;
        pass += ok;
        if (!ok) keys[p] = 0u;
    }
    pass = block_sum_i(pass, sh.red);
    if (pass == 0) {
        // no page clears the threshold: keep the argmax estimated max (lowest id)
        for (int p = threadIdx.x; p < np; p += blockDim.x) {
            const int n = min(kv.P, len - p * kv.P);
            const float m = src[2 * p], s = src[2 * p + 1];
            keys[p] = float_key(n > 1 ? fmaf(sqrtf(2.f * logf(static_cast<float>(n))), s, m) : m);
        }
    }
    // the k largest keys (failing pages hold 0, below every passing key), in
    // page order, with the register-resident radix boundary of the top-k
    // selection: pages [tid KPT, (tid + 1) KPT) per thread
    const int k = pass > cap ? cap : (pass == 0 ? 1 : pass);
    for (int i = threadIdx.x; i < 2 * kTkBins; i += blockDim.x) (&tsh.hist[0][0])[i] = 0;
    __syncthreads();
    uint32_t key[KPT];
    uint32_t valid = 0u;
    uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
        const int p = threadIdx.x * KPT + j;
        key[j] = p < np ? keys[p] : 0u;
        if (p < np) {
            valid |= 1u << j;
            kmn = min(kmn, key[j]);
            kmx = max(kmx, key[j]);
        }
    }
    tk_minmax(kmn, kmx, tsh);
    int shift, takeB;
    uint64_t bhi;
    uint32_t tmin, nmax;
    tk_boundary<KPT>(key, valid, np, k, kmn, kmx, tsh, shift, bhi, takeB);
    int32_t* dst = sel + (int64_t)bh * cap;
    tk_place<KPT>(key, valid, shift, bhi, takeB, tsh,
                  [&](int j, int pos) { dst[pos] = threadIdx.x * KPT + j; }, tmin, nmax);
    if (threadIdx.x == 0) {
        n_sel[bh] = k;
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

template <int KPT, int PG>
static cudaError_t launch_topk_reg(const float* bound, const KV& kv, int Hq, int kp,
                                   int32_t* sel, int32_t* n_sel, float* aux, int gs, int units,
                                   int csize, const WS& ws, const DecodeLayout& L,
                                   cudaStream_t s) {
    const int chunk = ((kv.maxp + csize - 1) / csize + 3) & ~3;   // as the kernel rounds
    if (chunk > kTkThreads * KPT) return kShapeUnsupported;
    const int slot = std::min(kp, chunk);
    if (csize > 1 && csize * slot > kTkThreads * KPT) return kShapeUnsupported;
    size_t smem = (size_t)kp * 4 + (csize > 1 ? (size_t)csize * slot * 8 : 0);
    if (PG > 0)   // [PG][nwm] bitmaps, [max_pages] page -> block (16-byte aligned)
        smem = ((smem + (size_t)PG * ((kv.maxp + 31) / 32) * 4 + 15) & ~size_t(15)) +
               (size_t)kv.maxp * 4;
    if (smem > 96 * 1024) return kShapeUnsupported;
    auto kernel = select_topk_reg_kernel<KPT, PG>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int cl = PG > 1 && gs == 0 ? PG : csize;     // CTAs per cluster
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(units * csize);
    cfg.blockDim = dim3(kTkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cl > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, bound, kv, Hq, kp, sel, n_sel, aux, gs, csize, ws, L);
}

template <int KPT>
static cudaError_t launch_topk_reg_plan(const float* bound, const KV& kv, int Hq, int kp,
                                        int32_t* sel, int32_t* n_sel, float* aux, int gs,
                                        int units, int csize, const WS* ws,
                                        const DecodeLayout* L, bool* planned, cudaStream_t s) {
    if (ws && csize == 1) {
        const int G = Hq / kv.hkv;
        cudaError_t e = kShapeUnsupported;
        switch (G) {
            case 1: e = launch_topk_reg<KPT, 1>(bound, kv, Hq, kp, sel, n_sel, aux, gs, units, 1, *ws, *L, s); break;
            case 2: e = launch_topk_reg<KPT, 2>(bound, kv, Hq, kp, sel, n_sel, aux, gs, units, 1, *ws, *L, s); break;
            case 4: e = launch_topk_reg<KPT, 4>(bound, kv, Hq, kp, sel, n_sel, aux, gs, units, 1, *ws, *L, s); break;
            case 8: e = launch_topk_reg<KPT, 8>(bound, kv, Hq, kp, sel, n_sel, aux, gs, units, 1, *ws, *L, s); break;
            default: break;
        }
        if (e != kShapeUnsupported) {
            if (e == cudaSuccess) *planned = true;
            return e;
        }
    }
    return launch_topk_reg<KPT, 0>(bound, kv, Hq, kp, sel, n_sel, aux, gs, units, csize, WS{},
                                   DecodeLayout{}, s);
}

cudaError_t launch_select_topk(const float* bound, const KV& kv, int Hq, int kp, int32_t* sel,
                               int32_t* n_sel, float* aux, bool shared, cudaStream_t s,
                               void* plan_ws, const DecodeLayout* plan_layout, bool* planned) {
    const int gs = shared ? Hq / kv.hkv : 0;
    const int units = shared ? kv.B * kv.hkv : kv.B * Hq;
    WS wsv{};
    const WS* ws = nullptr;
    if (plan_ws && plan_layout && planned) {
        wsv = ws_views(plan_ws, *plan_layout);
        ws = &wsv;
        *planned = false;
    }
    // register-resident keys: at most 4096 pages per CTA, longer sequences
    // split over a cluster of up to 8 CTAs
    int csize = 1;
    while (csize < kTkMaxCluster && (kv.maxp + csize - 1) / csize > 4096) csize *= 2;
    const int chunk = ((kv.maxp + csize - 1) / csize + 3) & ~3;
    cudaError_t e = kShapeUnsupported;
    if (chunk <= kTkThreads * 4)
        e = launch_topk_reg_plan<4>(bound, kv, Hq, kp, sel, n_sel, aux, gs, units, csize, ws,
                                    plan_layout, planned, s);
    else if (chunk <= kTkThreads * 8)
        e = launch_topk_reg_plan<8>(bound, kv, Hq, kp, sel, n_sel, aux, gs, units, csize, ws,
                                    plan_layout, planned, s);
    if (e == kShapeUnsupported && chunk <= kTkThreads * 16)
        e = launch_topk_reg_plan<16>(bound, kv, Hq, kp, sel, n_sel, aux, gs, units, csize, ws,
                                     plan_layout, planned, s);
    if (e != kShapeUnsupported) return e;

    // large budgets: keys in shared memory, one CTA per head
    const int threads = shared ? 1024 : (kv.maxp <= 8192 ? 512 : 1024);
    const size_t smem = (size_t)kv.maxp * 4 + (size_t)kp * 4;
    if ((int)smem > max_optin_smem() - 4096) return kShapeUnsupported;
    e = cudaFuncSetAttribute(select_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(select_topk_kernel, dim3(units), dim3(threads), smem, s, bound, kv, Hq,
                         kp, sel, n_sel, aux, gs);
}

template <int E, int KPT>
static cudaError_t launch_gauss_t(const float* ms, const KV& kv, int Hq, int cap, float alpha,
                                  float delta, int32_t* sel, int32_t* n_sel, float* aux, size_t smem,
                                  cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(select_gauss_kernel<E, KPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel_pdl(select_gauss_kernel<E, KPT>, dim3(kv.B * Hq), dim3(kSelThreads), smem,
                             s, ms, kv, Hq, cap, alpha, delta, sel, n_sel, aux);
}

cudaError_t launch_select_gauss(const float* ms, const KV& kv, int Hq, int cap, float alpha,
                                float delta, int32_t* sel, int32_t* n_sel, float* aux,
                                cudaStream_t s) {
    const size_t smem = sizeof(TkShared) + (size_t)kv.maxp * 16;
    if ((int)smem > max_optin_smem() - 1024 || kv.maxp > kSelThreads * 24) return kShapeUnsupported;
    const bool e2 = fabsf(alpha - 1.5f) < 1e-6f;
    if (kv.maxp <= kSelThreads * 8)
        return e2 ? launch_gauss_t<2, 8>(ms, kv, Hq, cap, alpha, delta, sel, n_sel, aux, smem, s)
                  : launch_gauss_t<1, 8>(ms, kv, Hq, cap, alpha, delta, sel, n_sel, aux, smem, s);
    if (kv.maxp <= kSelThreads * 16)
        return e2 ? launch_gauss_t<2, 16>(ms, kv, Hq, cap, alpha, delta, sel, n_sel, aux, smem, s)
                  : launch_gauss_t<1, 16>(ms, kv, Hq, cap, alpha, delta, sel, n_sel, aux, smem, s);
    return e2 ? launch_gauss_t<2, 24>(ms, kv, Hq, cap, alpha, delta, sel, n_sel, aux, smem, s)
              : launch_gauss_t<1, 24>(ms, kv, Hq, cap, alpha, delta, sel, n_sel, aux, smem, s);
}

}  // namespace ekv
