// alpha-entmax attention over the selected pages [EntmaxKV §2.C].
//
// Work unit u = (sequence b, kv head): its G query heads each selected their
// own pages; the unit reads the UNION of those pages once.
//
//   plan  (1 CTA per unit)      bitmaps of each head's pages -> union list in
//                               ascending page order, per-page head mask and
//                               each head's rank of the page.
//   qk    (CH pages per CTA)    bulk-copies K pages (cp.async.bulk, mbarrier
//                               pipeline) into shared memory; z' = (alpha-1)
//                               s q.k for the G heads with fp32 FMA (G <= 8
//                               rows are far too few for a tensor-core tile);
//                               each head's scores land in its own list.
//   tau   (1 CTA per head)      exact threshold: candidates z' > max - 1 are
//                               sorted (bitonic, shared memory); the closed
//                               form on the top-k prefix (alpha 2: sparsemax;
//                               alpha 1.5: quadratic) picks tau, polished by
//                               Newton steps on sum (z'-tau)_+^e = 1; other
//                               alpha: bisection.
//   pv    (CH pages per CTA)    p = (z' - tau)_+^(1/(alpha-1)); V pages with no
//                               positive weight for any head are never read;
//                               split-K partial sums, and the last CTA of the
//                               unit (atomic ticket) merges them in a fixed
//                               order: out = sum p v / sum p.  tau is global,
//                               so the merge is a plain sum.
#include "common.cuh"

EKV_DEFINE_STATUS(decode)

namespace ekv {

constexpr int kChunkPages = 16;   // union pages per qk / pv CTA
constexpr int kQkThreads = 256;
constexpr int kPvThreads = 256;
constexpr int kPlanThreads = 512;
constexpr int kTauThreads = 512;

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

DecodeLayout decode_layout(int B, int Hq, int Hkv, int D, int P, int max_pages, int cap) {
    DecodeLayout L{};
    L.U = B * Hkv;
    L.G = Hq / Hkv;
    L.Umax = std::min(L.G * cap, max_pages);
    L.CH = kChunkPages;
    L.Smax = (L.Umax + L.CH - 1) / L.CH;
    L.zcap = cap * P;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
    L.union_count = take(sizeof(int) * L.U);
    L.head_count = take(sizeof(int) * (size_t)B * Hq);
    L.counter = take(sizeof(int) * L.U);
    L.vpages = take(sizeof(int) * L.U);
    L.union_page = take(sizeof(int) * (size_t)L.U * L.Umax);
    L.union_mask = take(sizeof(int) * (size_t)L.U * L.Umax);
    L.union_rank = take(sizeof(int) * (size_t)L.U * L.Umax * L.G);
    L.z = take(sizeof(float) * (size_t)B * Hq * L.zcap);
    L.tau = take(sizeof(float) * (size_t)B * Hq);
    L.partial = take(sizeof(float) * (size_t)L.U * L.Smax * L.G * (D + 1));
    L.total = o;
    return L;
}

// Workspace views (device addresses).
struct WS {
    int* union_count;
    int* head_count;
    int* counter;
    int* vpages;
    int* union_page;
    int* union_mask;
    int* union_rank;
    float* z;
    float* tau;
    float* partial;
};
static WS ws_views(void* base, const DecodeLayout& L) {
    char* c = static_cast<char*>(base);
    return WS{reinterpret_cast<int*>(c + L.union_count), reinterpret_cast<int*>(c + L.head_count),
              reinterpret_cast<int*>(c + L.counter), reinterpret_cast<int*>(c + L.vpages),
              reinterpret_cast<int*>(c + L.union_page),
              reinterpret_cast<int*>(c + L.union_mask), reinterpret_cast<int*>(c + L.union_rank),
              reinterpret_cast<float*>(c + L.z), reinterpret_cast<float*>(c + L.tau),
              reinterpret_cast<float*>(c + L.partial)};
}

__device__ __forceinline__ int pages_of(const KV& kv, int b) {
    return min(kv.maxp, (kv.sl[b] + kv.P - 1) / kv.P);
}

// ---------------------------------------------------------------------------
// plan: union of the group's selections
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(KV kv, int Hq, const int32_t* __restrict__ sel, const int32_t* __restrict__ n_sel,
            int cap, WS ws, DecodeLayout L) {
    extern __shared__ __align__(16) uint32_t s_plan[];
    __shared__ int red[40];
    const int nwm = (kv.maxp + 31) / 32;
    uint32_t* bits = s_plan;                                        // [G][nwm]
    int* pre = reinterpret_cast<int*>(bits + (size_t)G * nwm);     // [G+1][nwm]

    const int u = blockIdx.x;
    const int b = u / kv.hkv;
    const int kvh = u % kv.hkv;
    const int np = pages_of(kv, b);
    const int nw = (np + 31) / 32;
    for (int i = threadIdx.x; i < G * nwm; i += blockDim.x) bits[i] = 0u;
    __syncthreads();
    for (int h = 0; h < G; ++h) {
        const int bh = b * Hq + kvh * G + h;
        int ns = n_sel[bh];
        if (ns < 0 || ns > cap) {
            if (threadIdx.x == 0) flag_bad_data();
            ns = max(0, min(ns, cap));
        }
        for (int r = threadIdx.x; r < ns; r += blockDim.x) {
            const int p = sel[(int64_t)bh * cap + r];
            if (p >= 0 && p < np) atomicOr(&bits[h * nwm + (p >> 5)], 1u << (p & 31));
            else flag_bad_data();
        }
    }
    __syncthreads();

    const int seg = (nw + blockDim.x - 1) / blockDim.x;
    const int w0 = min(nw, threadIdx.x * seg), w1 = min(nw, w0 + seg);
    int totals[G + 1];
#pragma unroll
    for (int a = 0; a <= G; ++a) {
        int local = 0;
        for (int w = w0; w < w1; ++w) {
            uint32_t word = 0;
            if (a < G) word = bits[a * nwm + w];
            else
#pragma unroll
                for (int h = 0; h < G; ++h) word |= bits[h * nwm + w];
            local += __popc(word);
        }
        int run = block_exclusive_scan(local, red, &totals[a]);
        for (int w = w0; w < w1; ++w) {
            uint32_t word = 0;
            if (a < G) word = bits[a * nwm + w];
            else
#pragma unroll
                for (int h = 0; h < G; ++h) word |= bits[h * nwm + w];
            pre[a * nwm + w] = run;
            run += __popc(word);
        }
    }
    if (threadIdx.x == 0) {
        ws.union_count[u] = totals[G];
        ws.counter[u] = 0;
        ws.vpages[u] = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) ws.head_count[b * Hq + kvh * G + h] = totals[h];
    }
    __syncthreads();
    int* upage = ws.union_page + (int64_t)u * L.Umax;
    int* umask = ws.union_mask + (int64_t)u * L.Umax;
    int* urank = ws.union_rank + (int64_t)u * L.Umax * G;
    for (int w = w0; w < w1; ++w) {
        uint32_t hw[G];
        uint32_t uw = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) { hw[h] = bits[h * nwm + w]; uw |= hw[h]; }
        int idx = pre[G * nwm + w];
        while (uw) {
            const int bit = __ffs(uw) - 1;
            uw &= uw - 1;
            const uint32_t below = (1u << bit) - 1u;
            int mask = 0;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const bool in = (hw[h] >> bit) & 1u;
                mask |= in ? (1 << h) : 0;
                urank[(int64_t)idx * G + h] = in ? pre[h * nwm + w] + __popc(hw[h] & below) : -1;
            }
            upage[idx] = w * 32 + bit;
            umask[idx] = mask;
            ++idx;
        }
    }
}

// ---------------------------------------------------------------------------
// qk: scores of the union pages
// ---------------------------------------------------------------------------
template <int D, int G, typename T>
struct QkShape {
    static constexpr int EPC = Elem<T>::kPer16;
    static constexpr int RC = D / EPC;                       // 16-byte chunks per key row
    static constexpr int LPT0 = (G * D / 64) < 2 ? 2 : (G * D / 64);
    static constexpr int LPT = LPT0 > RC ? RC : LPT0;       // lanes per token
    static constexpr int CPL = RC / LPT;                     // chunks per lane
    static constexpr int TPW = 32 / LPT;                     // tokens per warp pass
    static constexpr int NW = kQkThreads / 32;
    static constexpr int TPP = NW * TPW;                     // tokens per CTA pass
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kQkThreads)
qk_kernel(const float* __restrict__ q, int Hq, float qscale, KV kv, WS ws, DecodeLayout L,
          int sp, int nstages) {
    using S = QkShape<D, G, T>;
    extern __shared__ __align__(128) unsigned char s_raw[];
    __shared__ __align__(8) uint64_t bars[8];
    __shared__ int s_blk[kChunkPages], s_valid[kChunkPages], s_mask[kChunkPages];
    __shared__ int s_rank[kChunkPages][G];

    const int u = blockIdx.y;
    const int c = blockIdx.x;
    const int ucnt = ws.union_count[u];
    const int i0 = c * L.CH;
    if (i0 >= ucnt) return;
    const int npg = min(ucnt, i0 + L.CH) - i0;
    const int b = u / kv.hkv;
    const int kvh = u % kv.hkv;
    const int P = kv.P;
    const int len = kv.sl[b];
    const int tid = threadIdx.x;

    if (tid < npg) {
        const int idx = u * L.Umax + i0 + tid;
        const int page = ws.union_page[idx];
        int blk = kv.pt[(int64_t)b * kv.maxp + page];
        int valid = min(P, len - page * P);
        if (blk < 0 || blk >= kv.nb) { flag_bad_data(); blk = 0; valid = 0; }
        s_blk[tid] = blk;
        s_valid[tid] = valid;
        s_mask[tid] = ws.union_mask[idx];
#pragma unroll
        for (int h = 0; h < G; ++h) s_rank[tid][h] = ws.union_rank[(int64_t)idx * G + h];
    }
    if (tid == 0) {
        for (int s = 0; s < nstages; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    const int lane = tid & 31, wid = tid >> 5;
    const int lt = lane % S::LPT;                  // lane within its token group
    float qr[G][S::CPL][S::EPC];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int cc = 0; cc < S::CPL; ++cc)
#pragma unroll
            for (int e = 0; e < S::EPC; ++e)
                qr[h][cc][e] = qscale *
                    q[((int64_t)b * Hq + kvh * G + h) * D + (lt + cc * S::LPT) * S::EPC + e];
    __syncthreads();

    const size_t page_elems = (size_t)P * D;
    const uint32_t page_bytes = (uint32_t)(page_elems * sizeof(T));
    const int n_st = (npg + sp - 1) / sp;
    T* stage0 = reinterpret_cast<T*>(s_raw);
    const T* kbase = static_cast<const T*>(kv.k);
    auto issue = [&](int s) {
        const int slot = s % nstages;
        const int j0 = s * sp, j1 = min(npg, j0 + sp);
        mbar_arrive_expect_tx(&bars[slot], page_bytes * (uint32_t)(j1 - j0));
        for (int j = j0; j < j1; ++j) {
            const T* src = kbase + ((int64_t)s_blk[j] * kv.hkv + kvh) * page_elems;
            bulk_g2s(stage0 + (size_t)slot * sp * page_elems + (size_t)(j - j0) * page_elems, src,
                     page_bytes, &bars[slot]);
        }
    };
    if (tid == 0)
        for (int s = 0; s < min(nstages, n_st); ++s) issue(s);

    float* zb = ws.z + ((int64_t)b * Hq + kvh * G) * L.zcap;
    const int stage_tokens = sp * P;
    for (int s = 0; s < n_st; ++s) {
        const int slot = s % nstages;
        const bool ok = mbar_wait(&bars[slot], (uint32_t)((s / nstages) & 1));
        if (!__syncthreads_and(ok)) {
            if (tid == 0) flag_bad_data();
            return;
        }
        const T* st = stage0 + (size_t)slot * sp * page_elems;
        const int pages_here = min(npg, (s + 1) * sp) - s * sp;
        for (int t0 = 0; t0 < stage_tokens; t0 += S::TPP) {
            const int ts = t0 + wid * S::TPW + lane / S::LPT;     // token within stage
            const int jp = ts / P, t = ts - jp * P;
            const bool live = ts < stage_tokens && jp < pages_here;
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = 0.f;
            if (live) {
                const T* row = st + (size_t)ts * D;
#pragma unroll
                for (int cc = 0; cc < S::CPL; ++cc) {
                    const uint4 raw =
                        *reinterpret_cast<const uint4*>(row + (lt + cc * S::LPT) * S::EPC);
                    float x[S::EPC];
                    Elem<T>::widen(raw, x);
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int e = 0; e < S::EPC; ++e) acc[h] = fmaf(qr[h][cc][e], x[e], acc[h]);
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = group_sum<S::LPT>(acc[h]);
            if (live && lt < G) {
                const int pg = s * sp + jp;
                float mine = 0.f;
#pragma unroll
                for (int h = 0; h < G; ++h) if (lt == h) mine = acc[h];
                if ((s_mask[pg] >> lt) & 1) {
                    const int rank = s_rank[pg][lt];
                    zb[(int64_t)lt * L.zcap + (int64_t)rank * P + t] = t < s_valid[pg] ? mine : -INFINITY;
                }
            }
        }
        __syncthreads();
        if (tid == 0 && s + nstages < n_st) issue(s + nstages);
    }
}

// ---------------------------------------------------------------------------
// tau: exact alpha-entmax threshold per query head
// ---------------------------------------------------------------------------
__device__ __forceinline__ float pow_e(float a, int E, float ex) {
    return E == 2 ? a * a : (E == 1 ? a : powf(a, ex));
}

template <int E>   // 2: alpha = 1.5, 1: alpha = 2, 0: any other alpha
__global__ void __launch_bounds__(kTauThreads)
tau_kernel(float alpha, int P, WS ws, DecodeLayout L, float* __restrict__ tau_out,
           int32_t* __restrict__ support_out) {
    extern __shared__ __align__(16) float s_buf[];
    __shared__ float fred[40];
    __shared__ float2 f2red[32];
    __shared__ int ired[40];
    __shared__ int s_m;
    __shared__ float s_pref[2];
    __shared__ int s_kstar;

    const int bh = blockIdx.x;
    const int n = ws.head_count[bh] * P;
    const float* z = ws.z + (int64_t)bh * L.zcap;
    const int tid = threadIdx.x;
    if (n <= 0) {
        if (tid == 0) {
            ws.tau[bh] = INFINITY;
            if (tau_out) tau_out[bh] = INFINITY;
            if (support_out) support_out[bh] = 0;
        }
        return;
    }
    float mx = -INFINITY;
    for (int i = tid; i < n; i += blockDim.x) mx = fmaxf(mx, z[i]);
    mx = block_max(mx, fred);
    if (tid == 0) s_m = 0;
    __syncthreads();
    // candidates: x = z' - max > -1 (anything lower has zero weight)
    for (int i = tid; i < n; i += blockDim.x) {
        const float x = z[i] - mx;
        if (x > -1.f) s_buf[atomicAdd(&s_m, 1)] = x;
    }
    __syncthreads();
    const int m = s_m;
    const float ex = 1.f / (alpha - 1.f);
    float t;
    if (E == 0) {
        float lo = -1.f, hi = -powf(static_cast<float>(m), 1.f - alpha);
        for (int it = 0; it < 48; ++it) {
            const float mid = 0.5f * (lo + hi);
            float f = 0.f;
            for (int i = tid; i < m; i += blockDim.x) {
                const float a = s_buf[i] - mid;
                if (a > 0.f) f += powf(a, ex);
            }
            f = block_sum(f, fred) - 1.f;
            if (f >= 0.f) lo = mid; else hi = mid;
        }
        t = 0.5f * (lo + hi);
    } else {
        int M = 1;
        while (M < m) M <<= 1;
        for (int i = m + tid; i < M; i += blockDim.x) s_buf[i] = -INFINITY;
        __syncthreads();
        // bitonic sort, descending
        for (int k = 2; k <= M; k <<= 1) {
            for (int j = k >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < M; i += blockDim.x) {
                    const int ij = i ^ j;
                    if (ij > i) {
                        const float a = s_buf[i], c = s_buf[ij];
                        const bool desc = (i & k) == 0;
                        if (desc ? (a < c) : (a > c)) { s_buf[i] = c; s_buf[ij] = a; }
                    }
                }
                __syncthreads();
            }
        }
        // prefix sums over contiguous segments of the sorted candidates
        const int seg = (m + blockDim.x - 1) / blockDim.x;
        const int k0 = min(m, tid * seg), k1 = min(m, k0 + seg);
        float a1 = 0.f, a2 = 0.f;
        for (int i = k0; i < k1; ++i) { a1 += s_buf[i]; a2 = fmaf(s_buf[i], s_buf[i], a2); }
        const float inc1 = block_inclusive_scan_f(a1, fred);
        const float inc2 = block_inclusive_scan_f(a2, fred);
        float S1 = inc1 - a1, S2 = inc2 - a2;
        int best = 1;
        for (int i = k0; i < k1; ++i) {
            const float x = s_buf[i];
            S1 += x;
            S2 = fmaf(x, x, S2);
            const int kk = i + 1;
            bool valid;
            if (E == 1) {
                valid = x > (S1 - 1.f) / kk;
            } else {
                const float Mk = S1 / kk;
                const float ss = fmaxf(S2 - S1 * Mk, 0.f);
                valid = ss <= 1.f && (Mk - sqrtf((1.f - ss) / kk)) <= x;
            }
            if (valid) best = kk;
        }
        // k* = largest valid prefix length
        int kstar = best;
        {
            int v = kstar;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
            __syncthreads();
            if ((tid & 31) == 0) ired[tid >> 5] = v;
            __syncthreads();
            v = (tid & 31) < (int)(blockDim.x >> 5) ? ired[tid & 31] : 0;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
            kstar = v;
        }
        if (kstar - 1 >= k0 && kstar - 1 < k1) {
            // the owner of position k* recomputes its prefix sums
            float P1 = inc1 - a1, P2 = inc2 - a2;
            for (int i = k0; i < kstar; ++i) { P1 += s_buf[i]; P2 = fmaf(s_buf[i], s_buf[i], P2); }
            s_pref[0] = P1;
            s_pref[1] = P2;
            s_kstar = kstar;
        }
        __syncthreads();
        const float P1 = s_pref[0], P2 = s_pref[1];
        if (E == 1) {
            t = (P1 - 1.f) / kstar;
        } else {
            const float Mk = P1 / kstar;
            const float ss = fmaxf(P2 - P1 * Mk, 0.f);
            t = Mk - sqrtf(fmaxf(1.f - ss, 0.f) / kstar);
        }
        // Newton polish on f(t) = sum (x - t)_+^e - 1 (exact piecewise form)
        for (int it = 0; it < 3; ++it) {
            float2 acc = make_float2(0.f, 0.f);
            for (int i = tid; i < m; i += blockDim.x) {
                const float a = s_buf[i] - t;
                if (a > 0.f) {
                    if (E == 2) { acc.x = fmaf(a, a, acc.x); acc.y += 2.f * a; }
                    else { acc.x += a; acc.y += 1.f; }
                }
            }
            acc = block_sum2(acc, f2red);
            if (acc.y > 0.f) t += (acc.x - 1.f) / acc.y;
        }
    }
    int sup = 0;
    for (int i = tid; i < m; i += blockDim.x) sup += s_buf[i] > t;
    sup = block_sum_i(sup, ired);
    if (tid == 0) {
        const float tau = t + mx;
        ws.tau[bh] = tau;
        if (tau_out) tau_out[bh] = tau;
        if (support_out) support_out[bh] = sup;
    }
}

// ---------------------------------------------------------------------------
// pv: weights, value accumulation over the support pages, merge
// ---------------------------------------------------------------------------
template <typename T, int D, int G, int E>
__global__ void __launch_bounds__(kPvThreads)
pv_kernel(int Hq, float alpha, KV kv, WS ws, DecodeLayout L, float* __restrict__ out,
          int nstages) {
    constexpr int EPC = Elem<T>::kPer16;
    constexpr int LPR = D / EPC;          // lanes per value row
    constexpr int RPW = 32 / LPR;         // rows per warp pass
    constexpr int NW = kPvThreads / 32;
    constexpr int RPP = NW * RPW;         // rows per CTA pass
    extern __shared__ __align__(128) unsigned char s_raw[];
    __shared__ __align__(8) uint64_t bars[8];
    __shared__ int s_blk[kChunkPages], s_page_ok[kChunkPages], s_act[kChunkPages];
    __shared__ float s_tau[G];
    __shared__ float s_psum[G];
    __shared__ int s_nact, s_last;

    const int u = blockIdx.y;
    const int c = blockIdx.x;
    const int b = u / kv.hkv;
    const int kvh = u % kv.hkv;
    const int P = kv.P;
    const int tid = threadIdx.x;
    const int ucnt = ws.union_count[u];
    const int nchunks = (ucnt + L.CH - 1) / L.CH;
    float* outb = out + ((int64_t)b * Hq + kvh * G) * D;
    if (ucnt == 0) {
        if (c == 0)
            for (int i = tid; i < G * D; i += blockDim.x) outb[i] = 0.f;
        return;
    }
    if (c >= nchunks) return;
    const int i0 = c * L.CH;
    const int npg = min(ucnt, i0 + L.CH) - i0;
    const int len = kv.sl[b];

    // shared layout: weights [CH][P][G], reduction [RPP][G][D], V stages
    float* s_w = reinterpret_cast<float*>(s_raw);
    float* s_red = s_w + (size_t)kChunkPages * P * G;
    T* stage0 = reinterpret_cast<T*>(s_red + (size_t)RPP * G * D);

    if (tid < G) {
        s_tau[tid] = ws.tau[b * Hq + kvh * G + tid];
        s_psum[tid] = 0.f;
    }
    if (tid < kChunkPages) s_page_ok[tid] = 0;
    if (tid < npg) {
        const int idx = u * L.Umax + i0 + tid;
        const int page = ws.union_page[idx];
        int blk = kv.pt[(int64_t)b * kv.maxp + page];
        if (blk < 0 || blk >= kv.nb) blk = -1;
        s_blk[tid] = blk;
    }
    if (tid == 0) {
        for (int s = 0; s < nstages; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncthreads();

    const float ex = 1.f / (alpha - 1.f);
    const float* zb = ws.z + ((int64_t)b * Hq + kvh * G) * L.zcap;
    float ps[G];
#pragma unroll
    for (int h = 0; h < G; ++h) ps[h] = 0.f;
    for (int i = tid; i < npg * P; i += blockDim.x) {
        const int pg = i / P, t = i - pg * P;
        const int idx = u * L.Umax + i0 + pg;
        const int mask = ws.union_mask[idx];
        const int page = ws.union_page[idx];
        const bool tok_ok = s_blk[pg] >= 0 && t < min(P, len - page * P);
        bool any = false;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float w = 0.f;
            if (tok_ok && ((mask >> h) & 1)) {
                const int rank = ws.union_rank[(int64_t)idx * G + h];
                const float a = zb[(int64_t)h * L.zcap + (int64_t)rank * P + t] - s_tau[h];
                if (a > 0.f) w = pow_e(a, E, ex);
            }
            s_w[((size_t)pg * P + t) * G + h] = w;
            ps[h] += w;
            any |= w > 0.f;
        }
        if (any) s_page_ok[pg] = 1;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float v = warp_sum(ps[h]);
        if ((tid & 31) == 0) atomicAdd(&s_psum[h], v);
    }
    __syncthreads();
    if (tid == 0) {
        int n = 0;
        for (int j = 0; j < npg; ++j)
            if (s_page_ok[j]) s_act[n++] = j;
        s_nact = n;
        if (n) atomicAdd(&ws.vpages[u], n);
    }
    __syncthreads();
    const int nact = s_nact;

    const size_t page_elems = (size_t)P * D;
    const uint32_t page_bytes = (uint32_t)(page_elems * sizeof(T));
    const T* vbase = static_cast<const T*>(kv.v);
    auto issue = [&](int s) {
        const int slot = s % nstages;
        mbar_arrive_expect_tx(&bars[slot], page_bytes);
        const T* src = vbase + ((int64_t)s_blk[s_act[s]] * kv.hkv + kvh) * page_elems;
        bulk_g2s(stage0 + (size_t)slot * page_elems, src, page_bytes, &bars[slot]);
    };
    if (tid == 0)
        for (int s = 0; s < min(nstages, nact); ++s) issue(s);

    const int lane = tid & 31, wid = tid >> 5;
    const int lr = lane % LPR;
    const int rg = wid * RPW + lane / LPR;
    float acc[G][EPC];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < EPC; ++e) acc[h][e] = 0.f;
    bool failed = false;
    for (int s = 0; s < nact; ++s) {
        const int slot = s % nstages;
        const bool ok = mbar_wait(&bars[slot], (uint32_t)((s / nstages) & 1));
        if (!__syncthreads_and(ok)) { failed = true; break; }
        const T* st = stage0 + (size_t)slot * page_elems;
        const float* wp = s_w + (size_t)s_act[s] * P * G;
        for (int t = rg; t < P; t += RPP) {
            float x[EPC];
            Elem<T>::widen(*reinterpret_cast<const uint4*>(st + (size_t)t * D + lr * EPC), x);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float w = wp[t * G + h];
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[h][e] = fmaf(w, x[e], acc[h][e]);
            }
        }
        __syncthreads();
        if (tid == 0 && s + nstages < nact) issue(s + nstages);
    }
    if (failed) {
        if (tid == 0) flag_bad_data();
        return;
    }
    // reduce over the RPP row groups
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < EPC; ++e) s_red[((size_t)rg * G + h) * D + lr * EPC + e] = acc[h][e];
    __syncthreads();
    float* part = ws.partial + ((int64_t)u * L.Smax + c) * G * (D + 1);
    for (int i = tid; i < G * D; i += blockDim.x) {
        float sacc = 0.f;
        for (int g = 0; g < RPP; ++g) sacc += s_red[(size_t)g * G * D + i];
        part[i] = sacc;
    }
    if (tid < G) part[G * D + tid] = s_psum[tid];
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int ticket = atomicAdd(&ws.counter[u], 1);
        s_last = ticket == nchunks - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const float* part0 = ws.partial + (int64_t)u * L.Smax * G * (D + 1);
    for (int i = tid; i < G * D; i += blockDim.x) {
        const int h = i / D;
        float so = 0.f, sp = 0.f;
        for (int cc = 0; cc < nchunks; ++cc) {
            const float* pc = part0 + (int64_t)cc * G * (D + 1);
            so += __ldcg(pc + i);
            sp += __ldcg(pc + G * D + h);
        }
        outb[i] = sp > 0.f ? so / sp : 0.f;
    }
    if (tid == 0) ws.counter[u] = 0;
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
static cudaEvent_t g_stage_events[5];
static int g_n_stage_events = 0;

void set_decode_stage_events(const cudaEvent_t* events, int n) {
    g_n_stage_events = (events && n == 5) ? 5 : 0;
    for (int i = 0; i < g_n_stage_events; ++i) g_stage_events[i] = events[i];
}

static void stage_mark(int i, cudaStream_t s) {
    if (g_n_stage_events) cudaEventRecord(g_stage_events[i], s);
}

cudaError_t read_decode_counts(const void* ws_base, const DecodeLayout& L, int32_t* union_pages,
                               int32_t* v_pages, cudaStream_t s) {
    const char* c = static_cast<const char*>(ws_base);
    cudaError_t e = cudaSuccess;
    if (union_pages)
        e = cudaMemcpyAsync(union_pages, c + L.union_count, sizeof(int32_t) * L.U,
                            cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && v_pages)
        e = cudaMemcpyAsync(v_pages, c + L.vpages, sizeof(int32_t) * L.U, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}
template <typename T, int D, int G>
static cudaError_t launch_decode_t(const float* q, int Hq, float scale, const KV& kv,
                                   const int32_t* sel, const int32_t* n_sel, int cap, float alpha,
                                   float* out, float* tau_out, int32_t* support_out, const WS& ws,
                                   const DecodeLayout& L, cudaStream_t s) {
    cudaError_t e;
    // plan
    {
        const int nwm = (kv.maxp + 31) / 32;
        const size_t smem = (size_t)(2 * G + 1) * nwm * 4;
        e = cudaFuncSetAttribute(plan_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        stage_mark(0, s);
        plan_kernel<G><<<L.U, kPlanThreads, smem, s>>>(kv, Hq, sel, n_sel, cap, ws, L);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // qk
    {
        using S = QkShape<D, G, T>;
        const int sp = std::max(1, S::TPP / kv.P);
        const size_t stage_bytes = (size_t)sp * kv.P * D * sizeof(T);
        const int nst = (int)std::max<size_t>(2, std::min<size_t>(8, (64 * 1024) / stage_bytes));
        const size_t smem = stage_bytes * nst;
        e = cudaFuncSetAttribute(qk_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        dim3 grid(L.Smax, L.U);
        stage_mark(1, s);
        qk_kernel<T, D, G><<<grid, kQkThreads, smem, s>>>(q, Hq, (alpha - 1.f) * scale, kv, ws, L,
                                                          sp, nst);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // tau
    {
        int M = 1;
        while (M < L.zcap) M <<= 1;
        const size_t smem = (size_t)M * sizeof(float);
        const float a = alpha;
        const int E = fabsf(a - 1.5f) < 1e-6f ? 2 : (fabsf(a - 2.f) < 1e-6f ? 1 : 0);
        const dim3 grid(kv.B * Hq);
        stage_mark(2, s);
        if (E == 2) {
            e = cudaFuncSetAttribute(tau_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e == cudaSuccess)
                tau_kernel<2><<<grid, kTauThreads, smem, s>>>(alpha, kv.P, ws, L, tau_out, support_out);
        } else if (E == 1) {
            e = cudaFuncSetAttribute(tau_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e == cudaSuccess)
                tau_kernel<1><<<grid, kTauThreads, smem, s>>>(alpha, kv.P, ws, L, tau_out, support_out);
        } else {
            e = cudaFuncSetAttribute(tau_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e == cudaSuccess)
                tau_kernel<0><<<grid, kTauThreads, smem, s>>>(alpha, kv.P, ws, L, tau_out, support_out);
        }
        if (e != cudaSuccess) return e;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // pv
        constexpr int EPC = Elem<T>::kPer16;
        constexpr int RPP = (kPvThreads / 32) * (32 / (D / EPC));
        const size_t page_bytes = (size_t)kv.P * D * sizeof(T);
        const int nst = (int)std::max<size_t>(2, std::min<size_t>(8, (64 * 1024) / page_bytes));
        const size_t pv_smem = (size_t)kChunkPages * kv.P * G * 4 + (size_t)RPP * G * D * 4 +
                               page_bytes * nst;
        dim3 pgrid(L.Smax, L.U);
        stage_mark(3, s);
        if (E == 2) {
            e = cudaFuncSetAttribute(pv_kernel<T, D, G, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pv_smem);
            if (e == cudaSuccess)
                pv_kernel<T, D, G, 2><<<pgrid, kPvThreads, pv_smem, s>>>(Hq, alpha, kv, ws, L, out, nst);
        } else if (E == 1) {
            e = cudaFuncSetAttribute(pv_kernel<T, D, G, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pv_smem);
            if (e == cudaSuccess)
                pv_kernel<T, D, G, 1><<<pgrid, kPvThreads, pv_smem, s>>>(Hq, alpha, kv, ws, L, out, nst);
        } else {
            e = cudaFuncSetAttribute(pv_kernel<T, D, G, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pv_smem);
            if (e == cudaSuccess)
                pv_kernel<T, D, G, 0><<<pgrid, kPvThreads, pv_smem, s>>>(Hq, alpha, kv, ws, L, out, nst);
        }
        if (e != cudaSuccess) return e;
        stage_mark(4, s);
    }
    return cudaGetLastError();
}

cudaError_t launch_decode(const float* q, int Hq, float scale, const KV& kv, const int32_t* sel,
                          const int32_t* n_sel, int cap, float alpha, float* out, float* tau_out,
                          int32_t* support_out, void* ws_base, const DecodeLayout& L,
                          cudaStream_t s) {
    const WS ws = ws_views(ws_base, L);
    const int G = L.G;
    EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
        return launch_decode_t<T, kD, kG>(q, Hq, scale, kv, sel, n_sel, cap, alpha, out, tau_out,
                                           support_out, ws, L, s);
    })))
    return cudaErrorInvalidValue;
}

}  // namespace ekv
