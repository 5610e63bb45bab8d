// alpha-entmax attention over the selected pages [EntmaxKV §2.C].
//
// Work unit u = (sequence b, kv head): its G query heads each selected their
// own pages; the unit reads the UNION of those pages once.
//
//   plan  (1 CTA per unit)      bitmaps of each head's pages -> union list in
//                               ascending page order with a per-page head mask;
//                               resets the unit's per-call state.
//   qk                          the flattened union lists of all units are cut
//                               into one contiguous range per warp; K pages go
//                               through a private ring of bulk copies per warp
//                               and z' = (alpha-1) s q.k is computed for the G
//                               heads (bf16 K: tensor cores, see qk_mma_kernel;
//                               fp32 K: FMA).  Scores are stored per unit in
//                               union order, -inf where a head did not select
//                               the page; per-head maxima go out through atomics
//                               and each page's physical block is recorded.
//   tpv   (1 CTA per head)      candidates z' > max - 1 (all others have zero
//                               weight) are compacted; tau solves
//                               sum (z' - tau)_+^(1/(alpha-1)) = 1 by Newton from
//                               the left (alpha 1.5 and 2: the function is convex,
//                               so the iterates rise monotonically to the root)
//                               or by bisection (other alpha); then only the V
//                               rows of the support tokens are read and
//                               out = sum p v / sum p.
#include <cuda_bf16.h>

#include "common.cuh"

EKV_DEFINE_STATUS(decode)

#include "plan.cuh"

namespace ekv {

constexpr int kPlanThreads = 512;
constexpr int kQkConsumers = 12;                       // consumer warps per qk CTA
constexpr int kQkThreads = 32 * (kQkConsumers + 1);    // + one producer warp
constexpr int kQkGroup = 16;                           // pages resolved per producer step
constexpr int kQkMaxSlots = 48;
constexpr int kQkSmemBudget = 220 * 1024;
constexpr int kMaxUnits = 8192;                        // qk keeps a prefix over units in smem
constexpr int kTpvThreads = 256;
constexpr int kTpvgThreads = 512;                      // the global-candidate variant
constexpr int kTpvVec = 2;                             // float4 per thread per score tile (short: tpv's code runs cold)
constexpr int kTpvTile = kTpvThreads * kTpvVec * 4;    // scores per tile
constexpr int kTpvgTile = kTpvgThreads * kTpvVec * 4;
constexpr int kTpvgRows = 8;                           // V rows in flight per row group (tpv kernels)

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

DecodeLayout decode_layout(int B, int Hq, int Hkv, int D, int P, int max_pages, int cap,
                           bool candidates) {
    (void)D;
    DecodeLayout L{};
    L.U = B * Hkv;
    L.G = Hq / Hkv;
    L.Umax = std::min(L.G * cap, max_pages);
    L.nvw = (L.Umax * P + 31) / 32;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
    L.union_count = take(sizeof(int) * L.U);
    L.head_max = take(sizeof(uint32_t) * (size_t)B * Hq);
    L.union_page = take(sizeof(int) * (size_t)L.U * L.Umax);
    L.union_mask = take(sizeof(int) * (size_t)L.U * L.Umax);
    L.union_blk = take(sizeof(int) * (size_t)L.U * L.Umax);
    L.vtok = take(sizeof(uint32_t) * (size_t)L.U * L.nvw);
    L.vrows = take(sizeof(int) * L.U);
    L.z = take(sizeof(float) * (size_t)L.U * L.G * L.Umax * P);
    L.pmax = take(sizeof(float) * (size_t)L.U * L.G * L.Umax);
    L.tau = take(sizeof(float) * (size_t)B * Hq);
    L.ccap = cap * P;
    L.cand_x = L.cand_pos = L.plist = 0;
    if (candidates && L.ccap > kTpvSmemCand) {
        L.cand_x = take(sizeof(float) * (size_t)B * Hq * L.ccap);
        L.cand_pos = take(sizeof(int) * (size_t)B * Hq * L.ccap);
        L.plist = take(sizeof(int) * (size_t)B * Hq * L.Umax);
    }
    L.recs = 0;
    L.nrec = 0;
    L.total = o;
    return L;
}

DecodeLayout softmax_layout(int B, int Hq, int Hkv, int D, int P, int max_pages, int cap) {
    DecodeLayout L = decode_layout(B, Hq, Hkv, D, P, max_pages, cap, false);
    L.nrec = kPvMaxWarps + L.U;
    L.recs = L.total;
    L.total = align256(L.recs + sizeof(float) * (size_t)L.nrec * L.G * (D + 1));
    return L;
}

// ---------------------------------------------------------------------------
// plan: union of the group's selections
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(KV kv, int Hq, const int32_t* __restrict__ sel, const int32_t* __restrict__ n_sel,
            int cap, WS ws, DecodeLayout L) {
    extern __shared__ __align__(16) uint32_t s_plan[];   // bitmaps, then union pages
    __shared__ int red[40];
    __shared__ int s_ns[G];
    const int nwm = (kv.maxp + 31) / 32;
    int* s_upage = reinterpret_cast<int*>(s_plan + (size_t)G * nwm);
    pdl_wait();                         // the selection is the previous kernel's output
    pdl_trigger();                      // the q.K kernel's CTAs may take their places
    build_plan<G>(kv, Hq, sel, n_sel, cap, ws, L, blockIdx.x, s_plan, s_upage, s_upage + L.Umax,
                  red, s_ns);
}

// Plan of the full-cache decode: the union of unit u is every valid page of
// its sequence, selected by all G heads.  Grid (U, chunks): chunk c writes
// pages [c kPlanAllChunk, +kPlanAllChunk) and resets its share of the unit's
// per-call state (as build_plan does).
constexpr int kPlanAllChunk = 1024;

__global__ void __launch_bounds__(kPlanThreads)
plan_all_kernel(KV kv, int Hq, WS ws, DecodeLayout L) {
    const int u = blockIdx.x, c = blockIdx.y, nc = gridDim.y;
    const int b = u / kv.hkv, kvh = u - b * kv.hkv;
    const int G = L.G;
    const int np = pages_of(kv, b);
    if (c == 0 && threadIdx.x < G) ws.head_max[b * Hq + kvh * G + threadIdx.x] = 0u;
    const int wpc = (L.nvw + nc - 1) / nc;
    for (int i = c * wpc + threadIdx.x; i < min(L.nvw, (c + 1) * wpc); i += blockDim.x)
        ws.vtok[(int64_t)u * L.nvw + i] = 0u;
    int* upage = ws.union_page + (int64_t)u * L.Umax;
    int* umask = ws.union_mask + (int64_t)u * L.Umax;
    int* ublk = ws.union_blk + (int64_t)u * L.Umax;
    const int i1 = min(np, (c + 1) * kPlanAllChunk);
    for (int i = c * kPlanAllChunk + threadIdx.x; i < i1; i += blockDim.x) {
        int blk = kv.pt[(int64_t)b * kv.maxp + i];
        if (blk < 0 || blk >= kv.nb) {
            flag_bad_data();
            blk = -1;
        }
        upage[i] = i;
        umask[i] = (1 << G) - 1;
        ublk[i] = blk;
    }
    if (c == 0 && threadIdx.x == 0) ws.union_count[u] = np;
}

// ---------------------------------------------------------------------------
// qk: scores of the union pages
// ---------------------------------------------------------------------------
template <typename T, int D, int G>
struct QkCfg {
    static constexpr int EPC = Elem<T>::kPer16;             // elements per 16-byte chunk
    static constexpr int RC = D / EPC;                      // chunks per key row
    static constexpr int C0 = (RC / G) < 2 ? (RC / G) : 2;
    static constexpr int C1 = 64 / (G * EPC);               // keeps q at <= 64 registers
    static constexpr int CPL = C1 < C0 ? C1 : C0;           // chunks per lane
    static constexpr int LPT = RC / CPL;                    // lanes per token (>= G)
    static constexpr int TPW = 32 / LPT;                    // tokens per warp pass
    static constexpr int DUP = LPT / G;                     // lanes left holding each head's sum
    static_assert(CPL >= 1 && LPT >= G && LPT <= 32, "unsupported qk shape");
};

// Sums a[0..C) over the M*2 lanes of an aligned lane group, handing each
// lane one head: at every level a lane keeps half of its values (the upper
// half if its lane bit is set) and adds its partner's copy of that half, so
// C values cost C-1 shuffles instead of C*log2(lanes).  On return a[0] holds
// the complete sum of value index lt / (lanes / C) for lane-in-group lt.
template <int C, int M>
struct XReduce {
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
                XReduce<H, M / 2>::run(a, lt);
            } else {
                a[0] += __shfl_xor_sync(0xFFFFFFFFu, a[0], M);
                XReduce<1, M / 2>::run(a, lt);
            }
        }
    }
};

struct QkInfo { int u, i, valid, mask; };

template <typename T, int D, int G>
__global__ void __launch_bounds__(kQkThreads, 1)
qk_kernel(const float* __restrict__ q, int Hq, float qscale, KV kv, WS ws, DecodeLayout L,
          int nslots, int group, int write_pm) {
    using C = QkCfg<T, D, G>;
    extern __shared__ __align__(128) unsigned char s_raw[];
    __shared__ int red[40];
    const int P = kv.P;
    const uint32_t page_bytes = static_cast<uint32_t>(P * D * sizeof(T));
    // shared layout: ring [nslots][page] | staging [consumers][G * P] floats |
    // prefix [U + 1] ints | info [nslots] | full, empty barriers [nslots] each
    unsigned char* ring = s_raw;
    float* stage = reinterpret_cast<float*>(s_raw + (size_t)nslots * page_bytes);
    int* prefix = reinterpret_cast<int*>(stage + kQkConsumers * G * P);
    QkInfo* info = reinterpret_cast<QkInfo*>(prefix + ((L.U + 1 + 3) & ~3));
    uint64_t* full = reinterpret_cast<uint64_t*>(info + nslots);
    uint64_t* empty = full + nslots;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    {
        // exclusive prefix over units of the union sizes
        const int U = L.U;
        const int seg = (U + blockDim.x - 1) / blockDim.x;
        const int a0 = min(U, tid * seg), a1 = min(U, a0 + seg);
        int c = 0;
        for (int a = a0; a < a1; ++a) c += ws.union_count[a];
        int tot;
        int run = block_exclusive_scan(c, red, &tot);
        for (int a = a0; a < a1; ++a) {
            prefix[a] = run;
            run += ws.union_count[a];
        }
        if (tid == 0) prefix[U] = tot;
    }
    if (tid == 0) {
        for (int s = 0; s < nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_fence_init();
    }
    __syncthreads();
    const int total = prefix[L.U];
    const int f0 = (int)((int64_t)total * blockIdx.x / gridDim.x);
    const int f1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
    const int nloc = f1 - f0;
    if (nloc <= 0) return;

    if (warp == 0) {
        // ---- producer: page k (0-based within this CTA) goes to slot k % nslots
        int lo = 0, hi = L.U - 1;       // last unit whose range starts at or before f0
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= f0) lo = mid; else hi = mid - 1;
        }
        int cu = lo, ci = f0 - prefix[lo];
        const T* kbase = static_cast<const T*>(kv.k);
        for (int g = 0; g < nloc; g += group) {
            const int k = g + lane;
            const bool act = lane < group && k < nloc;
            int uu = cu, ii = ci + lane;
            if (act)
                while (ii >= prefix[uu + 1] - prefix[uu]) { ii -= prefix[uu + 1] - prefix[uu]; ++uu; }
            ci += group;
            while (cu < L.U && ci >= prefix[cu + 1] - prefix[cu]) { ci -= prefix[cu + 1] - prefix[cu]; ++cu; }
            if (act) {
                const int idx = uu * L.Umax + ii;
                const int page = ws.union_page[idx];
                const int mask = ws.union_mask[idx];
                const int blk = ws.union_blk[idx];         // validated by the plan
                const int b = uu / kv.hkv;
                const int kvh = uu - b * kv.hkv;
                int valid = min(P, kv.sl[b] - page * P);
                if (blk < 0) valid = 0;
                const int slot = k % nslots;
                const int use = k / nslots;
                if (use > 0 && !mbar_wait(&empty[slot], (uint32_t)((use - 1) & 1))) {
                    flag_timeout();      // a consumer stalled: hand over an empty page
                    valid = 0;
                }
                info[slot] = QkInfo{uu, ii, valid, mask};
                if (valid > 0) {
                    mbar_arrive_expect_tx(&full[slot], page_bytes);
                    bulk_g2s(ring + (size_t)slot * page_bytes,
                             kbase + ((int64_t)blk * kv.hkv + kvh) * P * D, page_bytes, &full[slot]);
                } else {
                    mbar_arrive(&full[slot]);
                }
            }
            // Lanes move to the next group together.  A lane running ahead
            // could otherwise wait on a slot's empty barrier two phases early,
            // and a parity wait would take the still-open phase as complete.
            __syncwarp();
        }
        return;
    }

    // ---- consumers: warp cw takes pages k = cw (mod consumers); nslots is a
    // multiple of the consumer count, so every slot has a single owner warp
    const int cw = warp - 1;
    const int lt = lane % C::LPT;
    const int tok = lane / C::LPT;
    float* st = stage + cw * G * P;
    float qr[G][C::CPL][C::EPC];
    float hm[G];
    int cur_u = -1;
#define EKV_QK_FLUSH_MAX()                                                                     \
    do {                                                                                       \
        const int fb = cur_u / kv.hkv;                                                         \
        const int fk = cur_u - fb * kv.hkv;                                                    \
        _Pragma("unroll") for (int h = 0; h < G; ++h) {                                        \
            const float m = warp_max(hm[h]);                                                   \
            if (lane == 0 && m > -INFINITY)                                                    \
                atomicMax(&ws.head_max[fb * Hq + fk * G + h], float_key(m));                   \
        }                                                                                      \
    } while (0)
    for (int k = cw; k < nloc; k += kQkConsumers) {
        const int slot = k % nslots;
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&full[slot], (uint32_t)((k / nslots) & 1)));
        if (!ok) {
            if (lane == 0) flag_timeout();
            break;
        }
        const QkInfo in = info[slot];
        if (in.u != cur_u) {
            if (cur_u >= 0) EKV_QK_FLUSH_MAX();
            cur_u = in.u;
            const int b = cur_u / kv.hkv;
            const int kvh = cur_u - b * kv.hkv;
            const float* qb = q + ((int64_t)b * Hq + kvh * G) * D;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                hm[h] = -INFINITY;
#pragma unroll
                for (int cc = 0; cc < C::CPL; ++cc)
#pragma unroll
                    for (int e = 0; e < C::EPC; ++e)
                        qr[h][cc][e] = qscale * qb[h * D + (lt + cc * C::LPT) * C::EPC + e];
            }
        }
        const T* pg = reinterpret_cast<const T*>(ring + (size_t)slot * page_bytes);
        for (int t0 = 0; t0 < P; t0 += C::TPW) {
            const int t = t0 + tok;
            const T* row = pg + (size_t)t * D;
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
            for (int cc = 0; cc < C::CPL; ++cc) {
                const uint4 raw = *reinterpret_cast<const uint4*>(row + (lt + cc * C::LPT) * C::EPC);
                float x[C::EPC];
                Elem<T>::widen(raw, x);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < C::EPC; ++e) acc[h] = fmaf(qr[h][cc][e], x[e], acc[h]);
            }
            XReduce<G, C::LPT / 2>::run(acc, lt);
            if (lt % C::DUP == 0) st[(lt / C::DUP) * P + t] = acc[0];
        }
        __syncwarp();
        for (int e = lane * 4; e < G * P; e += 128) {
            const int h = e / P, t = e - h * P;
            float4 v = *reinterpret_cast<const float4*>(st + e);
            const bool hin = (in.mask >> h) & 1;
            v.x = (hin && t + 0 < in.valid) ? v.x : -INFINITY;
            v.y = (hin && t + 1 < in.valid) ? v.y : -INFINITY;
            v.z = (hin && t + 2 < in.valid) ? v.z : -INFINITY;
            v.w = (hin && t + 3 < in.valid) ? v.w : -INFINITY;
            *reinterpret_cast<float4*>(ws.z + (((int64_t)in.u * G + h) * L.Umax + in.i) * P + t) = v;
            const float m4 = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
#pragma unroll
            for (int hh = 0; hh < G; ++hh)
                if (hh == h) hm[hh] = fmaxf(hm[hh], m4);
        }
        if (write_pm && lane < G) {           // head `lane`'s largest z' on this page
            float pm = -INFINITY;
            if ((in.mask >> lane) & 1)
                for (int t = 0; t < in.valid; ++t) pm = fmaxf(pm, st[lane * P + t]);
            ws.pmax[((int64_t)in.u * G + lane) * L.Umax + in.i] = pm;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
    if (cur_u >= 0) EKV_QK_FLUSH_MAX();
#undef EKV_QK_FLUSH_MAX
}

// ---------------------------------------------------------------------------
// qk for bf16 K on the tensor cores (mma.sync m16n8k16, fp32 accumulate).
//
// A = q of the group as 3G bf16 rows: each fp32 q (times (alpha-1) s) is split
// exactly into hi + mid + lo bf16 terms, so that the bf16 x bf16 products are
// exact and the three rows of a head sum to the fp32 score.  B = the K page:
// n = tokens, k = head dimensions.  The contraction order over k is free, so
// the k positions are permuted (identically in A and B) such that one 16-byte
// read of 8 consecutive dimensions of one token fills the B fragments of two
// k-steps: lane (g, t) reads token g, dimensions [32 dg + 8 t, +8).
//
// Every warp streams its own contiguous range of the flattened union lists
// through a private ring of NS page stages in shared memory: one bulk copy per
// page on the warp's own mbarriers (no handshake between warps), the copy of
// page k + NS - 1 issued as soon as page k - 1 has been consumed.
// ---------------------------------------------------------------------------
constexpr int kQmWarps = 4;                  // warps per CTA
constexpr int kQmCtasPerSm = 2;
constexpr int kQmStageBytes = 24 * 1024;     // ring bytes per warp

template <int D, int G>
struct QmCfg {
    static constexpr int NR = 3 * G;              // (split, head) rows of A
    static constexpr int MT = (NR + 15) / 16;     // m-tiles
    static constexpr int KS = D / 16;             // k-steps
};

struct PgDesc { int blk, u, i, valid, mask; };

__device__ __forceinline__ PgDesc resolve_page(int f, int f1, const int* prefix, const KV& kv,
                                               const WS& ws, const DecodeLayout& L) {
    PgDesc d{-1, 0, 0, 0, 0};
    if (f >= f1) return d;
    int lo = 0, hi = L.U - 1;    // last unit whose range starts at or before f
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= f) lo = mid; else hi = mid - 1;
    }
    d.u = lo;
    d.i = f - prefix[lo];
    const int idx = lo * L.Umax + d.i;
    // one round trip: page, head mask and the block the plan validated
    const int page = __ldcg(ws.union_page + idx);
    d.mask = __ldcg(ws.union_mask + idx);
    d.blk = __ldcg(ws.union_blk + idx);
    const int b = lo / kv.hkv;
    d.valid = d.blk >= 0 ? min(kv.P, kv.sl[b] - page * kv.P) : 0;
    return d;
}

__device__ __forceinline__ PgDesc shfl_desc(const PgDesc& d, int src) {
    return PgDesc{__shfl_sync(0xFFFFFFFFu, d.blk, src), __shfl_sync(0xFFFFFFFFu, d.u, src),
                  __shfl_sync(0xFFFFFFFFu, d.i, src), __shfl_sync(0xFFFFFFFFu, d.valid, src),
                  __shfl_sync(0xFFFFFFFFu, d.mask, src)};
}

template <int D, int G, bool kPM>      // kPM: also write each head's page maxima
__global__ void __launch_bounds__(kQmWarps * 32, kQmCtasPerSm)
qk_mma_kernel(const float* __restrict__ q, int Hq, float qscale, KV kv, WS ws, DecodeLayout L,
              int ns) {
    using C = QmCfg<D, G>;
    extern __shared__ __align__(128) unsigned char s_qm[];
    __shared__ int red[40];
    __shared__ __align__(8) uint64_t s_bar[kQmWarps][8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int P = kv.P;
    const uint32_t page_bytes = static_cast<uint32_t>(P * D * 2);
    // shared layout: per-warp rings [warps][ns][page] | unit prefix [U + 1]
    unsigned char* ring = s_qm + (size_t)warp * ns * page_bytes;
    int* s_prefix = reinterpret_cast<int*>(s_qm + (size_t)kQmWarps * ns * page_bytes);
    uint64_t* bar = s_bar[warp];
    for (int i = tid * 32; i < L.U; i += blockDim.x * 32) prefetch_l2_line(ws.union_count + i);
    pdl_wait();                 // the union plan is the previous kernel's output
    {
        const int U = L.U;
        const int seg = (U + blockDim.x - 1) / blockDim.x;
        const int a0 = min(U, tid * seg), a1 = min(U, a0 + seg);
        int c = 0;
        for (int a = a0; a < a1; ++a) c += __ldcg(ws.union_count + a);
        int tot;
        int run = block_exclusive_scan(c, red, &tot);
        for (int a = a0; a < a1; ++a) {
            s_prefix[a] = run;
            run += __ldcg(ws.union_count + a);
        }
        if (tid == 0) s_prefix[U] = tot;
    }
    if (lane == 0) {
        for (int st = 0; st < ns; ++st) mbar_init(&bar[st], 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int total = s_prefix[L.U];
    const int64_t nwg = (int64_t)gridDim.x * kQmWarps;
    const int wg = blockIdx.x * kQmWarps + warp;
    const int f0 = (int)((int64_t)total * wg / nwg);
    const int f1 = (int)((int64_t)total * (wg + 1) / nwg);
    const int npg = f1 - f0;
    if (npg <= 0) return;
    const unsigned char* kbase = static_cast<const unsigned char*>(kv.k);
    const uint64_t evict_first = l2_evict_first_policy();

    PgDesc cur = resolve_page(f0 + lane, f1, s_prefix, kv, ws, L);
    PgDesc nxt{-1, 0, 0, 0, 0};
    if (npg > 32) nxt = resolve_page(f0 + 32 + lane, f1, s_prefix, kv, ws, L);
    int cur_base = 0;
    // Issues page k into stage k % ns; returns its descriptor.
    auto issue = [&](int k) -> PgDesc {
        PgDesc dsc{-1, 0, 0, 0, 0};
        if (k >= npg) return dsc;
        if (k >= cur_base + 32) {
            cur = nxt;
            cur_base += 32;
            if (npg > cur_base + 32) nxt = resolve_page(f0 + cur_base + 32 + lane, f1, s_prefix, kv, ws, L);
        }
        dsc = shfl_desc(cur, k - cur_base);
        if (lane == 0) {
            const int st = k % ns;
            if (dsc.blk >= 0) {
                mbar_arrive_expect_tx(&bar[st], page_bytes);
                bulk_g2s_hint(ring + (size_t)st * page_bytes,
                              kbase + (((int64_t)dsc.blk * kv.hkv + dsc.u % kv.hkv) * P * D) * 2,
                              page_bytes, &bar[st], evict_first);
            } else {
                mbar_arrive(&bar[st]);
            }
        }
        return dsc;
    };

    uint32_t a[C::MT][C::KS][4];
    float hm = -INFINITY;                 // running max of head g (lanes g < G)
    int cur_u = -1;
    PgDesc dq[8];            // descriptor of the page held by each stage (ns <= 8)
#pragma unroll
    for (int x = 0; x < 8; ++x)
        if (x < ns - 1) dq[x] = issue(x);
    bool failed = false;
    for (int k = 0; k < npg; ++k) {
        const int st = k % ns;
        // stage (k - 1) % ns was consumed in the previous iteration
        {
            const PgDesc nd = issue(k + ns - 1);
            const int nst = (k + ns - 1) % ns;
#pragma unroll
            for (int x = 0; x < 8; ++x)
                if (x == nst) dq[x] = nd;
        }
        PgDesc d{};
#pragma unroll
        for (int x = 0; x < 8; ++x)
            if (x == st) d = dq[x];
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[st], (uint32_t)((k / ns) & 1)))) {
            failed = true;
            break;
        }
        if (d.u != cur_u) {
            if (cur_u >= 0) {
                float m = fmaxf(hm, __shfl_xor_sync(0xFFFFFFFFu, hm, 1));
                m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
                const int fb = cur_u / kv.hkv, fk = cur_u - fb * kv.hkv;
                if (t == 0 && g < G && m > -INFINITY)
                    atomicMax(&ws.head_max[fb * Hq + fk * G + g], float_key(m));
            }
            cur_u = d.u;
            hm = -INFINITY;
            const int b = cur_u / kv.hkv, kvh = cur_u - b * kv.hkv;
            const float* qb = q + ((int64_t)b * Hq + kvh * G) * D;
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int kk = 0; kk < C::KS; ++kk)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int row = mt * 16 + g + ((r & 1) ? 8 : 0);
                        const int dim = 32 * (kk >> 1) + 8 * t + 4 * (kk & 1) + ((r & 2) ? 2 : 0);
                        uint32_t v = 0;
                        if (row < C::NR) {
                            const int sp = row / G, hh2 = row - sp * G;
                            const float x0 = qscale * __ldg(qb + hh2 * D + dim);
                            const float x1 = qscale * __ldg(qb + hh2 * D + dim + 1);
                            v = split_term(x0, sp) | (split_term(x1, sp) << 16);
                        }
                        a[mt][kk][r] = v;
                    }
        }
        const unsigned char* pg = ring + (size_t)st * page_bytes;
        float pgm = -INFINITY;               // head g's largest z' on this page (this lane's tokens)
        for (int nt = 0; nt < P / 8; ++nt) {
            float c[C::MT][4];
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) c[mt][e] = 0.f;
            const unsigned char* row = pg + (size_t)(nt * 8 + g) * D * 2 + 16 * t;
#pragma unroll
            for (int dg = 0; dg < D / 32; ++dg) {
                const uint4 v = *reinterpret_cast<const uint4*>(row + 64 * dg);
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    mma_bf16(c[mt], a[mt][2 * dg], v.x, v.y);
                    mma_bf16(c[mt], a[mt][2 * dg + 1], v.z, v.w);
                }
            }
            // z(head g, token) = sum over the three split rows s G + g
            float z0 = 0.f, z1 = 0.f;
#pragma unroll
            for (int sp = 0; sp < 3; ++sp) {
                const int r0 = sp * G;                 // row of head 0 in this split
                const int mt = r0 / 16, hf = (r0 % 16) / 8;
                float v0 = c[mt][2 * hf], v1 = c[mt][2 * hf + 1];
                if ((r0 % 8) != 0) {
                    const int src = (((r0 + g) % 8) << 2) | t;
                    v0 = __shfl_sync(0xFFFFFFFFu, v0, src);
                    v1 = __shfl_sync(0xFFFFFFFFu, v1, src);
                }
                z0 += v0;
                z1 += v1;
            }
            if (g < G) {
                const int tok = nt * 8 + 2 * t;
                const bool hin = (d.mask >> g) & 1;
                z0 = (hin && tok < d.valid) ? z0 : -INFINITY;
                z1 = (hin && tok + 1 < d.valid) ? z1 : -INFINITY;
                *reinterpret_cast<float2*>(ws.z + (((int64_t)d.u * G + g) * L.Umax + d.i) * P + tok) =
                    make_float2(z0, z1);
                pgm = fmaxf(pgm, fmaxf(z0, z1));
            }
        }
        if constexpr (kPM) {
            pgm = fmaxf(pgm, __shfl_xor_sync(0xFFFFFFFFu, pgm, 1));
            pgm = fmaxf(pgm, __shfl_xor_sync(0xFFFFFFFFu, pgm, 2));
            if (g < G && t == 0) ws.pmax[((int64_t)d.u * G + g) * L.Umax + d.i] = pgm;
        }
        hm = fmaxf(hm, pgm);
        __syncwarp();        // every lane is done with stage st before it is refilled
    }
    pdl_trigger();
    if (failed) {
        if (lane == 0) flag_timeout();
        return;
    }
    {
        float m = fmaxf(hm, __shfl_xor_sync(0xFFFFFFFFu, hm, 1));
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
        const int fb = cur_u / kv.hkv, fk = cur_u - fb * kv.hkv;
        if (cur_u >= 0 && t == 0 && g < G && m > -INFINITY)
            atomicMax(&ws.head_max[fb * Hq + fk * G + g], float_key(m));
    }
}

// ---------------------------------------------------------------------------
// tpv: exact alpha-entmax threshold and value accumulation, one CTA per head
// ---------------------------------------------------------------------------
constexpr int kTpvPmVec = 8;          // page maxima per thread per round trip
constexpr int kTpvPruneTokens = 4096;  // candidate pages' tokens above which t is first bounded

// Union pages i < ucnt of a head whose largest z' exceeds max - 1 (only those
// can hold a token with nonzero weight), written to list[] in a fixed thread
// order (and, with list_x, their maxima minus max); returns their count.  pm[] holds the first round of maxima (entries
// j * blockDim + tid); later rounds are read from pmr (page i at pmr[i]).
// Every thread calls it.
__device__ int list_candidate_pages(float (&pm)[kTpvPmVec], const float* __restrict__ pmr,
                                    int ucnt, float mx, int* list, int* ired,
                                    float* list_x = nullptr) {
    const int tid = threadIdx.x, nt = blockDim.x;
    int npl = 0;
    for (int p0 = 0; p0 < ucnt; p0 += kTpvPmVec * nt) {
        if (p0 > 0) {
#pragma unroll
            for (int j = 0; j < kTpvPmVec; ++j) {
                const int i = p0 + j * nt + tid;
                pm[j] = i < ucnt ? __ldcg(pmr + i) : -INFINITY;
            }
        }
        int c = 0;
#pragma unroll
        for (int j = 0; j < kTpvPmVec; ++j) c += (p0 + j * nt + tid < ucnt) && pm[j] - mx > -1.f;
        int tot;
        int pos = npl + block_exclusive_scan(c, ired, &tot);
#pragma unroll
        for (int j = 0; j < kTpvPmVec; ++j) {
            const int i = p0 + j * nt + tid;
            if (i < ucnt && pm[j] - mx > -1.f) {
                if (list_x) list_x[pos] = pm[j] - mx;
                list[pos++] = i;
            }
        }
        npl += tot;
    }
    __syncthreads();
    return npl;
}
__device__ __forceinline__ float pow_e(float a, int E, float ex) {
    return E == 2 ? a * a : (E == 1 ? a : powf(a, ex));
}

// One step of the threshold solve f(t) = sum_i (x_i - t)_+^e - 1 = 0, x
// relative to the max, on the bracket lo <= t < hi with f(lo) >= 0 > f(hi)
// (initially [-1, 0]: the max alone gives f(-1) >= 0, and f(0) = -1).  f is
// convex and decreasing; d = -f'(t), h = f''(t) (e = 2: 2 #{x_i > t}; e = 1:
// 0, where Halley's step is Newton's).  Left of the root the step is
// Halley's, right of it Newton's (the tangent of a convex f meets 0 left of
// the root), and a step that leaves the bracket bisects it.  Returns true once
// t is the root to 1e-7, at least one unit in the last place on [-1, 0].
__device__ __forceinline__ bool threshold_step(float f, float d, float h, float& t, float& lo,
                                               float& hi) {
    if (f >= 0.f) lo = t; else hi = t;
    float nxt = lo;                                // no slope: bisect
    if (d > 0.f) {
        const float den = 2.f * d * d - f * h;
        const float step = f > 0.f && den > 0.f ? 2.f * f * d / den : f / d;
        nxt = t + step;
        if (fabsf(step) <= 1e-7f) {
            if (nxt > lo && nxt < hi) t = nxt;
            return true;
        }
    }
    if (hi - lo <= 1e-7f) return true;
    t = nxt > lo && nxt < hi ? nxt : 0.5f * (lo + hi);
    return false;
}

// The threshold t of the m candidates x (relative to the max; e = 1, 2) by
// threshold_step, by one warp for m <= 32 * NR candidates (NR per lane in
// registers, shuffle-only reductions), from the bracket [t0, 0] (f(t0) >= 0).
template <int E, int NR>
__device__ float warp_threshold_n(const float* s_vals, int m, float t0) {
    const int lane = threadIdx.x & 31;
    float xr[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int i = j * 32 + lane;
        xr[j] = i < m ? s_vals[i] : -INFINITY;
    }
    float tt = t0, lo = t0, hi = 0.f;
    for (int it = 0; it < 64; ++it) {
        float s0 = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const float a = xr[j] - tt;
            if (a > 0.f) {
                if (E == 2) { s0 = fmaf(a, a, s0); s1 += a; s2 += 1.f; }
                else { s0 += a; s1 += 1.f; }
            }
        }
        s0 = warp_sum(s0);
        s1 = warp_sum(s1);
        if (E == 2) s2 = warp_sum(s2);
        if (threshold_step(s0 - 1.f, E == 2 ? 2.f * s1 : s1, E == 2 ? 2.f * s2 : 0.f, tt, lo, hi))
            break;
    }
    return tt;
}
// m <= 1024: as few registers per lane as the candidates need
template <int E>
__device__ float warp_threshold(const float* s_vals, int m, float t0) {
    if (m <= 64) return warp_threshold_n<E, 2>(s_vals, m, t0);
    if (m <= 256) return warp_threshold_n<E, 8>(s_vals, m, t0);
    return warp_threshold_n<E, 32>(s_vals, m, t0);
}

// The same with every thread of the block taking part (any m).
template <int E, bool kGlobal>
__device__ float solve_threshold(const float* x, int m, float4* red, float t0 = -1.f) {
    float t = t0, lo = t0, hi = 0.f;
    for (int it = 0; it < 64; ++it) {
        float3 acc = make_float3(0.f, 0.f, 0.f);
        for (int i = threadIdx.x; i < m; i += blockDim.x) {
            const float a = (kGlobal ? __ldcg(x + i) : x[i]) - t;
            if (a > 0.f) {
                if (E == 2) { acc.x = fmaf(a, a, acc.x); acc.y += a; acc.z += 1.f; }
                else { acc.x += a; acc.y += 1.f; }
            }
        }
        acc = block_sum3(acc, red);
        if (threshold_step(acc.x - 1.f, E == 2 ? 2.f * acc.y : acc.y, E == 2 ? 2.f * acc.z : 0.f,
                           t, lo, hi))
            break;
    }
    return t;
}

// Weights w = (x - t)_+^e of the m candidates, with the support compacted to
// the front of each warp's contiguous segment of [0, m): x[] takes its
// weights, pos[] keeps its score indices.  A warp writes an entry only at or
// below one it has already read, so no second buffer is needed.  Marks the
// support tokens in `vtok`, adds the weights to `wsum` and returns the warp's
// support count (the same in every lane).
template <int E>
__device__ __forceinline__ int weigh_support(float* x, int* pos, int m, float t, float ex,
                                             uint32_t* vtok, float& wsum) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int seg = (m + nw - 1) / nw;
    const int s0 = min(m, wid * seg), s1 = min(m, s0 + seg);
    int cnt = 0;
    for (int i0 = s0; i0 < s1; i0 += 32) {
        const int i = i0 + lane;
        float w = 0.f;
        int p = 0;
        if (i < s1) {
            const float a = x[i] - t;
            if (a > 0.f) {
                w = pow_e(a, E, ex);
                p = pos[i];
            }
        }
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, w > 0.f);
        __syncwarp();                          // the chunk is read before any write
        if (w > 0.f) {
            const int dst = s0 + cnt + __popc(bal & ((1u << lane) - 1u));
            x[dst] = w;
            pos[dst] = p;
            wsum += w;
            atomicOr(&vtok[p >> 5], 1u << (p & 31));
        }
        cnt += __popc(bal);
    }
    return cnt;
}

// Score index -> V row (-1 for a page without a block) of the warp's
// compacted support entries; independent loads, one round trip per 128.
__device__ __forceinline__ void resolve_support_rows(int* pos, int m, int cnt,
                                                     const int* __restrict__ ublk, int P, int Hkv,
                                                     int kvh) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int s0 = min(m, wid * ((m + nw - 1) / nw));
#pragma unroll 4
    for (int j = s0 + lane; j < s0 + cnt; j += 32) {
        const int p = pos[j];
        const int ui = p / P;
        const int blk = __ldcg(ublk + ui);
        pos[j] = blk >= 0 ? ((blk * Hkv + kvh) * P + (p - ui * P)) : -1;
    }
}

// Index in the candidate arrays of support entry j (0 <= j < the support's
// size), given the warps' support counts.
__device__ __forceinline__ int support_index(int j, const int* wcnt, int m) {
    const int nw = blockDim.x >> 5;
    const int seg = (m + nw - 1) / nw;
    int w = 0;
    while (j >= wcnt[w]) { j -= wcnt[w]; ++w; }
    return w * seg + j;
}

// sum_j w_j V[row_j] over the support (entries taken by row groups of LPR
// lanes, kTpvgRows rows in flight per group), reduced across row groups into
// s_red[0 .. D) by the caller.
template <typename T, int D, int RG, bool kGlobal>
__device__ __forceinline__ void accumulate_support_rows(const float* x, const int* pos, int m,
                                                        int sup, const int* wcnt, const T* vbase,
                                                        float* s_red) {
    constexpr int EPC = Elem<T>::kPer16;
    constexpr int LPR = D / EPC;
    const int lr = threadIdx.x % LPR;
    const int rg = threadIdx.x / LPR;
    float acc[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) acc[e] = 0.f;
    for (int j0 = rg; j0 < sup; j0 += RG * kTpvgRows) {
        float w[kTpvgRows];
        int row[kTpvgRows];
#pragma unroll
        for (int k = 0; k < kTpvgRows; ++k) {
            const int j = j0 + k * RG;
            w[k] = 0.f;
            row[k] = -1;
            if (j < sup) {
                const int i = support_index(j, wcnt, m);
                w[k] = kGlobal ? __ldcg(x + i) : x[i];
                row[k] = kGlobal ? __ldcg(pos + i) : pos[i];
            }
        }
        uint4 r[kTpvgRows];
#pragma unroll
        for (int k = 0; k < kTpvgRows; ++k)
            if (row[k] >= 0) r[k] = ld_nc_v4(vbase + (int64_t)row[k] * D + lr * EPC);
#pragma unroll
        for (int k = 0; k < kTpvgRows; ++k)
            if (row[k] >= 0) {
                float v[EPC];
                Elem<T>::widen(r[k], v);
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[e] = fmaf(w[k], v[e], acc[e]);
            }
    }
#pragma unroll
    for (int e = 0; e < EPC; ++e) s_red[rg * D + lr * EPC + e] = acc[e];
}

// Weights w = (x - t)_+^e of the m candidates of tpv_kernel, the support
// compacted to the front of each warp's contiguous segment of [0, m) in place
// (a warp writes an entry only at or below one it has already read): x[] takes
// the weights and pos[] the V rows.  pos[] holds a candidate's index f into
// the head's candidate pages (page f >> pshift of the list, token f & (P - 1)),
// s_pl / s_pb those pages' union positions and physical blocks.  Marks the
// support tokens in `vtok`, adds the weights to `wsum` and returns the warp's
// support count (the same in every lane).
template <int E>
__device__ __forceinline__ int weigh_listed_support(float* x, int* pos, int m, float t, float ex,
                                                    const int* s_pl, const int* s_pb, int pshift,
                                                    int Hkv, int kvh, uint32_t* vtok,
                                                    float& wsum) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int P = 1 << pshift;
    const int seg = (m + nw - 1) / nw;
    const int s0 = min(m, wid * seg), s1 = min(m, s0 + seg);
    int cnt = 0;
    for (int i0 = s0; i0 < s1; i0 += 32) {
        const int i = i0 + lane;
        float w = 0.f;
        int row = -1, zi = 0;
        if (i < s1) {
            const float a = x[i] - t;
            if (a > 0.f) {
                w = pow_e(a, E, ex);
                const int f = pos[i];
                const int k = f >> pshift, tok = f & (P - 1);
                const int blk = s_pb[k];
                row = blk >= 0 ? (blk * Hkv + kvh) * P + tok : -1;
                zi = (s_pl[k] << pshift) + tok;
            }
        }
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, w > 0.f);
        __syncwarp();                          // the chunk is read before any write
        if (w > 0.f) {
            const int dst = s0 + cnt + __popc(bal & ((1u << lane) - 1u));
            x[dst] = w;
            pos[dst] = row;
            wsum += w;
            atomicOr(&vtok[zi >> 5], 1u << (zi & 31));
        }
        cnt += __popc(bal);
    }
    return cnt;
}

// Threshold and values, one CTA per head, from the per-page maxima qk wrote:
//   1. one round trip for the union size and the head's pmax row: the head's
//      max and the union pages whose maximum is above max - 1 -- only they can
//      hold a token with nonzero weight, since tau >= max - 1;
//   2. one round trip for those pages' scores and physical blocks; the
//      candidates z' - max > -1 are compacted (fixed thread order);
//   3. tau solves sum (z' - tau)_+^(1/(alpha-1)) = 1 by a safeguarded Halley
//      iteration (alpha 1.5 and 2; one warp with the candidates in registers
//      when there are at most 1024) or by bisection (other alpha);
//   4. the weights, the support compacted per warp, and one round trip for its
//      V rows only: out = sum p v / sum p.
template <typename T, int D, int E>   // E: 2 alpha = 1.5, 1 alpha = 2, 0 any other alpha
__global__ void __launch_bounds__(kTpvThreads)
tpv_kernel(int Hq, float alpha, int cand_cap, KV kv, WS ws, DecodeLayout L,
           float* __restrict__ out, float* __restrict__ tau_out, int32_t* __restrict__ support_out) {
    constexpr int EPC = Elem<T>::kPer16;
    constexpr int LPR = D / EPC;              // lanes per V row
    constexpr int RG = kTpvThreads / LPR;     // V rows per pass
    extern __shared__ __align__(16) float s_x[];                      // [cand_cap] x, then weights
    int* s_pos = reinterpret_cast<int*>(s_x + cand_cap);              // [cand_cap] candidate, then V row
    float* s_red = reinterpret_cast<float*>(s_pos + cand_cap);        // [RG][D]
    int* s_pl = reinterpret_cast<int*>(s_red + RG * D);               // [Umax] candidate pages
    int* s_pb = s_pl + L.Umax;                                        // [Umax] their blocks
    __shared__ float fred[40];
    __shared__ float4 f4red[32];
    __shared__ int ired[40];
    __shared__ int s_wcnt[32];
    __shared__ float s_t;

    const int G = L.G;
    const int Hkv = Hq / G;
    const int bh = blockIdx.x;
    const int b = bh / Hq;
    const int h = bh - b * Hq;
    const int kvh = h / G;
    const int hg = h - kvh * G;
    const int u = b * Hkv + kvh;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int P = kv.P;
    const int pshift = P == 32 ? 5 : 4;                               // page sizes are 16 or 32
    const float* z = ws.z + ((int64_t)u * G + hg) * L.Umax * P;
    const float* pmr = ws.pmax + ((int64_t)u * G + hg) * L.Umax;
    float* outb = out + (int64_t)bh * D;

    // 1. the union size and the head's per-page maxima
    for (int i = tid * 32; i < L.Umax; i += kTpvThreads * 32) prefetch_l2_line(pmr + i);
    if (tid == 0) prefetch_l2_line(ws.union_count + u);
    pdl_wait();                               // the scores are the previous kernel's output
    const int ucnt = __ldcg(ws.union_count + u);
    // the head's largest z', which q.K accumulated from the same scores as the
    // page maxima (0: the head has no selected token)
    const uint32_t hkey = __ldcg(ws.head_max + bh);
    float pm[kTpvPmVec];
#pragma unroll
    for (int j = 0; j < kTpvPmVec; ++j) {
        const int i = j * kTpvThreads + tid;
        pm[j] = i < L.Umax ? __ldcg(pmr + i) : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < kTpvPmVec; ++j)
        if (j * kTpvThreads + tid >= ucnt) pm[j] = -INFINITY;
    const float mx = hkey ? key_float(hkey) : -INFINITY;
    if (!(mx > -INFINITY)) {                  // no selected token
        for (int i = tid; i < D; i += blockDim.x) outb[i] = 0.f;
        if (tid == 0) {
            ws.tau[bh] = INFINITY;
            if (tau_out) tau_out[bh] = INFINITY;
            if (support_out) support_out[bh] = 0;
        }
        return;
    }
    // the pages' maxima go to s_x as well when it can hold every union page
    int npl = list_candidate_pages(pm, pmr, ucnt, mx, s_pl, ired,
                                   L.Umax <= cand_cap ? s_x : nullptr);   // ends with a barrier

    // 1b. many candidate tokens: a lower bound of t from the candidate pages'
    // maxima (scores of tokens of the head): their own threshold t_S solves
    // f_S(t_S) = 0 with f_S <= f, so t_S <= t.  Pages whose maximum is at most
    // t_S hold no token of the support and are dropped, tokens at or below it
    // are not candidates, and the solve below starts from t_S.
    float tlo = -1.f;
    if (E != 0 && (npl << pshift) > kTpvPruneTokens && L.Umax <= cand_cap) {
        float ts;
        if (npl <= 1024) {
            if (wid == 0) {
                const float tt = warp_threshold<E>(s_x, npl, -1.f);
                if (lane == 0) s_t = tt;
            }
            __syncthreads();
            ts = s_t;
        } else {
            ts = solve_threshold<E, false>(s_x, npl, f4red);
        }
        tlo = ts - 1e-6f;                     // a margin for the rounding of t_S
        int nl = 0;                           // kept pages, in order, through s_pb
        for (int base = 0; base < npl; base += kTpvThreads) {
            const int k = base + tid;
            const bool keep = k < npl && s_x[k] > tlo;
            int tot;
            const int pos = nl + block_exclusive_scan(keep ? 1 : 0, ired, &tot);
            if (keep) s_pb[pos] = s_pl[k];
            nl += tot;
        }
        __syncthreads();
        for (int k = tid; k < nl; k += kTpvThreads) s_pl[k] = s_pb[k];
        npl = nl;
        __syncthreads();
    }

    // 2. the candidate pages' scores and blocks (all loads in flight before any
    // is used); candidates x = z' - max > tlo in a fixed thread order, pos =
    // index into the candidate pages' tokens
    const int ne = npl << pshift;
    const int* ublk = ws.union_blk + (int64_t)u * L.Umax;
    int m = 0;
    for (int t0 = 0; t0 < ne; t0 += kTpvTile) {
        float v[kTpvVec * 4];
#pragma unroll
        for (int j = 0; j < kTpvVec * 4; ++j) {
            const int f = t0 + j * kTpvThreads + tid;
            v[j] = f < ne ? __ldcg(z + ((int64_t)s_pl[f >> pshift] << pshift) + (f & (P - 1))) : -INFINITY;
        }
        if (t0 == 0) {
            const int blk0 = tid < npl ? __ldcg(ublk + s_pl[tid]) : -1;
            for (int k = tid + kTpvThreads; k < npl; k += kTpvThreads) s_pb[k] = __ldcg(ublk + s_pl[k]);
            if (tid < npl) s_pb[tid] = blk0;
        }
#pragma unroll
        for (int j = 0; j < kTpvVec * 4; ++j) v[j] -= mx;
        int c = 0;
#pragma unroll
        for (int j = 0; j < kTpvVec * 4; ++j) c += v[j] > tlo;
        int tot;
        int pos = m + block_exclusive_scan(c, ired, &tot);
#pragma unroll
        for (int j = 0; j < kTpvVec * 4; ++j) {
            if (v[j] > tlo) {
                if (pos < cand_cap) {
                    s_x[pos] = v[j];
                    s_pos[pos] = t0 + j * kTpvThreads + tid;
                }
                ++pos;
            }
        }
        m += tot;
    }
    m = min(m, cand_cap);                     // the candidates are selected tokens: m <= cand_cap
    __syncthreads();

    // 3. threshold t (relative to the max): f(t) = sum (x - t)_+^e - 1 = 0
    float t;
    if (E != 0 && m <= 1024) {
        if (wid == 0) {
            const float tt = warp_threshold<E>(s_x, m, tlo);
            if (lane == 0) s_t = tt;
        }
        __syncthreads();
        t = s_t;
    } else if (E != 0) {
        t = solve_threshold<E, false>(s_x, m, f4red, tlo);
    } else {
        const float ex = 1.f / (alpha - 1.f);
        float lo = -1.f, hi = -powf(static_cast<float>(m), 1.f - alpha);
        for (int it = 0; it < 48; ++it) {
            const float mid = 0.5f * (lo + hi);
            float f = 0.f;
            for (int i = tid; i < m; i += blockDim.x) {
                const float a = s_x[i] - mid;
                if (a > 0.f) f += powf(a, ex);
            }
            f = block_sum(f, fred) - 1.f;
            if (f >= 0.f) lo = mid; else hi = mid;
        }
        t = 0.5f * (lo + hi);
    }

    // 4. weights, the support compacted per warp (V rows resolved from the
    // candidate pages' blocks), then the support's V rows
    const float ex = 1.f / (alpha - 1.f);
    float wsum = 0.f;
    const int cnt = weigh_listed_support<E>(s_x, s_pos, m, t, ex, s_pl, s_pb, pshift, Hkv, kvh,
                                            ws.vtok + (int64_t)u * L.nvw, wsum);
    if (lane == 0) s_wcnt[wid] = cnt;
    wsum = block_sum(wsum, fred);      // includes a barrier: weights, rows and counts are visible
    int sup = 0;
    for (int w = 0; w < kTpvThreads / 32; ++w) sup += s_wcnt[w];
    accumulate_support_rows<T, D, RG, false>(s_x, s_pos, m, sup, s_wcnt,
                                             static_cast<const T*>(kv.v), s_red);
    __syncthreads();
    for (int d = tid; d < D; d += blockDim.x) {
        float o = 0.f;
        for (int r = 0; r < RG; ++r) o += s_red[r * D + d];
        outb[d] = wsum > 0.f ? o / wsum : 0.f;
    }
    if (tid == 0) {
        const float tau = t + mx;
        ws.tau[bh] = tau;
        if (tau_out) tau_out[bh] = tau;
        if (support_out) support_out[bh] = sup;
    }
}

__global__ void count_rows_kernel(WS ws, DecodeLayout L) {
    const int u = blockIdx.x;
    int c = 0;
    for (int i = threadIdx.x; i < L.nvw; i += blockDim.x) c += __popc(ws.vtok[(int64_t)u * L.nvw + i]);
    c = warp_sum_i(c);
    __shared__ int part[32];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        int s = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += part[w];
        ws.vrows[u] = s;
    }
}

// ---------------------------------------------------------------------------
// tpv over global candidate buffers: the same steps as tpv_kernel for heads
// whose selection (or the whole cache) holds more candidates than shared
// memory does.  Candidates, then weights, live in the head's ccap-entry slice
// of cand_x / cand_pos; every threshold iteration re-reads them (L2).
// ---------------------------------------------------------------------------

template <typename T, int D, int E>
__global__ void __launch_bounds__(kTpvgThreads)
tpv_global_kernel(int Hq, float alpha, KV kv, WS ws, DecodeLayout L, float* __restrict__ out,
                  float* __restrict__ tau_out, int32_t* __restrict__ support_out) {
    constexpr int EPC = Elem<T>::kPer16;
    constexpr int LPR = D / EPC;              // lanes per V row
    constexpr int RG = kTpvgThreads / LPR;     // row groups
    __shared__ float s_red[RG * D];
    __shared__ float fred[40];
    __shared__ float4 f4red[32];
    __shared__ int ired[40];
    __shared__ int s_wcnt[32];

    const int G = L.G;
    const int Hkv = Hq / G;
    const int bh = blockIdx.x;
    const int b = bh / Hq;
    const int h = bh - b * Hq;
    const int kvh = h / G;
    const int hg = h - kvh * G;
    const int u = b * Hkv + kvh;
    const int tid = threadIdx.x;
    const int P = kv.P;
    const float* z = ws.z + ((int64_t)u * G + hg) * L.Umax * P;
    float* cx = ws.cand_x + (int64_t)bh * L.ccap;
    int* cp = ws.cand_pos + (int64_t)bh * L.ccap;
    float* outb = out + (int64_t)bh * D;

    const uint32_t key = __ldcg(ws.head_max + bh);
    const int ucnt = __ldcg(ws.union_count + u);
    const float* pmr = ws.pmax + ((int64_t)u * G + hg) * L.Umax;     // head-major
    float pm[kTpvPmVec];
#pragma unroll
    for (int j = 0; j < kTpvPmVec; ++j) {
        const int i = j * kTpvgThreads + tid;
        pm[j] = i < L.Umax ? __ldcg(pmr + i) : -INFINITY;
    }
    const int n = ucnt * P;
    if (key == 0u || n == 0) {
        for (int i = tid; i < D; i += blockDim.x) outb[i] = 0.f;
        if (tid == 0) {
            ws.tau[bh] = INFINITY;
            if (tau_out) tau_out[bh] = INFINITY;
            if (support_out) support_out[bh] = 0;
        }
        return;
    }
    const float mx = key_float(key);

    // pages that can hold a candidate, then their candidates x = z' - max >
    // -1, compacted in a fixed thread order
    int* pl = ws.plist + (int64_t)bh * L.Umax;
    const int npl = list_candidate_pages(pm, pmr, ucnt, mx, pl, ired);   // ends with a barrier
    int m = 0;
    const int ne = npl * P;
    for (int t0 = 0; t0 < ne; t0 += kTpvgTile) {
        float v[kTpvVec * 4];
        int zi[kTpvVec];
#pragma unroll
        for (int j = 0; j < kTpvVec; ++j) {
            const int e = t0 + (j * kTpvgThreads + tid) * 4;
            zi[j] = e < ne ? __ldcg(pl + e / P) * P + e % P : 0;
            const float4 f = e < ne ? __ldcg(reinterpret_cast<const float4*>(z + zi[j]))
                                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            v[4 * j] = f.x - mx; v[4 * j + 1] = f.y - mx; v[4 * j + 2] = f.z - mx; v[4 * j + 3] = f.w - mx;
        }
        int c = 0;
#pragma unroll
        for (int j = 0; j < kTpvVec * 4; ++j) c += v[j] > -1.f;
        int tot;
        int pos = m + block_exclusive_scan(c, ired, &tot);
#pragma unroll
        for (int j = 0; j < kTpvVec * 4; ++j) {
            if (v[j] > -1.f) {
                if (pos < L.ccap) {
                    cx[pos] = v[j];
                    cp[pos] = zi[j >> 2] + (j & 3);
                }
                ++pos;
            }
        }
        m += tot;
    }
    if (m > L.ccap) {                  // cannot happen: candidates are selected tokens
        if (tid == 0) flag_bad_data();
        m = L.ccap;
    }
    __syncthreads();                   // the block's candidate writes are visible

    // threshold t (relative to the max): f(t) = sum (x - t)_+^e - 1 = 0
    float t;
    if (E != 0) {
        t = solve_threshold<E, true>(cx, m, f4red);
    } else {
        const float ex = 1.f / (alpha - 1.f);
        float lo = -1.f, hi = -powf(static_cast<float>(m), 1.f - alpha);
        for (int it = 0; it < 48; ++it) {
            const float mid = 0.5f * (lo + hi);
            float f = 0.f;
            for (int i = tid; i < m; i += blockDim.x) {
                const float a = __ldcg(cx + i) - mid;
                if (a > 0.f) f += powf(a, ex);
            }
            f = block_sum(f, fred) - 1.f;
            if (f >= 0.f) lo = mid; else hi = mid;
        }
        t = 0.5f * (lo + hi);
    }

    // weights, the support compacted per warp, then its V rows
    const float ex = 1.f / (alpha - 1.f);
    float wsum = 0.f;
    const int cnt = weigh_support<E>(cx, cp, m, t, ex, ws.vtok + (int64_t)u * L.nvw, wsum);
    resolve_support_rows(cp, m, cnt, ws.union_blk + (int64_t)u * L.Umax, P, Hkv, kvh);
    if ((tid & 31) == 0) s_wcnt[tid >> 5] = cnt;
    __syncthreads();                   // (global) weights and rows visible to the block
    wsum = block_sum(wsum, fred);
    int sup = 0;
    for (int w = 0; w < kTpvgThreads / 32; ++w) sup += s_wcnt[w];
    accumulate_support_rows<T, D, RG, true>(cx, cp, m, sup, s_wcnt, static_cast<const T*>(kv.v),
                                            s_red);
    __syncthreads();
    for (int d = tid; d < D; d += blockDim.x) {
        float o = 0.f;
        for (int r = 0; r < RG; ++r) o += s_red[r * D + d];
        outb[d] = wsum > 0.f ? o / wsum : 0.f;
    }
    if (tid == 0) {
        const float tau = t + mx;
        ws.tau[bh] = tau;
        if (tau_out) tau_out[bh] = tau;
        if (support_out) support_out[bh] = sup;
    }
}

// ---------------------------------------------------------------------------
// softmax attention over the union pages (the comparison method)
//
// pv_softmax: the flattened union lists are cut into one contiguous range per
// warp, as for qk; each warp streams its V pages through a private ring of
// bulk copies and, per page, forms the weights e^(z - m_h) of the G heads (z
// from qk, m_h the head's max) and accumulates sum_t w v_t (lane: D / 32
// dimensions of every head) and sum_t w.  A warp flushes one partial record
// per segment of its range inside one unit: segments that start a unit go to
// slot kPvMaxWarps + u, a segment that starts the warp's range inside a unit
// to slot `warp`.  softmax_merge recomputes the segment starts of each unit
// and adds its records in order, so the result does not depend on timing.
// ---------------------------------------------------------------------------
constexpr int kPvWarps = 4;
constexpr int kPvCtasPerSm = 2;
constexpr int kPvStageBytes = 24 * 1024;

template <typename T, int DPL>
__device__ __forceinline__ void load_dpl(const unsigned char* p, float (&x)[DPL]) {
    if constexpr (sizeof(T) == 4) {
        if constexpr (DPL == 4) {
            const float4 f = *reinterpret_cast<const float4*>(p);
            x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
        } else {
            const float2 f = *reinterpret_cast<const float2*>(p);
            x[0] = f.x; x[1] = f.y;
        }
    } else {
        if constexpr (DPL == 4) {
            const uint2 r = *reinterpret_cast<const uint2*>(p);
            x[0] = __uint_as_float(r.x << 16); x[1] = __uint_as_float(r.x & 0xFFFF0000u);
            x[2] = __uint_as_float(r.y << 16); x[3] = __uint_as_float(r.y & 0xFFFF0000u);
        } else {
            const uint32_t r = *reinterpret_cast<const uint32_t*>(p);
            x[0] = __uint_as_float(r << 16); x[1] = __uint_as_float(r & 0xFFFF0000u);
        }
    }
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kPvWarps * 32, kPvCtasPerSm)
pv_softmax_kernel(int Hq, KV kv, WS ws, DecodeLayout L, int ns) {
    constexpr int DPL = D / 32;
    constexpr int NW = (32 * G + 31) / 32;        // weights per lane per page (P <= 32)
    extern __shared__ __align__(128) unsigned char s_pv[];
    __shared__ int red[40];
    __shared__ __align__(8) uint64_t s_bar[kPvWarps][8];
    __shared__ __align__(16) float s_w[kPvWarps][32 * G];     // [token][head]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = kv.P;
    const uint32_t page_bytes = static_cast<uint32_t>(P * D * sizeof(T));
    unsigned char* ring = s_pv + (size_t)warp * ns * page_bytes;
    int* s_prefix = reinterpret_cast<int*>(s_pv + (size_t)kPvWarps * ns * page_bytes);
    uint64_t* bar = s_bar[warp];
    {
        const int U = L.U;
        const int seg = (U + blockDim.x - 1) / blockDim.x;
        const int a0 = min(U, tid * seg), a1 = min(U, a0 + seg);
        int c = 0;
        for (int a = a0; a < a1; ++a) c += __ldcg(ws.union_count + a);
        int tot;
        int run = block_exclusive_scan(c, red, &tot);
        for (int a = a0; a < a1; ++a) {
            s_prefix[a] = run;
            run += __ldcg(ws.union_count + a);
        }
        if (tid == 0) s_prefix[U] = tot;
    }
    if (lane == 0) {
        for (int st = 0; st < ns; ++st) mbar_init(&bar[st], 1);
        mbar_fence_init();
    }
    __syncthreads();
    const int total = s_prefix[L.U];
    const int64_t nwg = (int64_t)gridDim.x * kPvWarps;
    const int wg = blockIdx.x * kPvWarps + warp;
    const int f0 = (int)((int64_t)total * wg / nwg);
    const int f1 = (int)((int64_t)total * (wg + 1) / nwg);
    const int npg = f1 - f0;
    if (npg <= 0) return;
    const unsigned char* vbase = static_cast<const unsigned char*>(kv.v);
    const uint64_t evict_first = l2_evict_first_policy();

    PgDesc cur = resolve_page(f0 + lane, f1, s_prefix, kv, ws, L);
    PgDesc nxt{-1, 0, 0, 0, 0};
    if (npg > 32) nxt = resolve_page(f0 + 32 + lane, f1, s_prefix, kv, ws, L);
    int cur_base = 0;
    auto issue = [&](int k) -> PgDesc {
        PgDesc dsc{-1, 0, 0, 0, 0};
        if (k >= npg) return dsc;
        if (k >= cur_base + 32) {
            cur = nxt;
            cur_base += 32;
            if (npg > cur_base + 32) nxt = resolve_page(f0 + cur_base + 32 + lane, f1, s_prefix, kv, ws, L);
        }
        dsc = shfl_desc(cur, k - cur_base);
        if (lane == 0) {
            const int st = k % ns;
            if (dsc.blk >= 0) {
                mbar_arrive_expect_tx(&bar[st], page_bytes);
                bulk_g2s_hint(ring + (size_t)st * page_bytes,
                              vbase + ((int64_t)dsc.blk * kv.hkv + dsc.u % kv.hkv) * page_bytes,
                              page_bytes, &bar[st], evict_first);
            } else {
                mbar_arrive(&bar[st]);
            }
        }
        return dsc;
    };

    float2 acc[G][DPL / 2];       // coordinate pairs (paired FMAs)
    float lsum[NW];               // this lane's share of sum_t w for head (lane + 32 j) / 32 ... see below
    float mh[G];
    int cur_u = -1, slot = -1;
    auto flush = [&]() {
        float* rec = ws.recs + (int64_t)slot * G * (D + 1);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < DPL / 2; ++e) {
                rec[g * D + lane * DPL + 2 * e] = acc[g][e].x;
                rec[g * D + lane * DPL + 2 * e + 1] = acc[g][e].y;
            }
        // weight index x = lane + 32 j covers head x / 32 (token x % 32)
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const float l = warp_sum(lsum[j]);
            if (lane == 0 && j < G) rec[G * D + j] = l;
        }
    };
    // scores of a page for this lane's weights: entry j = head j, token lane
    // (-inf where the head did not select the page or the token is past the end)
    auto load_z = [&](const PgDesc& dd, float (&zz)[NW]) {
        const float* zrow = ws.z + ((int64_t)dd.u * G) * L.Umax * P + (int64_t)dd.i * P;
#pragma unroll
        for (int j = 0; j < NW; ++j)
            zz[j] = (dd.blk >= 0 && j < G && lane < P && lane < dd.valid && ((dd.mask >> j) & 1))
                        ? __ldcg(zrow + (int64_t)j * L.Umax * P + lane) : -INFINITY;
    };
    PgDesc dq[8];
#pragma unroll
    for (int x = 0; x < 8; ++x)
        if (x < ns - 1) dq[x] = issue(x);
    float zc[NW];                 // the current page's scores, loaded one page ahead
    load_z(dq[0], zc);
    bool failed = false;
    for (int k = 0; k < npg; ++k) {
        const int st = k % ns;
        {
            const PgDesc nd = issue(k + ns - 1);
            const int nst = (k + ns - 1) % ns;
#pragma unroll
            for (int x = 0; x < 8; ++x)
                if (x == nst) dq[x] = nd;
        }
        PgDesc d{}, dn{};
        const int nxs = (k + 1) % ns;
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            if (x == st) d = dq[x];
            if (x == nxs) dn = dq[x];
        }
        float zn[NW];
        if (k + 1 < npg) load_z(dn, zn);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bar[st], (uint32_t)((k / ns) & 1)))) {
            failed = true;
            break;
        }
        if (d.u != cur_u) {
            if (cur_u >= 0) flush();
            cur_u = d.u;
            slot = (f0 + k == s_prefix[d.u]) ? kPvMaxWarps + d.u : wg;
            const int b = cur_u / kv.hkv, kvh = cur_u - b * kv.hkv;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint32_t key = __ldcg(ws.head_max + b * Hq + kvh * G + g);
                mh[g] = key == 0u ? 0.f : key_float(key);      // no score: every weight is 0
#pragma unroll
                for (int e = 0; e < DPL / 2; ++e) acc[g][e] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < NW; ++j) lsum[j] = 0.f;
        }
        // weights of the page: entry j is head j, token lane
#pragma unroll
        for (int j = 0; j < NW; ++j) {
            const float w = (j < G && lane < P) ? __expf(zc[j] - mh[j]) : 0.f;   // e^-inf = 0
            if (j < G && lane < P) s_w[warp][lane * G + j] = w;
            lsum[j] += w;
            zc[j] = zn[j];
        }
        __syncwarp();
        const unsigned char* pg = ring + (size_t)st * page_bytes + (size_t)lane * DPL * sizeof(T);
        const int nt = d.blk >= 0 ? d.valid : 0;
#pragma unroll 4
        for (int t = 0; t < nt; ++t) {
            float v[DPL];
            load_dpl<T, DPL>(pg + (size_t)t * D * sizeof(T), v);
            const float* wt = &s_w[warp][t * G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float w = wt[g];
#pragma unroll
                for (int e = 0; e < DPL / 2; ++e)
                    fma2(acc[g][e], make_float2(w, w), make_float2(v[2 * e], v[2 * e + 1]));
            }
        }
        __syncwarp();        // every lane is done with stage st and s_w before they are refilled
    }
    if (failed) {
        if (lane == 0) flag_timeout();
        return;
    }
    if (cur_u >= 0) flush();
}

// out = sum of the unit's records / sum of their weights; lse = m + log(l).
__global__ void __launch_bounds__(128)
softmax_merge_kernel(int Hq, KV kv, WS ws, DecodeLayout L, int nwg, float* __restrict__ out,
                     float* __restrict__ lse_out) {
    __shared__ int red[40];
    __shared__ int s_w[1024];
    __shared__ int s_n;
    const int G = L.G, D = kv.D;
    const int bh = blockIdx.x;
    const int b = bh / Hq, h = bh - b * Hq;
    const int kvh = h / G, g = h - kvh * G;
    const int u = b * kv.hkv + kvh;
    const int tid = threadIdx.x;
    // a = pages of the units before u, e = a + count_u, total = all pages
    int ca = 0, ct = 0;
    for (int x = tid; x < L.U; x += blockDim.x) {
        const int c = __ldcg(ws.union_count + x);
        ct += c;
        if (x < u) ca += c;
    }
    const int a = block_sum_i(ca, red);
    const int total = block_sum_i(ct, red);
    const int cnt = __ldcg(ws.union_count + u);
    const int e = a + cnt;
    // warps whose range starts strictly inside [a, e) and is not empty, ascending
    if (tid == 0) s_n = 0;
    __syncthreads();
    if (cnt > 0 && total > 0) {
        const int w_lo = (int)(((int64_t)a * nwg) / total);
        const int w_hi = min(nwg - 1, (int)(((int64_t)e * nwg) / total) + 1);
        for (int w = w_lo + tid; w <= w_hi; w += blockDim.x) {
            const int fw = (int)((int64_t)total * w / nwg);
            const int fn = (int)((int64_t)total * (w + 1) / nwg);
            if (fw > a && fw < e && fn > fw) {
                const int at = atomicAdd(&s_n, 1);
                if (at < 1024) s_w[at] = w;
            }
        }
    }
    __syncthreads();
    const int n = min(s_n, 1024);
    if (s_n > 1024 && tid == 0) flag_bad_data();
    // ascending warp order (n is small): one thread sorts
    if (tid == 0)
        for (int i = 1; i < n; ++i) {
            const int v = s_w[i];
            int j = i - 1;
            while (j >= 0 && s_w[j] > v) { s_w[j + 1] = s_w[j]; --j; }
            s_w[j + 1] = v;
        }
    __syncthreads();
    float l = 0.f;
    if (cnt > 0) {
        const float* r0 = ws.recs + (int64_t)(kPvMaxWarps + u) * G * (D + 1);
        l = __ldcg(r0 + G * D + g);
        for (int i = 0; i < n; ++i)
            l += __ldcg(ws.recs + (int64_t)s_w[i] * G * (D + 1) + G * D + g);
    }
    for (int dd = tid; dd < D; dd += blockDim.x) {
        float o = 0.f;
        if (cnt > 0) {
            o = __ldcg(ws.recs + (int64_t)(kPvMaxWarps + u) * G * (D + 1) + g * D + dd);
            for (int i = 0; i < n; ++i)
                o += __ldcg(ws.recs + (int64_t)s_w[i] * G * (D + 1) + g * D + dd);
        }
        out[(int64_t)bh * D + dd] = l > 0.f ? o / l : 0.f;
    }
    if (tid == 0 && lse_out) {
        const uint32_t key = __ldcg(ws.head_max + bh);
        lse_out[bh] = (l > 0.f && key != 0u) ? key_float(key) + logf(l) : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// kept mass: sum over a head's kept tokens of (z' - tau)_+^(1/(alpha-1)) for a
// given threshold tau (e.g. the full-cache one), from the scores a sparse
// decode left in its workspace.  One CTA per head.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
kept_mass_kernel(int Hq, float alpha, int P, WS ws, DecodeLayout L, const float* __restrict__ tau,
                 float* __restrict__ mass) {
    __shared__ float red[40];
    const int G = L.G;
    const int bh = blockIdx.x;
    const int b = bh / Hq, h = bh - b * Hq;
    const int kvh = h / G, hg = h - kvh * G;
    const int u = b * (Hq / G) + kvh;
    const int n = __ldcg(ws.union_count + u) * P;
    const float* z = ws.z + ((int64_t)u * G + hg) * L.Umax * P;
    const float t = __ldg(tau + bh);
    const float ex = 1.f / (alpha - 1.f);
    const int E = fabsf(alpha - 1.5f) < 1e-6f ? 2 : (fabsf(alpha - 2.f) < 1e-6f ? 1 : 0);
    float acc = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float a = __ldcg(z + i) - t;
        if (a > 0.f) acc += pow_e(a, E, ex);
    }
    acc = block_sum(acc, red);
    if (threadIdx.x == 0) mass[bh] = acc;
}

cudaError_t launch_kept_mass(int Hq, float alpha, int P, void* ws_base, const DecodeLayout& L,
                             const float* tau, float* mass, int BH, cudaStream_t s) {
    const WS ws = ws_views(ws_base, L);
    kept_mass_kernel<<<BH, 256, 0, s>>>(Hq, alpha, P, ws, L, tau, mass);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
static cudaEvent_t g_stage_events[4];
static int g_n_stage_events = 0;

void set_decode_stage_events(const cudaEvent_t* events, int n) {
    g_n_stage_events = (events && n == 4) ? 4 : 0;
    for (int i = 0; i < g_n_stage_events; ++i) g_stage_events[i] = events[i];
}

// Under stream capture the marks become event-record nodes of the graph
// (external records), so a replayed graph still times its stages.
static void stage_mark(int i, cudaStream_t s) {
    if (!g_n_stage_events) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(g_stage_events[i], s, cudaEventRecordExternal);
    else
        cudaEventRecord(g_stage_events[i], s);
}

cudaError_t read_decode_counts(void* ws_base, const DecodeLayout& L, int32_t* union_pages,
                               int32_t* v_rows, cudaStream_t s) {
    const WS ws = ws_views(ws_base, L);
    cudaError_t e = cudaSuccess;
    if (union_pages)
        e = cudaMemcpyAsync(union_pages, ws.union_count, sizeof(int32_t) * L.U,
                            cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && v_rows) {
        count_rows_kernel<<<L.U, 256, 0, s>>>(ws, L);
        e = cudaGetLastError();
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(v_rows, ws.vrows, sizeof(int32_t) * L.U, cudaMemcpyDeviceToHost, s);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}

static int sm_count() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
    int v = 148;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) cached[dev] = v;
    return v;
}

template <int E, typename T, int D>
static cudaError_t launch_tpv(float alpha, int Hq, const KV& kv, const WS& ws,
                              const DecodeLayout& L, int cap, float* out, float* tau_out,
                              int32_t* support_out, cudaStream_t s) {
    constexpr int RG = kTpvThreads / (D / Elem<T>::kPer16);
    const int cand_cap = cap * kv.P;
    cudaError_t e;
    if (cand_cap > kTpvSmemCand) {
        if (!ws.cand_x || !ws.plist || L.ccap < cand_cap) return kShapeUnsupported;
        stage_mark(2, s);
        e = launch_kernel(tpv_global_kernel<T, D, E>, dim3(kv.B * Hq), dim3(kTpvgThreads), 0, s, Hq,
                          alpha, kv, ws, L, out, tau_out, support_out);
        if (e != cudaSuccess) return e;
        stage_mark(3, s);
        return cudaSuccess;
    }
    const size_t smem = (size_t)cand_cap * 8 + (size_t)RG * D * sizeof(float) + (size_t)L.Umax * 8;
    e = cudaFuncSetAttribute(tpv_kernel<T, D, E>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    stage_mark(2, s);
    e = launch_kernel_pdl(tpv_kernel<T, D, E>, dim3(kv.B * Hq), dim3(kTpvThreads), smem, s, Hq, alpha,
                      cand_cap, kv, ws, L, out, tau_out, support_out);
    if (e != cudaSuccess) return e;
    stage_mark(3, s);
    return cudaSuccess;
}

// qk after a plan: z = qscale q.k of the union pages, and each head's max;
// with pm also each head's maximum on every union page.
template <typename T, int D, int G>
static cudaError_t launch_qk(const float* q, int Hq, float qscale, const KV& kv, const WS& ws,
                             const DecodeLayout& L, bool pm, cudaStream_t s) {
    cudaError_t e;
    if constexpr (sizeof(T) == 2) {
        const int page_bytes = kv.P * D * 2;
        const int ns = std::min(8, kQmStageBytes / page_bytes);
        const size_t smem = (size_t)kQmWarps * ns * page_bytes + (size_t)(L.U + 1) * sizeof(int);
        if (ns < 2) return kShapeUnsupported;
        auto kernel = pm ? qk_mma_kernel<D, G, true> : qk_mma_kernel<D, G, false>;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        stage_mark(1, s);
        e = launch_kernel_pdl(kernel, dim3(sm_count() * kQmCtasPerSm), dim3(kQmWarps * 32), smem, s, q, Hq,
                          qscale, kv, ws, L, ns);
        if (e != cudaSuccess) return e;
    } else {
        const size_t page_bytes = (size_t)kv.P * D * sizeof(T);
        const size_t fixed = (size_t)kQkConsumers * G * kv.P * 4 + (size_t)((L.U + 1 + 3) & ~3) * 4;
        const size_t per_slot = page_bytes + sizeof(QkInfo) + 16;
        int ns = (int)std::min<size_t>(kQkMaxSlots, (kQkSmemBudget - fixed) / per_slot);
        ns = (ns / kQkConsumers) * kQkConsumers;
        if (ns < kQkConsumers) return kShapeUnsupported;
        const size_t smem = fixed + (size_t)ns * per_slot;
        e = cudaFuncSetAttribute(qk_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        stage_mark(1, s);
        e = launch_kernel(qk_kernel<T, D, G>, dim3(sm_count()), dim3(kQkThreads), smem, s, q, Hq,
                          qscale, kv, ws, L, ns, std::min(kQkGroup, ns), pm ? 1 : 0);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// qk and tpv after a plan: scores of the union pages, then threshold and values.
template <typename T, int D, int G>
static cudaError_t launch_qk_tpv(const float* q, int Hq, float scale, const KV& kv, int cap,
                                 float alpha, float* out, float* tau_out, int32_t* support_out,
                                 const WS& ws, const DecodeLayout& L, cudaStream_t s) {
    // both threshold kernels start from each head's per-page maxima
    cudaError_t e = launch_qk<T, D, G>(q, Hq, (alpha - 1.f) * scale, kv, ws, L, true, s);
    if (e != cudaSuccess) return e;
    const int E = fabsf(alpha - 1.5f) < 1e-6f ? 2 : (fabsf(alpha - 2.f) < 1e-6f ? 1 : 0);
    if (E == 2) return launch_tpv<2, T, D>(alpha, Hq, kv, ws, L, cap, out, tau_out, support_out, s);
    if (E == 1) return launch_tpv<1, T, D>(alpha, Hq, kv, ws, L, cap, out, tau_out, support_out, s);
    return launch_tpv<0, T, D>(alpha, Hq, kv, ws, L, cap, out, tau_out, support_out, s);
}

template <typename T, int D, int G>
static cudaError_t launch_decode_t(const float* q, int Hq, float scale, const KV& kv,
                                   const int32_t* sel, const int32_t* n_sel, int cap, float alpha,
                                   float* out, float* tau_out, int32_t* support_out, const WS& ws,
                                   const DecodeLayout& L, cudaStream_t s, bool planned) {
    cudaError_t e;
    if (L.U > kMaxUnits || cap > kPlanSelRegs * kPlanThreads / G) return kShapeUnsupported;
    stage_mark(0, s);
    if (!planned) {
        const size_t smem = plan_smem_bytes(G, kv.maxp, L.Umax, cap);
        e = cudaFuncSetAttribute(plan_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        e = launch_kernel_pdl(plan_kernel<G>, dim3(L.U), dim3(kPlanThreads), smem, s, kv, Hq, sel,
                          n_sel, cap, ws, L);
        if (e != cudaSuccess) return e;
    }
    return launch_qk_tpv<T, D, G>(q, Hq, scale, kv, cap, alpha, out, tau_out, support_out, ws, L, s);
}

template <typename T, int D, int G>
static cudaError_t launch_decode_full_t(const float* q, int Hq, float scale, const KV& kv,
                                        float alpha, float* out, float* tau_out,
                                        int32_t* support_out, const WS& ws, const DecodeLayout& L,
                                        cudaStream_t s) {
    if (L.U > kMaxUnits || L.Umax != kv.maxp) return kShapeUnsupported;
    stage_mark(0, s);
    const int chunks = (kv.maxp + kPlanAllChunk - 1) / kPlanAllChunk;
    cudaError_t e = launch_kernel(plan_all_kernel, dim3(L.U, chunks), dim3(kPlanThreads), 0, s, kv, Hq,
                                  ws, L);
    if (e != cudaSuccess) return e;
    return launch_qk_tpv<T, D, G>(q, Hq, scale, kv, kv.maxp, alpha, out, tau_out, support_out, ws,
                                  L, s);
}

cudaError_t launch_decode(const float* q, int Hq, float scale, const KV& kv, const int32_t* sel,
                          const int32_t* n_sel, int cap, float alpha, float* out, float* tau_out,
                          int32_t* support_out, void* ws_base, const DecodeLayout& L,
                          cudaStream_t s, bool planned) {
    const WS ws = ws_views(ws_base, L);
    const int G = L.G;
    EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
        return launch_decode_t<T, kD, kG>(q, Hq, scale, kv, sel, n_sel, cap, alpha, out, tau_out,
                                           support_out, ws, L, s, planned);
    })))
    return kShapeUnsupported;
}

template <typename T, int D, int G>
static cudaError_t launch_decode_softmax_t(const float* q, int Hq, float scale, const KV& kv,
                                           const int32_t* sel, const int32_t* n_sel, int cap,
                                           bool full, float* out, float* lse_out, const WS& ws,
                                           const DecodeLayout& L, cudaStream_t s) {
    cudaError_t e;
    if (L.U > kMaxUnits || !ws.recs) return kShapeUnsupported;
    stage_mark(0, s);
    if (full) {
        if (L.Umax != kv.maxp) return kShapeUnsupported;
        const int chunks = (kv.maxp + kPlanAllChunk - 1) / kPlanAllChunk;
        e = launch_kernel(plan_all_kernel, dim3(L.U, chunks), dim3(kPlanThreads), 0, s, kv, Hq, ws, L);
    } else {
        if (cap > kPlanSelRegs * kPlanThreads / G) return kShapeUnsupported;
        const size_t smem = plan_smem_bytes(G, kv.maxp, L.Umax, cap);
        e = cudaFuncSetAttribute(plan_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = launch_kernel_pdl(plan_kernel<G>, dim3(L.U), dim3(kPlanThreads), smem, s, kv, Hq, sel, n_sel,
                          cap, ws, L);
    }
    if (e != cudaSuccess) return e;
    e = launch_qk<T, D, G>(q, Hq, scale, kv, ws, L, false, s);
    if (e != cudaSuccess) return e;
    const int page_bytes = kv.P * D * (int)sizeof(T);
    const int ns = std::max(2, std::min(8, kPvStageBytes / page_bytes));   // 16 KiB fp32 pages: 2
    const int grid = std::min(sm_count() * kPvCtasPerSm, kPvMaxWarps / kPvWarps);
    const size_t smem = (size_t)kPvWarps * ns * page_bytes + (size_t)(L.U + 1) * sizeof(int);
    e = cudaFuncSetAttribute(pv_softmax_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    stage_mark(2, s);
    e = launch_kernel(pv_softmax_kernel<T, D, G>, dim3(grid), dim3(kPvWarps * 32), smem, s, Hq, kv, ws,
                      L, ns);
    if (e != cudaSuccess) return e;
    e = launch_kernel(softmax_merge_kernel, dim3(kv.B * Hq), dim3(128), 0, s, Hq, kv, ws, L,
                      grid * kPvWarps, out, lse_out);
    if (e != cudaSuccess) return e;
    stage_mark(3, s);
    return cudaSuccess;
}

cudaError_t launch_decode_softmax(const float* q, int Hq, float scale, const KV& kv,
                                  const int32_t* sel, const int32_t* n_sel, int cap, bool full,
                                  float* out, float* lse_out, void* ws_base, const DecodeLayout& L,
                                  cudaStream_t s) {
    const WS ws = ws_views(ws_base, L);
    const int G = L.G;
    EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
        return launch_decode_softmax_t<T, kD, kG>(q, Hq, scale, kv, sel, n_sel, cap, full, out,
                                                   lse_out, ws, L, s);
    })))
    return kShapeUnsupported;
}

cudaError_t launch_decode_full(const float* q, int Hq, float scale, const KV& kv, float alpha,
                               float* out, float* tau_out, int32_t* support_out, void* ws_base,
                               const DecodeLayout& L, cudaStream_t s) {
    const WS ws = ws_views(ws_base, L);
    const int G = L.G;
    EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
        return launch_decode_full_t<T, kD, kG>(q, Hq, scale, kv, alpha, out, tau_out, support_out,
                                                ws, L, s);
    })))
    return kShapeUnsupported;
}

}  // namespace ekv
