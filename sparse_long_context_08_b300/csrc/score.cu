// Query-aware page scoring [EntmaxKV §2.A].
//
//   bbox:  U_p = s * sum_j max(q_j kmin_j, q_j kmax_j)   (upper bound on s q.k)
//   gauss: m_p = s q.mean_p,  s_p = s sqrt(sum_j q_j^2 var_pj)
//
// Two kernels.  bf16 metadata with 4 or 8 kv heads takes the bbox bound on
// the tensor cores (score_bbox_tc_kernel, described where it is defined).
// Every other case -- fp32 metadata, the Gaussian statistics, other head
// layouts -- takes score_kernel, an HBM-bound streaming kernel on the CUDA
// cores.  Its valid pages of all sequences, in
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
#include <climits>

#include "common.cuh"

EKV_DEFINE_STATUS(score)

namespace ekv {

constexpr int kScoreWarps = 8;
constexpr int kScoreThreads = 32 * kScoreWarps;
constexpr int kScoreCtasPerSm = 2;   // fp32 rows with G <= 4 take ScoreCfg::CTAS = 3
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
    // CTAs per SM: a third for fp32 rows of up to 4 heads per kv head (they fit
    // 80 registers; more warps hide the per-row chain of shuffles)
    static constexpr int CTAS = (ES == 4 && G <= 4) ? 3 : kScoreCtasPerSm;
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
// Arrive-on `bar` triggered when all of this thread's earlier cp.async copies
// have completed; the barrier's expected count includes it (no increment).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
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
__global__ void __launch_bounds__(kScoreThreads, (ScoreCfg<T, D, G, kGauss>::CTAS))
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
                pdl_wait();                    // q may be the previous kernel's output
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
    pdl_trigger();                      // the selection's CTAs may take their places
}

// ---------------------------------------------------------------------------
// The bbox bound on the tensor cores (bf16 metadata).
//
// The bound of page p for query head h of kv head g is
//     U_ph = sum_k A_(p,g)k B_(g,h)k,
//     A_(p,g) = [kmin_pg | kmax_pg],   B_(g,h) = [s min(q_h, 0) | s max(q_h, 0)]
// (K = 2D): the product of the metadata rows (one per page and kv head) with
// the query columns.  B is fp32; every column is the exact sum of three bf16
// terms (split_term), so the bf16 operands lose nothing.
//
// A tile is PPT = 128 / HKV consecutive pages of one sequence with all HKV kv
// heads (M = 128 rows, row = g * PPT + page), so the copies read each page's
// metadata block whole: the HKV rows of a block are contiguous (2 KB of kmin
// and 2 KB of kmax per block at D = 128, 8 kv heads), where one kv head's
// 256-byte row per page would be a random access into a scattered page table.
// B holds the columns of every kv head of the sequence (N = HKV * 3G, padded
// to 16): the MMA also forms the products of a row with the other kv heads'
// columns, which are not read (the tensor core has the cycles to spare).
//
// A CTA (one per SM) takes a contiguous range of tiles:
//   warps 0-7  per K half of a tile (kmin, then kmax): resolve the tile's
//              pages in the page table (prefetched one tile ahead) and copy
//              the rows with 16-byte cp.async, 512 contiguous bytes per warp
//              instruction, each chunk straight to its place in the
//              128B-swizzled K-major operand layout.  The stage's barrier
//              completes through cp.async arrive-on as the copies land, so a
//              producer never waits on its own copies.  When the tile's
//              sequence changes, B is rebuilt once the MMAs of the earlier
//              stages are done.  (Copies of one kv head's rows per tile ran at
//              half the speed; TMA gathers of the 128-byte row segments were
//              slower still: the copy engine takes the small rows one by one.)
//   warp 8     owns the TMEM columns (two accumulators); one thread fences the
//              landed copies for the tensor core, issues the D / 16 MMAs of a
//              stage (M = 128, K = 16 each) and commits them to the stage's
//              "empty" and, after the second half, the accumulator's "full"
//              barrier;
//   warps 9-12 read their 32 rows' window of the accumulator (TMEM lane =
//              row), add each head's three terms and store the bounds.
// Every hand-over is an mbarrier and every wait is bounded: a wait that gives
// up flags the score status and ends the CTA's loops.
// ---------------------------------------------------------------------------
static int sm_count_score();

constexpr int kTcRows = 128;
constexpr int kTcProdWarps = 8;                               // copy warps
constexpr int kTcProd = 32 * kTcProdWarps;
constexpr int kTcMmaWarp = kTcProdWarps;                      // then 4 epilogue warps
constexpr int kTcThreads = 32 * (kTcProdWarps + 5);
constexpr int kTcMaxSeqs = 1024;
constexpr int kTcSmemBudget = 216 * 1024;

template <int D, int G, int HKV>
struct TcCfg {
    static constexpr int PPT = kTcRows / HKV;                   // pages per tile
    static constexpr int KPW = 32 / PPT;                        // kv heads per 32 rows
    static constexpr int N = ((HKV * 3 * G + 15) / 16) * 16;    // MMA columns
    static constexpr int NW = ((KPW * 3 * G + 15) / 16) * 16;   // columns an epilogue warp reads
    static constexpr int KBH = D / 64;                          // 64-element K blocks per half
    static constexpr int A_BYTES = kTcRows * D * 2;             // one K half of a tile
    static constexpr int B_HALF = N * D * 2;
    static constexpr int B_BYTES = 2 * B_HALF;
    static constexpr int SA = (kTcSmemBudget - B_BYTES) / A_BYTES;
    static constexpr int S = SA < 8 ? SA : 8;
    // the last warp's window of the second accumulator ends past 2N when N is small
    static constexpr int MAXC = 2 * N > N + 3 * KPW * 3 * G + NW ? 2 * N : N + 3 * KPW * 3 * G + NW;
    static constexpr int TMEM_COLS = MAXC <= 32 ? 32 : MAXC <= 64 ? 64 : MAXC <= 128 ? 128
                                   : MAXC <= 256 ? 256 : 512;
    static_assert(PPT >= 1 && PPT <= 32 && 32 % PPT == 0, "tile rows");
    static_assert(N <= 256, "MMA columns");
    static_assert(S >= 2, "stage ring");
    static_assert(A_BYTES % 1024 == 0 && (N * 128) % 1024 == 0, "1024-byte aligned atoms");
    static_assert(N + (3 * KPW * 3 * G) + NW <= TMEM_COLS, "epilogue window inside the columns");
};

struct TcSh {
    uint64_t full[8], bfull[8], empty[8], accf[2], acce[2], binit;
    uint32_t tmem;
    int abort;
};

// Tile t (< B * tps, tps = ceil(max_pages / PPT) tiles per sequence) ->
// sequence, first page, pages of the sequence in the tile (<= 0: none).  The
// fixed number of tiles per sequence lets a CTA find its tiles without the
// sequence lengths, so its first page-table loads need not wait for them.
template <int PPT>
__device__ __forceinline__ void tc_tile(int t, int tps, const KV& kv, int& b, int& p0, int& npg) {
    b = t / tps;
    p0 = (t - b * tps) * PPT;
    const int np = min(kv.maxp, (__ldg(kv.sl + b) + kv.P - 1) / kv.P);
    npg = min(PPT, np - p0);
}

// B (N x 2D, K-major, 128B swizzle, two K halves) for sequence b: row
// g * 3G + 3h + term holds term `term` of s min(q, 0) (half 0, against kmin)
// and s max(q, 0) (half 1, against kmax) of query head g * G + h.  A thread
// takes (head, 8-coordinate chunk) pairs, loads of all its pairs in flight
// together, and writes the six chunks (two halves x three terms) each one
// feeds; padding rows are zero.
template <int D, int G, int HKV, int NT>
__device__ __forceinline__ void tc_build_b(unsigned char* bs, const float* __restrict__ q,
                                           float scale, int b, int t) {
    using C = TcCfg<D, G, HKV>;
    constexpr int nt = NT;                         // threads taking part
    constexpr int CH = D / 8;                      // chunks per head and half
    constexpr int PAIRS = HKV * G * CH;
    constexpr int PER = (PAIRS + NT - 1) / NT;     // pairs per thread
    const float* qb = q + (int64_t)b * HKV * G * D;
    float4 v[PER][2];
#pragma unroll
    for (int x = 0; x < PER; ++x) {
        const int pr = t + x * nt;
        if (pr < PAIRS) {
            const float4* src = reinterpret_cast<const float4*>(qb + (pr / CH) * D + (pr % CH) * 8);
            v[x][0] = __ldg(src);
            v[x][1] = __ldg(src + 1);
        }
    }
#pragma unroll
    for (int x = 0; x < PER; ++x) {
        const int pr = t + x * nt;
        if (pr >= PAIRS) continue;
        const int qh = pr / CH, k0 = (pr % CH) * 8;
        const int kb = k0 / 64, cin = (k0 % 64) / 8;
        const float e8[8] = {v[x][0].x, v[x][0].y, v[x][0].z, v[x][0].w,
                             v[x][1].x, v[x][1].y, v[x][1].z, v[x][1].w};
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int term = 0; term < 3; ++term) {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float sv = scale * e8[e];
                    const float xv = half ? fmaxf(sv, 0.f) : fminf(sv, 0.f);
                    w[e >> 1] |= split_term(xv, term) << ((e & 1) * 16);
                }
                const int n = qh * 3 + term;
                unsigned char* dst = bs + half * C::B_HALF + kb * (C::N * 128) + n * 128 +
                                     ((cin ^ (n & 7)) * 16);
                *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            }
    }
    // padding rows
    constexpr int PADC = (C::N - HKV * 3 * G) * 2 * CH;
    for (int c = t; c < PADC; c += nt) {
        const int n = HKV * 3 * G + c / (2 * CH), kc = c % (2 * CH);
        const int half = kc / CH, k0 = (kc % CH) * 8;
        *reinterpret_cast<uint4*>(bs + half * C::B_HALF + (k0 / 64) * (C::N * 128) + n * 128 +
                                  ((((k0 % 64) / 8) ^ (n & 7)) * 16)) = make_uint4(0u, 0u, 0u, 0u);
    }
}

template <int D, int G, int HKV>
__global__ void __launch_bounds__(kTcThreads, 1)
score_bbox_tc_kernel(const bf16raw* __restrict__ kmin, const bf16raw* __restrict__ kmax,
                     const float* __restrict__ q, float scale, KV kv, float* __restrict__ out) {
    using C = TcCfg<D, G, HKV>;
    constexpr int S = C::S, PPT = C::PPT;
    constexpr int Hq = HKV * G;
    extern __shared__ unsigned char s_raw[];
    unsigned char* bbuf = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(s_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char* ring = bbuf + C::B_BYTES;
    __shared__ TcSh sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tps = (kv.maxp + PPT - 1) / PPT;       // tiles per sequence

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&sh.full[i], kTcProd);
            mbar_init(&sh.bfull[i], kTcProd);
            mbar_init(&sh.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) { mbar_init(&sh.accf[i], 1); mbar_init(&sh.acce[i], 128); }
        mbar_init(&sh.binit, 128);
        sh.abort = 0;
        mbar_fence_init();
    }
    if (warp == kTcMmaWarp) tmem_alloc(&sh.tmem, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem;
    const int total = kv.B * tps;
    const int t0 = (int)((int64_t)total * blockIdx.x / gridDim.x);
    const int t1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
    const int nt = t1 - t0;
    volatile int* abort = &sh.abort;

    if (warp < kTcProdWarps) {
        // ---- producers: one K half of a tile per iteration
        constexpr int CPH = D * 2 / 16;                // 16-byte chunks per row
        constexpr int RPI = 32 / CPH;                  // rows (kv heads) per warp instruction
        constexpr int PPW = PPT / kTcProdWarps;        // pages per producer warp
        constexpr int IPP = HKV / RPI;                 // instructions per page
        static_assert(PPW >= 1 && PPT % kTcProdWarps == 0 && HKV % RPI == 0, "producer mapping");
        const int sub = lane / CPH, c = lane % CPH;
        const int kb = (c * 8) / 64, cin = c % 8;
        // the metadata is read once: its lines go first, so the bounds this
        // kernel writes are still in L2 for the selection
        const uint64_t evict_first = l2_evict_first_policy();
        // this lane's page (warp * PPW + lane, lanes < PPW) of tile i: its page
        // table entry, checked only when used (the load stays in flight)
        constexpr int kNoPage = INT_MIN;               // lane without a page in the tile
        // tile i: its sequence (returned) and this lane's page table entry
        auto page_block = [&](int i, int& blk) {
            const int t = t0 + i;
            const int b = t / tps;
            const int p = (t - b * tps) * PPT + warp * PPW + lane;
            // the entry (inside the table row) is loaded with the sequence
            // length; it is kept only for a page of the sequence
            const int e = (lane < PPW && p < kv.maxp) ? __ldg(kv.pt + (int64_t)b * kv.maxp + p) : 0;
            int bb, p0, npg;
            tc_tile<PPT>(t, tps, kv, bb, p0, npg);
            blk = (lane < PPW && warp * PPW + lane < npg) ? e : kNoPage;
            return b;
        };
        auto checked = [&](int blk) {
            if (blk == kNoPage) return -1;
            if (blk < 0 || blk >= kv.nb) { flag_bad_data(); return -1; }
            return blk;
        };
        int blk_cur = -1, blk_next = kNoPage, b_cur = -1, b_next = -1;
        if (nt > 0) {
            b_cur = page_block(0, blk_cur);
            blk_cur = checked(blk_cur);
        }
        int bseq = b_cur;                              // sequence whose columns B holds
                                                       // (the first: built by the epilogue warps)
        int j = 0;
        for (; j < 2 * nt && !*abort; ++j) {
            const int i = j >> 1, half = j & 1, s = j % S, u = j / S;
            if (half == 0) {                           // the next tile's pages, one tile ahead
                if (i > 0) {
                    blk_cur = checked(blk_next);
                    b_cur = b_next;
                }
                if (i + 1 < nt) b_next = page_block(i + 1, blk_next);
            }
            if (u > 0 && !mbar_wait(&sh.empty[s], (u - 1) & 1)) {
                *abort = 1;
                if (lane == 0) flag_timeout();
                break;
            }
            unsigned char* st = ring + (size_t)s * C::A_BYTES;
            const bf16raw* msrc = half ? kmax : kmin;
#pragma unroll 4
            for (int x = 0; x < PPW * IPP; ++x) {
                const int pw = x / IPP;                // page within the warp's
                const int g = (x % IPP) * RPI + sub;   // kv head
                const int blk = __shfl_sync(0xFFFFFFFFu, blk_cur, pw);
                const int r = g * PPT + warp * PPW + pw;   // row within the tile
                const bf16raw* src = msrc + ((int64_t)(blk >= 0 ? blk : 0) * HKV + g) * D + c * 8;
                unsigned char* dst = st + kb * (kTcRows * 128) + r * 128 + ((cin ^ (r & 7)) * 16);
                cp_async16_zfill_hint(dst, src, blk >= 0 ? 16 : 0, evict_first);
            }
            cp_async_arrive_noinc(&sh.full[s]);        // arrives once this thread's copies land
            // B for the tile's sequence, built while the copies are in flight
            if (b_cur != bseq) {
                // the MMAs of every earlier stage (issued in order) must be done
                if (j > 0 && !mbar_wait(&sh.empty[(j - 1) % S], ((j - 1) / S) & 1)) {
                    *abort = 1;
                    if (lane == 0) flag_timeout();
                    break;
                }
                pdl_wait();                            // q may be the previous kernel's output
                tc_build_b<D, G, HKV, kTcProd>(bbuf, q, scale, b_cur, tid);
                bseq = b_cur;
                fence_proxy_async_smem();              // B, written by this thread
            }
            mbar_arrive(&sh.bfull[s]);
        }
        cp_async_wait_all();                           // nothing stays in flight past the loop
    } else if (warp == kTcMmaWarp) {
        // ---- MMA issue (one thread)
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16_f32<kTcRows, C::N>();
            const uint32_t sbb = smem_u32(bbuf);
            int issued = 0;
            if (nt > 0 && !mbar_wait(&sh.binit, 0)) { *abort = 1; flag_timeout(); }
            for (int j = 0; j < 2 * nt && !*abort; ++j) {
                const int i = j >> 1, half = j & 1, s = j % S, u = j / S, a = i & 1, v = i >> 1;
                if (!mbar_wait(&sh.full[s], u & 1) || !mbar_wait(&sh.bfull[s], u & 1) ||
                    (half == 0 && v > 0 && !mbar_wait(&sh.acce[a], (v - 1) & 1))) {
                    *abort = 1;
                    flag_timeout();
                    break;
                }
                // the copies landed through the generic proxy: order them before
                // the tensor core's (async proxy) reads of the stage
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t sa = smem_u32(ring + (size_t)s * C::A_BYTES);
                const uint32_t sb = sbb + half * C::B_HALF;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int kb = ks >> 2, kin = ks & 3;
                    umma_bf16(tmem + a * C::N,
                              umma_desc_sw128(sa + kb * (kTcRows * 128) + kin * 32),
                              umma_desc_sw128(sb + kb * (C::N * 128) + kin * 32), idesc,
                              half > 0 || ks > 0);
                }
                umma_commit(&sh.empty[s]);
                if (half == 1) {
                    umma_commit(&sh.accf[a]);
                    issued = i + 1;
                }
            }
            // every issued MMA has completed before the columns are freed
            if (issued > 0) mbar_wait(&sh.accf[(issued - 1) & 1], ((issued - 1) >> 1) & 1);
        }
        __syncwarp();
    } else {
        // ---- epilogue: TMEM lane = row = kv head * PPT + page of the tile
        const int quarter = warp & 3;
        const int m = quarter * 32 + lane;
        const int g = m / PPT, pi = m % PPT;
        const int go = lane / PPT;                     // kv head within the warp's window
        const int col0 = (quarter * 32 / PPT) * 3 * G;
        if (nt > 0) {                                  // B of the first tile's sequence
            int b, p0, npg;
            tc_tile<PPT>(t0, tps, kv, b, p0, npg);
            pdl_wait();                                // q may be the previous kernel's output
            tc_build_b<D, G, HKV, 128>(bbuf, q, scale, b, tid - (kTcMmaWarp + 1) * 32);
            fence_proxy_async_smem();
            mbar_arrive(&sh.binit);
        }
        for (int i = 0; i < nt && !*abort; ++i) {
            const int a = i & 1, v = i >> 1;
            if (!mbar_wait(&sh.accf[a], v & 1)) {
                *abort = 1;
                if (lane == 0) flag_timeout();
                break;
            }
            tc_fence_after();
            uint32_t r[C::NW];
#pragma unroll
            for (int x = 0; x < C::NW; x += 16)
                tmem_ld16(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * C::N + col0 + x,
                          *reinterpret_cast<uint32_t(*)[16]>(r + x));
            tc_fence_before();
            mbar_arrive(&sh.acce[a]);
            int b, p0, npg;
            tc_tile<PPT>(t0 + i, tps, kv, b, p0, npg);
            if (pi < npg) {
                const int p = p0 + pi;
                const int blk = __ldg(kv.pt + (int64_t)b * kv.maxp + p);
                const bool live = blk >= 0 && blk < kv.nb;
#pragma unroll
                for (int o = 0; o < C::KPW; ++o) {
                    if (o != go) continue;
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        const int x = o * 3 * G + 3 * h;
                        const float ub = (__uint_as_float(r[x + 2]) + __uint_as_float(r[x + 1])) +
                                         __uint_as_float(r[x]);
                        out[((int64_t)b * Hq + g * G + h) * kv.maxp + p] = live ? ub : -INFINITY;
                    }
                }
            }
        }
    }
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// cudaErrorNotSupported: this shape takes the CUDA-core kernel.
template <int D, int G, int HKV>
static cudaError_t launch_score_tc_t(const float* q, float scale, const KV& kv, const void* kmin,
                                     const void* kmax, float* out, cudaStream_t s) {
    using C = TcCfg<D, G, HKV>;
    if (kv.B > kTcMaxSeqs || (reinterpret_cast<uintptr_t>(kmin) & 15) ||
        (reinterpret_cast<uintptr_t>(kmax) & 15))
        return cudaErrorNotSupported;
    const size_t smem = 1024 + C::B_BYTES + (size_t)C::S * C::A_BYTES;
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        smem + sizeof(TcSh) + 256 > (size_t)optin)
        return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(score_bbox_tc_kernel<D, G, HKV>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel_pdl(score_bbox_tc_kernel<D, G, HKV>, dim3(sm_count_score()), dim3(kTcThreads),
                         smem, s, static_cast<const bf16raw*>(kmin),
                         static_cast<const bf16raw*>(kmax), q, scale, kv, out);
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
    if (kv.B > kScoreMaxSeqs || kv.maxp >= (1 << 17)) return kShapeUnsupported;
    using C = ScoreCfg<T, D, G, kGauss>;
    const int grid = sm_count_score() * C::CTAS;
    const int64_t total_max = (int64_t)kv.B * kv.maxp;
    const int nloc_max = (int)((total_max + grid - 1) / grid) + 1;
    const size_t ring_bytes = (size_t)kScoreWarps * kScoreStages * 2 * 32 * C::DPL * sizeof(T);
    const size_t smem = ring_bytes + (size_t)(kv.B + 1 + 2 * nloc_max) * sizeof(int);
    if (smem > 110 * 1024) return kShapeUnsupported;
    cudaError_t e = cudaFuncSetAttribute(score_kernel<T, D, G, kGauss>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel_pdl(score_kernel<T, D, G, kGauss>, dim3(grid), dim3(kScoreThreads), smem, s, q, Hq,
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
        if (kv.dtype == 1) {
            // bf16 metadata: the tensor-core kernel, unless the shape is outside it
            cudaError_t e = cudaErrorNotSupported;
            if (kv.hkv == 8 && G <= 8) {
                EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
                    e = launch_score_tc_t<kD, kG, 8>(q, scale, kv, kmin, kmax, out, s);
                }))
            } else if (kv.hkv == 4) {
                EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
                    e = launch_score_tc_t<kD, kG, 4>(q, scale, kv, kmin, kmax, out, s);
                }))
            }
            if (e != cudaErrorNotSupported) return e;
        }
        EKV_DISPATCH_T(kv.dtype, EKV_DISPATCH_D(kv.D, EKV_DISPATCH_G(G, {
            return launch_score_t<T, kD, kG, false>(q, Hq, scale, kv, kmin, kmax, out, s);
        })))
    }
    return kShapeUnsupported;
}

}  // namespace ekv
