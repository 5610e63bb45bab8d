// Decode workspace views and the per-unit union plan of the decode kernels.
//
// Include after EKV_DEFINE_STATUS(...): build_plan reports malformed
// selections through the translation unit's flag_bad_data().
#pragma once

#include "common.cuh"

namespace ekv {

constexpr int kPlanSelRegs = 32;       // selection entries held per thread while planning

// Workspace views (device addresses).
struct WS {
    int* union_count;
    uint32_t* head_max;   // order-preserving keys of each head's max z'
    int* union_page;      // [U][Umax] logical pages of the unit's union, ascending
    int* union_mask;      // [U][Umax] heads (bits) that selected the page
    int* union_blk;       // [U][Umax] physical block of the page (-1: bad page-table entry)
    uint32_t* vtok;       // [U][nvw] tokens whose V row was read
    int* vrows;           // per-unit popcount of vtok (measurement)
    float* z;             // [U][G][Umax * P]
    float* pmax;          // [U][Umax][G] largest z' of each union page per head
    float* tau;
    float* cand_x;        // [B * Hq][ccap] candidates, then weights (large selections only)
    int* cand_pos;        // [B * Hq][ccap] their score index, then V row
    int* plist;           // [B * Hq][Umax] pages that may hold candidates (large selections)
    float* recs;          // [nrec][G][D + 1] softmax partial sums (softmax decode only)
};
inline WS ws_views(void* base, const DecodeLayout& L) {
    char* c = static_cast<char*>(base);
    return WS{reinterpret_cast<int*>(c + L.union_count), reinterpret_cast<uint32_t*>(c + L.head_max),
              reinterpret_cast<int*>(c + L.union_page), reinterpret_cast<int*>(c + L.union_mask),
              reinterpret_cast<int*>(c + L.union_blk), reinterpret_cast<uint32_t*>(c + L.vtok),
              reinterpret_cast<int*>(c + L.vrows), reinterpret_cast<float*>(c + L.z),
              reinterpret_cast<float*>(c + L.pmax), reinterpret_cast<float*>(c + L.tau),
              L.cand_x ? reinterpret_cast<float*>(c + L.cand_x) : nullptr,
              L.cand_pos ? reinterpret_cast<int*>(c + L.cand_pos) : nullptr,
              L.plist ? reinterpret_cast<int*>(c + L.plist) : nullptr,
              L.recs ? reinterpret_cast<float*>(c + L.recs) : nullptr};
}

__device__ __forceinline__ int pages_of(const KV& kv, int b) {
    return min(kv.maxp, (kv.sl[b] + kv.P - 1) / kv.P);
}

// Shared memory build_plan needs: [G][ceil(max_pages/32)] bitmap words plus
// [Umax] union pages (ints).
inline size_t plan_smem_bytes(int G, int max_pages, int Umax) {
    return (size_t)G * ((max_pages + 31) / 32) * 4 + (size_t)Umax * 4;
}

// Union plan of unit u = (sequence b, kv head): the ascending union of the G
// heads' selected pages, each page's head mask and physical block; also resets
// the unit's per-call state (head maxima, V-row marks).  Called by every
// thread of the block; needs G * cap <= kPlanSelRegs * blockDim.x.  `s_bits`
// and `s_upage` as sized by plan_smem_bytes, `red` >= 40 ints, `s_ns` >= G.
template <int G>
__device__ void build_plan(const KV& kv, int Hq, const int32_t* __restrict__ sel,
                           const int32_t* __restrict__ n_sel, int cap, const WS& ws,
                           const DecodeLayout& L, int u, uint32_t* s_bits, int* s_upage,
                           int* red, int* s_ns) {
    const int nwm = (kv.maxp + 31) / 32;
    const int b = u / kv.hkv;
    const int kvh = u - b * kv.hkv;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh0 = b * Hq + kvh * G;
    // one round trip: the counts and, speculatively, every selection row in
    // full (entries past a head's count are read but not used)
    if (tid < G) s_ns[tid] = __ldcg(n_sel + bh0 + tid);
    int pv[kPlanSelRegs];
#pragma unroll
    for (int k = 0; k < kPlanSelRegs; ++k) {
        const int e = tid + k * nt;
        pv[k] = e < G * cap ? __ldcg(sel + (int64_t)bh0 * cap + e) : -1;
    }
    const int np = pages_of(kv, b);
    const int nw = (np + 31) / 32;
    for (int i = tid; i < G * nw; i += nt) {
        const int h = i / nw;
        s_bits[h * nwm + (i - h * nw)] = 0u;
    }
    if (tid < G) ws.head_max[bh0 + tid] = 0u;
    for (int i = tid; i < L.nvw; i += nt) ws.vtok[(int64_t)u * L.nvw + i] = 0u;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPlanSelRegs; ++k) {
        const int e = tid + k * nt;
        if (e < G * cap) {
            const int h = e / cap, r = e - h * cap;
            int ns = s_ns[h];
            if (ns < 0 || ns > cap) {
                if (r == 0) flag_bad_data();
                ns = max(0, min(ns, cap));
            }
            if (r < ns) {
                const int p = pv[k];
                if (p >= 0 && p < np) atomicOr(&s_bits[h * nwm + (p >> 5)], 1u << (p & 31));
                else flag_bad_data();
            }
        }
    }
    __syncthreads();

    const int seg = (nw + nt - 1) / nt;
    const int w0 = min(nw, tid * seg), w1 = min(nw, w0 + seg);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) {
        uint32_t x = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) x |= s_bits[h * nwm + w];
        cnt += __popc(x);
    }
    int total;
    int idx = block_exclusive_scan(cnt, red, &total);
    int* upage = ws.union_page + (int64_t)u * L.Umax;
    int* umask = ws.union_mask + (int64_t)u * L.Umax;
    for (int w = w0; w < w1; ++w) {
        uint32_t hw[G];
        uint32_t uw = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) { hw[h] = s_bits[h * nwm + w]; uw |= hw[h]; }
        while (uw) {
            const int bit = __ffs(uw) - 1;
            uw &= uw - 1;
            int mask = 0;
#pragma unroll
            for (int h = 0; h < G; ++h) mask |= static_cast<int>((hw[h] >> bit) & 1u) << h;
            upage[idx] = w * 32 + bit;
            umask[idx] = mask;
            s_upage[idx] = w * 32 + bit;
            ++idx;
        }
    }
    __syncthreads();
    // physical blocks of the union pages (one parallel page-table round trip)
    int* ublk = ws.union_blk + (int64_t)u * L.Umax;
    for (int i = tid; i < total; i += nt) {
        int blk = kv.pt[(int64_t)b * kv.maxp + s_upage[i]];
        if (blk < 0 || blk >= kv.nb) {
            flag_bad_data();
            blk = -1;
        }
        ublk[i] = blk;
    }
    if (tid == 0) ws.union_count[u] = total;
}

}  // namespace ekv
