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
    float* pmax;          // [U][G][Umax] largest z' of each union page per head
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

// Shared memory build_plan needs: [G][ceil(max_pages/32)] bitmap words,
// [Umax] union pages and [G * cap] staged selection entries (ints).
inline size_t plan_smem_bytes(int G, int max_pages, int Umax, int cap) {
    return (size_t)G * ((max_pages + 31) / 32) * 4 + (size_t)Umax * 4 + (size_t)G * cap * 4;
}

// The union plan of unit u = (sequence b, kv head) from its G heads' page
// bitmaps s_bits ([G][nwm] words, nwm = ceil(max_pages / 32); words past the
// sequence's pages are not read): the ascending union of the pages, each
// page's head mask and physical block, and the union size.  Called by every
// thread of the block; `red` >= 40 ints.  s_pblk (nullable): the sequence's
// page-table row in shared memory; without it the blocks are read from the
// page table in global memory, and s_upage ([Umax]) is scratch.  Entries
// outside [0, num_blocks) are flagged and planned as -1.
template <int G>
__device__ void plan_from_bits(const KV& kv, const WS& ws, const DecodeLayout& L, int u,
                               const uint32_t* s_bits, int* s_upage, int* red,
                               const int* s_pblk = nullptr) {
    const int nwm = (kv.maxp + 31) / 32;
    const int b = u / kv.hkv;
    const int tid = threadIdx.x, nt = blockDim.x;
    // bitmap bytes (8 pages each) split over the threads: a thread emits at
    // most 8 pages per byte it holds
    const int nb8 = (pages_of(kv, b) + 7) / 8;
    const int seg = (nb8 + nt - 1) / nt;
    const int y0 = min(nb8, tid * seg), y1 = min(nb8, y0 + seg);
    auto head_byte = [&](int h, int y) -> uint32_t {
        return (s_bits[h * nwm + (y >> 2)] >> (8 * (y & 3))) & 0xFFu;
    };
    int cnt = 0;
    for (int y = y0; y < y1; ++y) {
        uint32_t x = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) x |= head_byte(h, y);
        cnt += __popc(x);
    }
    int total;
    int idx = block_exclusive_scan(cnt, red, &total);
    int* upage = ws.union_page + (int64_t)u * L.Umax;
    int* umask = ws.union_mask + (int64_t)u * L.Umax;
    int* ublk = ws.union_blk + (int64_t)u * L.Umax;
    for (int y = y0; y < y1; ++y) {
        uint32_t hw[G];
        uint32_t uw = 0;
#pragma unroll
        for (int h = 0; h < G; ++h) { hw[h] = head_byte(h, y); uw |= hw[h]; }
        while (uw) {
            const int bit = __ffs(uw) - 1;
            uw &= uw - 1;
            int mask = 0;
#pragma unroll
            for (int h = 0; h < G; ++h) mask |= static_cast<int>((hw[h] >> bit) & 1u) << h;
            const int page = y * 8 + bit;
            upage[idx] = page;
            umask[idx] = mask;
            if (s_pblk) {
                int blk = s_pblk[page];
                if (blk < 0 || blk >= kv.nb) {
                    flag_bad_data();
                    blk = -1;
                }
                ublk[idx] = blk;
            } else {
                s_upage[idx] = page;
            }
            ++idx;
        }
    }
    if (tid == 0) ws.union_count[u] = total;
    if (s_pblk) return;
    __syncthreads();
    // physical blocks of the union pages (one parallel page-table round trip)
    for (int i = tid; i < total; i += nt) {
        int blk = kv.pt[(int64_t)b * kv.maxp + s_upage[i]];
        if (blk < 0 || blk >= kv.nb) {
            flag_bad_data();
            blk = -1;
        }
        ublk[i] = blk;
    }
}

// The union plan of unit u from its G heads' selection rows already in
// shared memory (s_sel [G][cap], s_ns [G] counts, each in [0, cap]): the
// rows are set into the bitmaps s_bits ([G][nwm] words, scratch), then
// plan_from_bits.  s_upage ([Umax]) is scratch; `red` >= 40 ints.  Pages
// outside the sequence are skipped and flagged.
template <int G>
__device__ void plan_from_rows(const KV& kv, int cap, const WS& ws, const DecodeLayout& L, int u,
                               const int* s_sel, const int* s_ns, uint32_t* s_bits, int* s_upage,
                               int* red) {
    const int nwm = (kv.maxp + 31) / 32;
    const int b = u / kv.hkv;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int np = pages_of(kv, b);
    const int nw = (np + 31) / 32;
    for (int i = tid; i < G * nw; i += nt) {
        const int h = i / nw;
        s_bits[h * nwm + (i - h * nw)] = 0u;
    }
    __syncthreads();
    for (int e = tid; e < G * cap; e += nt) {
        const int h = e / cap, r = e - h * cap;
        if (r < s_ns[h]) {
            const int p = s_sel[e];
            if (p >= 0 && p < np) atomicOr(&s_bits[h * nwm + (p >> 5)], 1u << (p & 31));
            else flag_bad_data();
        }
    }
    __syncthreads();
    plan_from_bits<G>(kv, ws, L, u, s_bits, s_upage, red);
}

// Resets unit u's per-call state: its heads' maxima and V-row marks.
__device__ __forceinline__ void plan_reset_unit(int Hq, int G, const WS& ws, const DecodeLayout& L,
                                                const KV& kv, int u) {
    const int b = u / kv.hkv, kvh = u - b * kv.hkv;
    const int tid = threadIdx.x, nt = blockDim.x;
    if (tid < G) ws.head_max[b * Hq + kvh * G + tid] = 0u;
    for (int i = tid; i < L.nvw; i += nt) ws.vtok[(int64_t)u * L.nvw + i] = 0u;
}

// Union plan of unit u = (sequence b, kv head) from the selection in global
// memory: the counts and every row entry are staged in shared memory in one
// round trip (entries past a head's count are read but not used), then
// plan_from_rows; also resets the unit's per-call state.  Needs G * cap <=
// kPlanSelRegs * blockDim.x; `s_bits`, `s_upage` and `s_sel` as sized by
// plan_smem_bytes, `red` >= 40 ints, `s_ns` >= G.
template <int G>
__device__ void build_plan(const KV& kv, int Hq, const int32_t* __restrict__ sel,
                           const int32_t* __restrict__ n_sel, int cap, const WS& ws,
                           const DecodeLayout& L, int u, uint32_t* s_bits, int* s_upage,
                           int* s_sel, int* red, int* s_ns) {
    const int b = u / kv.hkv;
    const int kvh = u - b * kv.hkv;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int bh0 = b * Hq + kvh * G;
    const int ns_reg = tid < G ? __ldcg(n_sel + bh0 + tid) : 0;
    int pv[kPlanSelRegs];
#pragma unroll
    for (int k = 0; k < kPlanSelRegs; ++k) {
        const int e = tid + k * nt;
        pv[k] = e < G * cap ? __ldcg(sel + (int64_t)bh0 * cap + e) : -1;
    }
    plan_reset_unit(Hq, G, ws, L, kv, u);
    // the entries go to shared memory before the barrier: their loads complete
    // here, in one round trip with the counts
#pragma unroll
    for (int k = 0; k < kPlanSelRegs; ++k) {
        const int e = tid + k * nt;
        if (e < G * cap) s_sel[e] = pv[k];
    }
    if (tid < G) {
        int ns = ns_reg;
        if (ns < 0 || ns > cap) {
            flag_bad_data();
            ns = max(0, min(ns, cap));
        }
        s_ns[tid] = ns;
    }
    __syncthreads();
    plan_from_rows<G>(kv, cap, ws, L, u, s_sel, s_ns, s_bits, s_upage, red);
}

}  // namespace ekv
