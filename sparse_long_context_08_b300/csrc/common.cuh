// Shared device helpers for the EntmaxKV kernels (sm_103a): element widening,
// warp/block reductions, order-preserving float keys, and the mbarrier + bulk
// copy (TMA, cp.async.bulk) primitives used to stage K/V pages.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "internal.h"

namespace ekv {

// ---------------------------------------------------------------------------
// elements: fp32, or bf16 stored as raw 16-bit patterns (widened exactly)
// ---------------------------------------------------------------------------
struct bf16raw { uint16_t bits; };

template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int kPer16 = 4;   // elements per 16-byte chunk
    __device__ __forceinline__ static void widen(const uint4& r, float* o) {
        o[0] = __uint_as_float(r.x); o[1] = __uint_as_float(r.y);
        o[2] = __uint_as_float(r.z); o[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static float one(const float* p, int64_t i) { return p[i]; }
    __device__ __forceinline__ static void store(float* p, int64_t i, float v) { p[i] = v; }
};
template <> struct Elem<bf16raw> {
    static constexpr int kPer16 = 8;
    __device__ __forceinline__ static void widen(const uint4& r, float* o) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = __uint_as_float(w[i] << 16);
            o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static float one(const bf16raw* p, int64_t i) {
        return __uint_as_float(static_cast<uint32_t>(p[i].bits) << 16);
    }
    // only used for values that are themselves widened bf16 (exact)
    __device__ __forceinline__ static void store(bf16raw* p, int64_t i, float v) {
        p[i].bits = static_cast<uint16_t>(__float_as_uint(v) >> 16);
    }
};

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// ---------------------------------------------------------------------------
// reductions
// ---------------------------------------------------------------------------
template <int kLanes>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ uint32_t warp_max_u(uint32_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Block-wide reductions; `red` is shared scratch of >= 32 entries.  Every
// thread of the block must call them; all threads receive the result.
__device__ __forceinline__ float block_max(float v, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    v = lane < nw ? red[lane] : -INFINITY;
    return warp_max(v);
}
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    v = lane < nw ? red[lane] : 0.f;
    return warp_sum(v);
}
__device__ __forceinline__ float2 block_sum2(float2 v, float2* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v.x = warp_sum(v.x);
    v.y = warp_sum(v.y);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    v = lane < nw ? red[lane] : make_float2(0.f, 0.f);
    v.x = warp_sum(v.x);
    v.y = warp_sum(v.y);
    return v;
}
// Block-wide sum of a float3; `red` >= 32 float4.
__device__ __forceinline__ float3 block_sum3(float3 v, float4* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v.x = warp_sum(v.x);
    v.y = warp_sum(v.y);
    v.z = warp_sum(v.z);
    __syncthreads();
    if (lane == 0) red[wid] = make_float4(v.x, v.y, v.z, 0.f);
    __syncthreads();
    const float4 r = lane < nw ? red[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    return make_float3(warp_sum(r.x), warp_sum(r.y), warp_sum(r.z));
}
__device__ __forceinline__ int block_sum_i(int v, int* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_sum_i(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    v = lane < nw ? red[lane] : 0;
    return warp_sum_i(v);
}
__device__ __forceinline__ uint32_t block_max_u(uint32_t v, uint32_t* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    v = warp_max_u(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    v = lane < nw ? red[lane] : 0u;
    return warp_max_u(v);
}

// Exclusive block scan of one int per thread; returns the prefix and writes
// the block total to *total.  `red` needs >= 33 ints.
__device__ __forceinline__ int block_exclusive_scan(int v, int* red, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) red[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int s = lane < nw ? red[lane] : 0;
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xFFFFFFFFu, si, o);
            if (lane >= o) si += n;
        }
        if (lane < nw) red[lane] = si - s;
        if (lane == 31) red[32] = si;
    }
    __syncthreads();
    int r = red[wid] + incl - v;
    *total = red[32];
    return r;
}

// Same for floats (inclusive prefix of one value per thread).
__device__ __forceinline__ float block_inclusive_scan_f(float v, float* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    float incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) red[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        float s = lane < nw ? red[lane] : 0.f;
        float si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float n = __shfl_up_sync(0xFFFFFFFFu, si, o);
            if (lane >= o) si += n;
        }
        if (lane < nw) red[lane] = si - s;
    }
    __syncthreads();
    float r = red[wid] + incl;
    __syncthreads();
    return r;
}

// ---------------------------------------------------------------------------
// order-preserving uint32 keys of floats (-0 folded into +0, NaN to -inf)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t float_key(float f) {
    if (f != f) f = -INFINITY;
    f = f + 0.0f;
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}

// ---------------------------------------------------------------------------
// mbarrier + 1-D bulk async copy (TMA engine), with bounded waits
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Plain arrival (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase with the given parity; gives up after limit_ns and
// returns false (the caller records a timeout and stops issuing work).
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    return mbar_wait_for(bar, parity, kWaitLimitNs);
}
// Global -> shared bulk copy, completion signalled on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------------------
// kernel launch
// ---------------------------------------------------------------------------
// The kernels of a step run back to back in stream order.  Launching them with
// programmatic dependent launch (the successor's blocks resident early, waiting
// on griddepcontrol) measured slower at the 128K workload: 116.6-119.0 us per
// step against 113.4-114.3 us without (means of the step graph); the waiting
// blocks of the big score and value kernels cost more than the launch latency
// they hide.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Programmatic dependent launch: a kernel launched with launch_kernel_pdl may
// start while the previous kernel in the stream is still running; it calls
// pdl_wait() before its first read of that kernel's output (the wait returns
// once the previous grid has completed and its memory is visible; without the
// launch attribute it returns at once).  A kernel calls pdl_trigger() when its
// main work is done, so that the next kernel's CTAs can be placed on SMs it
// frees while its last CTAs finish.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// cp.async of 16 bytes global -> shared, of which src_bytes (0 or 16) are
// read and the rest zero-filled; cp_async_wait_all waits for all of this
// thread's copies.
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// The same with an L2 cache policy (createpolicy) for the read lines.
__device__ __forceinline__ void cp_async16_zfill_hint(void* dst, const void* src, int src_bytes,
                                                      uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes), "l"(policy) : "memory");
}

// Requests the 128-byte line holding p into L2 (and its address translation);
// no value is read, so the line may still be written by another kernel.
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// L2 policy for data read once (the K/V pools and page metadata streams): the
// lines are the first to go, so the small per-step arrays written between the
// kernels (bounds, scores) stay in L2 for the next kernel.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// ---------------------------------------------------------------------------
// exact bf16 splitting and the bf16 tensor-core product
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// 5th-generation tensor core (tcgen05) primitives
// ---------------------------------------------------------------------------

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (TMA, tensor core operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle
// layout: 8-row atoms of 128-byte rows, atoms 1024 bytes apart (stride byte
// offset), the leading byte offset unused; start address >> 4 in bits 0-13,
// descriptor version 1 in bits 46-48, swizzle mode 2 (128 B) in bits 61-63.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B (both
// K-major), fp32 accumulator, M x N.
template <int M, int N>
__device__ __forceinline__ constexpr uint32_t umma_idesc_bf16_f32() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, one thread issues.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, int accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on bar when every tcgen05 operation this thread issued before
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}
// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes (lane i of the
// warp reads TMEM lane (taddr >> 16) + i), then waits for the load.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t bf16_rn_bits(float x) {
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// Term s (0 hi, 1 mid, 2 lo) of the three-way bf16 split of x: hi + mid + lo
// == x exactly for normal x (8 + 8 + 8 significand bits cover fp32's 24).
__device__ __forceinline__ uint32_t split_term(float x, int s) {
    const uint32_t hi = bf16_rn_bits(x);
    const float r1 = x - __uint_as_float(hi << 16);
    const uint32_t mid = bf16_rn_bits(r1);
    const float r2 = r1 - __uint_as_float(mid << 16);
    const uint32_t lo = bf16_rn_bits(r2);
    return s == 0 ? hi : (s == 1 ? mid : lo);
}

// d = a * b + d on both lanes of a float pair, one rounding each (paired fp32 FMA).
__device__ __forceinline__ void fma2(float2& d, float2 a, float2 b) {
    unsigned long long dd = *reinterpret_cast<unsigned long long*>(&d);
    const unsigned long long aa = *reinterpret_cast<unsigned long long*>(&a);
    const unsigned long long bb = *reinterpret_cast<unsigned long long*>(&b);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(dd) : "l"(aa), "l"(bb));
    d = *reinterpret_cast<float2*>(&dd);
}

// c += A (16 x 16, row) * B (16 x 8, col), bf16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace ekv
