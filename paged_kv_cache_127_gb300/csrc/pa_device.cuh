// pa_device.cuh -- small sm_103a device helpers used by the libpa kernels:
// mbarrier + 1-D bulk (TMA) copy wrappers in inline PTX, ex2, and 16-byte
// chunk -> fp32 unpacking for the three storage types.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "../../include/pa.h"

namespace pa {

// Polls of a bounded mbarrier wait before a kernel reports a timeout.
constexpr uint32_t kWaitLimit = 1u << 22;

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    uint64_t state;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
                 : "=l"(state)
                 : "r"(bar), "r"(bytes)
                 : "memory");
    (void)state;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    uint64_t state;
    asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(state) : "r"(bar) : "memory");
    (void)state;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after `limit` polls (each try_wait may itself
// suspend for a while).  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// 1-D bulk copy global -> shared, completing `bytes` transaction bytes on
// `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Same with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------ math
// 2^x with the hardware approximation (ex2.approx, flush-to-zero); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// ------------------------------------------------------------------ storage types
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kBytes = 4;
    static constexpr int kVec = 4;  // elements per 16-byte chunk
    static __device__ __forceinline__ void unpack(const uint4 &c, float *f) {
        f[0] = __uint_as_float(c.x);
        f[1] = __uint_as_float(c.y);
        f[2] = __uint_as_float(c.z);
        f[3] = __uint_as_float(c.w);
    }
};

template <>
struct Elem<__half> {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
    static __device__ __forceinline__ float2 pair(uint32_t w) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
    static __device__ __forceinline__ void unpack(const uint4 &c, float *f) {
        float2 a = pair(c.x), b = pair(c.y), d = pair(c.z), e = pair(c.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = d.x; f[5] = d.y; f[6] = e.x; f[7] = e.y;
    }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    static constexpr int kVec = 8;
    // bfloat16 is the top half of a binary32: widening is a shift / mask.
    static __device__ __forceinline__ void unpack(const uint4 &c, float *f) {
        f[0] = __uint_as_float(c.x << 16); f[1] = __uint_as_float(c.x & 0xffff0000u);
        f[2] = __uint_as_float(c.y << 16); f[3] = __uint_as_float(c.y & 0xffff0000u);
        f[4] = __uint_as_float(c.z << 16); f[5] = __uint_as_float(c.z & 0xffff0000u);
        f[6] = __uint_as_float(c.w << 16); f[7] = __uint_as_float(c.w & 0xffff0000u);
    }
};

__device__ __forceinline__ void set_error(unsigned int *err, unsigned int bit) {
    if (err) atomicOr(err, bit);
}

// Exclusive scan of hist[hi], hist[hi - 1], ..., hist[hi - nb + 1] (largest
// bin first) into start[]; returns the total.  Every thread of a 1024-thread block calls it; nb <= 1024.
__device__ __forceinline__ int scan_bins_desc(const int *hist, int *start, int hi, int nb, int *warp_sums) {
    const int t = threadIdx.x;
    const int lane = t & 31, wid = t >> 5;
    const int v = t < nb ? hist[hi - t] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += u;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    if (t < nb) start[hi - t] = (wid > 0 ? warp_sums[wid - 1] : 0) + incl - v;
    const int total = warp_sums[31];
    __syncthreads();
    return total;
}

}  // namespace pa
