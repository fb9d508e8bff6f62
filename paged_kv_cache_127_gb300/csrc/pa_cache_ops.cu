// pa_cache_ops.cu -- the two companion kernels of paged decode, plus the
// cross-partition merge of the split-K decode.
//
//  - write_kv (reshape-and-cache): each new token's K and V rows go to its slot,
//    k_cache[slot / B, h, slot % B, :] = k[t, h, :].  ("PagedAttention: Virtual
//    Memory for the KV Cache", "Sharing a prefix and copying a partial block":
//    the engine writes the new entry into the block its table points at.)
//  - copy_blocks: copy-on-write copy of whole physical blocks, src -> dst, in
//    both caches (same section; "Paged Attention and vLLM", "Continuous
//    Batching and Scheduler", the copy-on-write rule).
//  - merge: o = sum_b 2^(m_b - m*) acc_b / sum_b 2^(m_b - m*) l_b with
//    m* = max_b m_b, over the partitions of one (sequence, query head)
//    ("Paged Attention and vLLM", "Paged Attention CUDA Kernel", merge
//    equation; m is kept in log2 units, so the weights are powers of two).
//
// The copies move 16-byte vectors; every row is a multiple of 16 bytes.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void write_kv_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                const int64_t *__restrict__ slots, int Hkv, int row_chunks, int B,
                                int N, uint4 *__restrict__ kc, uint4 *__restrict__ vc,
                                unsigned int *err) {
    // Launched as a programmatic dependent: wait for the previous kernel in the
    // stream (it may still be reading the caches), then let the next one start
    // its set-up -- it waits for this grid before it reads the caches.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int t = blockIdx.x;
    const int64_t slot = slots[t];
    if (slot < 0) return;
    if (slot >= (int64_t)N * B) {
        if (threadIdx.x == 0) set_error(err, PA_DEVERR_BAD_SLOT);
        return;
    }
    const int64_t blk = slot / B;
    const int64_t off = slot % B;
    const int per_cache = Hkv * row_chunks;
    for (int c = threadIdx.x; c < 2 * per_cache; c += blockDim.x) {
        const bool is_v = c >= per_cache;
        const int cc = is_v ? c - per_cache : c;
        const int h = cc / row_chunks;
        const int w = cc - h * row_chunks;
        const size_t src = ((size_t)t * Hkv + h) * row_chunks + w;
        const size_t dst = (((size_t)blk * Hkv + h) * B + off) * row_chunks + w;
        if (is_v)
            vc[dst] = v[src];
        else
            kc[dst] = k[src];
    }
}

// Copy `chunks` 16-byte chunks of one block (source and destination blocks
// are distinct, so the ranges do not overlap).  The CTA's slice (blockIdx.z
// of gridDim.z) is copied kCopyUnroll chunks per thread at a time: all loads
// first, then all stores, so each thread keeps kCopyUnroll reads in flight
// (a read of pinned host memory crosses the CPU-GPU link, with a long latency).
constexpr int kCopyUnroll = 8;

__device__ __forceinline__ void copy_chunks(const uint4 *__restrict__ from, uint4 *__restrict__ to, int64_t chunks) {
    const int64_t stride = (int64_t)blockDim.x * gridDim.z;
    for (int64_t i0 = threadIdx.x + (int64_t)blockIdx.z * blockDim.x; i0 < chunks; i0 += stride * kCopyUnroll) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < chunks) v[u] = from[i];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < chunks) to[i] = v[u];
        }
    }
}

// grid: (pair, 2 * layer + {0: K, 1: V}, slice of the block)
__global__ void copy_blocks_kernel(uint4 *kc, uint4 *vc, const int64_t *__restrict__ pairs,
                                   int64_t chunks, int64_t layer_chunks, int N, unsigned int *err) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int p = blockIdx.x;
    const int64_t src = pairs[2 * p];
    const int64_t dst = pairs[2 * p + 1];
    if (src < 0 || src >= N || dst < 0 || dst >= N) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_error(err, PA_DEVERR_BAD_PAIR);
        return;
    }
    uint4 *base = ((blockIdx.y & 1) ? vc : kc) + (int64_t)(blockIdx.y >> 1) * layer_chunks;
    copy_chunks(base + src * chunks, base + dst * chunks, chunks);
}

// Block swap between a device pool and a host pool (pinned host memory the
// GPU reads and writes directly over the CPU-GPU link).  grid: (pair,
// 2 * layer + {0: K, 1: V}, slice).  pairs[i] = (source block, destination
// block) in the direction's (from, to) pools.
__global__ void swap_blocks_kernel(const uint4 *from_k, const uint4 *from_v, uint4 *to_k, uint4 *to_v,
                                   const int64_t *__restrict__ pairs, int64_t chunks, int64_t from_layer,
                                   int64_t to_layer, int from_n, int to_n, unsigned int *err) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int p = blockIdx.x;
    const int64_t src = pairs[2 * p];
    const int64_t dst = pairs[2 * p + 1];
    if (src < 0 || src >= from_n || dst < 0 || dst >= to_n) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_error(err, PA_DEVERR_BAD_PAIR);
        return;
    }
    const int64_t layer = blockIdx.y >> 1;
    const uint4 *from = ((blockIdx.y & 1) ? from_v : from_k) + layer * from_layer + src * chunks;
    uint4 *to = ((blockIdx.y & 1) ? to_v : to_k) + layer * to_layer + dst * chunks;
    copy_chunks(from, to, chunks);
}

cudaError_t launch_swap_blocks(const void *from_k, const void *from_v, void *to_k, void *to_v,
                               const int64_t *pairs, int P, int64_t block_bytes, int layers, int64_t from_layer_bytes,
                               int64_t to_layer_bytes, int from_n, int to_n, unsigned int *err, cudaStream_t st) {
    if (P == 0 || layers == 0) return cudaSuccess;
    const int64_t chunks = block_bytes / 16;
    const int threads = 256;
    int z = (int)((chunks + threads * 8 - 1) / (threads * 8));
    if (z < 1) z = 1;
    if (z > 64) z = 64;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P, 2u * (unsigned)layers, (unsigned)z);
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, swap_blocks_kernel, static_cast<const uint4 *>(from_k),
                              static_cast<const uint4 *>(from_v), static_cast<uint4 *>(to_k),
                              static_cast<uint4 *>(to_v), pairs, chunks, from_layer_bytes / 16, to_layer_bytes / 16,
                              from_n, to_n, err);
}

// One warp per (sequence, query head); lane i owns D/32 consecutive outputs.
// Partials are read kU partitions per round trip.  The kernel may be launched
// as a programmatic dependent of the decode kernel: it waits for that grid
// (and so for every partial) before reading.
template <int D>
__global__ void decode_merge_kernel(const DecodeArgs a) {
    constexpr int kPer = D / 32;
    constexpr int kU = 4;
#ifndef PA_MERGE_FAST_PARTS
#define PA_MERGE_FAST_PARTS 8
#endif
    constexpr int kFastParts = PA_MERGE_FAST_PARTS;  // rows with at most this many partitions merge in one round trip
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int gw = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (gw >= a.S * a.Hq) return;
    const int s = gw / a.Hq;
    int len = a.context_lens[s];
    const int cap = a.max_blocks * a.B;
    len = len < 0 ? 0 : (len > cap ? cap : len);
    const int np = (len + a.partition_size - 1) / a.partition_size;
    if (np <= 1) return;  // finished in place by the partition kernel
    const size_t r0 = (size_t)gw * a.max_parts;
    const float *ml = a.ws_ml + 2 * r0;
    const float *acc = a.ws_acc + r0 * D;
    if (kFastParts > 0 && np <= kFastParts) {
        // one round trip: every lane loads all (m, l) pairs (broadcast) and its
        // slice of every partial sum together, then combines them in registers
        float2 w[kFastParts > 0 ? kFastParts : 1];
        float x[kFastParts > 0 ? kFastParts : 1][kPer];
#pragma unroll
        for (int p = 0; p < kFastParts; ++p) {
            if (p < np) {
                w[p] = *reinterpret_cast<const float2 *>(ml + 2 * p);
#pragma unroll
                for (int i = 0; i < kPer; ++i) x[p][i] = acc[(size_t)p * D + lane * kPer + i];
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int p = 0; p < kFastParts; ++p)
            if (p < np) M = fmaxf(M, w[p].x);
        float L = 0.f, o[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) o[i] = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int p = 0; p < kFastParts; ++p) {
                if (p < np) {
                    const float wt = ex2(w[p].x - M);
                    L += wt * w[p].y;
#pragma unroll
                    for (int i = 0; i < kPer; ++i) o[i] += wt * x[p][i];
                }
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        float *dst = a.out + (size_t)gw * D + lane * kPer;
#pragma unroll
        for (int i = 0; i < kPer; ++i) dst[i] = o[i] * inv;
        return;
    }
    float M = -INFINITY;
    for (int p = lane; p < np; p += 32) M = fmaxf(M, ml[2 * p]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    float o[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) o[i] = 0.f;
    if (M != -INFINITY) {
        for (int p0 = 0; p0 < np; p0 += kU) {
            float2 w[kU];
            float x[kU][kPer];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int p = p0 + u < np ? p0 + u : p0;
                w[u] = p0 + u < np ? *reinterpret_cast<const float2 *>(ml + 2 * p) : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int i = 0; i < kPer; ++i) x[u][i] = acc[(size_t)p * D + lane * kPer + i];
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const float wt = ex2(w[u].x - M);  // 0 for the padding entries
                L += wt * w[u].y;
#pragma unroll
                for (int i = 0; i < kPer; ++i) o[i] += wt * x[u][i];
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float *dst = a.out + (size_t)gw * D + lane * kPer;
#pragma unroll
    for (int i = 0; i < kPer; ++i) dst[i] = o[i] * inv;
}

cudaError_t launch_decode_merge(const DecodeArgs &a, cudaStream_t st) {
    const int warps = a.S * a.Hq;
    const int per_block = 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + per_block - 1) / per_block));
    cfg.blockDim = dim3(per_block * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.D == 64) return cudaLaunchKernelEx(&cfg, decode_merge_kernel<64>, a);
    if (a.D == 128) return cudaLaunchKernelEx(&cfg, decode_merge_kernel<128>, a);
    return cudaErrorNotSupported;
}

cudaError_t launch_write_kv(const void *k, const void *v, const int64_t *slots, int T, int Hkv,
                            int row_bytes, int B, int N, void *k_cache, void *v_cache,
                            unsigned int *err, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)T);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, write_kv_kernel, static_cast<const uint4 *>(k), static_cast<const uint4 *>(v),
                              slots, Hkv, row_bytes / 16, B, N, static_cast<uint4 *>(k_cache),
                              static_cast<uint4 *>(v_cache), err);
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int P,
                               int64_t block_bytes, int N, int layers, int64_t layer_bytes, unsigned int *err,
                               cudaStream_t st) {
    if (P == 0 || layers == 0) return cudaSuccess;
    const int64_t chunks = block_bytes / 16;
    const int threads = 256;
    int z = (int)((chunks + threads * 8 - 1) / (threads * 8));  // ~8 vectors per thread
    if (z < 1) z = 1;
    if (z > 64) z = 64;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P, 2u * (unsigned)layers, (unsigned)z);
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_blocks_kernel, static_cast<uint4 *>(k_cache),
                              static_cast<uint4 *>(v_cache), pairs, chunks, layer_bytes / 16, N, err);
}

}  // namespace pa
