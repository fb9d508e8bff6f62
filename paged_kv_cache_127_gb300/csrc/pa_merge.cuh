// pa_merge.cuh -- the cross-partition merge of split-K attention partials
// ("Paged Attention and vLLM", "Paged Attention CUDA Kernel", the merge
// equation):
//
//   o = sum_b 2^(m_b - m*) acc_b / sum_b 2^(m_b - m*) l_b,   m* = max_b m_b,
//
// with m kept in log2 units, so the weights are powers of two.  A partition
// that saw no key has m_b = -inf and weight 0.
//
// Launch shape: one block of kMergeWarps warps per output row (a query token
// of chunk attention).  The block reads the row's
// partition count np once; a row with a single partition was written in place
// by the partition kernel and costs one load.  Otherwise warp w merges heads
// w, w + kMergeWarps, ...: H heads at a time with H * np <= 8, so every (m, l)
// pair and partial sum of those H heads is loaded in one round trip within a
// fixed register budget (rows with more than 8 partitions take a looped path).
#pragma once

#include <cmath>

#include "pa_device.cuh"

namespace pa {

constexpr int kMergeWarps = 8;

template <int D>
struct MergeVec {
    static constexpr int kPer = D / 32;  // floats of one partial sum per lane
    static_assert(kPer == 2 || kPer == 4, "head_dim 64 or 128");
    float v[kPer];
    __device__ __forceinline__ void load(const float *p) {
        if constexpr (kPer == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(p);
            v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2 *>(p);
            v[0] = t.x, v[1] = t.y;
        }
    }
    __device__ __forceinline__ void store(float *p) const {
        if constexpr (kPer == 4) *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
        else *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
    }
};

// Merge heads h0 + j * kMergeWarps (j < H, those below Hq) of row r, whose
// np <= F partials sit at ((r * Hq + h) * max_parts + p) in ws_ml (pairs) and
// ws_acc (D floats each): all loads first, then the sums in partition order.
template <int D, int H, int F>
__device__ __forceinline__ void merge_heads(int r, int h0, int np, int Hq, int max_parts, const float *ws_ml,
                                            const float *ws_acc, float *out) {
    using V = MergeVec<D>;
    constexpr int kPer = V::kPer;
    const int lane = threadIdx.x & 31;
    float2 w[H][F];
    V x[H][F];
    float M[H];
#pragma unroll
    for (int j = 0; j < H; ++j) {
        M[j] = -INFINITY;
        const int h = h0 + j * kMergeWarps;
        const size_t q = ((size_t)r * Hq + h) * max_parts;
#pragma unroll
        for (int p = 0; p < F; ++p)
            if (h < Hq && p < np) {
                w[j][p] = *reinterpret_cast<const float2 *>(ws_ml + 2 * (q + p));
                x[j][p].load(ws_acc + (q + p) * D + lane * kPer);
                M[j] = fmaxf(M[j], w[j][p].x);
            }
    }
#pragma unroll
    for (int j = 0; j < H; ++j) {
        const int h = h0 + j * kMergeWarps;
        if (h >= Hq) continue;
        float L = 0.f;
        V o;
#pragma unroll
        for (int k = 0; k < kPer; ++k) o.v[k] = 0.f;
        if (M[j] != -INFINITY) {
#pragma unroll
            for (int p = 0; p < F; ++p)
                if (p < np) {
                    const float wt = ex2(w[j][p].x - M[j]);  // 0 for a partition that saw no key
                    L += wt * w[j][p].y;
#pragma unroll
                    for (int k = 0; k < kPer; ++k) o.v[k] += wt * x[j][p].v[k];
                }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int k = 0; k < kPer; ++k) o.v[k] *= inv;
        o.store(out + ((size_t)r * Hq + h) * D + lane * kPer);
    }
}

// Rows with more than 8 partitions: one head at a time, 4 partitions per
// round trip.
template <int D>
__device__ __forceinline__ void merge_head_long(int r, int h, int np, int Hq, int max_parts, const float *ws_ml,
                                                const float *ws_acc, float *out) {
    using V = MergeVec<D>;
    constexpr int kPer = V::kPer;
    constexpr int kU = 4;
    const int lane = threadIdx.x & 31;
    const size_t q = ((size_t)r * Hq + h) * max_parts;
    float M = -INFINITY, L = 0.f;
    for (int p = lane; p < np; p += 32) M = fmaxf(M, ws_ml[2 * (q + p)]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    V o;
#pragma unroll
    for (int k = 0; k < kPer; ++k) o.v[k] = 0.f;
    if (M != -INFINITY) {
        for (int p0 = 0; p0 < np; p0 += kU) {
            float2 w[kU];
            V x[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int p = p0 + u < np ? p0 + u : p0;
                w[u] = p0 + u < np ? *reinterpret_cast<const float2 *>(ws_ml + 2 * (q + p)) : make_float2(-INFINITY, 0.f);
                x[u].load(ws_acc + (q + p) * D + lane * kPer);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const float wt = ex2(w[u].x - M);  // 0 for the padding entries
                L += wt * w[u].y;
#pragma unroll
                for (int k = 0; k < kPer; ++k) o.v[k] += wt * x[u].v[k];
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) o.v[k] *= inv;
    o.store(out + ((size_t)r * Hq + h) * D + lane * kPer);
}

// Merge every head of row r (np >= 2 partitions).  Called by the whole block.
template <int D>
__device__ __forceinline__ void merge_row(int r, int np, int Hq, int max_parts, const float *ws_ml, const float *ws_acc,
                                          float *out) {
    const int warp = threadIdx.x >> 5;
    if (np <= 2) {
        for (int h0 = warp; h0 < Hq; h0 += 4 * kMergeWarps) merge_heads<D, 4, 2>(r, h0, np, Hq, max_parts, ws_ml, ws_acc, out);
    } else if (np <= 4) {
        for (int h0 = warp; h0 < Hq; h0 += 2 * kMergeWarps) merge_heads<D, 2, 4>(r, h0, np, Hq, max_parts, ws_ml, ws_acc, out);
    } else if (np <= 8) {
        for (int h0 = warp; h0 < Hq; h0 += kMergeWarps) merge_heads<D, 1, 8>(r, h0, np, Hq, max_parts, ws_ml, ws_acc, out);
    } else {
        for (int h = warp; h < Hq; h += kMergeWarps) merge_head_long<D>(r, h, np, Hq, max_parts, ws_ml, ws_acc, out);
    }
}

}  // namespace pa
