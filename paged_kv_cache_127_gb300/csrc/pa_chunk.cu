// pa_chunk.cu -- work list and split-K merge of chunk attention (several query
// tokens per sequence; the tensor-core partition kernel is in pa_chunk_mma.cuh).
//
// The plan (one CTA) checks that query_start is non-decreasing within [0, T],
// maps every query row to its sequence (-1 where none, or where the sequence
// is skipped because n_s > context length or n_s > max_query_len), and lists
// the work: on the mma.sync path every (sequence, partition, row block) whose
// rows see at least one key of the partition, with the partition's token count
// up to the block's last row position, largest first (a counting sort on the
// block count); on the tcgen05 path every (sequence, group of 128-row tiles)
// with its step count, longest first.  The merge
// combines, for each query row, the partitions 0 .. pos / partition_size it
// sees ("Paged Attention and vLLM", "Paged Attention CUDA Kernel", the merge
// equation).
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

__device__ __forceinline__ int clamp_len(int len, int cap) { return len < 0 ? 0 : (len > cap ? cap : len); }

// Tokens of partition p that row block rb of sequence (n, len) needs: up to the
// block's last row position; 0 when that row ends before the partition.
__device__ __forceinline__ int block_tokens(int n, int len, int G, int rows_per_block, int rb, int p, int Pt) {
    const int rows = n * G;
    const int r_last = min(rows, (rb + 1) * rows_per_block) - 1;
    const int pos_max = len - n + r_last / G;
    const int nt = pos_max + 1 - p * Pt;
    return nt <= 0 ? 0 : (nt > Pt ? Pt : nt);
}

}  // namespace

// tcgen05 path: steps of the CTA that serves tile group g of a sequence with n
// queries and context len (up to its last row's position), kN keys per step.
__device__ __forceinline__ int umma_steps(int n, int len, int G, int rows_cta, int g) {
    const int t_last = min(n - 1, (g * rows_cta + rows_cta - 1) / G);
    return (len - n + t_last) / PA_CHUNK_UMMA_KEYS + 1;
}

__global__ void __launch_bounds__(1024) chunk_plan_kernel(const ChunkArgs a) {
    constexpr int kBins = kUmmaStepBins > kMaxPartitionBlocks + 1 ? kUmmaStepBins : kMaxPartitionBlocks + 1;
    constexpr int kQsCache = 4096;
    __shared__ int hist[kBins];
    __shared__ int start[kBins];
    __shared__ int qs_cache[kQsCache];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x;
    const int Pt = a.partition_size;
    const int B = a.B;
    const int cap = a.max_blocks * B;
    const int maxpb = Pt / B;
    const int G = a.Hq / a.Hkv;
    const int rpb = a.row_warps * 16;
    for (int i = tid; i < kBins; i += blockDim.x) hist[i] = 0;
    int my_bad = 0;
    if (tid == 0) {
        a.plan_hdr[1] = 0;
        my_bad = (a.query_start[0] < 0 || a.query_start[a.S] > a.T) ? 1 : 0;
    }
    for (int s = tid; s < a.S; s += blockDim.x)
        if (a.query_start[s] > a.query_start[s + 1]) my_bad = 1;
    if (__syncthreads_or(my_bad)) {
        if (tid == 0) {
            set_error(a.err, PA_DEVERR_BAD_LEN);
            a.plan_hdr[0] = 0;
        }
        for (int i = tid; i < a.T; i += blockDim.x) a.tok_seq[i] = -1;
        return;
    }
    // query row -> sequence (read by the split-K merge; the tcgen05 path has
    // none): the last s with query_start[s] <= i, if i is inside its range.  The
    // binary search runs over a shared-memory copy of query_start when it fits.
    if (a.umma_rows == 0) {
        const bool cached = a.S + 1 <= kQsCache;
        if (cached)
            for (int i = tid; i <= a.S; i += blockDim.x) qs_cache[i] = a.query_start[i];
        __syncthreads();
        const int *qsv = cached ? qs_cache : a.query_start;
        for (int i = tid; i < a.T; i += blockDim.x) {
            int lo = 0, hi = a.S;  // invariant: query_start[lo] <= i (or lo == 0), answer in [lo, hi)
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (qsv[mid] <= i) lo = mid; else hi = mid;
            }
            int s = -1;
            if (a.S > 0 && qsv[lo] <= i && i < qsv[lo + 1]) {
                const int n = qsv[lo + 1] - qsv[lo];
                const int len = a.context_lens[lo];
                if (len >= 0 && len <= cap && n <= len && n <= a.max_query_len) s = lo;
            }
            a.tok_seq[i] = s;
        }
    }
    if (a.umma_rows > 0) {
        // tcgen05 path: one entry per (sequence, tile group), by step count, longest first
        const int R = a.umma_rows;
        for (int s = tid; s < a.S; s += blockDim.x) {
            const int raw = a.context_lens[s];
            const int len = clamp_len(raw, cap);
            const int n = a.query_start[s + 1] - a.query_start[s];
            if (raw != len || n > len || n > a.max_query_len) {
                set_error(a.err, PA_DEVERR_BAD_LEN);
                continue;
            }
            for (int g = 0; g * R < n * G; ++g)
                atomicAdd(&hist[min(umma_steps(n, len, G, R, g), kBins - 1)], 1);
        }
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int z = kBins - 1; z >= 0; --z) {
                start[z] = acc;
                acc += hist[z];
            }
            a.plan_hdr[0] = acc;
        }
        __syncthreads();
        for (int s = tid; s < a.S; s += blockDim.x) {
            const int raw = a.context_lens[s];
            const int len = clamp_len(raw, cap);
            const int n = a.query_start[s + 1] - a.query_start[s];
            if (raw != len || n > len || n > a.max_query_len) continue;
            for (int g = 0; g * R < n * G; ++g) {
                const int steps = umma_steps(n, len, G, R, g);
                const int pos = atomicAdd(&start[min(steps, kBins - 1)], 1);
                a.plan_list[pos] = make_int4(s, g, steps, 0);
            }
        }
        return;
    }
    for (int s = tid; s < a.S; s += blockDim.x) {
        const int raw = a.context_lens[s];
        const int len = clamp_len(raw, cap);
        const int n = a.query_start[s + 1] - a.query_start[s];
        if (raw != len || n > len || n > a.max_query_len) {
            set_error(a.err, PA_DEVERR_BAD_LEN);
            continue;
        }
        const int nrb = (n * G + rpb - 1) / rpb;
        for (int rb = 0; rb < nrb; ++rb)
            for (int p = 0;; ++p) {
                const int nt = block_tokens(n, len, G, rpb, rb, p, Pt);
                if (nt == 0) break;
                atomicAdd(&hist[(nt + B - 1) / B], 1);
            }
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int z = maxpb; z >= 1; --z) {
            start[z] = acc;
            acc += hist[z];
        }
        a.plan_hdr[0] = acc * (a.Hkv / a.head_group);  // items: (sequence, partition, row block, head group)
    }
    __syncthreads();
    for (int s = tid; s < a.S; s += blockDim.x) {
        const int raw = a.context_lens[s];
        const int len = clamp_len(raw, cap);
        const int n = a.query_start[s + 1] - a.query_start[s];
        if (raw != len || n > len || n > a.max_query_len) continue;
        const int nrb = (n * G + rpb - 1) / rpb;
        for (int rb = 0; rb < nrb; ++rb)
            for (int p = 0;; ++p) {
                const int nt = block_tokens(n, len, G, rpb, rb, p, Pt);
                if (nt == 0) break;
                const int pos = atomicAdd(&start[(nt + B - 1) / B], 1);
                a.plan_list[pos] = make_int4(s, p, nt, rb);
            }
    }
}

cudaError_t launch_chunk_plan(const ChunkArgs &a, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(1024);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chunk_plan_kernel, a);
}

// One warp per (query row, query head): combine the row's partitions.
template <int D>
__global__ void chunk_merge_kernel(const ChunkArgs a) {
    constexpr int kPer = D / 32;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int gw = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (gw >= a.T * a.Hq) return;
    const int i = gw / a.Hq;
    const int s = a.tok_seq[i];
    if (s < 0) return;
    const int qs = a.query_start[s];
    const int n = a.query_start[s + 1] - qs;
    const int len = clamp_len(a.context_lens[s], a.max_blocks * a.B);
    const int pos = len - n + (i - qs);
    const int np = pos / a.partition_size + 1;
    if (np <= 1) return;  // written in place by the partition kernel
    const size_t r0 = (size_t)gw * a.max_parts;
    const float *ml = a.ws_ml + 2 * r0;
    const float *acc = a.ws_acc + r0 * D;
    float M = -INFINITY;
    for (int p = lane; p < np; p += 32) M = fmaxf(M, ml[2 * p]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    float o[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) o[k] = 0.f;
    if (M != -INFINITY) {
        for (int p = 0; p < np; ++p) {
            const float2 w = *reinterpret_cast<const float2 *>(ml + 2 * p);
            const float wt = ex2(w.x - M);  // 0 for a partition that saw no key
            L += wt * w.y;
#pragma unroll
            for (int k = 0; k < kPer; ++k) o[k] += wt * acc[(size_t)p * D + lane * kPer + k];
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float *dst = a.out + (size_t)gw * D + lane * kPer;
#pragma unroll
    for (int k = 0; k < kPer; ++k) dst[k] = o[k] * inv;
}

cudaError_t launch_chunk_merge(const ChunkArgs &a, cudaStream_t st) {
    const long long warps = (long long)a.T * a.Hq;
    if (warps == 0) return cudaSuccess;
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
    if (a.D == 64) return cudaLaunchKernelEx(&cfg, chunk_merge_kernel<64>, a);
    if (a.D == 128) return cudaLaunchKernelEx(&cfg, chunk_merge_kernel<128>, a);
    return cudaErrorNotSupported;
}

}  // namespace pa
