// pa_chunk.cu -- work list and split-K merge of chunk attention (several query
// tokens per sequence; the tensor-core partition kernel is in pa_chunk_mma.cuh).
//
// The plan (one CTA) checks that query_start is non-decreasing within [0, T],
// records for every query row how many partitions it sees (0 where the row
// has no sequence, or where the sequence is skipped because n_s > context
// length or n_s > max_query_len), and lists
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
#include "pa_merge.cuh"

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
    static_assert(kBins <= 1024, "one bin per thread in the scan");
    constexpr int kCache = 4096;
    __shared__ int hist[kBins];
    __shared__ int start[kBins];
    __shared__ int warp_sums[32];
    __shared__ int qs_cache[kCache + 1];
    __shared__ int len_cache[kCache];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x;
    const int Pt = a.partition_size;
    const int B = a.B;
    const int cap = a.max_blocks * B;
    const int maxpb = Pt / B;
    const int G = a.Hq / a.Hkv;
    const int rpb = a.row_warps * 16;
    // query_start and context_lens are read once, into shared memory when they fit
    const bool cached = a.S <= kCache;
    if (cached) {
        for (int i = tid; i <= a.S; i += blockDim.x) qs_cache[i] = a.query_start[i];
        for (int i = tid; i < a.S; i += blockDim.x) len_cache[i] = a.context_lens[i];
    }
    for (int i = tid; i < kBins; i += blockDim.x) hist[i] = 0;
    if (tid == 0) a.plan_hdr[1] = 0;
    __syncthreads();
    const int *qsv = cached ? qs_cache : a.query_start;
    const int *lenv = cached ? len_cache : a.context_lens;
    int my_bad = 0;
    if (tid == 0) my_bad = (qsv[0] < 0 || qsv[a.S] > a.T) ? 1 : 0;
    for (int s = tid; s < a.S; s += blockDim.x)
        if (qsv[s] > qsv[s + 1]) my_bad = 1;
    if (__syncthreads_or(my_bad)) {
        if (tid == 0) {
            set_error(a.err, PA_DEVERR_BAD_LEN);
            a.plan_hdr[0] = 0;
        }
        for (int i = tid; i < a.T; i += blockDim.x) a.row_parts[i] = 0;
        return;
    }
    // Partitions each query row sees (read by the split-K merge; the tcgen05
    // path has none): 0 where the row has no sequence, else pos / Pt + 1 for
    // the row's position pos.  The row's sequence is the last s with
    // query_start[s] <= i, if i is inside its range (a binary search).
    if (a.umma_rows == 0) {
        for (int i = tid; i < a.T; i += blockDim.x) {
            int lo = 0, hi = a.S;  // invariant: query_start[lo] <= i (or lo == 0), answer in [lo, hi)
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (qsv[mid] <= i) lo = mid; else hi = mid;
            }
            int np = 0;
            if (qsv[lo] <= i && i < qsv[lo + 1]) {
                const int n = qsv[lo + 1] - qsv[lo];
                const int len = lenv[lo];
                if (len >= 0 && len <= cap && n <= len && n <= a.max_query_len)
                    np = (len - n + (i - qsv[lo])) / Pt + 1;
            }
            a.row_parts[i] = np;
        }
    }
    if (a.umma_rows > 0) {
        // tcgen05 path: one entry per (sequence, tile group), by step count, longest first
        const int R = a.umma_rows;
        for (int s = tid; s < a.S; s += blockDim.x) {
            const int raw = lenv[s];
            const int len = clamp_len(raw, cap);
            const int n = qsv[s + 1] - qsv[s];
            if (raw != len || n > len || n > a.max_query_len) {
                set_error(a.err, PA_DEVERR_BAD_LEN);
                continue;
            }
            for (int g = 0; g * R < n * G; ++g)
                atomicAdd(&hist[min(umma_steps(n, len, G, R, g), kBins - 1)], 1);
        }
        __syncthreads();
        const int total = scan_bins_desc(hist, start, kBins - 1, kBins, warp_sums);
        if (tid == 0) a.plan_hdr[0] = total;
        for (int s = tid; s < a.S; s += blockDim.x) {
            const int raw = lenv[s];
            const int len = clamp_len(raw, cap);
            const int n = qsv[s + 1] - qsv[s];
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
        const int raw = lenv[s];
        const int len = clamp_len(raw, cap);
        const int n = qsv[s + 1] - qsv[s];
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
    // bins maxpb .. 1 (a partition's block count), largest first
    const int total = scan_bins_desc(hist, start, maxpb, maxpb, warp_sums);
    if (tid == 0) a.plan_hdr[0] = total * (a.Hkv / a.head_group);  // items: (sequence, partition, row block, head group)
    for (int s = tid; s < a.S; s += blockDim.x) {
        const int raw = lenv[s];
        const int len = clamp_len(raw, cap);
        const int n = qsv[s + 1] - qsv[s];
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

// One block per query row (pa_merge.cuh): the plan stored how many
// partitions the row sees; a row with one was written in place.
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32, 3) chunk_merge_kernel(const ChunkArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int i = blockIdx.x;
    const int np = a.row_parts[i];
    if (np <= 1) return;  // no sequence, or written in place by the partition kernel
    merge_row<D>(i, np, a.Hq, a.max_parts, a.ws_ml, a.ws_acc, a.out);
}

cudaError_t launch_chunk_merge(const ChunkArgs &a, cudaStream_t st) {
    if (a.T == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.T);
    cfg.blockDim = dim3(kMergeWarps * 32);
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
