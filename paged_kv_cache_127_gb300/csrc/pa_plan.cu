// pa_plan.cu -- work list for the tensor-core decode.
//
// One CTA lists every (sequence, partition) pair of the batch -- with the
// partition's token count and the sequence's partition count -- largest
// partition first (a counting sort on the partition's block count), so the
// persistent decode kernel hands out big items before small ones and its
// tail is short.  Partition 0 of the first min(S, ctas / groups) sequences is
// left out: decode CTA b takes it directly (sequence b / groups, head group
// b % groups), so the decode kernel need not wait for this list before its
// first item.  It also resets the claim counters, writes the all-zero output
// rows of empty contexts (of every layer the list will serve), and flags
// context lengths outside [0, max_blocks * B].
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kLenCache = 4096;

__global__ void __launch_bounds__(1024) decode_plan_kernel(const DecodeArgs a) {
    __shared__ int hist[kMaxPartitionBlocks + 1];
    __shared__ int start[kMaxPartitionBlocks + 1];
    __shared__ int warp_sums[32];
    __shared__ int len_cache[kLenCache];  // context_lens, read once when they fit
    // Wait for the work before this one in the stream (the workspace and
    // context_lens are only touched after it), then let the decode kernel
    // start: everything before this grid is complete, so it may read the caches,
    // tables and lengths for its first items; it waits for this grid before it
    // reads the list.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int Pt = a.partition_size;
    const int B = a.B;
    const int cap = a.max_blocks * B;
    const int maxpb = Pt / B;
    const int groups = a.Hkv / a.head_group;
    const int nstatic = min(a.S, a.ctas / groups);  // sequences whose partition 0 the CTAs take directly
    for (int i = tid; i <= maxpb; i += blockDim.x) hist[i] = 0;
    if (tid == 0) {
        a.plan_hdr[1] = 0;
        a.plan_hdr[2] = 0;
    }
    const bool cached = a.S <= kLenCache;
    if (cached)
        for (int s = tid; s < a.S; s += blockDim.x) len_cache[s] = a.context_lens[s];
    __syncthreads();
    const int *lenv = cached ? len_cache : a.context_lens;
    for (int s = tid; s < a.S; s += blockDim.x) {
        int len = lenv[s];
        if (len < 0 || len > cap) {
            set_error(a.err, PA_DEVERR_BAD_LEN);
            len = len < 0 ? 0 : cap;
        }
        if (len == 0) {
            for (int l = 0; l < a.zero_layers; ++l) {
                float4 *row = reinterpret_cast<float4 *>(a.out + l * a.out_layer_floats + (size_t)s * a.Hq * a.D);
                for (int i = 0; i < a.Hq * a.D / 4; ++i) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            continue;
        }
        const int np = (len + Pt - 1) / Pt;
        for (int p = s < nstatic ? 1 : 0; p < np; ++p) {
            const int nt = min(Pt, len - p * Pt);
            atomicAdd(&hist[(nt + B - 1) / B], 1);
        }
    }
    __syncthreads();
    // list positions by block count, largest first
    const int total = scan_bins_desc(hist, start, maxpb, maxpb, warp_sums);
    if (tid == 0) a.plan_hdr[0] = total * groups;  // items: (sequence, partition, head group)
    for (int s = tid; s < a.S; s += blockDim.x) {
        int len = lenv[s];
        len = len < 0 ? 0 : (len > cap ? cap : len);
        const int np = (len + Pt - 1) / Pt;
        for (int p = s < nstatic ? 1 : 0; p < np; ++p) {
            const int nt = min(Pt, len - p * Pt);
            const int pos = atomicAdd(&start[(nt + B - 1) / B], 1);
            a.plan_list[pos] = make_int4(s, p, nt, np);
        }
    }
}

cudaError_t launch_decode_plan(const DecodeArgs &a, cudaStream_t st) {
    // launched as a programmatic dependent: its launch overlaps the tail of the
    // previous kernel in the stream, and it waits for that kernel before work
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(1024);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_plan_kernel, a);
}

}  // namespace pa
