// pa_internal.h -- host-side interface between the C-ABI entry points
// (pa_api.cu) and the per-dtype kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/pa.h"

namespace pa {

// A launch constant of the current device (a grid size; 1 for "attributes
// set"), computed by compute(dev, &value) on the first launch there and cached.
// Host threads that race on a first launch compute and store the same value.
constexpr int kMaxLaunchDevices = 64;
template <typename Compute>
cudaError_t per_device_value(std::atomic<int> (&cache)[kMaxLaunchDevices], int *value, Compute compute) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxLaunchDevices) return cudaErrorInvalidDevice;
    int v = cache[dev].load(std::memory_order_acquire);
    if (v == 0) {
        e = compute(dev, &v);
        if (e != cudaSuccess) return e;
        cache[dev].store(v, std::memory_order_release);
    }
    *value = v;
    return cudaSuccess;
}

// Everything a decode launch needs, already validated by the entry point.
struct DecodeArgs {
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *out;
    float *ws_ml;    // [S, Hq, P, 2]  (m in log2 units, l)
    float *ws_acc;   // [S, Hq, P, D]
    int *plan_hdr;   // [0] work items, [1] claim counter, [2] CTAs done claiming
    int4 *plan_list; // (sequence, partition, tokens, partitions of the sequence) per item, largest first
    unsigned int *err;
    int S, Hq, Hkv, D, B, N, max_blocks, partition_size, max_parts;
    int head_group;  // KV heads per tensor-core work item (decode_head_group)
    float scale;
    // The plan writes the zero rows of empty contexts into `zero_layers`
    // outputs, out + l * out_layer_floats (a step over several layers runs the
    // plan once: the work list depends only on the tables and lengths).
    int zero_layers;
    long long out_layer_floats;
    // Tensor-core path: CTAs of the decode grid, and whether the decode may
    // start before its predecessor completes (early != 0 only right after this
    // call's own plan kernel, which lets it start once everything before the
    // plan is complete).  The first sequences' partition 0 is taken by CTAs
    // directly, without the plan's list: sequences s < min(S, ctas / groups).
    int ctas;
    int early;
};

// Everything a chunk-attention launch needs (several query tokens per sequence).
struct ChunkArgs {
    const void *q;                  // [T, Hq, D]
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start;     // [S + 1]
    float *out;                     // [T, Hq, D]
    float *ws_ml;                   // [T, Hq, P, 2]
    float *ws_acc;                  // [T, Hq, P, D]
    int *plan_hdr;                  // [0] work items, [1] claim counter
    int4 *plan_list;                // (sequence, partition, tokens, row block), largest first
    int32_t *row_parts;             // [T]: partitions each query row sees, 0 if the row has no sequence
    unsigned int *err;
    int S, T, Hq, Hkv, D, B, N, max_blocks, partition_size, max_parts, max_query_len;
    int head_group;                 // KV heads per work item
    int row_warps;                  // 16-row query tiles per KV head per work item (1 or 2)
    int umma_rows;                  // tcgen05 path: query rows per CTA (128 or 256); 0 on the mma.sync path
    float scale;
};

// Row warps of a chunk-attention work item: two 16-row tiles per KV head when
// a sequence can have more than 16 (query token, query head) rows, else one.
inline int chunk_row_warps(int max_query_len, int G) { return (long long)max_query_len * G > 16 ? 2 : 1; }

// Chunk attention on the tcgen05 path: when a sequence can have at least this
// many (query token, query head) rows per KV head, 128-row tiles with the
// accumulators in tensor memory replace the mma.sync kernel (and its split-K).
#ifndef PA_CHUNK_UMMA_MIN_ROWS
#define PA_CHUNK_UMMA_MIN_ROWS 64
#endif
inline bool chunk_uses_umma(int max_query_len, int G) {
    return (long long)max_query_len * G >= PA_CHUNK_UMMA_MIN_ROWS;
}
// Keys per step of the tcgen05 kernel, and its rows per CTA: two 128-row tiles
// once a sequence can fill them.
#ifndef PA_CHUNK_UMMA_KEYS
#define PA_CHUNK_UMMA_KEYS 64
#endif
#ifndef PA_CHUNK_UMMA_PAIR_ROWS
#define PA_CHUNK_UMMA_PAIR_ROWS 256
#endif
inline int chunk_umma_rows(int max_query_len, int G) {
    return (long long)max_query_len * G >= PA_CHUNK_UMMA_PAIR_ROWS ? 256 : 128;
}
// Step-count bins of the tcgen05 work list (longer CTAs are binned together).
constexpr int kUmmaStepBins = 1024;

// KV heads that one tensor-core work item (one CTA) covers: PA_MMA_HEAD_GROUP
// (4 by default) when they divide Hkv, else the largest power of two that does.
#ifndef PA_MMA_HEAD_GROUP
#define PA_MMA_HEAD_GROUP 4
#endif
inline int decode_head_group(int Hkv) {
    int hg = PA_MMA_HEAD_GROUP;
    while (hg > 1 && Hkv % hg != 0) hg /= 2;
    return hg;
}

// Tokens per partition upper bound (table slice staged in shared memory).
constexpr int kMaxPartitionBlocks = 256;

// Token rows per tensor-core decode stage: one TMA box is this many rows of one
// (physical block, KV head); a block of B slots is B / kChunkRows boxes.
constexpr int kChunkRows = 16;

// Launchers return cudaSuccess, cudaErrorNotSupported for a shape that is not
// compiled, or the launch error.
// CUDA-core decode (fp32 caches).
cudaError_t launch_decode_f32(const DecodeArgs &a, cudaStream_t st);

// Cross-partition merge of the split-K partials (dtype independent).
cudaError_t launch_decode_merge(const DecodeArgs &a, cudaStream_t st);

// Work list for the tensor-core decode (f16 / bf16 path).  The decode kernel
// leaves the claim counters as the plan set them (the last CTA to finish
// claiming resets them), so one plan serves several launches over the same
// tables and lengths, in stream order.
cudaError_t launch_decode_plan(const DecodeArgs &a, cudaStream_t st);

// Tensor-core decode: f16 / bf16 caches, K and V read through 2-D tensor maps
// ([N*Hkv*B rows, D columns], 64x B boxes, 128-byte swizzle).
cudaError_t launch_decode_mma_f16(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                  cudaStream_t st);
cudaError_t launch_decode_mma_bf16(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   cudaStream_t st);
// CTAs the tensor-core decode launches for these shapes on the current device
// (a persistent grid: SMs x resident CTAs per SM).
cudaError_t decode_mma_ctas_f16(const DecodeArgs &a, int *ctas);
cudaError_t decode_mma_ctas_bf16(const DecodeArgs &a, int *ctas);

// pa_decode with its launches split: kPlanAndRun is pa_decode; kPlanOnly
// writes the work list (and the zero rows of `zero_layers` outputs spaced
// out_layer_floats apart); kRunOnly runs the decode and merge kernels on a list
// an earlier kPlanOnly / kPlanAndRun left in the same workspace, for the same
// tables and lengths.  Validation and statuses as for pa_decode.
enum class DecodePhase { kPlanAndRun, kPlanOnly, kRunOnly };
int32_t decode_call(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *context_lens, float scale, float *out,
                    void *workspace, size_t workspace_bytes, void *stream, DecodePhase phase, int zero_layers,
                    long long out_layer_floats);

// Encode the tensor map of one cache [N, Hkv, B, D] of 16-bit elements as a
// 3-D tensor {D, B, N*Hkv}; a box is 64 columns x kChunkRows rows x head_group
// (block, head) pairs.
cudaError_t make_cache_tensor_map(CUtensorMap *map, const void *cache, bool bf16, int D, int B,
                                  long long block_heads, int head_group);

// Encode the tensor map of the queries q [T, Hq, D] of 16-bit elements as a
// 3-D tensor {D, Hq, T}; a box is 64 columns x G heads x 128 / G tokens: the
// 128 (query token, query head) rows of one tcgen05 tile of a KV head, the
// left or right half of D, landing with the 128-byte swizzle.
cudaError_t make_query_tensor_map(CUtensorMap *map, const void *q, bool bf16, int D, int Hq, long long T, int G);
cudaError_t make_output_tensor_map(CUtensorMap *map, float *out, int D, int Hq, long long T, int G);

// Process-unique id of the calling thread's current CUDA context, or 0 when
// no context is current or the driver cannot say.  A device reset destroys
// the primary context; the one created after it has a new id, so addresses
// cached under the old id are known to be stale.
unsigned long long current_context_id();

// Chunk attention: work list, tensor-core partition kernel, split-K merge.
cudaError_t launch_chunk_plan(const ChunkArgs &a, cudaStream_t st);
cudaError_t launch_chunk_mma_f16(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                 cudaStream_t st);
cudaError_t launch_chunk_mma_bf16(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                  cudaStream_t st);
cudaError_t launch_chunk_merge(const ChunkArgs &a, cudaStream_t st);
// tcgen05 path: one CTA per (128-row tile, KV head, sequence); tensor maps with
// one (block, head) per box (make_cache_tensor_map with head_group 1).
cudaError_t launch_chunk_umma_f16(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                  const CUtensorMap &tmq, const CUtensorMap &tmo, cudaStream_t st);
cudaError_t launch_chunk_umma_bf16(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   const CUtensorMap &tmq, const CUtensorMap &tmo, cudaStream_t st);

cudaError_t launch_write_kv(const void *k, const void *v, const int64_t *slots, int T, int Hkv,
                            int row_bytes, int B, int N, void *k_cache, void *v_cache,
                            unsigned int *err, cudaStream_t st);

// Copy whole blocks for `layers` caches laid out layer_bytes apart (K and V).
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int P,
                               int64_t block_bytes, int N, int layers, int64_t layer_bytes, unsigned int *err,
                               cudaStream_t st);

// Copy whole blocks between two pools (device <-> pinned host), `layers` deep.
cudaError_t launch_swap_blocks(const void *from_k, const void *from_v, void *to_k, void *to_v,
                               const int64_t *pairs, int P, int64_t block_bytes, int layers, int64_t from_layer_bytes,
                               int64_t to_layer_bytes, int from_n, int to_n, unsigned int *err, cudaStream_t st);

}  // namespace pa
