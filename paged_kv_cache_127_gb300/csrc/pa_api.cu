// pa_api.cu -- C-ABI entry points of libpa for the GPU calls: argument
// validation, workspace sizing, the per-device error word, dtype / shape
// dispatch.  See include/pa.h for the contract of each call.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

// Sticky PA_DEVERR_* bits; every device that loads the library has its own copy.
__device__ unsigned int g_device_error_word;

constexpr int kMaxDevices = 64;
constexpr int kDefaultPartition = 512;

// The error word's device address in the current context, looked up with
// cudaGetSymbolAddress and cached per device together with the context id, so
// a context created after a device reset gets a fresh lookup.
unsigned int *error_word() {
    static std::mutex mu;
    static unsigned long long ctx_of[kMaxDevices] = {};
    static unsigned int *cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = pa::current_context_id();
    if (!cache[dev] || ctx == 0 || ctx != ctx_of[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned int *>(p);
        ctx_of[dev] = pa::current_context_id();   // the lookup makes the primary context current
    }
    return cache[dev];
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(int dtype) { return dtype == PA_F32 ? 4 : 2; }

// Checks shared by all GPU calls (cache geometry).
int32_t check_cache_dims(const pa_dims *d) {
    if (!d) return PA_ERR_INVALID;
    if (d->num_kv_heads <= 0 || d->head_dim <= 0 || d->block_size <= 0 || d->num_blocks <= 0)
        return PA_ERR_INVALID;
    if (d->kv_dtype < PA_F32 || d->kv_dtype > PA_BF16) return PA_ERR_INVALID;
    if ((d->head_dim * elem_bytes(d->kv_dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// partition_size 0: pick by the (sequence, KV head group of 4) pairs of the
// batch, so that a small batch still yields enough work items for every SM
// (measured on a 32-layer step: 8 sequences run 1.7x faster at 128 tokens than
// at 512, 32 sequences 1.4x faster at 256; 256 sequences are best at 512).
int32_t effective_partition(const pa_dims *d) {
    if (d->partition_size > 0) return d->partition_size;
    const int64_t pairs = (int64_t)d->num_seqs * (d->num_kv_heads > 0 ? d->num_kv_heads : 1) / 4;
    if (pairs >= 256) return kDefaultPartition;
    if (pairs >= 32) return 256;
    return 128;
}

// partition_size 0 for chunk attention: four times the decode choice, at most
// 2048 tokens.  A chunk item carries several query rows per KV head, so each
// key costs more arithmetic and fewer, longer partitions pay: fewer items to
// set up and fewer partials to merge (measured on 256 sequences x 5 queries,
// 8B-shaped: 512 tokens 4.54 TB/s, 1024 4.79, 2048 4.99).
int32_t chunk_partition(const pa_dims *d) {
    if (d->partition_size > 0) return d->partition_size;
    const int32_t pt = 4 * effective_partition(d);
    const int32_t cap = pa::kMaxPartitionBlocks * (d->block_size > 0 ? d->block_size : 1);
    return pt < 2048 ? (pt < cap ? pt : cap) : (2048 < cap ? 2048 : cap);
}

// Full decode checks for partitions of pt tokens; fills max_parts.
int32_t check_decode_dims_pt(const pa_dims *d, int32_t pt, int32_t *max_parts) {
    int32_t rc = check_cache_dims(d);
    if (rc != PA_OK) return rc;
    if (d->num_seqs < 0 || d->num_q_heads <= 0 || d->max_blocks_per_seq <= 0) return PA_ERR_INVALID;
    if (d->num_q_heads % d->num_kv_heads != 0) return PA_ERR_INVALID;
    if (d->partition_size < 0) return PA_ERR_INVALID;
    const int32_t G = d->num_q_heads / d->num_kv_heads;
    if (pt % d->block_size != 0 || pt / d->block_size > pa::kMaxPartitionBlocks) return PA_ERR_INVALID;
    if (!(d->head_dim == 64 || d->head_dim == 128) || !(d->block_size == 16 || d->block_size == 32) ||
        !(G == 1 || G == 2 || G == 4 || G == 8))
        return PA_ERR_UNSUPPORTED;
    const int64_t cap = (int64_t)d->max_blocks_per_seq * d->block_size;
    if (cap > INT32_MAX) return PA_ERR_INVALID;
    // cache rows (N * Hkv * B) are addressed with 32-bit coordinates
    if ((int64_t)d->num_blocks * d->num_kv_heads * d->block_size > INT32_MAX) return PA_ERR_INVALID;
    const int64_t parts = (cap + pt - 1) / pt;
    if (parts > 65535) return PA_ERR_INVALID;
    if ((int64_t)d->num_seqs * d->num_kv_heads > INT32_MAX) return PA_ERR_INVALID;
    *max_parts = (int32_t)parts;
    return PA_OK;
}

int32_t check_decode_dims(const pa_dims *d, int32_t *max_parts) {
    if (!d) return PA_ERR_INVALID;
    return check_decode_dims_pt(d, effective_partition(d), max_parts);
}

// Workspace layout, each part 256-byte aligned:
//   header    2 ints: work items, claim counter
//   list      int4 [S * P]: (sequence, partition, tokens, partitions) work items, largest first
//   acc       float [S, Hq, P, D]: split-K partial sums          (only if P > 1)
//   ml        float [S, Hq, P, 2]: partial (max in log2 units, sum) (only if P > 1)
struct WsLayout {
    size_t list, acc, ml, total;
};

WsLayout workspace_layout(const pa_dims *d, int32_t max_parts) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t S = (size_t)d->num_seqs;
    WsLayout L{};
    size_t off = 256;
    L.list = off;
    off += up(S * max_parts * 4 * sizeof(int));
    L.acc = off;
    off += max_parts > 1 ? up(S * d->num_q_heads * max_parts * d->head_dim * sizeof(float)) : 0;
    L.ml = off;
    off += max_parts > 1 ? up(S * d->num_q_heads * max_parts * 2 * sizeof(float)) : 0;
    L.total = off;
    return L;
}

size_t workspace_bytes_for(const pa_dims *d, int32_t max_parts) {
    return d->num_seqs > 0 ? workspace_layout(d, max_parts).total : 0;
}

// Chunk-attention checks: the decode checks, 16-bit caches only, and a token
// count and query-length bound whose scratch sizes stay addressable.
int32_t check_chunk_dims(const pa_dims *d, int32_t T, int32_t max_q, int32_t *max_parts) {
    if (!d) return PA_ERR_INVALID;
    int32_t rc = check_decode_dims_pt(d, chunk_partition(d), max_parts);
    if (rc != PA_OK) return rc;
    if (d->kv_dtype == PA_F32) return PA_ERR_UNSUPPORTED;
    if (T < 0 || max_q < 1 || max_q > (1 << 20)) return PA_ERR_INVALID;
    if ((int64_t)T * d->num_q_heads > INT32_MAX) return PA_ERR_INVALID;
    if (d->num_seqs > 65535) return PA_ERR_INVALID;  // the tcgen05 grid's z extent
    return PA_OK;
}

// Chunk workspace, each part 256-byte aligned:
//   header    2 ints: work items, claim counter
//   list      int4 [S * P * R]: (sequence, partition, tokens, row block)
//   tok       int32 [T]: partitions each query row sees (0: no sequence)
//   acc, ml   float [T, Hq, P, D] and [T, Hq, P, 2]   (only if P > 1)
struct ChunkLayout {
    size_t list, tok, acc, ml, total;
};

ChunkLayout chunk_layout(const pa_dims *d, int32_t T, int32_t max_q, int32_t max_parts) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const int64_t G = d->num_q_heads / d->num_kv_heads;
    const int64_t rpb = 16 * pa::chunk_row_warps(max_q, (int)G);
    const int64_t R = ((int64_t)max_q * G + rpb - 1) / rpb;
    ChunkLayout L{};
    size_t off = 256;
    L.list = off;
    off += up((size_t)d->num_seqs * max_parts * R * 4 * sizeof(int));
    L.tok = off;
    off += up((size_t)T * sizeof(int32_t));
    // split-K partials only on the mma.sync path (the tcgen05 path walks a tile's whole context)
    const bool partials = max_parts > 1 && !pa::chunk_uses_umma(max_q, (int)G);
    L.acc = off;
    off += partials ? up((size_t)T * d->num_q_heads * max_parts * d->head_dim * sizeof(float)) : 0;
    L.ml = off;
    off += partials ? up((size_t)T * d->num_q_heads * max_parts * 2 * sizeof(float)) : 0;
    L.total = off;
    return L;
}

// Tensor maps of the two caches, re-encoded only when the cache or its shape
// changes (per host thread).
struct TmapEntry {
    const void *ptr = nullptr;
    long long block_heads = 0;
    int D = 0, B = 0, hg = 0;
    bool bf16 = false;
    CUtensorMap map;
};

cudaError_t cache_tensor_map(const void *ptr, bool bf16, int D, int B, long long block_heads, int hg,
                             CUtensorMap *out) {
    thread_local TmapEntry cache[4];
    thread_local int next = 0;
    for (auto &e : cache)
        if (e.ptr == ptr && e.block_heads == block_heads && e.D == D && e.B == B && e.hg == hg &&
            e.bf16 == bf16) {
            *out = e.map;
            return cudaSuccess;
        }
    TmapEntry &e = cache[next];
    next = (next + 1) % 4;
    cudaError_t rc = pa::make_cache_tensor_map(&e.map, ptr, bf16, D, B, block_heads, hg);
    if (rc != cudaSuccess) {
        e.ptr = nullptr;
        return rc;
    }
    e.ptr = ptr;
    e.block_heads = block_heads;
    e.D = D;
    e.B = B;
    e.hg = hg;
    e.bf16 = bf16;
    *out = e.map;
    return cudaSuccess;
}

// The query tensor map of the tcgen05 chunk path, re-encoded only when the
// queries' pointer or shape changes (per host thread).
cudaError_t query_tensor_map(const void *q, bool bf16, int D, int Hq, long long T, int G, CUtensorMap *out) {
    struct Entry {
        const void *ptr = nullptr;
        long long T = 0;
        int D = 0, Hq = 0, G = 0;
        bool bf16 = false;
        CUtensorMap map;
    };
    thread_local Entry cache[2];
    thread_local int next = 0;
    for (auto &e : cache)
        if (e.ptr == q && e.T == T && e.D == D && e.Hq == Hq && e.G == G && e.bf16 == bf16) {
            *out = e.map;
            return cudaSuccess;
        }
    Entry &e = cache[next];
    next = (next + 1) % 2;
    cudaError_t rc = pa::make_query_tensor_map(&e.map, q, bf16, D, Hq, T, G);
    if (rc != cudaSuccess) {
        e.ptr = nullptr;
        return rc;
    }
    e.ptr = q;
    e.T = T;
    e.D = D;
    e.Hq = Hq;
    e.G = G;
    e.bf16 = bf16;
    *out = e.map;
    return cudaSuccess;
}

// The output tensor map of the tcgen05 chunk path, likewise cached.
cudaError_t output_tensor_map(float *o, int D, int Hq, long long T, int G, CUtensorMap *out) {
    struct Entry {
        const float *ptr = nullptr;
        long long T = 0;
        int D = 0, Hq = 0, G = 0;
        CUtensorMap map;
    };
    thread_local Entry cache[2];
    thread_local int next = 0;
    for (auto &e : cache)
        if (e.ptr == o && e.T == T && e.D == D && e.Hq == Hq && e.G == G) {
            *out = e.map;
            return cudaSuccess;
        }
    Entry &e = cache[next];
    next = (next + 1) % 2;
    cudaError_t rc = pa::make_output_tensor_map(&e.map, o, D, Hq, T, G);
    if (rc != cudaSuccess) {
        e.ptr = nullptr;
        return rc;
    }
    e.ptr = o;
    e.T = T;
    e.D = D;
    e.Hq = Hq;
    e.G = G;
    *out = e.map;
    return cudaSuccess;
}

int32_t to_status(cudaError_t e) {
    if (e == cudaSuccess) return PA_OK;
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    return PA_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t pa_decode_workspace_bytes(const pa_dims *dims) {
    int32_t parts = 0;
    if (check_decode_dims(dims, &parts) != PA_OK) return 0;
    return workspace_bytes_for(dims, parts);
}

}  // extern "C"

namespace pa {

int32_t decode_call(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *context_lens, float scale, float *out,
                    void *workspace, size_t workspace_bytes, void *stream, DecodePhase phase, int zero_layers,
                    long long out_layer_floats) {
    int32_t parts = 0;
    int32_t rc = check_decode_dims(dims, &parts);
    if (rc != PA_OK) return rc;
    if (dims->num_seqs == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID;
    const size_t need = workspace_bytes_for(dims, parts);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PA_ERR_INVALID;
    const WsLayout L = workspace_layout(dims, parts);

    pa::DecodeArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = out;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.plan_hdr = reinterpret_cast<int *>(ws);
    a.plan_list = reinterpret_cast<int4 *>(ws + L.list);
    a.ws_acc = parts > 1 ? reinterpret_cast<float *>(ws + L.acc) : nullptr;
    a.ws_ml = parts > 1 ? reinterpret_cast<float *>(ws + L.ml) : nullptr;
    a.err = error_word();
    if (!a.err) return PA_ERR_CUDA;
    a.S = dims->num_seqs;
    a.Hq = dims->num_q_heads;
    a.Hkv = dims->num_kv_heads;
    a.D = dims->head_dim;
    a.B = dims->block_size;
    a.N = dims->num_blocks;
    a.max_blocks = dims->max_blocks_per_seq;
    a.partition_size = effective_partition(dims);
    a.max_parts = parts;
    a.head_group = pa::decode_head_group(dims->num_kv_heads);
    a.scale = scale;
    a.zero_layers = zero_layers;
    a.out_layer_floats = out_layer_floats;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dims->kv_dtype == PA_F32) {
        if (phase == DecodePhase::kPlanOnly) return PA_OK;  // the CUDA-core path has no plan
        // fp32 caches: CUDA-core kernel, then the merge kernel for split-K
        e = pa::launch_decode_f32(a, st);
        if (e != cudaSuccess) return to_status(e);
        if (parts > 1) {
            e = pa::launch_decode_merge(a, st);
            if (e != cudaSuccess) return to_status(e);
        }
        return PA_OK;
    }
    // f16 / bf16 caches: work list, the persistent tensor-core kernel, then the
    // split-K merge (each launch a programmatic dependent of the previous one)
    const bool bf16 = dims->kv_dtype == PA_BF16;
    const long long block_heads = (long long)dims->num_blocks * dims->num_kv_heads;
    CUtensorMap tmk, tmv;
    e = cache_tensor_map(k_cache, bf16, dims->head_dim, dims->block_size, block_heads, a.head_group, &tmk);
    if (e == cudaSuccess)
        e = cache_tensor_map(v_cache, bf16, dims->head_dim, dims->block_size, block_heads, a.head_group, &tmv);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    e = bf16 ? pa::decode_mma_ctas_bf16(a, &a.ctas) : pa::decode_mma_ctas_f16(a, &a.ctas);
    if (e != cudaSuccess) return to_status(e);
    a.early = phase == DecodePhase::kPlanAndRun ? 1 : 0;  // the decode kernel follows its own plan
    if (phase != DecodePhase::kRunOnly) {
        e = pa::launch_decode_plan(a, st);
        if (e != cudaSuccess) return to_status(e);
        if (phase == DecodePhase::kPlanOnly) return PA_OK;
    }
    e = bf16 ? pa::launch_decode_mma_bf16(a, tmk, tmv, st) : pa::launch_decode_mma_f16(a, tmk, tmv, st);
    if (e != cudaSuccess) return to_status(e);
    if (parts > 1) e = pa::launch_decode_merge(a, st);
    return to_status(e);
}

}  // namespace pa

extern "C" {

int32_t pa_decode(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, const int32_t *context_lens, float scale, float *out,
                  void *workspace, size_t workspace_bytes, void *stream) {
    return pa::decode_call(dims, q, k_cache, v_cache, block_tables, context_lens, scale, out, workspace,
                           workspace_bytes, stream, pa::DecodePhase::kPlanAndRun, 1, 0);
}

size_t pa_chunk_workspace_bytes(const pa_dims *dims, int32_t num_tokens, int32_t max_query_len) {
    int32_t parts = 0;
    if (check_chunk_dims(dims, num_tokens, max_query_len, &parts) != PA_OK) return 0;
    return chunk_layout(dims, num_tokens, max_query_len, parts).total;
}

int32_t pa_chunk_attention(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens, const int32_t *query_start,
                           int32_t num_tokens, int32_t max_query_len, float scale, float *out, void *workspace,
                           size_t workspace_bytes, void *stream) {
    int32_t parts = 0;
    int32_t rc = check_chunk_dims(dims, num_tokens, max_query_len, &parts);
    if (rc != PA_OK) return rc;
    if (dims->num_seqs == 0 || num_tokens == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out) return PA_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(query_start, 4))
        return PA_ERR_INVALID;
    const ChunkLayout L = chunk_layout(dims, num_tokens, max_query_len, parts);
    if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256)) return PA_ERR_INVALID;

    pa::ChunkArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.out = out;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.plan_hdr = reinterpret_cast<int *>(ws);
    a.plan_list = reinterpret_cast<int4 *>(ws + L.list);
    a.row_parts = reinterpret_cast<int32_t *>(ws + L.tok);
    a.ws_acc = parts > 1 ? reinterpret_cast<float *>(ws + L.acc) : nullptr;
    a.ws_ml = parts > 1 ? reinterpret_cast<float *>(ws + L.ml) : nullptr;
    a.err = error_word();
    if (!a.err) return PA_ERR_CUDA;
    a.S = dims->num_seqs;
    a.T = num_tokens;
    a.Hq = dims->num_q_heads;
    a.Hkv = dims->num_kv_heads;
    a.D = dims->head_dim;
    a.B = dims->block_size;
    a.N = dims->num_blocks;
    a.max_blocks = dims->max_blocks_per_seq;
    a.partition_size = chunk_partition(dims);
    a.max_parts = parts;
    a.max_query_len = max_query_len;
    a.head_group = pa::decode_head_group(dims->num_kv_heads);
    a.row_warps = pa::chunk_row_warps(max_query_len, dims->num_q_heads / dims->num_kv_heads);
    a.scale = scale;

    const bool bf16 = dims->kv_dtype == PA_BF16;
    const bool umma = pa::chunk_uses_umma(max_query_len, dims->num_q_heads / dims->num_kv_heads);
    a.umma_rows = umma ? pa::chunk_umma_rows(max_query_len, dims->num_q_heads / dims->num_kv_heads) : 0;
    const int box_heads = umma ? 1 : a.head_group;
    const long long block_heads = (long long)dims->num_blocks * dims->num_kv_heads;
    CUtensorMap tmk, tmv;
    cudaError_t e = cache_tensor_map(k_cache, bf16, dims->head_dim, dims->block_size, block_heads, box_heads, &tmk);
    if (e == cudaSuccess)
        e = cache_tensor_map(v_cache, bf16, dims->head_dim, dims->block_size, block_heads, box_heads, &tmv);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = pa::launch_chunk_plan(a, st);
    if (e != cudaSuccess) return to_status(e);
    if (umma) {
        // the tcgen05 kernel loads its query tiles and stores its output with TMA as well
        CUtensorMap tmq, tmo;
        e = query_tensor_map(q, bf16, dims->head_dim, dims->num_q_heads, num_tokens,
                             dims->num_q_heads / dims->num_kv_heads, &tmq);
        if (e == cudaSuccess)
            e = output_tensor_map(out, dims->head_dim, dims->num_q_heads, num_tokens,
                                  dims->num_q_heads / dims->num_kv_heads, &tmo);
        if (e != cudaSuccess) return PA_ERR_CUDA;
        e = bf16 ? pa::launch_chunk_umma_bf16(a, tmk, tmv, tmq, tmo, st)
                 : pa::launch_chunk_umma_f16(a, tmk, tmv, tmq, tmo, st);
        return to_status(e);
    }
    e = bf16 ? pa::launch_chunk_mma_bf16(a, tmk, tmv, st) : pa::launch_chunk_mma_f16(a, tmk, tmv, st);
    if (e != cudaSuccess) return to_status(e);
    if (parts > 1) e = pa::launch_chunk_merge(a, st);
    return to_status(e);
}

int32_t pa_write_kv(const pa_dims *dims, const void *k, const void *v, const int64_t *slot_mapping,
                    int32_t num_tokens, void *k_cache, void *v_cache, void *stream) {
    int32_t rc = check_cache_dims(dims);
    if (rc != PA_OK) return rc;
    if (num_tokens < 0) return PA_ERR_INVALID;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PA_ERR_INVALID;
    unsigned int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    return to_status(pa::launch_write_kv(k, v, slot_mapping, num_tokens, dims->num_kv_heads,
                                         dims->head_dim * elem_bytes(dims->kv_dtype), dims->block_size,
                                         dims->num_blocks, k_cache, v_cache, err,
                                         static_cast<cudaStream_t>(stream)));
}

int32_t pa_copy_blocks(const pa_dims *dims, void *k_cache, void *v_cache, const int64_t *src_dst_pairs,
                       int32_t num_pairs, void *stream) {
    const int64_t layer_bytes = dims ? (int64_t)dims->num_blocks * dims->num_kv_heads * dims->block_size *
                                           dims->head_dim * elem_bytes(dims->kv_dtype)
                                     : 0;
    return pa_copy_blocks_layers(dims, k_cache, v_cache, 1, layer_bytes, src_dst_pairs, num_pairs, stream);
}

// Layers one copy or swap launch covers: its grid has 2 * num_layers rows (K and V).
constexpr int32_t kMaxCopyLayers = 32767;

int32_t pa_copy_blocks_layers(const pa_dims *dims, void *k_caches, void *v_caches, int32_t num_layers,
                              int64_t layer_stride_bytes, const int64_t *src_dst_pairs, int32_t num_pairs,
                              void *stream) {
    int32_t rc = check_cache_dims(dims);
    if (rc != PA_OK) return rc;
    // the copy grid's y extent is 2 * num_layers, at most 65535
    if (num_pairs < 0 || num_layers < 0 || num_layers > kMaxCopyLayers) return PA_ERR_INVALID;
    if (num_pairs == 0 || num_layers == 0) return PA_OK;
    const int64_t block_bytes =
        (int64_t)dims->num_kv_heads * dims->block_size * dims->head_dim * elem_bytes(dims->kv_dtype);
    const int64_t pool_bytes = block_bytes * dims->num_blocks;
    if (!k_caches || !v_caches || !src_dst_pairs || !aligned(k_caches, 16) || !aligned(v_caches, 16) ||
        !aligned(src_dst_pairs, 8))
        return PA_ERR_INVALID;
    if (num_layers > 1 && (layer_stride_bytes < pool_bytes || layer_stride_bytes % 16 != 0)) return PA_ERR_INVALID;
    unsigned int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    return to_status(pa::launch_copy_blocks(k_caches, v_caches, src_dst_pairs, num_pairs, block_bytes,
                                            dims->num_blocks, num_layers, layer_stride_bytes, err,
                                            static_cast<cudaStream_t>(stream)));
}

namespace {
// The device-side address of host memory the GPU can access directly (pinned
// or registered), or nullptr.
void *device_alias_of_host(void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost) return nullptr;
    return at.devicePointer;
}
}  // namespace

int32_t pa_swap_blocks(const pa_dims *dims, void *k_cache, void *v_cache, void *host_k, void *host_v,
                       int32_t num_host_blocks, int32_t num_layers, int64_t dev_layer_stride_bytes,
                       int64_t host_layer_stride_bytes, const int64_t *pairs, int32_t num_pairs, int32_t direction,
                       void *stream) {
    int32_t rc = check_cache_dims(dims);
    if (rc != PA_OK) return rc;
    if (num_pairs < 0 || num_layers < 0 || num_layers > kMaxCopyLayers || num_host_blocks <= 0 ||
        (direction != PA_SWAP_OUT && direction != PA_SWAP_IN))
        return PA_ERR_INVALID;
    if (num_pairs == 0 || num_layers == 0) return PA_OK;
    const int64_t block_bytes =
        (int64_t)dims->num_kv_heads * dims->block_size * dims->head_dim * elem_bytes(dims->kv_dtype);
    if (!k_cache || !v_cache || !host_k || !host_v || !pairs || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(host_k, 16) || !aligned(host_v, 16) || !aligned(pairs, 8))
        return PA_ERR_INVALID;
    if (num_layers > 1 && (dev_layer_stride_bytes < block_bytes * dims->num_blocks || dev_layer_stride_bytes % 16 ||
                           host_layer_stride_bytes < block_bytes * num_host_blocks || host_layer_stride_bytes % 16))
        return PA_ERR_INVALID;
    void *hk = device_alias_of_host(host_k);
    void *hv = device_alias_of_host(host_v);
    if (!hk || !hv) return PA_ERR_INVALID;  // not pinned / registered host memory
    unsigned int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (direction == PA_SWAP_OUT)
        return to_status(pa::launch_swap_blocks(k_cache, v_cache, hk, hv, pairs, num_pairs, block_bytes, num_layers,
                                                dev_layer_stride_bytes, host_layer_stride_bytes, dims->num_blocks,
                                                num_host_blocks, err, st));
    return to_status(pa::launch_swap_blocks(hk, hv, k_cache, v_cache, pairs, num_pairs, block_bytes, num_layers,
                                            host_layer_stride_bytes, dev_layer_stride_bytes, num_host_blocks,
                                            dims->num_blocks, err, st));
}

int32_t pa_copy_to_device(void *dst_device, const void *src_host, size_t bytes, void *stream) {
    if (bytes == 0) return PA_OK;
    if (!dst_device || !src_host) return PA_ERR_INVALID;
    return cudaMemcpyAsync(dst_device, src_host, bytes, cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int32_t pa_copy_to_host(void *dst_host, const void *src_device, size_t bytes, void *stream) {
    if (bytes == 0) return PA_OK;
    if (!dst_host || !src_device) return PA_ERR_INVALID;
    return cudaMemcpyAsync(dst_host, src_device, bytes, cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int32_t pa_device_errors(uint32_t *flags, int32_t clear) {
    if (!flags) return PA_ERR_INVALID;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_error_word, sizeof v) != cudaSuccess) return PA_ERR_CUDA;
    *flags = v;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof zero) != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

const char *pa_version(void) { return "pa 0.1.0 sm_103a"; }

}  // extern "C"
