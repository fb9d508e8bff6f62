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

unsigned int *error_word() {
    static std::mutex mu;
    static unsigned int *cache[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<unsigned int *>(p);
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

int32_t effective_partition(const pa_dims *d) {
    return d->partition_size > 0 ? d->partition_size : kDefaultPartition;
}

// Full decode checks; fills max_parts.
int32_t check_decode_dims(const pa_dims *d, int32_t *max_parts) {
    int32_t rc = check_cache_dims(d);
    if (rc != PA_OK) return rc;
    if (d->num_seqs < 0 || d->num_q_heads <= 0 || d->max_blocks_per_seq <= 0) return PA_ERR_INVALID;
    if (d->num_q_heads % d->num_kv_heads != 0) return PA_ERR_INVALID;
    if (d->partition_size < 0) return PA_ERR_INVALID;
    const int32_t G = d->num_q_heads / d->num_kv_heads;
    const int32_t pt = effective_partition(d);
    if (pt % d->block_size != 0 || pt / d->block_size > pa::kMaxPartitionBlocks) return PA_ERR_INVALID;
    if (!(d->head_dim == 64 || d->head_dim == 128) || !(d->block_size == 16 || d->block_size == 32) ||
        !(G == 1 || G == 2 || G == 4 || G == 8))
        return PA_ERR_UNSUPPORTED;
    const int64_t cap = (int64_t)d->max_blocks_per_seq * d->block_size;
    if (cap > INT32_MAX) return PA_ERR_INVALID;
    const int64_t parts = (cap + pt - 1) / pt;
    if (parts > 65535) return PA_ERR_INVALID;
    if ((int64_t)d->num_seqs * d->num_kv_heads > INT32_MAX) return PA_ERR_INVALID;
    *max_parts = (int32_t)parts;
    return PA_OK;
}

size_t workspace_bytes_for(const pa_dims *d, int32_t max_parts) {
    if (max_parts <= 1) return 0;
    const size_t rows = (size_t)d->num_seqs * d->num_q_heads * max_parts;
    const size_t bytes = rows * (size_t)(d->head_dim + 2) * sizeof(float);
    return (bytes + 255) & ~(size_t)255;
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

int32_t pa_decode(const pa_dims *dims, const void *q, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, const int32_t *context_lens, float scale, float *out,
                  void *workspace, size_t workspace_bytes, void *stream) {
    int32_t parts = 0;
    int32_t rc = check_decode_dims(dims, &parts);
    if (rc != PA_OK) return rc;
    if (dims->num_seqs == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID;
    const size_t need = workspace_bytes_for(dims, parts);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16))) return PA_ERR_INVALID;

    pa::DecodeArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = out;
    const size_t acc_floats = (size_t)dims->num_seqs * dims->num_q_heads * parts * dims->head_dim;
    a.ws_acc = need ? static_cast<float *>(workspace) : nullptr;
    a.ws_ml = need ? static_cast<float *>(workspace) + acc_floats : nullptr;
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
    a.scale = scale;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (dims->kv_dtype) {
        case PA_F32: e = pa::launch_decode_f32(a, st); break;
        case PA_F16: e = pa::launch_decode_f16(a, st); break;
        default: e = pa::launch_decode_bf16(a, st); break;
    }
    if (e != cudaSuccess) return to_status(e);
    if (parts > 1) {
        e = pa::launch_decode_merge(a, st);
        if (e != cudaSuccess) return to_status(e);
    }
    return PA_OK;
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
    int32_t rc = check_cache_dims(dims);
    if (rc != PA_OK) return rc;
    if (num_pairs < 0) return PA_ERR_INVALID;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !src_dst_pairs || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(src_dst_pairs, 8))
        return PA_ERR_INVALID;
    unsigned int *err = error_word();
    if (!err) return PA_ERR_CUDA;
    const int64_t block_bytes =
        (int64_t)dims->num_kv_heads * dims->block_size * dims->head_dim * elem_bytes(dims->kv_dtype);
    return to_status(pa::launch_copy_blocks(k_cache, v_cache, src_dst_pairs, num_pairs, block_bytes,
                                            dims->num_blocks, err, static_cast<cudaStream_t>(stream)));
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
