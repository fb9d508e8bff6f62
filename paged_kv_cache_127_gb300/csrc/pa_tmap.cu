// pa_tmap.cu -- tensor maps (TMA descriptors) for the KV caches.
//
// A cache [N, Hkv, B, D] of 16-bit elements is described as a 3-D tensor
// {D columns, B rows, N*Hkv (block, head) pairs}.  A box is 64 columns (128
// bytes) x 16 rows x HG consecutive (block, head) pairs: 16 token rows of HG
// KV heads of one physical block, the left or right half of D.  It lands in
// shared memory as [HG][16][128 bytes] with the 128-byte swizzle, so ldmatrix
// reads of 8 rows hit 8 different bank groups, and one copy moves HG x 2 KB.
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <class Fn>
Fn driver_fn(const char *name, unsigned int version) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<Fn>(p);
    return nullptr;
}
}  // namespace

unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        get_current = driver_fn<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
        get_id = driver_fn<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

cudaError_t make_cache_tensor_map(CUtensorMap *map, const void *cache, bool bf16, int D, int B,
                                  long long block_heads, int head_group) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)B, (cuuint64_t)block_heads};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)B * D * 2};
    const cuuint32_t box[3] = {64u, (cuuint32_t)kChunkRows, (cuuint32_t)head_group};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_query_tensor_map(CUtensorMap *map, const void *q, bool bf16, int D, int Hq, long long T, int G) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
    const cuuint32_t box[3] = {64u, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void *>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The fp32 output [T, Hq, D] of the tcgen05 chunk path, for TMA stores: a box
// is 32 columns (128 bytes, 128-byte swizzle) x G heads x 128 / G tokens, the
// 128 rows of one query tile in (token, head) order.
cudaError_t make_output_tensor_map(CUtensorMap *map, float *out, int D, int Hq, long long T, int G) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)Hq * D * 4};
    const cuuint32_t box[3] = {32u, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace pa
