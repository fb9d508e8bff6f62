// pa_chunk_bf16.cu -- tensor-core chunk-attention instantiations for bf16 KV
// caches (a translation unit of its own so the dtypes compile in parallel).
#include "pa_chunk_mma.cuh"

namespace pa {
cudaError_t launch_chunk_mma_bf16(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                  cudaStream_t st) {
    return dispatch_chunk_mma<__nv_bfloat16>(a, tmk, tmv, st);
}
}  // namespace pa
