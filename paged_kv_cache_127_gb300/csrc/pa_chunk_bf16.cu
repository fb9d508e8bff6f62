// pa_chunk_bf16.cu -- tensor-core chunk-attention instantiations (mma.sync and tcgen05) for bf16 KV
// caches (a translation unit of its own so the dtypes compile in parallel).
#include "pa_chunk_mma.cuh"
#include "pa_chunk_umma.cuh"

namespace pa {
cudaError_t launch_chunk_mma_bf16(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                  cudaStream_t st) {
    return dispatch_chunk_mma<__nv_bfloat16>(a, tmk, tmv, st);
}
cudaError_t launch_chunk_umma_bf16(const ChunkArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                  const CUtensorMap &tmq, const CUtensorMap &tmo, cudaStream_t st) {
    return dispatch_chunk_umma<__nv_bfloat16>(a, tmk, tmv, tmq, tmo, st);
}
}  // namespace pa
