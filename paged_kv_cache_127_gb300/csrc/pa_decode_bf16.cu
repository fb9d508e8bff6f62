// pa_decode_bf16.cu -- tensor-core decode instantiations for bf16 KV caches
// (a translation unit of its own so the dtypes compile in parallel).
#include "pa_decode_mma.cuh"

namespace pa {
cudaError_t launch_decode_mma_bf16(const DecodeArgs &a, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                 cudaStream_t st) {
    return dispatch_decode_mma<__nv_bfloat16>(a, tmk, tmv, st);
}
cudaError_t decode_mma_ctas_bf16(const DecodeArgs &a, int *ctas) {
    return dispatch_decode_mma_grid<__nv_bfloat16>(a, ctas);
}
}  // namespace pa
