// pa_decode_bf16.cu -- decode kernel instantiations for bf16 KV caches (kept in a
// translation unit of their own so the three dtypes compile in parallel).
#include "pa_decode.cuh"

namespace pa {
cudaError_t launch_decode_bf16(const DecodeArgs &a, cudaStream_t st) { return dispatch_decode<__nv_bfloat16>(a, st); }
}  // namespace pa
