// pa_decode_f32.cu -- decode kernel instantiations for f32 KV caches (kept in a
// translation unit of their own so the three dtypes compile in parallel).
#include "pa_decode.cuh"

namespace pa {
cudaError_t launch_decode_f32(const DecodeArgs &a, cudaStream_t st) { return dispatch_decode<float>(a, st); }
}  // namespace pa
