// pa_decode_f16.cu -- decode kernel instantiations for f16 KV caches (kept in a
// translation unit of their own so the three dtypes compile in parallel).
#include "pa_decode.cuh"

namespace pa {
cudaError_t launch_decode_f16(const DecodeArgs &a, cudaStream_t st) { return dispatch_decode<__half>(a, st); }
}  // namespace pa
