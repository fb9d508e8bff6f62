// pa_noalloc.cu -- pa_decode for callers that cannot allocate device memory.
//
// Some callers have no way to hand pa_decode a workspace: code running inside
// a memory pool or arena that forbids further device allocations, plugin hosts
// that own every allocation, or setups where a cudaMalloc would synchronise
// the device at a bad moment.  For them, this entry point takes its split-K
// scratch from a fixed buffer compiled into the library instead of from the
// caller.
//
// The buffer is a file-scope __device__ array of PA_NOALLOC_SCRATCH_BYTES
// bytes.  Every GPU that loads the library holds it until the process exits.
// Host code cannot use the array's name as a device address, so the entry
// point looks up the real device address with cudaGetSymbolAddress the first
// time it runs on each device (with that device current) and caches it, keyed
// by the CUDA context so that a device reset leads to a fresh lookup.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch in the current context.  It is looked
// up once per device and cached with the context's id; when the id changes
// (the device was reset and its primary context rebuilt) it is looked up again.
void *scratch_for_current_device() {
    static std::mutex mu;
    static unsigned long long ctx_of[kMaxDevices] = {};
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = pa::current_context_id();
    if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = p;
        ctx_of[dev] = pa::current_context_id();   // the lookup makes the primary context current
    }
    return addr[dev];
}

}  // namespace

extern "C" int32_t pa_decode_noalloc(const pa_dims *dims, const void *q, const void *k_cache,
                                     const void *v_cache, const int32_t *block_tables,
                                     const int32_t *context_lens, float scale, float *out, void *stream) {
    if (!dims) return PA_ERR_INVALID;
    // pa_decode_workspace_bytes returns 0 both for "no scratch needed" and for
    // invalid dims; pa_decode itself reports the latter.
    const size_t need = pa_decode_workspace_bytes(dims);
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_TOO_LARGE;
    void *scratch = nullptr;
    if (need > 0) {
        scratch = scratch_for_current_device();
        if (!scratch) return PA_ERR_CUDA;
    }
    // pa_decode writes every scratch byte it later reads within the same call,
    // so whatever an earlier call left in the buffer does not matter.
    return pa_decode(dims, q, k_cache, v_cache, block_tables, context_lens, scale, out, scratch,
                     need > 0 ? (size_t)PA_NOALLOC_SCRATCH_BYTES : 0, stream);
}
