// moe_forward_static_scratch: the whole layer with its scratch in a fixed
// array inside this library instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they run the layer -- an inference-engine plugin whose enqueue step is
// handed fixed buffers and must not allocate, or a serving process that
// reserved its whole memory budget at start-up, so that a later cudaMalloc
// would fail or break its accounting.  They pass the tokens, the weights and
// the output buffer; the library supplies the scratch.  The kernels are
// enqueued directly on the caller's stream (the launch-graph cache of
// moe_forward is not used here, since building a graph takes driver
// resources).
//
// The array is MOE_STATIC_SCRATCH_BYTES per device and stays allocated, on
// every device that loads the library, until the process exits.  All calls on
// a device share it, so calls whose GPU work overlaps (different streams, or
// host threads racing) corrupt each other's scratch: serialise them.  A call
// leaves the previous call's contents behind; nothing needs to start at zero,
// since every scratch element a call reads was written earlier in that call.
#include <mutex>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[64];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is asked from
// the runtime once per device (with that device current) and cached.
int scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_forward_static_scratch(const void *x, const void *W_g,
                                          const float *router_bias, const void *const *W1,
                                          const void *const *W3, const void *const *W2, int T,
                                          int d, int ffn, int E, int k, int dtype, void *out,
                                          void *stream) {
    size_t need = 0;
    int rc = moe_workspace_bytes(T, d, ffn, E, k, dtype, &need);
    if (rc != MOE_OK) return rc;
    if (need > MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
    void *scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != MOE_OK) return rc;
    return moe::forward_direct(x, W_g, router_bias, W1, W3, W2, T, d, ffn, E, k, dtype, out,
                               scratch, MOE_STATIC_SCRATCH_BYTES,
                               static_cast<cudaStream_t>(stream));
}
