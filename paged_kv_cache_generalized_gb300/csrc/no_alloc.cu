// pa_forward_no_alloc: pa_forward for callers that cannot allocate device memory.
//
// Its scratch is a file-scope device array of fixed size, so the library (not the caller)
// provides it and nothing is allocated at call time.  Every device that loads the library holds
// this array (PA_NO_ALLOC_WORKSPACE_BYTES) until the process exits.
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace {

// The shared scratch.  Host code must not use this symbol as an address: it names a host-side
// stand-in, and a kernel given it would fault or (where the GPU can reach host memory) silently
// use the wrong memory.  The device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_no_alloc_ws[PA_NO_ALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_no_alloc_ws on the current device, looked up once per device (the first
// call on a device does this set-up, with that device current).
pa_status no_alloc_workspace(void **out) {
    static void *ptrs[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_no_alloc_ws) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        ptrs[dev] = p;
    }
    *out = ptrs[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_forward_no_alloc(const pa_dims *dims, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *ctx_lens, const int32_t *q_lens,
                                          float scale, void *out, pa_stream_t stream) {
    const size_t need = pa_forward_workspace_size(dims);
    if (need == 0) {
        // invalid or unsupported dims: let pa_forward report which, before any device work
        return pa_forward(dims, q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale, out,
                          nullptr, 0, stream);
    }
    if (need > (size_t)PA_NO_ALLOC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
    void *ws = nullptr;
    const pa_status st = no_alloc_workspace(&ws);
    if (st != PA_OK) return st;
    // pa_forward's workspace needs no initialisation: its planner writes everything it reads.
    return pa_forward(dims, q, k_cache, v_cache, block_tables, ctx_lens, q_lens, scale, out, ws,
                      (size_t)PA_NO_ALLOC_WORKSPACE_BYTES, stream);
}
