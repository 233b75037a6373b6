// decode_noalloc.cu -- the fused decode for callers that must not allocate.
//
// Some callers cannot call cudaMalloc at decode time: a runtime that hands out
// every byte of device memory from its own pool up front, code running inside
// a region where allocation is forbidden or would synchronise the device, or a
// plugin that may not own device allocations.  dattn_decode_f16_ex needs a
// workspace for its split-K partial states, and dattn_decode_f16 allocates one.
// This entry point instead uses a fixed scratch array that is part of the
// library image: a file-scope __device__ array, created on each GPU when this
// module is loaded there and held until the process exits.
//
// In host code, g_noalloc_scratch is only a host-side stand-in for the device
// array, not a device address.  The address of the array on the current
// device is looked up once per device with cudaGetSymbolAddress and passed to
// the kernels as their workspace.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "dattn.h"
#include "dattn_internal.h"

namespace {

constexpr size_t kScratchBytes = DATTN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (set up once per
// device, with that device current).
int scratch_address(void **addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
        return dattn::set_last_error(DATTN_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevices)
        return dattn::set_last_error(DATTN_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            char msg[256];
            snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(no-alloc scratch): %s",
                     cudaGetErrorString(e));
            return dattn::set_last_error(DATTN_ERR_CUDA, msg);
        }
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return DATTN_OK;
}

}  // namespace

extern "C" int dattn_decode_f16_noalloc(const void *Q, const void *K_cache, const void *V_cache,
                                        void *out, int batch, int n_heads, int head_dim,
                                        int seq_len, const uint32_t *current_pos,
                                        dattn_stream_t stream) {
    size_t need = 0;
    if (int st = dattn_decode_workspace_bytes(batch, n_heads, head_dim, seq_len, 0, &need))
        return st;
    if (need > kScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "this shape needs %zu bytes of scratch; the static no-alloc scratch holds %zu "
                 "(use dattn_decode_f16_ex with a workspace)",
                 need, kScratchBytes);
        return dattn::set_last_error(DATTN_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    if (int st = scratch_address(&scratch)) return st;
    // Nothing in the scratch has to start at zero: each call writes every
    // partial state before the combine reads it.
    return dattn_decode_f16_ex(Q, K_cache, V_cache, out, batch, n_heads, head_dim, seq_len,
                               current_pos, scratch, kScratchBytes, 0, stream);
}
