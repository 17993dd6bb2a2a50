// bsa_noalloc.cu -- the selector for callers that cannot allocate device
// memory.
//
// bsa_topk_select needs a caller-provided workspace when its launch policy
// splits long rows over several warps (the split path keeps per-chunk
// candidate lists and merge tickets there).  Some callers have no way to
// provide one: code that runs while a CUDA graph is being captured in a mode
// that forbids cudaMalloc, plugins hosted by an engine that owns all device
// memory and exposes no allocator to them, and real-time loops that must not
// call into the allocator at all.  For them this file keeps the scratch in a
// fixed file-scope device array and forwards to bsa_topk_select.
//
// The array's device address is looked up once per device (with that device
// current) by the first call made on it, whether or not that call needs
// scratch; that first call should therefore come before any stream capture.
// Every later call on the device reuses the same array, so calls that overlap
// on the GPU (other streams, other host threads) race on it.  The merge
// tickets the split path needs at zero are cleared by bsa_topk_select on every
// call; nothing else must start at zero.
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "../../include/bsa_topk.h"

namespace {

constexpr size_t kScratchBytes = BSA_NOALLOC_SCRATCH_BYTES;

// One copy per device that loads this library's code; held until exit.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_addr[kMaxDevices];
cudaError_t g_status[kMaxDevices];

// Device address of the current device's copy of g_scratch.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(g_once[dev], [dev] {
        void* p = nullptr;
        g_status[dev] = cudaGetSymbolAddress(&p, g_scratch);
        g_addr[dev] = p;
    });
    if (g_status[dev] != cudaSuccess) return g_status[dev];
    *out = g_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int bsa_topk_select_noalloc(const void* scores, int32_t dtype, int64_t T, int64_t H,
                                       int64_t M, int64_t token_stride, int64_t head_stride,
                                       const int32_t* num_valid_pages, int32_t K,
                                       int32_t num_init, int32_t num_local, int32_t* out_idx,
                                       void* stream) {
    const size_t need = bsa_topk_workspace_bytes(T, H, M, K, dtype);
    if (need > kScratchBytes) return BSA_ERR_CAPACITY;
    // Looked up on every call (a cached read after the first), so that the
    // lookup never waits for the first call that needs scratch.
    void* ws = nullptr;
    const cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) return (int)e;
    // token-major [T, H, K] output
    return bsa_topk_select(scores, dtype, T, H, M, token_stride, head_stride, num_valid_pages,
                           K, num_init, num_local, out_idx, H * (int64_t)K, (int64_t)K, ws,
                           need > 0 ? kScratchBytes : 0, stream);
}
