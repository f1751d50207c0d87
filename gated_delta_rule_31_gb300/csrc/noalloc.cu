// noalloc.cu - gdr_fwd_chunked_noalloc: the chunked forward without a caller-provided
// workspace, for callers that cannot allocate device memory themselves (see gdr.h).
//
// The scratch lives in a file-scope __device__ array, so it exists on every GPU that loads
// this library and stays there until the process exits. Host code cannot use the array's
// name as a device address (on the host it names a shadow variable), so the device address
// is looked up once per device with cudaGetSymbolAddress while that device is current, and
// cached. The call then runs the regular gdr_fwd_chunked path on that scratch.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gdr.h"

namespace {

constexpr size_t kScratchBytes = (size_t)GDR_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up on first use).
gdr_status scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDR_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GDR_OK;
}

}  // namespace

extern "C" gdr_status gdr_fwd_chunked_noalloc(const gdr_problem* p, const void* q, const void* k, const void* v,
                                              const float* g, const float* beta, const float* h0, void* o,
                                              float* ht, gdr_stream_t stream) {
    const size_t need = gdr_fwd_chunked_workspace(p);
    if (need == 0) {  // invalid or unsupported problem: let the regular call report which
        return gdr_fwd_chunked(p, q, k, v, g, beta, h0, o, ht, nullptr, 0, stream);
    }
    if (need > kScratchBytes) return GDR_ERR_WORKSPACE;  // larger than the built-in scratch
    void* ws = nullptr;
    gdr_status s = scratch_on_current_device(&ws);
    if (s != GDR_OK) return s;
    return gdr_fwd_chunked(p, q, k, v, g, beta, h0, o, ht, ws, kScratchBytes, stream);
}
