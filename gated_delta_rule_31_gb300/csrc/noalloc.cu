// noalloc.cu - gdr_fwd_chunked_noalloc: the chunked forward without a caller-provided
// workspace, for callers that cannot allocate device memory themselves (see gdr.h), and
// gdr_noalloc_status, which reads the status word of its built-in scratch.
//
// The scratch lives in a file-scope __device__ array, so it exists on every GPU that loads
// this library and stays there until the process exits. Host code cannot use the array's
// name as a device address (on the host it names a shadow variable), so the device address
// is looked up once per device with cudaGetSymbolAddress while that device is current, and
// cached. The call then runs the regular gdr_fwd_chunked path on that scratch, whose first
// 256 bytes hold the status word the chunk kernels write when a bounded wait expires.
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

// The device that runs work queued on `stream`; it must be the current device, because the
// scratch address is looked up (and the regular call launches) on the current device.
gdr_status stream_device(gdr_stream_t stream, int* dev) {
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur < 0 || cur >= kMaxDevices) return GDR_ERR_CUDA;
    int sd = cur;
    if (stream && cudaStreamGetDevice((cudaStream_t)stream, &sd) != cudaSuccess) return GDR_ERR_INVALID_ARG;
    if (sd != cur) return GDR_ERR_INVALID_ARG;
    *dev = cur;
    return GDR_OK;
}

// Device address of the scratch array on `dev` (the current device), looked up on first use.
// With lazy module loading this first lookup is also when the driver reserves the array.
gdr_status scratch_on_device(int dev, bool setup, void** out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev] && setup) {
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
    int dev = -1;
    gdr_status s = stream_device(stream, &dev);
    if (s != GDR_OK) return s;
    void* ws = nullptr;
    if ((s = scratch_on_device(dev, true, &ws)) != GDR_OK) return s;
    return gdr_fwd_chunked(p, q, k, v, g, beta, h0, o, ht, ws, kScratchBytes, stream);
}

extern "C" gdr_status gdr_noalloc_status(gdr_stream_t stream) {
    int dev = -1;
    gdr_status s = stream_device(stream, &dev);
    if (s != GDR_OK) return s;
    void* ws = nullptr;
    if ((s = scratch_on_device(dev, false, &ws)) != GDR_OK) return s;
    if (!ws) return GDR_OK;  // no call has run on this device
    return gdr_workspace_status(ws, 256, stream);
}
