// pad.cu - staging copies for head sizes below the tensor-core path's 128: a tensor viewed as
// [outer][rows][cols] is copied into [outer][rows_to][cols_to] with zeros in the added rows and
// columns, and results are cropped back. Zero key / query / value channels and zero state rows
// and columns contribute nothing to any product of the chunk algebra, so the padded problem's
// results in the original channels are those of the original problem.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace gdr {

namespace {

template <typename T>
__global__ void pad_kernel(const T* __restrict__ src, T* __restrict__ dst, size_t outer, int rs, int cs, int rd,
                           int cd) {
    const size_t n = outer * (size_t)rd * cd;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % cd);
        const size_t t = i / cd;
        const int r = (int)(t % rd);
        const size_t o = t / rd;
        dst[i] = (r < rs && c < cs) ? src[(o * rs + r) * cs + c] : T(0);
    }
}

template <typename T>
__global__ void crop_kernel(const T* __restrict__ src, T* __restrict__ dst, size_t outer, int rs, int cs, int rd,
                            int cd) {
    const size_t n = outer * (size_t)rd * cd;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % cd);
        const size_t t = i / cd;
        const int r = (int)(t % rd);
        const size_t o = t / rd;
        dst[i] = src[(o * rs + r) * cs + c];
    }
}

unsigned grid_for(size_t n) {
    const size_t b = (n + 255) / 256;
    return (unsigned)(b < 4096 ? (b ? b : 1) : 4096);
}

}  // namespace

cudaError_t launch_pad(const void* src, void* dst, int elem_bytes, size_t outer, int rs, int cs, int rd, int cd,
                       cudaStream_t s) {
    const size_t n = outer * (size_t)rd * cd;
    if (n == 0) return cudaSuccess;
    trace_begin("stage_pad", s);
    if (elem_bytes == 2)
        pad_kernel<uint16_t><<<grid_for(n), 256, 0, s>>>(static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst),
                                                        outer, rs, cs, rd, cd);
    else
        pad_kernel<float><<<grid_for(n), 256, 0, s>>>(static_cast<const float*>(src), static_cast<float*>(dst), outer,
                                                     rs, cs, rd, cd);
    trace_end(s);
    return cudaGetLastError();
}

cudaError_t launch_crop(const void* src, void* dst, int elem_bytes, size_t outer, int rs, int cs, int rd, int cd,
                        cudaStream_t s) {
    const size_t n = outer * (size_t)rd * cd;
    if (n == 0) return cudaSuccess;
    trace_begin("stage_crop", s);
    if (elem_bytes == 2)
        crop_kernel<uint16_t><<<grid_for(n), 256, 0, s>>>(static_cast<const uint16_t*>(src),
                                                         static_cast<uint16_t*>(dst), outer, rs, cs, rd, cd);
    else
        crop_kernel<float><<<grid_for(n), 256, 0, s>>>(static_cast<const float*>(src), static_cast<float*>(dst), outer,
                                                      rs, cs, rd, cd);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace gdr
