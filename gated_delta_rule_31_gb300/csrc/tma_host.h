// tma_host.h - host-side creation of TMA tensor maps (driver entry point fetched through
// the runtime, so the library does not link libcuda directly).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdr {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Map over a dense tensor [n3, n2, n1, n0] (n0 innermost) of `esize`-byte elements, moving
// boxes of box0 x 1 x box2 x 1 elements (box0 contiguous) with the given swizzle. Loads read
// elements outside the tensor as zero; stores skip them.
inline bool make_map_4d(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base, uint64_t n0,
                        uint64_t n1, uint64_t n2, uint64_t n3, uint32_t box0, uint32_t box2, CUtensorMapSwizzle swz) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {n0, n1, n2, n3};
    cuuint64_t strides[3] = {n0 * esize, n0 * n1 * esize, n0 * n1 * n2 * esize};
    cuuint32_t box[4] = {box0, 1, box2, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
inline bool make_map_4d_bf16(CUtensorMap* m, const void* base, uint64_t n0, uint64_t n1, uint64_t n2, uint64_t n3,
                             uint32_t box0, uint32_t box2, CUtensorMapSwizzle swz) {
    return make_map_4d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, n0, n1, n2, n3, box0, box2, swz);
}

}  // namespace gdr
