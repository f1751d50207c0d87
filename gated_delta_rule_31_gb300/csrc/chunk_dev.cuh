// chunk_dev.cuh - device helpers shared by the chunk kernels (prep for scalar and per-channel
// gates): bf16 packing, shared / global 16-byte stores, and the UT solve T = (I + A)^-1.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace gdr {

constexpr int LDA = 65;  // row stride (floats) of the fp32 [64 x 64] A / T tiles in shared memory

__device__ __forceinline__ void unpack8(const uint4& u, float* x) {
    x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
    x[4] = bf16lo(u.z); x[5] = bf16hi(u.z); x[6] = bf16lo(u.w); x[7] = bf16hi(u.w);
}
__device__ __forceinline__ uint4 pack8(const float* x, float s) {
    return make_uint4(pack_bf16(s * x[0], s * x[1]), pack_bf16(s * x[2], s * x[3]), pack_bf16(s * x[4], s * x[5]),
                      pack_bf16(s * x[6], s * x[7]));
}
__device__ __forceinline__ void st_chunk(uint32_t addr, const float* x, float s) {
    const uint4 u = pack8(x, s);
    st_shared_v4(addr, u.x, u.y, u.z, u.w);
}
__device__ __forceinline__ void st_global16(uint8_t* p, const uint4& u) { *reinterpret_cast<uint4*>(p) = u; }

// T = (I + A)^-1 for the strictly lower triangular fp32 A [64 x 64] (row stride LDA), by 16 x 16
// blocks. Phase 1 (160 threads, one column each): forward substitution with L_II = I + A_II
// gives the diagonal inverses T_II (right-hand side e_c) and Y_IK = T_II A_IK for I > K
// (right-hand side column c of A_IK). Then T_IJ = -sum_{J<=K<I} Y_IK T_KJ by block distance
// I - J = 1, 2, 3. Called by all 256 threads of the CTA; ends with a CTA barrier. T's blocks
// above the block diagonal are not written (they are zero). Xs: [6][16][17] fp32 scratch.
__device__ __forceinline__ void ut_solve(const float* Am, float* Tm, float* Xs, int tid) {
    if (tid < 160) {
        int I, K, cc;
        const bool diag = tid < 64;
        if (diag) {
            I = tid >> 4;
            K = I;
            cc = tid & 15;
        } else {
            const int pidx = (tid - 64) >> 4;  // pairs (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
            cc = (tid - 64) & 15;
            I = pidx == 0 ? 1 : (pidx < 3 ? 2 : 3);
            K = pidx - I * (I - 1) / 2;
        }
        const float* Ab = Am + (16 * I) * LDA + 16 * I;
        const float* Bc = Am + (16 * I) * LDA + 16 * K + cc;
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; i++) {
            float s = diag ? (i == cc ? 1.f : 0.f) : Bc[i * LDA];
#pragma unroll
            for (int j = 0; j < i; j++) s -= Ab[i * LDA + j] * y[j];
            y[i] = s;
        }
        if (diag) {
#pragma unroll
            for (int i = 0; i < 16; i++) Tm[(16 * I + i) * LDA + 16 * I + cc] = y[i];
        } else {
            float* yp = Xs + ((tid - 64) >> 4) * (16 * 17);
#pragma unroll
            for (int i = 0; i < 16; i++) yp[i * 17 + cc] = y[i];
        }
    }
    __syncthreads();
    // item J of a level is block (J + dlev, J); all sums are formed before any store
    for (int dlev = 1; dlev <= 3; dlev++) {
        const int nb = 4 - dlev;
        const int i = (tid >> 4) & 15, cc = tid & 15;
        float s[3] = {0.f, 0.f, 0.f};
#pragma unroll
        for (int J = 0; J < 3; J++) {
            if (J < nb) {
                const int I = J + dlev;
                for (int K = J; K < I; K++) {
                    const float* yr = Xs + (I * (I - 1) / 2 + K) * (16 * 17) + i * 17;
                    const float* tc = Tm + (16 * K) * LDA + 16 * J + cc;
#pragma unroll
                    for (int m = 0; m < 16; m++) s[J] += yr[m] * tc[m * LDA];
                }
            }
        }
#pragma unroll
        for (int J = 0; J < 3; J++)
            if (J < nb) Tm[(16 * (J + dlev) + i) * LDA + 16 * J + cc] = -s[J];
        __syncthreads();
    }
}

}  // namespace gdr
