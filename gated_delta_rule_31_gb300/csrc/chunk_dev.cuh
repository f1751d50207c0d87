// chunk_dev.cuh - device helpers shared by the chunk kernels: bf16 packing, shared / global
// 16-byte stores, the lane split of M=64 accumulator rows, and the UT solve T = (I + A)^-1.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"

namespace gdr {

// Row stride (floats) of the fp32 [64 x 64] A / T tiles in shared memory: rows start on 16-byte
// boundaries, so rows and 4-column strips move as float4.
constexpr int LDA = 68;
constexpr int LDY = 20;  // row stride of the [16 x 16] Y blocks of the solve scratch (float4 rows)
constexpr int SOLVE_SCRATCH_BYTES = 6 * 16 * LDY * 4;

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

// An M=64 accumulator row lives in lane l < 16 of its warp; lane l + 16 takes the upper half of
// the N columns read from TMEM: N = 16 -> w[0..7], N = 32 -> w[0..15].
template <int N>
__device__ __forceinline__ void split_cols(const float* v, float* w, int lane) {
#pragma unroll
    for (int e = 0; e < N / 2; e++) {
        const float hi = __shfl_sync(0xffffffffu, v[N / 2 + e], lane & 15);
        w[e] = (lane >> 4) ? hi : v[e];
    }
}

// The same split of N = 32 columns with the 4-column groups interleaved: lane l < 16 takes columns
// 8 q + 0..3 and lane l + 16 columns 8 q + 4..7 (q < 4), w[4 q + i]. A 16-byte store of group q by
// both lanes then fills one 32-byte sector of the row.
__device__ __forceinline__ void split_cols_sector(const float* v, float* w, int lane) {
#pragma unroll
    for (int q = 0; q < 4; q++)
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float hi = __shfl_sync(0xffffffffu, v[8 * q + 4 + i], lane & 15);
            w[4 * q + i] = (lane >> 4) ? hi : v[8 * q + i];
        }
}

// T = (I + A)^-1 for the strictly lower triangular fp32 A [64 x 64] (row stride LDA), by 16 x 16
// blocks. Phase 1 (160 threads, one column each): forward substitution with L_II = I + A_II
// gives the diagonal inverses T_II (right-hand side e_c) and Y_IK = T_II A_IK for I > K
// (right-hand side column c of A_IK); rows of L_II are read as float4. Then, by block distance
// I - J = 1, 2, 3, T_IJ = -sum_{J<=K<I} Y_IK T_KJ with one thread per (block, row, 4-column
// strip), reading Y rows and T strips as float4. Called by all 256 threads of the CTA; ends
// with a CTA barrier. T's blocks above the block diagonal are not written (they are zero).
// Xs: [6][16][LDY] fp32 scratch.
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
            float l[16];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                if (4 * q < i) {
                    const float4 f = *reinterpret_cast<const float4*>(Ab + i * LDA + 4 * q);
                    l[4 * q] = f.x; l[4 * q + 1] = f.y; l[4 * q + 2] = f.z; l[4 * q + 3] = f.w;
                }
            }
            float s = diag ? (i == cc ? 1.f : 0.f) : Bc[i * LDA];
#pragma unroll
            for (int j = 0; j < i; j++) s -= l[j] * y[j];
            y[i] = s;
        }
        if (diag) {
#pragma unroll
            for (int i = 0; i < 16; i++) Tm[(16 * I + i) * LDA + 16 * I + cc] = y[i];
        } else {
            float* yp = Xs + ((tid - 64) >> 4) * (16 * LDY);
#pragma unroll
            for (int i = 0; i < 16; i++) yp[i * LDY + cc] = y[i];
        }
    }
    __syncthreads();
    for (int dlev = 1; dlev <= 3; dlev++) {
        const int J = tid >> 6, i = (tid >> 2) & 15, c4 = tid & 3;  // block (J + dlev, J), row i, cols 4 c4..
        if (J < 4 - dlev) {
            const int I = J + dlev;
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            for (int K = J; K < I; K++) {
                const float* yr = Xs + (I * (I - 1) / 2 + K) * (16 * LDY) + i * LDY;
                float y[16];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float4 f = *reinterpret_cast<const float4*>(yr + 4 * q);
                    y[4 * q] = f.x; y[4 * q + 1] = f.y; y[4 * q + 2] = f.z; y[4 * q + 3] = f.w;
                }
                const float* tc = Tm + (16 * K) * LDA + 16 * J + 4 * c4;
#pragma unroll
                for (int m = 0; m < 16; m++) {
                    const float4 t = *reinterpret_cast<const float4*>(tc + m * LDA);
                    s[0] += y[m] * t.x; s[1] += y[m] * t.y; s[2] += y[m] * t.z; s[3] += y[m] * t.w;
                }
            }
            *reinterpret_cast<float4*>(Tm + (16 * I + i) * LDA + 16 * J + 4 * c4) =
                make_float4(-s[0], -s[1], -s[2], -s[3]);
        }
        __syncthreads();
    }
}

}  // namespace gdr
