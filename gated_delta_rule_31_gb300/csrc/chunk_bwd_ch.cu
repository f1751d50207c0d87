// chunk_bwd_ch.cu - backward (VJP) of the chunked gated delta rule with a per-channel gate
// (one decay per key channel, g [B,T,Hv,Dk]): the channelwise variant of "Two-pass
// optimization for channelwise gated delta rule kernel" (ExecuTorch PR #21020) in the chunked
// reverse mode of "Adding VJP for gated delta net" (MLX PR #4565, chunked case).
//
// Launch sequence: prep_ch (also keeps T, W and K^ .* Gamma per chunk) -> forward states scan
// -> reverse scan (chunk-end state gradients, dh0) -> grad_ch_mma -> grad_ch_simt -> the
// value-head sum with the norm backward.
//
// Per (b, hv, chunk), with E_rj,d = prod_{j<t<=r} a_t,d, Gamma_r,d = prod_{t<=r} a_t,d,
// b_r,d = Gamma_C,d / Gamma_r,d and the chunk algebra of chunk_fwd_ch.cu:
//   U  = U~ - W H0        dU = P^T dO + Kbar dH1          dW = -dU H0^T
//   X  = dO H0^T          Y  = U dH1^T                     Z  = T^T dW
//   dPs = scale tril(dO U^T)        dT = dU (diag(beta) V)^T + dW (diag(beta) K^ .* Gamma)^T
//   dA = -strict_lower(T^T dT T^T)  dv = diag(beta) T^T dU
// (the dense products, on tcgen05: grad_ch_mma). Then per element (r, d) (grad_ch_simt):
//   dq^ = scale Gamma X + sum_{j<=r} dPs_rj k^_j E_rj
//   dk^ = b Y + beta Gamma Z + beta_r sum_{j<r} dA_rj k^_j E_rj
//         + sum_{i>=r} dPs_ir q^_i E_ir + sum_{i>r} dA_ir beta_i k^_i E_ir
//   dgamma_r = every term above times its own factor of Gamma_r (+1), b_r (-1) or E (+1 on
//   the row side, -1 on the column side); dgamma_C = sum_r b k^ Y + Gamma_C <dH1, H0>_d;
//   dg = reverse cumulative sum of dgamma in the chunk (+ dgamma_C on every token);
//   dbeta = V . (T^T dU) + sum_d Gamma k^ Z + sum_d k^ (sum_{j<r} dA_rj k^_j E_rj).
// The decay-weighted contractions run on the CUDA cores with running products of the
// per-token factors a_t <= 1, so no decay can overflow however strong.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "chunk.h"
#include "chunk_dev.cuh"
#include "common.cuh"
#include "kernels.h"

namespace gdr {
namespace {

// ---------------------------------------------------------------- tensor-core pass
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t C_DO = 0;        // dO [64 x 128] (TMA, panels 8 KB)
constexpr uint32_t C_W = 16384;     // W image; then U image
constexpr uint32_t C_KB = 32768;    // Kbar image; then dU image
constexpr uint32_t C_H0 = 49152;    // H0 image [128 d x 128 v]; then dW image [64 x 128]
constexpr uint32_t C_DH = 81920;    // dH1 image; then dT (+0) and Yt (+8 KB) images [64 x 64]
constexpr uint32_t C_V = 114688;    // v [64 x 128] (TMA)
constexpr uint32_t C_KG = 131072;   // K^ .* Gamma image [64 x 128]
constexpr uint32_t C_P = 147456;    // P image [64 x 64]
constexpr uint32_t C_T = 155648;    // T image [64 x 64]
constexpr uint32_t C_SM = 163840;   // bet[64], dbp[4][64]
constexpr uint32_t C_BYTES = C_SM + 2048;
constexpr uint32_t TM1 = 0, TM2 = 128;  // TMEM columns of the two accumulators
constexpr int CH_THREADS = 512;

__device__ __forceinline__ void unpack8c(const uint4& u, float* x) {
    x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
    x[4] = bf16lo(u.z); x[5] = bf16hi(u.z); x[6] = bf16lo(u.w); x[7] = bf16hi(u.w);
}
// An M=64 accumulator row lives in lane l < 16 of its warp; lane l + 16 takes the upper half
// of the columns read: n = 16 -> w[0..7], n = 32 -> w[0..15].
template <int N>
__device__ __forceinline__ void split_cols(const float* v, float* w, int lane) {
#pragma unroll
    for (int e = 0; e < N / 2; e++) {
        const float hi = __shfl_sync(0xffffffffu, v[N / 2 + e], lane & 15);
        w[e] = (lane >> 4) ? hi : v[e];
    }
}
__device__ __forceinline__ void st_f4x(float* dst, const float* x, int n4) {
    for (int q = 0; q < n4; q++)
        reinterpret_cast<float4*>(dst)[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
}

__global__ void __launch_bounds__(CH_THREADS, 1)
    grad_ch_mma_kernel(const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                       GradChArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkProblem& P = a.p;
    const int c = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const int t0 = c * kChunk;
    const size_t idx = ((size_t)b * P.Hv + hv) * P.NC + c;
    const uint8_t* rec = a.rec + idx * REC_BYTES;
    const uint8_t* rec2 = a.rec2 + idx * REC2_BYTES_CH;
    float* chx = reinterpret_cast<float*>(a.chx + idx * CHX_BYTES);
    const int lg = warp & 3, qt = warp >> 2, hf = lane >> 4;
    const int r = 16 * lg + (lane & 15);
    const bool act = lane < 16;
    const int c32 = 32 * qt, c16 = 16 * qt;
    float* bet = reinterpret_cast<float*>(sm + C_SM);
    float* dbp = bet + 64;  // [4][64] V . (T^T dU) partials by column quarter
    uint32_t mph = 0;
    bool ok = true;

    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_sh, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_sh;
    const uint32_t tl = tmem_at(tm, 32 * lg, 0);
    if (tid == 0) {
        mbar_expect_tx(&bar_ld, 163840);
        tma_load_4d(sm + C_DO + 0, &mdo, 0, hv, t0, b, &bar_ld);
        tma_load_4d(sm + C_DO + 8192, &mdo, 64, hv, t0, b, &bar_ld);
        tma_load_4d(sm + C_V + 0, &mv, 0, hv, t0, b, &bar_ld);
        tma_load_4d(sm + C_V + 8192, &mv, 64, hv, t0, b, &bar_ld);
        bulk_load(sm + C_W, rec2 + REC2_W, 16384, &bar_ld);
        bulk_load(sm + C_KB, rec + REC_K, 16384, &bar_ld);
        bulk_load(sm + C_H0, a.hs + idx * STATE_IMG, 32768, &bar_ld);
        bulk_load(sm + C_DH, a.dhs + idx * STATE_IMG, 32768, &bar_ld);
        bulk_load(sm + C_KG, rec2 + REC2_KG, 16384, &bar_ld);
        bulk_load(sm + C_P, rec + REC_P, 8192, &bar_ld);
        bulk_load(sm + C_T, rec2 + REC2_T, 8192, &bar_ld);
    }
    if (tid < 64) bet[tid] = (t0 + tid < P.T) ? a.beta[((size_t)b * P.T + t0 + tid) * P.Hv + hv] : 0.f;
    if (tid < 256) dbp[tid] = 0.f;
    auto wait_mma = [&](int site) -> bool {
        bool w = mbar_wait(&bar_mma, mph, &abort_sh, a.status, site);
        mph ^= 1;
        w = !__syncthreads_or(!w);
        tc_fence_after();
        return w;
    };
    auto sync_for_mma = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    };
    auto mma = [&](uint32_t col, uint64_t ad, uint64_t bd, uint32_t id, bool acc) {
        mma_bf16(tm + col, ad, bd, id, acc ? 1u : 0u);
    };
    const uint32_t id64x128_kk = idesc_bf16(64, 128, 0, 0), id64x128_km = idesc_bf16(64, 128, 0, 1),
                   id64x128_mm = idesc_bf16(64, 128, 1, 1), id64x64_kk = idesc_bf16(64, 64, 0, 0),
                   id64x64_mm = idesc_bf16(64, 64, 1, 1);
    ok = mbar_wait(&bar_ld, 0, &abort_sh, a.status, 60);
    if (__syncthreads_or(!ok)) goto teardown;

    // ---------------------------------------------------------------- M1: W H0, dU
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kD; k0 += 16)
            mma(TM1, desc_kmajor(sb + C_W, 64, 0, k0), desc_mnmajor(sb + C_H0, 128, 0, k0), id64x128_km, k0 > 0);
        for (int k0 = 0; k0 < kChunk; k0 += 16)
            mma(TM2, desc_mnmajor(sb + C_P, 64, 0, k0), desc_mnmajor(sb + C_DO, 64, 0, k0), id64x128_mm, k0 > 0);
        for (int k0 = 0; k0 < kD; k0 += 16)
            mma(TM2, desc_kmajor(sb + C_KB, 64, 0, k0), desc_mnmajor(sb + C_DH, 128, 0, k0), id64x128_km, true);
        mma_commit(&bar_mma);
    }
    {  // <dH1, H0>_d per state row d over the two images (same layout): 4 threads per row
        const int d = tid >> 2, pp = tid & 3;
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            float x[8], y[8];
            unpack8c(ld_shared_v4(sb + C_H0 + sw128_chunk(d, 4 * pp + q, 128)), x);
            unpack8c(ld_shared_v4(sb + C_DH + sw128_chunk(d, 4 * pp + q, 128)), y);
#pragma unroll
            for (int e = 0; e < 8; e++) s += x[e] * y[e];
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (pp == 0) chx[CHX_HDH / 4 + d] = s;
    }
    uint4 utv[2];  // this lane's half of U~ slice qt (columns c32 + 16 hf ..)
#pragma unroll
    for (int q = 0; q < 2; q++)
        utv[q] = *reinterpret_cast<const uint4*>(rec + REC_U + qt * 4096 + sw64_chunk(r, 2 * hf + q));
    if (!wait_mma(61)) goto teardown;
    {  // U = U~ - W H0 -> U image (C_W);  dU -> dU image (C_KB)
        float x[32], w[16];
        const int q0 = 4 * qt + 2 * hf;
        tmem_ld32(tl + TM1 + c32, x);
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
#pragma unroll
        for (int q = 0; q < 2; q++) {
            float ut[8];
            unpack8c(utv[q], ut);
#pragma unroll
            for (int e = 0; e < 8; e++) ut[e] -= w[8 * q + e];
            st_chunk(sb + C_W + sw128_chunk(r, q0 + q, 64), ut, 1.f);
        }
        tmem_ld32(tl + TM2 + c32, x);
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
#pragma unroll
        for (int q = 0; q < 2; q++) st_chunk(sb + C_KB + sw128_chunk(r, q0 + q, 64), w + 8 * q, 1.f);
    }
    sync_for_mma();

    // ---------------------------------------------------------------- M2: dP = dO U^T, X = dO H0^T
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kD; k0 += 16) {
            mma(TM2, desc_kmajor(sb + C_DO, 64, 0, k0), desc_kmajor(sb + C_W, 64, 0, k0), id64x64_kk, k0 > 0);
            mma(TM1, desc_kmajor(sb + C_DO, 64, 0, k0), desc_kmajor(sb + C_H0, 128, 0, k0), id64x128_kk, k0 > 0);
        }
        mma_commit(&bar_mma);
    }
    if (!wait_mma(62)) goto teardown;
    {
        float x[32], w[16];
        tmem_ld32(tl + TM1 + c32, x);
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
        st_f4x(chx + CHX_X / 4 + r * kD + c32 + 16 * hf, w, 4);
        float v[16], u[8];
        tmem_ld16(tl + TM2 + c16, v);
        tmem_wait_ld();
        split_cols<16>(v, u, lane);
        const int j0 = c16 + 8 * hf;
#pragma unroll
        for (int e = 0; e < 8; e++) u[e] = (j0 + e <= r) ? P.scale * u[e] : 0.f;
        st_f4x(chx + CHX_DP / 4 + r * kChunk + j0, u, 2);
    }
    sync_for_mma();

    // ---------------------------------------------------------------- M3: Y = U dH1^T, dWn = dU H0^T
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kD; k0 += 16) {
            mma(TM1, desc_kmajor(sb + C_W, 64, 0, k0), desc_kmajor(sb + C_DH, 128, 0, k0), id64x128_kk, k0 > 0);
            mma(TM2, desc_kmajor(sb + C_KB, 64, 0, k0), desc_kmajor(sb + C_H0, 128, 0, k0), id64x128_kk, k0 > 0);
        }
        mma_commit(&bar_mma);
    }
    if (!wait_mma(63)) goto teardown;
    {
        float x[32], w[16];
        tmem_ld32(tl + TM1 + c32, x);
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
        st_f4x(chx + CHX_Y / 4 + r * kD + c32 + 16 * hf, w, 4);
        tmem_ld32(tl + TM2 + c32, x);  // dW = -dWn -> dW image (over H0, which is no longer read)
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
#pragma unroll
        for (int q = 0; q < 2; q++) st_chunk(sb + C_H0 + sw128_chunk(r, 4 * qt + 2 * hf + q, 64), w + 8 * q, -1.f);
    }
    sync_for_mma();

    // ---------------------------------------------------------------- M4: dU V^T, dW (K^ .* Gamma)^T, T^T dU
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kD; k0 += 16) {
            mma(TM1, desc_kmajor(sb + C_KB, 64, 0, k0), desc_kmajor(sb + C_V, 64, 0, k0), id64x64_kk, k0 > 0);
            mma(TM1 + 64, desc_kmajor(sb + C_H0, 64, 0, k0), desc_kmajor(sb + C_KG, 64, 0, k0), id64x64_kk, k0 > 0);
        }
        for (int k0 = 0; k0 < kChunk; k0 += 16)
            mma(TM2, desc_mnmajor(sb + C_T, 64, 0, k0), desc_mnmajor(sb + C_KB, 64, 0, k0), id64x128_mm, k0 > 0);
        mma_commit(&bar_mma);
    }
    if (!wait_mma(64)) goto teardown;
    {
        {  // dT_rj = beta_j (dU V^T + dW (K^ .* Gamma)^T)_rj -> dT image (C_DH)
            float d1[16], d2[16], w1[8], w2[8];
            tmem_ld16(tl + TM1 + c16, d1);
            tmem_ld16(tl + TM1 + 64 + c16, d2);
            tmem_wait_ld();
            split_cols<16>(d1, w1, lane);
            split_cols<16>(d2, w2, lane);
            const int jc = 2 * qt + hf;
#pragma unroll
            for (int e = 0; e < 8; e++) w1[e] = bet[8 * jc + e] * (w1[e] + w2[e]);
            st_chunk(sb + C_DH + sw128_chunk(r, jc, 64), w1, 1.f);
        }
        {  // T^T dU: dv = beta T^T dU;  V . (T^T dU) per row
            float x[32], w[16];
            tmem_ld32(tl + TM2 + c32, x);
            tmem_wait_ld();
            split_cols<32>(x, w, lane);
            float dot = 0.f;
#pragma unroll
            for (int q = 0; q < 2; q++) {
                float vv[8];
                unpack8c(ld_shared_v4(sb + C_V + sw128_chunk(r, 4 * qt + 2 * hf + q, 64)), vv);
#pragma unroll
                for (int e = 0; e < 8; e++) dot += vv[e] * w[8 * q + e];
            }
            dot += __shfl_xor_sync(0xffffffffu, dot, 16);
            if (act) dbp[qt * 64 + r] = dot;
            if (t0 + r < P.T) {
                const float bb = bet[r];
#pragma unroll
                for (int e = 0; e < 16; e++) w[e] *= bb;
                st_f4x(a.dv + (((size_t)b * P.T + t0 + r) * P.Hv + hv) * kD + c32 + 16 * hf, w, 4);
            }
        }
    }
    sync_for_mma();

    // ---------------------------------------------------------------- M5: Z = T^T dW, Yt = dT T^T
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kChunk; k0 += 16) {
            mma(TM2, desc_mnmajor(sb + C_T, 64, 0, k0), desc_mnmajor(sb + C_H0, 64, 0, k0), id64x128_mm, k0 > 0);
            mma(TM1, desc_kmajor(sb + C_DH, 64, 0, k0), desc_kmajor(sb + C_T, 64, 0, k0), id64x64_kk, k0 > 0);
        }
        mma_commit(&bar_mma);
    }
    if (!wait_mma(65)) goto teardown;
    {
        float x[32], w[16];
        tmem_ld32(tl + TM2 + c32, x);
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
        st_f4x(chx + CHX_Z / 4 + r * kD + c32 + 16 * hf, w, 4);
        float v[16], u[8];
        tmem_ld16(tl + TM1 + c16, v);
        tmem_wait_ld();
        split_cols<16>(v, u, lane);
        st_chunk(sb + C_DH + 8192 + sw128_chunk(r, 2 * qt + hf, 64), u, 1.f);
    }
    sync_for_mma();

    // ---------------------------------------------------------------- M6: T^T Yt -> dA
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kChunk; k0 += 16)
            mma(TM1, desc_mnmajor(sb + C_T, 64, 0, k0), desc_mnmajor(sb + C_DH + 8192, 64, 0, k0), id64x64_mm,
                k0 > 0);
        mma_commit(&bar_mma);
    }
    if (!wait_mma(66)) goto teardown;
    {
        float v[16], u[8];
        tmem_ld16(tl + TM1 + c16, v);
        tmem_wait_ld();
        split_cols<16>(v, u, lane);
        const int j0 = c16 + 8 * hf;
#pragma unroll
        for (int e = 0; e < 8; e++) u[e] = (j0 + e < r) ? -u[e] : 0.f;
        st_f4x(chx + CHX_DA / 4 + r * kChunk + j0, u, 2);
        if (tid < 64) chx[CHX_DB / 4 + tid] = dbp[tid] + dbp[64 + tid] + dbp[128 + tid] + dbp[192 + tid];
    }
teardown:
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0) {  // let copies still in flight land before the CTA exits
        volatile int never = 0;
        mbar_wait(&bar_ld, 0, &never, nullptr, 0);
        mbar_wait(&bar_mma, mph, &never, nullptr, 0);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// ---------------------------------------------------------------- CUDA-core pass
// shared memory (fp32): k^, q^, a_t, gamma [64][128]; dPs, dA row-major [64][64] and
// transposed [64][LDT]
constexpr int LDT = 68;
constexpr uint32_t S_KH = 0, S_QH = 32768, S_AL = 65536, S_GM = 98304;
constexpr uint32_t S_DPR = 131072, S_DAR = 147456, S_DPT = 163840, S_DAT = S_DPT + 64 * LDT * 4;
constexpr uint32_t S_SM = S_DAT + 64 * LDT * 4;  // bet[64], rk[64], rq[64], gcs[4][128], bt[4][128], dbr[4][64]
constexpr uint32_t S_BYTES = S_SM + (3 * 64 + 2 * 512 + 256) * 4;
static_assert(S_BYTES <= 232448, "grad_ch_simt smem");

__global__ void __launch_bounds__(CH_THREADS, 1) grad_ch_simt_kernel(GradChArgs a) {
    extern __shared__ __align__(16) uint8_t smem_s[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkProblem& P = a.p;
    const int c = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const int G = P.Hv / P.Hk, hk = hv / G;
    const int t0 = c * kChunk;
    const size_t idx = ((size_t)b * P.Hv + hv) * P.NC + c;
    const float* chx = reinterpret_cast<const float*>(a.chx + idx * CHX_BYTES);
    float* KH = reinterpret_cast<float*>(smem_s + S_KH);
    float* QH = reinterpret_cast<float*>(smem_s + S_QH);
    float* AL = reinterpret_cast<float*>(smem_s + S_AL);
    float* GM = reinterpret_cast<float*>(smem_s + S_GM);
    float* DPR = reinterpret_cast<float*>(smem_s + S_DPR);
    float* DAR = reinterpret_cast<float*>(smem_s + S_DAR);
    float* DPT = reinterpret_cast<float*>(smem_s + S_DPT);
    float* DAT = reinterpret_cast<float*>(smem_s + S_DAT);
    float* bet = reinterpret_cast<float*>(smem_s + S_SM);
    float* rk = bet + 64;
    float* rq = rk + 64;
    float* gcs = rq + 64;   // [4][128] sum_r b k^ Y by row block
    float* btot = gcs + 512; // [4][128] dgamma sums by row block
    float* dbr = btot + 512; // [4][64] dbeta partials by channel group
    const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);

    // raw k, q (zero past T), g (0 past T: a = 1, beta = 0), dPs and dA: every global load of
    // the thread is issued before the first shared-memory store
    {
        uint4 kr[2], qr[2];
        float4 gr[4], dp[2], da[2];
#pragma unroll
        for (int n = 0; n < 2; n++) {
            const int u = tid + CH_THREADS * n, rr = u >> 4, t = t0 + rr;
            const size_t xi = (((size_t)b * P.T + t) * P.Hk + hk) * kD + 8 * (u & 15);
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            kr[n] = t < P.T ? *reinterpret_cast<const uint4*>(kg + xi) : z;
            qr[n] = t < P.T ? *reinterpret_cast<const uint4*>(qg + xi) : z;
            dp[n] = reinterpret_cast<const float4*>(chx + CHX_DP / 4)[u];
            da[n] = reinterpret_cast<const float4*>(chx + CHX_DA / 4)[u];
        }
#pragma unroll
        for (int n = 0; n < 4; n++) {
            const int u = tid + CH_THREADS * n, rr = u >> 5, t = t0 + rr;
            gr[n] = t < P.T ? *reinterpret_cast<const float4*>(a.g + (((size_t)b * P.T + t) * P.Hv + hv) * kD +
                                                                4 * (u & 31))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float bv = (tid < 64 && t0 + tid < P.T) ? a.beta[((size_t)b * P.T + t0 + tid) * P.Hv + hv] : 0.f;
#pragma unroll
        for (int n = 0; n < 2; n++) {
            const int u = tid + CH_THREADS * n;
            float x[8];
            unpack8c(kr[n], x);
#pragma unroll
            for (int e = 0; e < 8; e++) KH[8 * u + e] = x[e];
            unpack8c(qr[n], x);
#pragma unroll
            for (int e = 0; e < 8; e++) QH[8 * u + e] = x[e];
            const int rr = u >> 4, j0 = 4 * (u & 15);
            reinterpret_cast<float4*>(DPR)[u] = dp[n];
            reinterpret_cast<float4*>(DAR)[u] = da[n];
            const float pv[4] = {dp[n].x, dp[n].y, dp[n].z, dp[n].w}, av[4] = {da[n].x, da[n].y, da[n].z, da[n].w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                DPT[(j0 + e) * LDT + rr] = pv[e];
                DAT[(j0 + e) * LDT + rr] = av[e];
            }
        }
#pragma unroll
        for (int n = 0; n < 4; n++) {
            const int u = tid + CH_THREADS * n;
            reinterpret_cast<float4*>(GM)[u] = gr[n];
            reinterpret_cast<float4*>(AL)[u] =
                make_float4(__expf(gr[n].x), __expf(gr[n].y), __expf(gr[n].z), __expf(gr[n].w));
        }
        if (tid < 64) bet[tid] = bv;
    }
    __syncthreads();
    {  // L2 norm factors: warp w takes rows 4w .. 4w + 3 of k and of q
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int rr = 4 * warp + i;
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int m = 0; m < 4; m++) {
                const float kv = KH[rr * kD + lane + 32 * m], qv = QH[rr * kD + lane + 32 * m];
                sk += kv * kv;
                sq += qv * qv;
            }
            sk = warp_sum(sk);
            sq = warp_sum(sq);
            if (lane == 0) {
                rk[rr] = P.use_norm ? 1.0f / sqrtf(sk + 1e-6f) : 1.0f;
                rq[rr] = P.use_norm ? 1.0f / sqrtf(sq + 1e-6f) : 1.0f;
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < kChunk * kD; i += CH_THREADS) {
        KH[i] *= rk[i >> 7];
        QH[i] *= rq[i >> 7];
    }
    if (tid < kD) {  // gamma_r,d: in-chunk cumulative log-decay of channel d = tid
        float s = 0.f;
        for (int rr = 0; rr < kChunk; rr++) {
            s += GM[rr * kD + tid];
            GM[rr * kD + tid] = s;
        }
    }
    __syncthreads();

    // thread <-> channel d (lanes: consecutive channels) and rows r0 .. r0 + 15
    const int d = 32 * (warp & 3) + lane, rb = warp >> 2, r0 = 16 * rb;
    const float gC = GM[(kChunk - 1) * kD + d];
    float dk[16], dgm[16];
    float gsum = 0.f;
    // row side: sum_j dPs_rj k^_j E_rj and sum_j dA_rj k^_j E_rj, j descending from the row; then
    // the terms of X, Y, Z of the same rows. dq^ and the dbeta partials are final here.
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const int ra = r0 + 8 * h;
        float xs[8], ys[8], zs[8];  // fetched now, used after the contraction
#pragma unroll
        for (int e = 0; e < 8; e++) {
            xs[e] = chx[CHX_X / 4 + (ra + e) * kD + d];
            ys[e] = chx[CHX_Y / 4 + (ra + e) * kD + d];
            zs[e] = chx[CHX_Z / 4 + (ra + e) * kD + d];
        }
        float E[8], X1[8], Y1[8];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            E[e] = 1.f;
            X1[e] = 0.f;
            Y1[e] = 0.f;
        }
        // the diagonal block (j = ra+7 .. ra) with per-row running products E_rj
        for (int j = ra + 7; j >= ra; j--) {
            const float kj = KH[j * kD + d];
            const float an = j + 1 < kChunk ? AL[(j + 1) * kD + d] : 1.f;
#pragma unroll
            for (int e = 0; e < 8; e++) {
                E[e] = (j < ra + e) ? E[e] * an : 1.f;
                const float w = kj * E[e];
                X1[e] += DPT[j * LDT + ra + e] * w;
                Y1[e] += DAT[j * LDT + ra + e] * w;
            }
        }
        // j < ra: E_rj = E_r,ra * F_j with F_j = prod_{j<t<=ra} a_t shared by the 8 rows, so
        // the rows accumulate sum_j M_rj k^_j F_j and take their own factor E_r,ra at the end
        {
            float X1f[8], Y1f[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                X1f[e] = 0.f;
                Y1f[e] = 0.f;
            }
            float F = 1.f;
            for (int j = ra - 1; j >= 0; j--) {
                F *= AL[(j + 1) * kD + d];
                const float w = KH[j * kD + d] * F;
                const float4 p0 = *reinterpret_cast<const float4*>(DPT + j * LDT + ra);
                const float4 p1 = *reinterpret_cast<const float4*>(DPT + j * LDT + ra + 4);
                const float4 a0 = *reinterpret_cast<const float4*>(DAT + j * LDT + ra);
                const float4 a1 = *reinterpret_cast<const float4*>(DAT + j * LDT + ra + 4);
                const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    X1f[e] += pv[e] * w;
                    Y1f[e] += av[e] * w;
                }
            }
#pragma unroll
            for (int e = 0; e < 8; e++) {
                X1[e] += E[e] * X1f[e];
                Y1[e] += E[e] * Y1f[e];
            }
        }
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int i = 8 * h + e, rr = ra + e;
            const float gm = GM[rr * kD + d];
            const float Gm = __expf(gm), bb = __expf(gC - gm);
            const float x = xs[e], y = ys[e], z = zs[e];
            const float kh = KH[rr * kD + d], qh = QH[rr * kD + d], br = bet[rr];
            const float dqv = P.scale * Gm * x + X1[e];
            dk[i] = bb * y + br * Gm * z + br * Y1[e];
            dgm[i] = P.scale * Gm * qh * x - bb * kh * y + br * Gm * kh * z + qh * X1[e] + br * kh * Y1[e];
            gsum += bb * kh * y;
            const float dbs = warp_sum(Gm * kh * z + kh * Y1[e]);
            if (lane == 0) dbr[(warp & 3) * 64 + rr] = dbs;
            if (t0 + rr < P.T) a.dqh[(((size_t)b * P.T + t0 + rr) * P.Hv + hv) * kD + d] = dqv;
        }
    }
    // column side: sum_i dPs_ij q^_i E_ij + sum_i dA_ij beta_i k^_i E_ij, i ascending from the row
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const int ja = r0 + 8 * h;
        float E[8], X2[8];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            E[e] = 1.f;
            X2[e] = 0.f;
        }
        // the diagonal block (i = ja .. ja+7) with per-column running products E_ij
        for (int i = ja; i < ja + 8; i++) {
            const float ai = AL[i * kD + d], qi = QH[i * kD + d], kbi = bet[i] * KH[i * kD + d];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                E[e] = (i > ja + e) ? E[e] * ai : 1.f;
                X2[e] += (DPR[i * kChunk + ja + e] * qi + DAR[i * kChunk + ja + e] * kbi) * E[e];
            }
        }
        // i > ja+7: E_ij = E_ja+7,j * F_i with F_i = prod_{ja+7<t<=i} a_t shared by the 8 columns
        {
            float X2f[8];
#pragma unroll
            for (int e = 0; e < 8; e++) X2f[e] = 0.f;
            float F = 1.f;
            for (int i = ja + 8; i < kChunk; i++) {
                F *= AL[i * kD + d];
                const float wq = QH[i * kD + d] * F, wk = bet[i] * KH[i * kD + d] * F;
                const float4 p0 = *reinterpret_cast<const float4*>(DPR + i * kChunk + ja);
                const float4 p1 = *reinterpret_cast<const float4*>(DPR + i * kChunk + ja + 4);
                const float4 a0 = *reinterpret_cast<const float4*>(DAR + i * kChunk + ja);
                const float4 a1 = *reinterpret_cast<const float4*>(DAR + i * kChunk + ja + 4);
                const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int e = 0; e < 8; e++) X2f[e] += pv[e] * wq + av[e] * wk;
            }
#pragma unroll
            for (int e = 0; e < 8; e++) X2[e] += E[e] * X2f[e];
        }
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const int i = 8 * h + e, jj = ja + e;
            dk[i] += X2[e];
            dgm[i] -= KH[jj * kD + d] * X2[e];
        }
    }
    // dgamma_C,d, block sums of dgamma, dbeta partials
    float suf[16];
    {
        float s = 0.f;
#pragma unroll
        for (int i = 15; i >= 0; i--) {
            s += dgm[i];
            suf[i] = s;
        }
        gcs[rb * kD + d] = gsum;
        btot[rb * kD + d] = s;
    }
    __syncthreads();
    {
        const float dgC = gcs[d] + gcs[kD + d] + gcs[2 * kD + d] + gcs[3 * kD + d] +
                          __expf(gC) * chx[CHX_HDH / 4 + d];
        float off = dgC;
        for (int k = rb + 1; k < 4; k++) off += btot[k * kD + d];
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const int t = t0 + r0 + i;
            if (t < P.T) {
                const size_t o = (((size_t)b * P.T + t) * P.Hv + hv) * kD + d;
                a.dg[o] = suf[i] + off;
                a.dkh[o] = dk[i];
            }
        }
    }
    if (tid < 64 && t0 + tid < P.T)
        a.dbeta[((size_t)b * P.T + t0 + tid) * P.Hv + hv] =
            chx[CHX_DB / 4 + tid] + dbr[tid] + dbr[64 + tid] + dbr[128 + tid] + dbr[192 + tid];
}

}  // namespace

cudaError_t launch_grad_ch(const GradChArgs& a, const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s) {
    const int smem1 = C_BYTES + 1024;
    cudaError_t e = cudaFuncSetAttribute(grad_ch_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(grad_ch_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(a.p.NC, a.p.Hv, a.p.B);
    trace_begin("chunk_grad_channel_mma", s);
    grad_ch_mma_kernel<<<grid, CH_THREADS, smem1, s>>>(mv, mdo, a);
    trace_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_begin("chunk_grad_channel_simt", s);
    grad_ch_simt_kernel<<<grid, CH_THREADS, S_BYTES, s>>>(a);
    trace_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // dq^, dk^ summed over the value heads of each key head, then the norm backward
    SeqBwdArgs f{};
    f.B = a.p.B; f.T = a.p.T; f.Hk = a.p.Hk; f.Hv = a.p.Hv; f.Dk = kD; f.Dv = kD;
    f.channel = 1;
    f.use_norm = a.p.use_norm;
    f.bf16 = 1;
    f.q = a.q; f.k = a.k;
    f.dq = a.dq; f.dk = a.dk;
    f.dqh = a.dqh; f.dkh = a.dkh;
    return launch_qk_norm_backward(f, s);
}

}  // namespace gdr
