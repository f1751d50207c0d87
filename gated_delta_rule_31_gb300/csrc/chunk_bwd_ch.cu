// chunk_bwd_ch.cu - backward (VJP) of the chunked gated delta rule with a per-channel gate
// (one decay per key channel, g [B,T,Hv,Dk]): the channelwise variant of "Two-pass
// optimization for channelwise gated delta rule kernel" (ExecuTorch PR #21020) in the chunked
// reverse mode of "Adding VJP for gated delta net" (MLX PR #4565, chunked case).
//
// Launch sequence: prep_ch (also keeps T and W per chunk) -> forward states scan
// -> reverse scan (chunk-end state gradients, dh0) -> grad_ch_mma -> grad_ch_contract -> the
// value-head sum with the norm backward.
//
// Per (b, hv, chunk), with E_rj,d = prod_{j<t<=r} a_t,d, Gamma_r,d = prod_{t<=r} a_t,d,
// b_r,d = Gamma_C,d / Gamma_r,d and the chunk algebra of chunk_fwd_ch.cu:
//   U  = U~ - W H0        dU = P^T dO + Kbar dH1          dW = -dU H0^T
//   X  = dO H0^T          Y  = U dH1^T                     Z  = T^T dW
//   dPs = scale tril(dO U^T)        dT = dU (diag(beta) V)^T + dW (diag(beta) K^ .* Gamma)^T
//   dA = -strict_lower(T^T dT T^T)  dv = diag(beta) T^T dU
// Since U~ = T diag(beta) V and W = T diag(beta) (K^ .* Gamma), T^T dT T^T equals
// (T^T dU) U~^T + (T^T dW) W^T: dA comes from T^T dU and Z = T^T dW, which are needed anyway,
// and the kept U~ and W, so dT is never formed.
// (the dense products, on tcgen05: grad_ch_mma). Then per element (r, d) (grad_ch_contract):
//   dq^ = scale Gamma X + sum_{j<=r} dPs_rj k^_j E_rj
//   dk^ = b Y + beta Gamma Z + beta_r sum_{j<r} dA_rj k^_j E_rj
//         + sum_{i>=r} dPs_ir q^_i E_ir + sum_{i>r} dA_ir beta_i k^_i E_ir
//   dgamma_r = every term above times its own factor of Gamma_r (+1), b_r (-1) or E (+1 on
//   the row side, -1 on the column side); dgamma_C = sum_r b k^ Y + Gamma_C <dH1, H0>_d;
//   dg = reverse cumulative sum of dgamma in the chunk (+ dgamma_C on every token);
//   dbeta = V . (T^T dU) + sum_d Gamma k^ Z + sum_d k^ (sum_{j<r} dA_rj k^_j E_rj).
// The decay-weighted contractions run by 16-row blocks: below the block diagonal as tcgen05
// products of operands scaled by products of per-token factors a_t <= 1, inside the diagonal
// blocks on the CUDA cores with running products; no decay can overflow however strong.
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
constexpr uint32_t C_DO = 0;        // dO [64 x 128] (TMA, panels 8 KB); then U~ (4 SW64 slices)
constexpr uint32_t C_W = 16384;     // W image [64 x 128]
constexpr uint32_t C_KB = 32768;    // Kbar image; then dU image; then T^T dU image
constexpr uint32_t C_H0 = 49152;    // H0 image [128 d x 128 v]; then dW, then T^T dW images [64 x 128]
constexpr uint32_t C_DH = 81920;    // dH1 image [128 d x 128 v]
constexpr uint32_t C_V = 114688;    // v [64 x 128] (TMA)
constexpr uint32_t C_U = 131072;    // U image [64 x 128]
constexpr uint32_t C_P = 147456;    // P image [64 x 64]
constexpr uint32_t C_T = 155648;    // T image [64 x 64]
constexpr uint32_t C_SM = 163840;   // bet[64], dbp[4][64]
constexpr uint32_t C_STG = C_SM + 2048;  // per warp 4 rows x 36 fp32: staging of the fp32 row stores
constexpr uint32_t C_BYTES = C_STG + 16 * 4 * 36 * 4;
constexpr uint32_t TM1 = 0, TM2 = 128;  // TMEM columns of the two accumulators
constexpr int CH_THREADS = 512;

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
    const uint8_t* rec2 = a.rec2 + idx * REC2_BYTES;
    float* chx = reinterpret_cast<float*>(a.chx + idx * CHX_BYTES);
    const int lg = warp & 3, qt = warp >> 2, hf = lane >> 4;
    const int r = 16 * lg + (lane & 15);
    const bool act = lane < 16;
    const int c32 = 32 * qt, c16 = 16 * qt;
    float* bet = reinterpret_cast<float*>(sm + C_SM);
    float* dbp = bet + 64;  // [4][64] V . (T^T dU) partials by column quarter
    float* stg = reinterpret_cast<float*>(sm + C_STG) + warp * 144;  // this warp's row-store staging
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
        mbar_expect_tx(&bar_ld, 147456);
        tma_load_4d(sm + C_DO + 0, &mdo, 0, hv, t0, b, &bar_ld);
        tma_load_4d(sm + C_DO + 8192, &mdo, 64, hv, t0, b, &bar_ld);
        tma_load_4d(sm + C_V + 0, &mv, 0, hv, t0, b, &bar_ld);
        tma_load_4d(sm + C_V + 8192, &mv, 64, hv, t0, b, &bar_ld);
        bulk_load(sm + C_W, rec2 + REC2_W, 16384, &bar_ld);
        bulk_load(sm + C_KB, rec + REC_K, 16384, &bar_ld);
        bulk_load(sm + C_H0, a.hs + idx * STATE_IMG, 32768, &bar_ld);
        bulk_load(sm + C_DH, a.dhs + idx * STATE_IMG, 32768, &bar_ld);
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
    // fp32 rows of a [64 x 128] result tile to global memory: this warp holds rows 16 lg .. + 15 of
    // column quarter qt, lane l (l & 15: the row) columns c32 + 16 (l >> 4) .. + 15. Four rows at
    // a time go through the warp's staging so that each store instruction writes four whole 128-byte
    // row segments (8 lanes each) instead of 64 bytes in each of 16 rows. The stores are issued after
    // the next products, because the proxy fence before those would otherwise wait for them.
    // g0: row 0 at column c32; rs: floats per row; rows at or past `rows` are not written.
    auto store_rows = [&](float* g0, size_t rs, const float* v, int rows) {
        const int rl = lane & 15, m = lane >> 3, cg = lane & 7;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            if ((rl >> 2) == i) {
#pragma unroll
                for (int q = 0; q < 4; q++)
                    *reinterpret_cast<float4*>(stg + (rl & 3) * 36 + 16 * hf + 4 * q) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
            __syncwarp();
            const int row = 16 * lg + 4 * i + m;
            const float4 x = *reinterpret_cast<const float4*>(stg + m * 36 + 4 * cg);
            if (row < rows) *reinterpret_cast<float4*>(g0 + (size_t)row * rs + 4 * cg) = x;
            __syncwarp();
        }
    };
    const uint32_t id64x128_kk = idesc_bf16(64, 128, 0, 0), id64x128_km = idesc_bf16(64, 128, 0, 1),
                   id64x128_mm = idesc_bf16(64, 128, 1, 1), id64x64_kk = idesc_bf16(64, 64, 0, 0);
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
            unpack8(ld_shared_v4(sb + C_H0 + sw128_chunk(d, 4 * pp + q, 128)), x);
            unpack8(ld_shared_v4(sb + C_DH + sw128_chunk(d, 4 * pp + q, 128)), y);
#pragma unroll
            for (int e = 0; e < 8; e++) s += x[e] * y[e];
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        if (pp == 0) chx[CHX_HDH / 4 + d] = s;
    }
    uint4 utv[2];  // this lane's half of U~ slice qt (columns c32 + 16 hf ..), kept for its image
#pragma unroll
    for (int q = 0; q < 2; q++)
        utv[q] = *reinterpret_cast<const uint4*>(rec + REC_U + qt * 4096 + sw64_chunk(r, 2 * hf + q));
    if (!wait_mma(61)) goto teardown;
    {  // U = U~ - W H0 -> U image (C_U);  dU -> dU image (C_KB)
        float x[32], w[16];
        const int q0 = 4 * qt + 2 * hf;
        tmem_ld32(tl + TM1 + c32, x);
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
#pragma unroll
        for (int q = 0; q < 2; q++) {
            float ut[8];
            unpack8(utv[q], ut);
#pragma unroll
            for (int e = 0; e < 8; e++) ut[e] -= w[8 * q + e];
            st_chunk(sb + C_U + sw128_chunk(r, q0 + q, 64), ut, 1.f);
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
            mma(TM2, desc_kmajor(sb + C_DO, 64, 0, k0), desc_kmajor(sb + C_U, 64, 0, k0), id64x64_kk, k0 > 0);
            mma(TM1, desc_kmajor(sb + C_DO, 64, 0, k0), desc_kmajor(sb + C_H0, 128, 0, k0), id64x128_kk, k0 > 0);
        }
        mma_commit(&bar_mma);
    }
    if (!wait_mma(62)) goto teardown;
    float wx[16], up[8];  // X and dPs, exported once M3 is issued
    {
#pragma unroll
        for (int q = 0; q < 2; q++)  // U~ slice images over dO, which M2 was the last to read
            *reinterpret_cast<uint4*>(sm + C_DO + qt * 4096 + sw64_chunk(r, 2 * hf + q)) = utv[q];
        float x[32];
        tmem_ld32(tl + TM1 + c32, x);
        tmem_wait_ld();
        split_cols<32>(x, wx, lane);
        float v[16];
        tmem_ld16(tl + TM2 + c16, v);
        tmem_wait_ld();
        split_cols<16>(v, up, lane);
        const int j0 = c16 + 8 * hf;
#pragma unroll
        for (int e = 0; e < 8; e++) up[e] = (j0 + e <= r) ? P.scale * up[e] : 0.f;
    }
    sync_for_mma();

    // ---------------------------------------------------------------- M3: Y = U dH1^T, dWn = dU H0^T
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kD; k0 += 16) {
            mma(TM1, desc_kmajor(sb + C_U, 64, 0, k0), desc_kmajor(sb + C_DH, 128, 0, k0), id64x128_kk, k0 > 0);
            mma(TM2, desc_kmajor(sb + C_KB, 64, 0, k0), desc_kmajor(sb + C_H0, 128, 0, k0), id64x128_kk, k0 > 0);
        }
        mma_commit(&bar_mma);
    }
    store_rows(chx + CHX_X / 4 + c32, kD, wx, kChunk);
    st_f4x(chx + CHX_DP / 4 + r * kChunk + c16 + 8 * hf, up, 2);
    if (!wait_mma(63)) goto teardown;
    float wy[16];  // Y, exported once M4 is issued
    {
        float x[32], w[16];
        tmem_ld32(tl + TM1 + c32, x);
        tmem_wait_ld();
        split_cols<32>(x, wy, lane);
        tmem_ld32(tl + TM2 + c32, x);  // dW = -dWn -> dW image (over H0, which is no longer read)
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
#pragma unroll
        for (int q = 0; q < 2; q++) st_chunk(sb + C_H0 + sw128_chunk(r, 4 * qt + 2 * hf + q, 64), w + 8 * q, -1.f);
    }
    sync_for_mma();

    // ---------------------------------------------------------------- M4: T^T dU, Z = T^T dW
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kChunk; k0 += 16) {
            mma(TM2, desc_mnmajor(sb + C_T, 64, 0, k0), desc_mnmajor(sb + C_KB, 64, 0, k0), id64x128_mm, k0 > 0);
            mma(TM1, desc_mnmajor(sb + C_T, 64, 0, k0), desc_mnmajor(sb + C_H0, 64, 0, k0), id64x128_mm, k0 > 0);
        }
        mma_commit(&bar_mma);
    }
    store_rows(chx + CHX_Y / 4 + c32, kD, wy, kChunk);
    if (!wait_mma(64)) goto teardown;
    float wv[16], wz[16];  // dv and Z, stored once M5 is issued
    {
        const int q0 = 4 * qt + 2 * hf;
        float x[32], w[16];
        tmem_ld32(tl + TM2 + c32, x);  // T^T dU: dv = beta T^T dU;  V . (T^T dU) per row; its image
        tmem_wait_ld();
        split_cols<32>(x, w, lane);
        float dot = 0.f;
#pragma unroll
        for (int q = 0; q < 2; q++) {
            float vv[8];
            unpack8(ld_shared_v4(sb + C_V + sw128_chunk(r, q0 + q, 64)), vv);
#pragma unroll
            for (int e = 0; e < 8; e++) dot += vv[e] * w[8 * q + e];
            st_chunk(sb + C_KB + sw128_chunk(r, q0 + q, 64), w + 8 * q, 1.f);
        }
        dot += __shfl_xor_sync(0xffffffffu, dot, 16);
        if (act) dbp[qt * 64 + r] = dot;
        const float bb = bet[r];
#pragma unroll
        for (int e = 0; e < 16; e++) wv[e] = bb * w[e];
        tmem_ld32(tl + TM1 + c32, x);  // Z and its image
        tmem_wait_ld();
        split_cols<32>(x, wz, lane);
#pragma unroll
        for (int q = 0; q < 2; q++) st_chunk(sb + C_H0 + sw128_chunk(r, q0 + q, 64), wz + 8 * q, 1.f);
    }
    sync_for_mma();

    // ---------------------------------------------------------------- M5: (T^T dU) U~^T + Z W^T -> dA
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kD; k0 += 16)
            mma(TM1, desc_kmajor(sb + C_KB, 64, 0, k0), desc_kmajor_sw64(sb + C_DO, 64, k0), id64x64_kk, k0 > 0);
        for (int k0 = 0; k0 < kD; k0 += 16)
            mma(TM1, desc_kmajor(sb + C_H0, 64, 0, k0), desc_kmajor(sb + C_W, 64, 0, k0), id64x64_kk, true);
        mma_commit(&bar_mma);
    }
    store_rows(a.dv + (((size_t)b * P.T + t0) * P.Hv + hv) * kD + c32, (size_t)P.Hv * kD, wv, P.T - t0);
    store_rows(chx + CHX_Z / 4 + c32, kD, wz, kChunk);
    if (!wait_mma(65)) goto teardown;
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

// ---------------------------------------------------------------- contraction pass
// The decay-weighted contractions by 16-row blocks (block I = rows 16I .. 16I + 15). A pair
// (r, j) with j in an earlier block than r factors through s = 16I - 1 (I the block of r):
//   E_rj = [prod_{16I<=t<=r} a_t] [prod_{j<t<16I} a_t]
// and a pair (i, j) with i in a later block than j through s = 16J + 15 (J the block of j):
//   E_ij = [prod_{j<t<=16J+15} a_t] [prod_{16J+16<=t<=i} a_t]
// every factor a product of per-token factors <= 1, so the parts below the block diagonal are
// tcgen05 products of decay-scaled bf16 operands:
//   row side     D_I = [dPs; dA] R_I,   R_I[j] = k^_j prod_{j<t<16I} a_t          (j < 16I)
//   column side  C_J = [dPs^T | dA^T] [Q_J; K_J],  Q_J[i] = q^_i prod_{16J+16<=t<=i} a_t,
//                K_J[i] = beta_i k^_i prod_{16J+16<=t<=i} a_t                      (i >= 16J + 16)
// after which each row takes its own factor. Inside the diagonal blocks the running decay is
// formed on the CUDA cores. Shared memory: k^, q^, a_t fp32 [64][128]; dPs, dA fp32 [64][64];
// a 64 KB region for the operand images and then the fp32 products staged by row; small arrays.
constexpr uint32_t X_KH = 0, X_QH = 32768, X_AL = 65536, X_DPR = 98304, X_DAR = 114688;
constexpr uint32_t X_IMG = 131072;
constexpr uint32_t X_AR = X_IMG, X_R1 = X_IMG + 16384, X_R2 = X_IMG + 20480, X_R3 = X_IMG + 28672;
constexpr uint32_t X_AC = X_IMG, X_B0 = X_IMG + 16384, X_B1 = X_IMG + 40960, X_B2 = X_IMG + 57344;
constexpr uint32_t X_DT = X_IMG + 40960;  // row side: transposed diagonal blocks of dPs, dA (8 KB)
constexpr int LST = 132;  // fp32 row stride of the staged products (rows of 16 lanes hit distinct banks)
constexpr uint32_t X_SM = X_IMG + 65536;
constexpr uint32_t X_BYTES = X_SM + (3 * 64 + 2 * 512 + 256 + 512) * 4;
static_assert(X_R1 % 1024 == 0 && X_R2 % 1024 == 0 && X_R3 % 1024 == 0 && X_B0 % 1024 == 0 &&
                  X_B1 % 1024 == 0 && X_B2 % 1024 == 0, "operand images need 1024-byte alignment");
static_assert(X_R3 + 48 * 256 <= X_DT && X_DT + 8192 <= X_SM && X_B2 + 32 * 256 <= X_SM, "operand images");
static_assert(3 * 32 * LST * 4 <= 65536, "staged products");
static_assert(X_BYTES + 1024 <= 232448, "contraction pass smem");

__global__ void __launch_bounds__(CH_THREADS, 1) grad_ch_contract_kernel(GradChArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkProblem& P = a.p;
    const int c = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const int G = P.Hv / P.Hk, hk = hv / G;
    const int t0 = c * kChunk;
    const size_t idx = ((size_t)b * P.Hv + hv) * P.NC + c;
    const float* chx = reinterpret_cast<const float*>(a.chx + idx * CHX_BYTES);
    float* KH = reinterpret_cast<float*>(sm + X_KH);
    float* QH = reinterpret_cast<float*>(sm + X_QH);
    float* AL = reinterpret_cast<float*>(sm + X_AL);
    float* DPR = reinterpret_cast<float*>(sm + X_DPR);
    float* DAR = reinterpret_cast<float*>(sm + X_DAR);
    float* ST = reinterpret_cast<float*>(sm + X_IMG);  // staged products (after the images are read)
    float* bet = reinterpret_cast<float*>(sm + X_SM);
    float* rk = bet + 64;
    float* rq = rk + 64;
    float* gcs = rq + 64;     // [4][128] sum_r b k^ Y by row block
    float* btot = gcs + 512;  // [4][128] dgamma sums by row block
    float* dbr = btot + 512;  // [4][64] dbeta partials by channel group
    float* bpr = dbr + 256;   // [4][128] prod of a_t over each 16-row block
    const __nv_bfloat16* kg = static_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
    uint32_t mph = 0;
    bool mma_pend = false;  // thread 0: products committed and not yet waited for
    bool ok = true;
    float pre, post, gsum, Gm, gC;  // per-channel decay products of this thread's rows (set below)

    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_mma, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_sh, 512);
        tmem_relinquish();
    }
    // raw k, q (zero past T), a_t = exp(g) (g = 0 past T), dPs and dA; every global load of the
    // thread is issued before its first shared-memory store. The 16 lanes holding a row of k (q)
    // sum its squares by shuffles, so k^ and q^ are stored already normalised.
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
            float x[8], y[8];
            unpack8(kr[n], x);
            unpack8(qr[n], y);
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int e = 0; e < 8; e++) {
                sk += x[e] * x[e];
                sq += y[e] * y[e];
            }
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) {
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
            }
            const float fk = P.use_norm ? 1.0f / sqrtf(sk + 1e-6f) : 1.0f;
            const float fq = P.use_norm ? 1.0f / sqrtf(sq + 1e-6f) : 1.0f;
            if ((u & 15) == 0) {
                rk[u >> 4] = fk;
                rq[u >> 4] = fq;
            }
            reinterpret_cast<float4*>(KH)[2 * u] = make_float4(fk * x[0], fk * x[1], fk * x[2], fk * x[3]);
            reinterpret_cast<float4*>(KH)[2 * u + 1] = make_float4(fk * x[4], fk * x[5], fk * x[6], fk * x[7]);
            reinterpret_cast<float4*>(QH)[2 * u] = make_float4(fq * y[0], fq * y[1], fq * y[2], fq * y[3]);
            reinterpret_cast<float4*>(QH)[2 * u + 1] = make_float4(fq * y[4], fq * y[5], fq * y[6], fq * y[7]);
            reinterpret_cast<float4*>(DPR)[u] = dp[n];
            reinterpret_cast<float4*>(DAR)[u] = da[n];
        }
#pragma unroll
        for (int n = 0; n < 4; n++) {
            const int u = tid + CH_THREADS * n;
            reinterpret_cast<float4*>(AL)[u] =
                make_float4(__expf(gr[n].x), __expf(gr[n].y), __expf(gr[n].z), __expf(gr[n].w));
        }
        if (tid < 64) bet[tid] = bv;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_sh;
    {  // the diagonal 16 x 16 blocks of dPs and dA transposed (row j, column r), for the row side
        float* DT = reinterpret_cast<float*>(sm + X_DT);
        for (int u = tid; u < 4 * 16 * 16; u += CH_THREADS) {
            const int blk = u >> 8, jj = (u >> 4) & 15, rr = u & 15;
            const int src = (16 * blk + rr) * kChunk + 16 * blk + jj;
            DT[u] = DPR[src];
            DT[1024 + u] = DAR[src];
        }
        const int d2 = tid & 127, blk = tid >> 7;  // block products of the per-token factors
        float p = 1.f;
        for (int t = 16 * blk; t < 16 * blk + 16; t++) p *= AL[t * kD + d2];
        bpr[blk * kD + d2] = p;
    }

    // ------------------------------------------------ row side
    {  // [dPs; dA] as a bf16 [128 x 64] K-major image, 8 columns per task
        for (int u = tid; u < 128 * 8; u += CH_THREADS) {
            const int row = u >> 3, ch = u & 7;
            const float4* src = reinterpret_cast<const float4*>((row < 64 ? DPR + row * 64 : DAR + (row - 64) * 64) + 8 * ch);
            const float4 v0 = src[0], v1 = src[1];
            const float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            st_chunk(sb + X_AR + sw128_chunk(row, ch, 128), x, 1.f);
        }
        const int d2 = tid & 127, I = tid >> 7;  // R_I rows j = 16 I - 1 .. 0 of channel d2
        if (I >= 1) {  // 16 rows' inputs loaded before their stores
            const uint32_t rb = I == 1 ? X_R1 : I == 2 ? X_R2 : X_R3;
            float sfx = 1.f;
#pragma unroll 1
            for (int jb = 16 * I - 16; jb >= 0; jb -= 16) {
                float av[16], kv[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    av[i] = AL[(jb + i) * kD + d2];
                    kv[i] = KH[(jb + i) * kD + d2];
                }
#pragma unroll
                for (int i = 15; i >= 0; i--) {
                    *reinterpret_cast<__nv_bfloat16*>(sm + rb + sw128_off(jb + i, d2, 16 * I)) =
                        __float2bfloat16_rn(kv[i] * sfx);
                    sfx *= av[i];
                }
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // D_I (M=128: dPs rows, then dA rows; N=128 channels; K = 16 I) at columns 128 (I - 1)
        tc_fence_after();
        const uint32_t id = idesc_bf16(128, 128, 0, 1);
        for (int I = 1; I <= 3; I++) {
            const uint32_t rb = I == 1 ? X_R1 : I == 2 ? X_R2 : X_R3;
            for (int k0 = 0; k0 < 16 * I; k0 += 16)
                mma_bf16(tm + 128 * (I - 1), desc_kmajor(sb + X_AR, 128, 0, k0), desc_mnmajor(sb + rb, 16 * I, 0, k0),
                         id, k0 > 0 ? 1u : 0u);
        }
        mma_commit(&bar_mma);
        mma_pend = true;
    }
    // thread <-> channel d (lanes: consecutive channels) and rows r0 .. r0 + 15 (= block rb)
    const int d = 32 * (warp & 3) + lane, rb = warp >> 2, r0 = 16 * rb;
    float X1[16], Y1[16];  // sum_{j<=r} dPs_rj k^_j E_rj, sum_{j<r} dA_rj k^_j E_rj
#pragma unroll
    const float* DTp = reinterpret_cast<const float*>(sm + X_DT) + 256 * rb;  // [j - r0][r - r0]
    for (int h = 0; h < 2; h++) {  // inside the diagonal block, 8 rows at a time
        const int ra = r0 + 8 * h;
        float E[8];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            E[e] = 1.f;
            X1[8 * h + e] = 0.f;
            Y1[8 * h + e] = 0.f;
        }
        for (int j = ra + 7; j >= ra; j--) {
            const float kj = KH[j * kD + d];
            const float an = j + 1 < kChunk ? AL[(j + 1) * kD + d] : 1.f;
            const float* pr = DTp + (j - r0) * 16 + 8 * h;
            const float4 p0 = *reinterpret_cast<const float4*>(pr), p1 = *reinterpret_cast<const float4*>(pr + 4);
            const float4 a0 = *reinterpret_cast<const float4*>(pr + 1024);
            const float4 a1 = *reinterpret_cast<const float4*>(pr + 1028);
            const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int e = 0; e < 8; e++) {
                E[e] = (j < ra + e) ? E[e] * an : 1.f;
                const float w = kj * E[e];
                X1[8 * h + e] += pv[e] * w;
                Y1[8 * h + e] += av[e] * w;
            }
        }
        if (h == 1) {  // j = r0 + 7 .. r0: E_rj = E_r,ra * prod_{j<t<=ra} a_t, the second factor shared by the 8 rows
            float X1f[8], Y1f[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                X1f[e] = 0.f;
                Y1f[e] = 0.f;
            }
            float F = 1.f;
            for (int j = ra - 1; j >= r0; j--) {
                F *= AL[(j + 1) * kD + d];
                const float w = KH[j * kD + d] * F;
                const float* pr = DTp + (j - r0) * 16 + 8;
                const float4 p0 = *reinterpret_cast<const float4*>(pr), p1 = *reinterpret_cast<const float4*>(pr + 4);
                const float4 a0 = *reinterpret_cast<const float4*>(pr + 1024);
                const float4 a1 = *reinterpret_cast<const float4*>(pr + 1028);
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
                X1[8 + e] += E[e] * X1f[e];
                Y1[8 + e] += E[e] * Y1f[e];
            }
        }
    }
    float xs[4], ys[4], zs[4];  // X, Y, Z of the next 4 rows, fetched ahead
#pragma unroll
    for (int e = 0; e < 4; e++) {
        xs[e] = chx[CHX_X / 4 + (r0 + e) * kD + d];
        ys[e] = chx[CHX_Y / 4 + (r0 + e) * kD + d];
        zs[e] = chx[CHX_Z / 4 + (r0 + e) * kD + d];
    }
    ok = mbar_wait(&bar_mma, mph, &abort_sh, a.status, 70);
    mph ^= 1;
    if (__syncthreads_or(!ok)) goto teardown;
    if (tid == 0) mma_pend = false;
    tc_fence_after();
    {  // stage D_I rows of block I (dPs part, dA part) as fp32 [I - 1][2][16][LST]
        const int sub = warp & 3, q32 = warp >> 2;
        const int row = 32 * sub + lane, rr = row & 63, part = row >> 6, rI = rr >> 4;
#pragma unroll 1
        for (int I = 1; I <= 3; I++) {
            float v[32];
            tmem_ld32(tmem_at(tm, 32 * sub, 128 * (I - 1) + 32 * q32), v);
            tmem_wait_ld();
            if (rI == I) st_f4x(ST + ((I - 1) * 32 + part * 16 + (rr - 16 * I)) * LST + 32 * q32, v, 8);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (rb >= 1) {  // below the block diagonal: each row's own factor prod_{16 rb<=t<=r} a_t
        float cpr = 1.f;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            cpr *= AL[(r0 + i) * kD + d];
            X1[i] += cpr * ST[((rb - 1) * 32 + i) * LST + d];
            Y1[i] += cpr * ST[((rb - 1) * 32 + 16 + i) * LST + d];
        }
    }
    // per-channel decays of this thread's rows: Gamma_r = prod_{t<=r} a_t, b_r = prod_{t>r} a_t
    pre = 1.f;
    post = 1.f;
    for (int k = 0; k < rb; k++) pre *= bpr[k * kD + d];
    for (int k = rb + 1; k < 4; k++) post *= bpr[k * kD + d];
    float bq[16];
    {
        float sfx = post;
#pragma unroll
        for (int i = 15; i >= 0; i--) {
            bq[i] = sfx;
            sfx *= AL[(r0 + i) * kD + d];
        }
    }
    float dk[16], dgm[16];
    gsum = 0.f;
    Gm = pre;
#pragma unroll
    for (int i4 = 0; i4 < 16; i4 += 4) {  // terms of X, Y, Z; dq^ and the dbeta partials are final here
        float xc[4], yc[4], zc[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            xc[e] = xs[e];
            yc[e] = ys[e];
            zc[e] = zs[e];
        }
        if (i4 + 4 < 16) {
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int rr = r0 + i4 + 4 + e;
                xs[e] = chx[CHX_X / 4 + rr * kD + d];
                ys[e] = chx[CHX_Y / 4 + rr * kD + d];
                zs[e] = chx[CHX_Z / 4 + rr * kD + d];
            }
        }
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int i = i4 + e, rr = r0 + i;
            Gm *= AL[rr * kD + d];
            const float bb = bq[i], x = xc[e], y = yc[e], z = zc[e];
            const float kh = KH[rr * kD + d], qh = QH[rr * kD + d], br = bet[rr];
            const float dqv = P.scale * Gm * x + X1[i];
            dk[i] = bb * y + br * Gm * z + br * Y1[i];
            dgm[i] = P.scale * Gm * qh * x - bb * kh * y + br * Gm * kh * z + qh * X1[i] + br * kh * Y1[i];
            gsum += bb * kh * y;
            X1[i] = Gm * kh * z + kh * Y1[i];  // this row's dbeta partial (X1[i] is no longer read)
            if (t0 + rr < P.T) a.dqh[(((size_t)b * P.T + t0 + rr) * P.Hv + hv) * kD + d] = dqv;
        }
    }
    {  // dbeta partials summed over the warp's 32 channels by a reduce-scatter: lanes 2m, 2m+1 get row m
        const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
        float w8[8], w4[4], w2[2];
#pragma unroll
        for (int e = 0; e < 8; e++)
            w8[e] = (b4 ? X1[8 + e] : X1[e]) + __shfl_xor_sync(0xffffffffu, b4 ? X1[e] : X1[8 + e], 16);
#pragma unroll
        for (int e = 0; e < 4; e++)
            w4[e] = (b3 ? w8[4 + e] : w8[e]) + __shfl_xor_sync(0xffffffffu, b3 ? w8[e] : w8[4 + e], 8);
#pragma unroll
        for (int e = 0; e < 2; e++)
            w2[e] = (b2 ? w4[2 + e] : w4[e]) + __shfl_xor_sync(0xffffffffu, b2 ? w4[e] : w4[2 + e], 4);
        float w1 = (b1 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2);
        w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
        const int row = (b4 ? 8 : 0) + (b3 ? 4 : 0) + (b2 ? 2 : 0) + (b1 ? 1 : 0);
        if ((lane & 1) == 0) dbr[(warp & 3) * 64 + r0 + row] = w1;
    }
    gC = Gm * post;  // Gamma_C of channel d
    __syncthreads();  // the staged row-side products are read

    // ------------------------------------------------ column side
    for (int u = tid; u < 64 * 16; u += CH_THREADS) {  // [dPs^T | dA^T] bf16 [64 x 128] K-major
        const int j = u & 63, ch = u >> 6;
        const float* M = ch < 8 ? DPR : DAR;
        const int i0 = 8 * (ch & 7);
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; e++) x[e] = M[(i0 + e) * kChunk + j];
        st_chunk(sb + X_AC + sw128_chunk(j, ch, 64), x, 1.f);
    }
    {
        const int d2 = tid & 127, J = tid >> 7;  // Q_J, K_J rows of channel d2
        if (J <= 2) {
            const int n = 48 - 16 * J;
            const uint32_t bb = J == 0 ? X_B0 : J == 1 ? X_B1 : X_B2;
            float pr = 1.f;
#pragma unroll 1
            for (int ib = 16 * J + 16; ib < kChunk; ib += 16) {  // 16 rows' inputs loaded before their stores
                float av[16], qv[16], kv[16];
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    av[e] = AL[(ib + e) * kD + d2];
                    qv[e] = QH[(ib + e) * kD + d2];
                    kv[e] = bet[ib + e] * KH[(ib + e) * kD + d2];
                }
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    pr *= av[e];
                    const int row = ib + e - 16 * J - 16;
                    *reinterpret_cast<__nv_bfloat16*>(sm + bb + sw128_off(row, d2, 2 * n)) =
                        __float2bfloat16_rn(qv[e] * pr);
                    *reinterpret_cast<__nv_bfloat16*>(sm + bb + sw128_off(n + row, d2, 2 * n)) =
                        __float2bfloat16_rn(kv[e] * pr);
                }
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // C_J (M=64 rows j; N=128; K = rows i >= 16J + 16 of both halves) at columns 128 J
        tc_fence_after();
        const uint32_t id = idesc_bf16(64, 128, 0, 1);
        for (int J = 0; J <= 2; J++) {
            const int n = 48 - 16 * J, i0 = 16 * J + 16;
            const uint32_t bb = J == 0 ? X_B0 : J == 1 ? X_B1 : X_B2;
            for (int kk = 0; kk < n; kk += 16)
                mma_bf16(tm + 128 * J, desc_kmajor(sb + X_AC, 64, 0, i0 + kk), desc_mnmajor(sb + bb, 2 * n, 0, kk), id,
                         kk > 0 ? 1u : 0u);
            for (int kk = 0; kk < n; kk += 16)
                mma_bf16(tm + 128 * J, desc_kmajor(sb + X_AC, 64, 0, 64 + i0 + kk),
                         desc_mnmajor(sb + bb, 2 * n, 0, n + kk), id, 1u);
        }
        mma_commit(&bar_mma);
        mma_pend = true;
    }
    float X2[16];  // sum_{i>=j} dPs_ij q^_i E_ij + sum_{i>j} dA_ij beta_i k^_i E_ij
#pragma unroll
    for (int h = 0; h < 2; h++) {  // inside the diagonal block, 8 columns at a time
        const int ja = r0 + 8 * h;
        float E[8];
#pragma unroll
        for (int e = 0; e < 8; e++) {
            E[e] = 1.f;
            X2[8 * h + e] = 0.f;
        }
        for (int i = ja; i < ja + 8; i++) {
            const float ai = AL[i * kD + d], qi = QH[i * kD + d], kbi = bet[i] * KH[i * kD + d];
            const float4 p0 = *reinterpret_cast<const float4*>(DPR + i * kChunk + ja);
            const float4 p1 = *reinterpret_cast<const float4*>(DPR + i * kChunk + ja + 4);
            const float4 a0 = *reinterpret_cast<const float4*>(DAR + i * kChunk + ja);
            const float4 a1 = *reinterpret_cast<const float4*>(DAR + i * kChunk + ja + 4);
            const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int e = 0; e < 8; e++) {
                E[e] = (i > ja + e) ? E[e] * ai : 1.f;
                X2[8 * h + e] += (pv[e] * qi + av[e] * kbi) * E[e];
            }
        }
        if (h == 0) {  // i = r0 + 8 .. r0 + 15: E_ij = E_ja+7,j * prod_{ja+7<t<=i} a_t, the second factor shared by the 8 columns
            float X2f[8];
#pragma unroll
            for (int e = 0; e < 8; e++) X2f[e] = 0.f;
            float F = 1.f;
            for (int i = ja + 8; i < r0 + 16; i++) {
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
    }
    ok = mbar_wait(&bar_mma, mph, &abort_sh, a.status, 71);
    mph ^= 1;
    if (__syncthreads_or(!ok)) goto teardown;
    if (tid == 0) mma_pend = false;
    tc_fence_after();
    {  // stage C_J (rows j of block J sit in lanes 0-15 of sub-partition J) as fp32 [J][16][LST]
        const int sub = warp & 3, q32 = warp >> 2;
        if (sub <= 2) {
            float v[32];
            tmem_ld32(tmem_at(tm, 32 * sub, 128 * sub + 32 * q32), v);
            tmem_wait_ld();
            if (lane < 16) st_f4x(ST + (sub * 16 + lane) * LST + 32 * q32, v, 8);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (rb <= 2) {  // above the block diagonal in i: each column's own factor prod_{j<t<=16 rb+15} a_t
        float fs = 1.f;
#pragma unroll
        for (int i = 15; i >= 0; i--) {
            X2[i] += fs * ST[(rb * 16 + i) * LST + d];
            fs *= AL[(r0 + i) * kD + d];
        }
    }
#pragma unroll
    for (int i = 0; i < 16; i++) {
        dk[i] += X2[i];
        dgm[i] -= KH[(r0 + i) * kD + d] * X2[i];
    }
    // dgamma_C,d, block sums of dgamma, dg as the in-chunk reverse cumulative sum
    float suf[16];
    {
        float sacc = 0.f;
#pragma unroll
        for (int i = 15; i >= 0; i--) {
            sacc += dgm[i];
            suf[i] = sacc;
        }
        gcs[rb * kD + d] = gsum;
        btot[rb * kD + d] = sacc;
    }
    __syncthreads();
    {
        const float dgC = gcs[d] + gcs[kD + d] + gcs[2 * kD + d] + gcs[3 * kD + d] + gC * chx[CHX_HDH / 4 + d];
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
teardown:
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0 && mma_pend) {  // products still in flight finish before TMEM is released
        volatile int never = 0;
        mbar_wait(&bar_mma, mph, &never, nullptr, 0);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

}  // namespace

cudaError_t launch_grad_ch(const GradChArgs& a, const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s) {
    const int smem1 = C_BYTES + 1024;
    cudaError_t e = cudaFuncSetAttribute(grad_ch_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(grad_ch_contract_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)X_BYTES + 1024);
    if (e != cudaSuccess) return e;
    dim3 grid(a.p.NC, a.p.Hv, a.p.B);
    trace_begin("chunk_grad_channel_mma", s);
    grad_ch_mma_kernel<<<grid, CH_THREADS, smem1, s>>>(mv, mdo, a);
    trace_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_begin("chunk_grad_channel_contract", s);
    grad_ch_contract_kernel<<<grid, CH_THREADS, X_BYTES + 1024, s>>>(a);
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
