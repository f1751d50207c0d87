// chunk_fwd_ch.cu - chunk operators of the gated delta rule with a per-channel gate (one decay
// per key channel, g [B,T,Hv,Dk]): the channelwise variant described in "Two-pass optimization
// for channelwise gated delta rule kernel" (ExecuTorch PR #21020, Summary), here in the chunked
// form of "Adding VJP for gated delta net" (MLX PR #4565). One CTA per (b, v-head, chunk).
//
// With a_t = exp(g_t) in R^Dk, Gamma_r = prod_{t<=r} a_t and E_rj = prod_{j<t<=r} a_t (per
// channel), the chunk algebra of chunk.h holds with every decay taken channel by channel:
//   A_rj = beta_r sum_d k^_rd k^_jd E_rj,d (j < r),   P_rj = scale sum_d q^_rd k^_jd E_rj,d (j <= r)
//   W = T diag(beta) (K^ .* Gamma),   U~ = T diag(beta) V,   Kbar = K^ .* (Gamma_C / Gamma_r)
//   Mneg = -Kbar^T W,   Qc = scale Q^ .* Gamma - P W,   H1 = diag(Gamma_C) H0 + Mneg H0 + Kbar^T U~
// so the record has the scalar-gate layout and the scan only scales state row d by Gamma_C,d.
// Decays are formed as products of per-token factors a_t <= 1 (never as exp of a difference
// of cumulative sums), so no factor can overflow however strong the decay. A and P are
// accumulated on the CUDA cores (the decay sits inside the contraction); the WY products,
// Mneg and P W run on tcgen05 from scaled bf16 operand images.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "chunk.h"
#include "chunk_dev.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace gdr {

// Shared memory (offsets from a 1024-aligned base), ~195 KB: one CTA per SM.
constexpr uint32_t CS_KQ = 0;         // k rows 0-63 / q rows 64-127 (TMA, panels 16 KB)
constexpr uint32_t CS_V = 32768;      // v [64 x 128] (panels 8 KB)
constexpr uint32_t CS_AL = 49152;     // a_t = exp(g_t) fp32 [64][128]; later prod_{t>r} a_t
constexpr uint32_t CS_GP = 81920;     // Gamma_r = prod_{t<=r} a_t fp32 [64][128]
constexpr uint32_t CS_A = 114688;     // A fp32 [64][LDA]; then the [Tw; Tu] image
constexpr uint32_t CS_T = 132096;     // T fp32 [64][LDA]; then the W image [64 x 128]
constexpr uint32_t CS_P = 149504;     // P image [64 x 64]
constexpr uint32_t CS_KG = 157696;    // K .* Gamma image [64 x 128]
constexpr uint32_t CS_KB = 174080;    // Kbar image [64 x 128]
constexpr uint32_t CS_SCR = 190464;   // solve scratch [6][16][LDY] fp32
constexpr uint32_t CS_SMALL = CS_SCR + SOLVE_SCRATCH_BYTES;  // bet[64], rho[128], safe[4]
constexpr uint32_t CS_R01 = 199680;   // R_1 [32 x 128] and R_0 [16 x 128] images (12 KB)
// while A and P are formed: the scaled [k; q] operand L over the K .* Gamma and Kbar images,
// R_2 over T, R_3 over v (which is fetched afterwards), R_1 and R_0 in their own region
constexpr uint32_t CS_L = CS_KG, CS_R2 = CS_T, CS_R3 = CS_V, CS_R1 = CS_R01, CS_R0 = CS_R01 + 8192;
constexpr uint32_t CS_BYTES = CS_R01 + 12288;
static_assert(CS_SMALL + 1024 <= CS_R01 && CS_R01 % 1024 == 0, "R_0 / R_1 region");
static_assert(CS_T + 12288 <= CS_P, "R_2 over T");
// A diagonal block's decays come from the tensor-core product when, on every key channel, the
// product of its 16 per-token factors is at least this (the largest B-side scale is then below
// 1e34, far inside the bf16 range); otherwise the running decay on the CUDA cores forms them.
constexpr float kDiagMinDecay = 1e-34f;
static_assert(CS_A % 1024 == 0 && CS_T % 1024 == 0 && CS_P % 1024 == 0 && CS_KG % 1024 == 0 &&
                  CS_KB % 1024 == 0, "operand images need 1024-byte alignment");
static_assert(CS_A + 64 * LDA * 4 <= CS_T && CS_T + 64 * LDA * 4 <= CS_P, "fp32 tiles");
static_assert(CS_BYTES + 1024 <= 232448, "prep_ch smem");

constexpr int PCH_THREADS = 512;  // 16 warps: the A/P loop is latency-bound

// Element (r, d) of the fp32 [64][128] per-token decay arrays (a_t, then prod_{t>r} a_t; Gamma_r).
// The 4-float group is XOR-ed with the row's low 3 bits, so 8 rows read at the same channels
// hit 8 different bank groups, while a row's float4 groups stay contiguous.
__device__ __forceinline__ int dix(int r, int d) { return r * kD + (d ^ ((r & 7) << 2)); }

__global__ void __launch_bounds__(PCH_THREADS, 1)
    prep_ch_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                   const __grid_constant__ CUtensorMap mv, PrepArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const ChunkProblem& P = a.p;
    const int hk = hv / (P.Hv / P.Hk);
    const int t0 = c * kChunk;
    const size_t bh = (size_t)b * P.Hv + hv;
    uint8_t* rec = a.rec + (bh * P.NC + c) * REC_BYTES;
    uint8_t* rec2 = a.rec2 ? a.rec2 + (bh * P.NC + c) * REC2_BYTES : nullptr;  // backward: T, W
    float* al = reinterpret_cast<float*>(sm + CS_AL);
    float* gp = reinterpret_cast<float*>(sm + CS_GP);
    float* Am = reinterpret_cast<float*>(sm + CS_A);
    float* Tm = reinterpret_cast<float*>(sm + CS_T);
    float* Xs = reinterpret_cast<float*>(sm + CS_SCR);
    float* bet = reinterpret_cast<float*>(sm + CS_SMALL);
    float* rho = bet + 64;  // [128] rows 0-63: k norm factors, 64-127: q norm factors
    int* safe = reinterpret_cast<int*>(rho + 128);  // [4][4]: per block and warp, diagonal block by MMA
    bool ok;
    uint32_t mph = 0;                        // bar_mma phase
    bool mma_pend = false, v_pend = false;   // (thread 0) products / v copy not yet waited for

    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_tma, 1);
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
    if (tid == 0) {
        mbar_expect_tx(&bar_tma, 4 * 8192);  // v follows once its region has served as R_3
        tma_load_4d(sm + CS_KQ + 0, &mk, 0, hk, t0, b, &bar_tma);
        tma_load_4d(sm + CS_KQ + 16384, &mk, 64, hk, t0, b, &bar_tma);
        tma_load_4d(sm + CS_KQ + 8192, &mq, 0, hk, t0, b, &bar_tma);
        tma_load_4d(sm + CS_KQ + 24576, &mq, 64, hk, t0, b, &bar_tma);
    }
    {  // a_t = exp(g_t) per channel (tokens past T: g = 0, beta = 0: the state passes unchanged)
        const int t = tid >> 3, q8 = tid & 7;
        const bool valid = t0 + t < P.T;
        const float4* src =
            reinterpret_cast<const float4*>(a.g + (((size_t)b * P.T + t0 + t) * P.Hv + hv) * kD + 16 * q8);
        float4 gv[4];
#pragma unroll
        for (int n = 0; n < 4; n++) gv[n] = valid ? src[n] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int n = 0; n < 4; n++)
            *reinterpret_cast<float4*>(al + dix(t, 16 * q8 + 4 * n)) =
                make_float4(__expf(gv[n].x), __expf(gv[n].y), __expf(gv[n].z), __expf(gv[n].w));
        if (tid < 64) bet[tid] = (t0 + tid < P.T) ? a.beta[((size_t)b * P.T + t0 + tid) * P.Hv + hv] : 0.f;
    }
    ok = mbar_wait(&bar_tma, 0, &abort_sh, a.status, 15);
    if (__syncthreads_or(!ok)) goto teardown;
    if (tid < 128) {  // Gamma_r, channel d = tid: running product over the chunk's tokens,
        float p = 1.f;  // 16 tokens' factors loaded before their products are stored
#pragma unroll 1
        for (int t0b = 0; t0b < kChunk; t0b += 16) {
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; i++) x[i] = al[dix(t0b + i, tid)];
#pragma unroll
            for (int i = 0; i < 16; i++) {
                p *= x[i];
                gp[dix(t0b + i, tid)] = p;
            }
        }
    } else if (tid < 256) {  // L2 norm factors: row tid-128 of the [k; q] tile (read order rotated by the row)
        const int row = tid - 128;
        float ss = 0.f;
#pragma unroll
        for (int ch = 0; ch < 16; ch++) {
            const int j = (ch + row) & 15;
            float x[8];
            unpack8(ld_shared_v4(sb + CS_KQ + sw128_chunk(row, j, 128)), x);
#pragma unroll
            for (int e = 0; e < 8; e++) ss += x[e] * x[e];
        }
        rho[row] = P.use_norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
    }
    if (tid < 256) {  // P image starts at zero (its upper triangle is never written)
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        st_shared_v4(sb + CS_P + tid * 32, z.x, z.y, z.z, z.w);
        st_shared_v4(sb + CS_P + tid * 32 + 16, z.x, z.y, z.z, z.w);
    }
    __syncthreads();

    // A and P by 16-row blocks I (rows 16I .. 16I + 15). For r in block I and j < 16I the decay
    // factors through s = 16I - 1 into two products of per-token factors, each <= 1:
    //   E_rj = [prod_{s<t<=r} a_t] [prod_{j<t<=s} a_t]
    // so the blocks below the block diagonal are tcgen05 products D_I = L R_I^T of scaled
    // operands: L = [k; q] with row r scaled by p_r = prod_{16I<=t<=r} a_t, R_I = rows j < 16I of
    // k scaled by prod_{j<t<16I} a_t. Inside the diagonal block (16I <= j <= r) E_rj = p_r / p_j,
    // so R_I continues with the block's own rows k_j / p_j (>= 1): N = 16 (I + 1). That factor is
    // bounded only while p_j stays in range, so a block whose 16-token product falls below
    // kDiagMinDecay on some channel takes its diagonal decays from the running product on the
    // CUDA cores instead (exact for any decay).
    {
        const int d = tid & 127, blk = tid >> 7;  // channel d, block blk
        const __nv_bfloat16* kqs = reinterpret_cast<const __nv_bfloat16*>(sm + CS_KQ);
        {  // L rows of block blk (k rows r, q rows 64 + r); all loads before the stores
            float av[16], kv[16], qv[16];
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const int r = 16 * blk + i;
                av[i] = al[dix(r, d)];
                kv[i] = __bfloat162float(kqs[sw128_off(r, d, 128) >> 1]);
                qv[i] = __bfloat162float(kqs[sw128_off(64 + r, d, 128) >> 1]);
            }
            const uint32_t rb = blk == 0 ? CS_R0 : blk == 1 ? CS_R1 : blk == 2 ? CS_R2 : CS_R3;
            const int nr = 16 * blk + 16;  // rows of R_blk
            float p = 1.f;
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const int r = 16 * blk + i;
                p *= av[i];
                *reinterpret_cast<__nv_bfloat16*>(sm + CS_L + sw128_off(r, d, 128)) = __float2bfloat16_rn(kv[i] * p);
                *reinterpret_cast<__nv_bfloat16*>(sm + CS_L + sw128_off(64 + r, d, 128)) =
                    __float2bfloat16_rn(qv[i] * p);
                // the diagonal block's B-side row k_j / p_j (zero where the block falls back)
                *reinterpret_cast<__nv_bfloat16*>(sm + rb + sw128_off(r, d, nr)) =
                    __float2bfloat16_rn(p >= kDiagMinDecay ? kv[i] / p : 0.f);
            }
            const bool ok_d = p >= kDiagMinDecay;  // p: the block's 16-token product on channel d
            const unsigned all_ok = __all_sync(0xffffffffu, ok_d);
            if (lane == 0) safe[4 * blk + (warp & 3)] = all_ok ? 1 : 0;
        }
        if (blk) {  // R_blk: rows j = 16 blk - 1 .. 0, 16 rows' inputs loaded before their stores
            const uint32_t rb = blk == 1 ? CS_R1 : blk == 2 ? CS_R2 : CS_R3;
            const int nr = 16 * blk + 16;
            float sfx = 1.f;
#pragma unroll 1
            for (int jb = 16 * blk - 16; jb >= 0; jb -= 16) {
                float av[16], kv[16];
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    av[i] = al[dix(jb + i, d)];
                    kv[i] = __bfloat162float(kqs[sw128_off(jb + i, d, 128) >> 1]);
                }
#pragma unroll
                for (int i = 15; i >= 0; i--) {
                    *reinterpret_cast<__nv_bfloat16*>(sm + rb + sw128_off(jb + i, d, nr)) =
                        __float2bfloat16_rn(kv[i] * sfx);
                    sfx *= av[i];
                }
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // D_I (M=128, N=16 (I + 1)) into TMEM columns 0, 16, 48, 96
        tc_fence_after();
#pragma unroll
        for (int I = 0; I <= 3; I++) {
            const uint32_t rb = I == 0 ? CS_R0 : I == 1 ? CS_R1 : I == 2 ? CS_R2 : CS_R3;
            const uint32_t id = idesc_bf16(128, 16 * I + 16, 0, 0);
            for (int k0 = 0; k0 < kD; k0 += 16)
                mma_bf16(tm + 8 * I * (I + 1), desc_kmajor(sb + CS_L, 128, 0, k0),
                         desc_kmajor(sb + rb, 16 * I + 16, 0, k0), id, k0 > 0);
        }
        mma_commit(&bar_mma);
        mma_pend = true;
    }
    // diagonal blocks on the CUDA cores. Lane = (column jsel = lane >> 4, channel group
    // cg = lane & 15); channel group cg owns channels 32 m + 4 (cg & 7) + x for m = (cg >> 3) +
    // {0, 2}, x < 4 (the 8 lanes sharing m read 8 consecutive 8-byte words of a row). Warp w
    // takes block I = w >> 2 and, with c = w & 3, the column pairs (16I + 2c, +1) and then
    // (16I + 14 - 2c, +1): both halves of the warp walk the same rows jb .. 16I + 15, so every
    // row load serves two columns, and every warp makes 18 steps.
    {
        const int jsel = lane >> 4, cg = lane & 15, mq = cg >> 3, c8 = cg & 7;
        const int I = warp >> 2, c = warp & 3, rend = 16 * I + 16;
        const bool by_mma = safe[4 * I] & safe[4 * I + 1] & safe[4 * I + 2] & safe[4 * I + 3];
        float kj[8], e[8];
        auto load_row8 = [&](int row, float* x) {
#pragma unroll
            for (int mm = 0; mm < 2; mm++) {
                const int m = mq + 2 * mm;
                const uint32_t off = CS_KQ + sw128_chunk(row, 4 * m + (c8 >> 1), 128) + 8 * (c8 & 1);
                const uint2 u = *reinterpret_cast<const uint2*>(sm + off);
                x[4 * mm] = bf16lo(u.x);
                x[4 * mm + 1] = bf16hi(u.x);
                x[4 * mm + 2] = bf16lo(u.y);
                x[4 * mm + 3] = bf16hi(u.y);
            }
        };
#pragma unroll 1
        for (int ph = 0; ph < (by_mma ? 0 : 2); ph++) {
            const int jb = 16 * I + (ph == 0 ? 2 * c : 14 - 2 * c);
            const int j = jb + jsel;
            load_row8(j, kj);
#pragma unroll
            for (int x = 0; x < 8; x++) e[x] = 1.f;
            for (int r = jb; r < rend; r++) {
                const bool past = r > j;  // E_rj = E_(r-1)j * a_r past the column's own row
#pragma unroll
                for (int mm = 0; mm < 2; mm++) {
                    const float4 f = *reinterpret_cast<const float4*>(al + dix(r, 32 * (mq + 2 * mm) + 4 * c8));
                    e[4 * mm] *= past ? f.x : 1.f;
                    e[4 * mm + 1] *= past ? f.y : 1.f;
                    e[4 * mm + 2] *= past ? f.z : 1.f;
                    e[4 * mm + 3] *= past ? f.w : 1.f;
                }
                float kr[8], qr[8];
                load_row8(r, kr);
                load_row8(64 + r, qr);
                float pa = 0.f, pp = 0.f;
#pragma unroll
                for (int x = 0; x < 8; x++) {
                    const float w = kj[x] * e[x];
                    pa += kr[x] * w;
                    pp += qr[x] * w;
                }
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    pa += __shfl_xor_sync(0xffffffffu, pa, o);
                    pp += __shfl_xor_sync(0xffffffffu, pp, o);
                }
                if (cg == 0 && r >= j) {
                    if (r > j) Am[r * LDA + j] = bet[r] * rho[r] * rho[j] * pa;
                    const __nv_bfloat16 pv = __float2bfloat16_rn(P.scale * rho[64 + r] * rho[j] * pp);
                    *reinterpret_cast<__nv_bfloat16*>(sm + CS_P + sw128_off(r, j, 64)) = pv;
                }
            }
        }
    }
    ok = mbar_wait(&bar_mma, mph, &abort_sh, a.status, 18);
    mph ^= 1;
    if (__syncthreads_or(!ok)) goto teardown;
    if (tid == 0) mma_pend = false;
    tc_fence_after();
    {  // D row 32 lg + lane (k rows, then q rows) into A / P: below the block diagonal, and the
       // diagonal blocks formed by the product. The lane group's rows lie in blocks I0 (lanes
       // 0-15) and I0 + 1; their 16-column panels (I, pc <= I) are shared out over the group's 4 warps.
        const int lg = warp & 3, sub = warp >> 2;
        const int row = 32 * lg + lane, rr = row & 63, rI = rr >> 4;
        const int I0 = 2 * (lg & 1), npan = 2 * I0 + 3;  // panels of blocks I0 and I0 + 1
        for (int n = sub; n < npan; n += 4) {
            const int I = n < I0 + 1 ? I0 : I0 + 1, pc = n < I0 + 1 ? n : n - I0 - 1;
            float v[16];
            tmem_ld16(tmem_at(tm, 32 * lg, 8 * I * (I + 1) + 16 * pc), v);
            tmem_wait_ld();
            const bool diag_mma = safe[4 * I] & safe[4 * I + 1] & safe[4 * I + 2] & safe[4 * I + 3];
            if (rI == I && (pc < I || diag_mma)) {
                const float4 r0 = *reinterpret_cast<const float4*>(rho + 16 * pc);
                const float4 r1 = *reinterpret_cast<const float4*>(rho + 16 * pc + 4);
                const float4 r2 = *reinterpret_cast<const float4*>(rho + 16 * pc + 8);
                const float4 r3 = *reinterpret_cast<const float4*>(rho + 16 * pc + 12);
                const float rj[16] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w,
                                      r2.x, r2.y, r2.z, r2.w, r3.x, r3.y, r3.z, r3.w};
                float x[16];
                if (row < 64) {  // A (strictly lower; zeros above are not read)
                    const float f = bet[rr] * rho[rr];
#pragma unroll
                    for (int e2 = 0; e2 < 16; e2++) x[e2] = 16 * pc + e2 < rr ? f * rj[e2] * v[e2] : 0.f;
                    float4* dst = reinterpret_cast<float4*>(Am + rr * LDA + 16 * pc);
#pragma unroll
                    for (int q = 0; q < 4; q++) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
                } else {  // P (lower with the diagonal; zeros above)
                    const float f = P.scale * rho[64 + rr];
#pragma unroll
                    for (int e2 = 0; e2 < 16; e2++) x[e2] = 16 * pc + e2 <= rr ? f * rj[e2] * v[e2] : 0.f;
                    st_chunk(sb + CS_P + sw128_chunk(rr, 2 * pc, 64), x, 1.f);
                    st_chunk(sb + CS_P + sw128_chunk(rr, 2 * pc + 1, 64), x + 8, 1.f);
                }
            }
        }
    }
    fence_proxy_async_smem();  // the P image leaves by a bulk copy
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // v into its region (R_3 is no longer read)
        mbar_expect_tx(&bar_tma, 2 * 8192);
        tma_load_4d(sm + CS_V + 0, &mv, 0, hv, t0, b, &bar_tma);
        tma_load_4d(sm + CS_V + 8192, &mv, 64, hv, t0, b, &bar_tma);
        v_pend = true;
    }
    __syncthreads();
    if (tid >= 256 && tid < 384) {  // prod_{t>r} a_t, channel d, in place of a_t (16 tokens read
        const int d = tid - 256;       // before written), by threads the solve's first phase leaves idle
        float p = 1.f;
#pragma unroll 1
        for (int t0b = kChunk - 16; t0b >= 0; t0b -= 16) {
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; i++) x[i] = al[dix(t0b + i, d)];
#pragma unroll
            for (int i = 15; i >= 0; i--) {
                al[dix(t0b + i, d)] = p;
                p *= x[i];
            }
        }
        a.gam[(bh * P.NC + c) * kD + d] = gp[dix(kChunk - 1, d)];  // Gamma_C per channel
    }
    if (tid == 0) {  // P to the record
        bulk_store(rec + REC_P, sm + CS_P, 8192);
        bulk_commit();
    }
    ut_solve(Am, Tm, Xs, tid);  // T = (I + A)^-1 (ends with a barrier; suffix products done)
    {  // [Tw; Tu]: Tw = T diag(beta rho_k), Tu = T diag(beta) (K-major A operand, over A)
        const int row = tid >> 2, qtr = tid & 3;  // 16 columns per thread
        const int i = row & 63;
        const bool isw = row < 64;
        const float* trow = Tm + i * LDA + 16 * qtr;
        float t[16], x[16];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const float4 f = *reinterpret_cast<const float4*>(trow + 4 * q);
            const float tv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int j = 16 * qtr + 4 * q + e;
                t[4 * q + e] = (j >> 4) <= (i >> 4) ? tv[e] : 0.f;
                x[4 * q + e] = t[4 * q + e] * bet[j] * (isw ? rho[j] : 1.f);
            }
        }
#pragma unroll
        for (int q = 0; q < 2; q++) st_chunk(sb + CS_A + sw128_chunk(row, 2 * qtr + q, 128), x + 8 * q, 1.f);
    }
    {  // K .* Gamma and Kbar = diag(rho_k) K .* prod_{t>r} a_t, 16 channels of row r each (a quarter
       // warp takes 8 rows at the same channels)
        const int r = (tid & 7) + 8 * (tid >> 6), q8 = (tid >> 3) & 7;
        const float rk = rho[r];
#pragma unroll
        for (int q = 0; q < 2; q++) {
            const int j = 2 * q8 + q;  // 8-channel chunk of the row
            float x[8], yg[8], yb[8];
            unpack8(ld_shared_v4(sb + CS_KQ + sw128_chunk(r, j, 128)), x);
            const float4 g0 = *reinterpret_cast<const float4*>(gp + dix(r, 8 * j));
            const float4 g1 = *reinterpret_cast<const float4*>(gp + dix(r, 8 * j + 4));
            const float4 b0 = *reinterpret_cast<const float4*>(al + dix(r, 8 * j));
            const float4 b1 = *reinterpret_cast<const float4*>(al + dix(r, 8 * j + 4));
            const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int e = 0; e < 8; e++) {
                yg[e] = x[e] * gg[e];
                yb[e] = rk * x[e] * bb[e];
            }
            const uint32_t off = sw128_chunk(r, j, 64);
            st_chunk(sb + CS_KG + off, yg, 1.f);
            const uint4 ub = pack8(yb, 1.f);
            st_shared_v4(sb + CS_KB + off, ub.x, ub.y, ub.z, ub.w);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // Kbar to the record, from its image
        bulk_store(rec + REC_K, sm + CS_KB, 16384);
        bulk_commit();
    }

    // W = Tw (K .* Gamma) and U~ = Tu V as two M=128 products of [Tw; Tu] (rows 0-63 of the
    // first, rows 64-127 of the second are the wanted ones); B operands MN-major
    ok = mbar_wait(&bar_tma, 1, &abort_sh, a.status, 19);
    if (__syncthreads_or(!ok)) goto teardown;
    if (tid == 0) {
        v_pend = false;
        tc_fence_after();
        const uint32_t id = idesc_bf16(128, 128, 0, 1);
        for (int k0 = 0; k0 < kChunk; k0 += 16) {
            mma_bf16(tm + 0, desc_kmajor(sb + CS_A, 128, 0, k0), desc_mnmajor(sb + CS_KG, 64, 0, k0), id, k0 > 0);
            mma_bf16(tm + 128, desc_kmajor(sb + CS_A, 128, 0, k0), desc_mnmajor(sb + CS_V, 64, 0, k0), id, k0 > 0);
        }
        mma_commit(&bar_mma);
        mma_pend = true;
    }
    if (rec2 && tid < 256) {  // T for the backward, from the tile still intact, stored once the
                              // products are issued: the proxy fence before them would wait for it
        const int i = tid >> 2, qtr = tid & 3;
        const float* trow = Tm + i * LDA + 16 * qtr;
#pragma unroll
        for (int q = 0; q < 2; q++) {
            float t[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const int j = 16 * qtr + 8 * q + e;
                t[e] = (j >> 4) <= (i >> 4) ? trow[8 * q + e] : 0.f;
            }
            st_global16(rec2 + REC2_T + sw128_chunk(i, 2 * qtr + q, 64), pack8(t, 1.f));
        }
    }
    ok = mbar_wait(&bar_mma, mph, &abort_sh, a.status, 16);
    mph ^= 1;
    if (__syncthreads_or(!ok)) goto teardown;
    if (tid == 0) mma_pend = false;
    tc_fence_after();
    if (warp < 8) {
        const int lg = warp & 3, h = warp >> 2;
        if (lg < 2) {  // W rows i = 32 lg + lane -> W image (over T)
            const int i = 32 * lg + lane;
            float w[64];
            tmem_ld32(tmem_at(tm, 32 * lg, 64 * h), w);
            tmem_ld32(tmem_at(tm, 32 * lg, 64 * h + 32), w + 32);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; q++) st_chunk(sb + CS_T + sw128_chunk(i, 8 * h + q, 64), w + 8 * q, 1.f);
        } else {  // U~ rows i = 32 lg + lane - 64 -> the record's slice images, staged over v (read)
            const int i = 32 * lg + lane - 64;
            float u[64];
            tmem_ld32(tmem_at(tm, 32 * lg, 128 + 64 * h), u);
            tmem_ld32(tmem_at(tm, 32 * lg, 128 + 64 * h + 32), u + 32);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 8; q++) {
                const int col = 64 * h + 8 * q;
                st_chunk(sb + CS_V + (col >> 5) * 4096 + sw64_chunk(i, q & 3), u + 8 * q, 1.f);
            }
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {  // U~ (and W for the backward) to the record, from their images
        bulk_store(rec + REC_U, sm + CS_V, 16384);
        if (rec2) bulk_store(rec2 + REC2_W, sm + CS_T, 16384);
        bulk_commit();
    }

    // Mneg = -Kbar^T W (M=128: A = Kbar image read MN-major) and P W (M=64)
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idm = idesc_bf16(128, 128, 1, 1);
        for (int k0 = 0; k0 < kChunk; k0 += 16)
            mma_bf16(tm + 0, desc_mnmajor(sb + CS_KB, 64, 0, k0), desc_mnmajor(sb + CS_T, 64, 0, k0), idm, k0 > 0);
        const uint32_t idp = idesc_bf16(64, 128, 0, 1);
        for (int k0 = 0; k0 < kChunk; k0 += 16)
            mma_bf16(tm + 128, desc_kmajor(sb + CS_P, 64, 0, k0), desc_mnmajor(sb + CS_T, 64, 0, k0), idp, k0 > 0);
        mma_commit(&bar_mma);
        mma_pend = true;
    }
    ok = mbar_wait(&bar_mma, mph, &abort_sh, a.status, 17);
    mph ^= 1;
    if (__syncthreads_or(!ok)) goto teardown;
    if (tid == 0) mma_pend = false;
    tc_fence_after();
    {  // 16 warps: lane group lg, column quarter h (32 columns)
        const int lg = warp & 3, h = warp >> 2;
        {  // Mneg rows d = 32 lg + lane
            const int d = 32 * lg + lane;
            float m[32];
            tmem_ld32(tmem_at(tm, 32 * lg, 32 * h), m);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; q++) st_chunk(sb + CS_AL + sw128_chunk(d, 4 * h + q, 128), m + 8 * q, -1.f);
        }
        {  // Qc = scale diag(rho_q) Q .* Gamma - P W, rows i = 16 lg + lane (M=64 layout)
            const int i = 16 * lg + (lane & 15);
            float pw[32];
            tmem_ld32(tmem_at(tm, 32 * lg, 128 + 32 * h), pw);
            tmem_wait_ld();
            if (lane < 16) {
                const float f = P.scale * rho[64 + i];
                uint4 qv[4];
#pragma unroll
                for (int q = 0; q < 4; q++)
                    qv[q] = ld_shared_v4(sb + CS_KQ + sw128_chunk(64 + i, 4 * h + q, 128));
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float x[8];
                    unpack8(qv[q], x);
                    const float4 g0 = *reinterpret_cast<const float4*>(gp + dix(i, 32 * h + 8 * q));
                    const float4 g1 = *reinterpret_cast<const float4*>(gp + dix(i, 32 * h + 8 * q + 4));
                    const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                    for (int e = 0; e < 8; e++) x[e] = f * x[e] * gg[e] - pw[8 * q + e];
                    st_chunk(sb + CS_A + sw128_chunk(i, 4 * h + q, 64), x, 1.f);
                }
            }
        }
    }
    // Mneg (over the decay products) and Qc (over [Tw; Tu]) to the record, from their images
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        bulk_store(rec + REC_M, sm + CS_AL, 32768);
        bulk_store(rec + REC_Q, sm + CS_A, 16384);
        bulk_commit();
    }
teardown:
    if (tid == 0) bulk_wait_all();  // record stores complete before the CTA exits
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0) {  // let copies and products still in flight finish before the CTA exits
        volatile int never = 0;
        mbar_wait(&bar_tma, 0, &never, nullptr, 0);
        if (v_pend) mbar_wait(&bar_tma, 1, &never, nullptr, 0);
        if (mma_pend) mbar_wait(&bar_mma, mph, &never, nullptr, 0);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

cudaError_t launch_prep_ch(const PrepArgs& a, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           cudaStream_t s) {
    const int smem = CS_BYTES + 1024;
    cudaError_t e = cudaFuncSetAttribute(prep_ch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.p.NC, a.p.Hv, a.p.B);
    trace_begin("chunk_prep_channel", s);
    prep_ch_kernel<<<grid, PCH_THREADS, smem, s>>>(mq, mk, mv, a);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace gdr
