// chunk_bwd.cu - backward (VJP) of the chunked gated delta rule, the "chunked case" of
// "Adding VJP for gated delta net" (MLX PR #4565): dq, dk, dv, dg, dbeta and dh0 for the
// loss <do, o> + <dht, ht>, through the in-kernel q/k L2 norm ("fold q/k L2-norm into the
// gated_delta_rule kernel": the kernel owns the normalisation, so no normalised q/k is
// ever stored). Launch sequence:
//   prep (also keeps T and W per chunk)  ->  forward scan storing the chunk-start states
//   ->  reverse scan storing the chunk-end state gradients (and dh0)  ->  grad_kernel.
// grad_kernel: one CTA per (b, key head, chunk); it loops over the value heads that share
// the key head, so dq and dk are summed over the group on chip (deterministic, no atomics).
// Per value head, with H0 the chunk-start state, dH1 the chunk-end state gradient:
//   U   = U~ - W H0                  dU  = P^T dO + Kbar dH1
//   dP  = dO U^T  -> dS = scale E .* dP, Z = dP .* P      X = dO H0^T
//   dQ^ += scale diag(Gamma) X + dS diag(rk) K            dK^ += (diag(rq) dS)^T Q
//   Y   = U dH1^T -> dK^ += diag(b) Y, db = rk .* rowsum(K .* Y)
//   dW  = -dU H0^T;  dT = dU V^T diag(beta) + dW K^T diag(beta Gamma rk)
//   dV  = diag(beta) T^T dU;  T^T dW -> dK^ += diag(beta Gamma) T^T dW
//   dA  = strict_lower(-T^T dT T^T) = strict_lower(-(T^T dU) U~^T - (T^T dW) W^T)   (U~ = T diag(beta) V
//         and W = T diag(beta Gamma rk) K, so dT itself is never formed)
//   dK^ += N K with N_rj = rk_j (M_rj + M_jr), M = beta_r E .* dA
//   dgamma from every Gamma, E, b, Gamma_C term;  dg = reverse cumsum of dgamma in the chunk
//   dq = rq (dQ^ - q^ (q^ . dQ^)), likewise dk (after the group sum).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "chunk.h"
#include "chunk_dev.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace gdr {

// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t G_KQ = 0;        // k rows 0-63, q rows 64-127 (panels 16 KB)      [whole CTA]
constexpr uint32_t G_V = 32768;     // U image [64 x 128]; then v; later M fp32 [64][64]
constexpr uint32_t G_DO = 49152;    // dO [64 x 128]; later dSq image [64 x 64]
constexpr uint32_t G_H0 = 65536;    // H0 image [128 d x 128 v]; later dW, then T^T dW images [64 x 128]
constexpr uint32_t G_DH = 98304;    // dH1 image; after M3 U~ as four SW64 slices [64 x 32] (the record's)
constexpr uint32_t G_T = 131072;    // T image [64 x 64]; after M5 (dA) the N image
constexpr uint32_t G_W = 139264;    // W image [64 x 128] (read again by M5)
constexpr uint32_t G_P = 155648;    // P image [64 x 64]; later dSk image
constexpr uint32_t G_KB = 163840;   // Kbar image [64 x 128]; later dU, then T^T dU images
constexpr uint32_t G_GF = 180224;   // G = K K^T fp32 [64][64]                            [whole CTA]
constexpr uint32_t G_ZS = 196608;   // fp32 [64][64] scratch (column sums)
constexpr uint32_t G_SM = 212992;   // small arrays
constexpr uint32_t G_SM_FLOATS = 64 * 4 + 256 * 4 + 64 + 272 + 4 + 128;  // see the carve-up in grad_kernel
constexpr uint32_t G_STG = G_SM + 7168;  // per warp 4 rows x 40 fp32: staging of the fp32 row stores
constexpr uint32_t G_BYTES = G_STG + 16 * 4 * 40 * 4;
static_assert(G_SM_FLOATS * 4 <= 7168, "small arrays");
static_assert(G_BYTES + 1024 <= 232448, "grad smem");

// TMEM columns: dQ^ accumulator, dK^ accumulator (both M=64 x 128), two temporaries.
constexpr uint32_t TM_DQ = 0, TM_DK = 128, TM_T1 = 256, TM_T2 = 384;

struct GradArgs {
    ChunkProblem p;
    const float *g, *beta;
    const uint8_t *rec, *rec2, *hs, *dhs;
    const float* gam;  // Gamma_C per chunk (unused here: recomputed)
    float *dq, *dk, *dv, *dg, *dbeta;
    float *dqh, *dkh;  // split gradient (kSplit): dq^, dk^ per value head, fp32 [B][T][Hv][Dk]
    int* status;
};

// fp32 [64][64] scratch element (r, j), columns XOR-swizzled by the row so that a warp
// touching one column across rows (or one row across columns) hits distinct banks
__device__ __forceinline__ int fsw(int r, int j) { return r * 64 + (j ^ (r & 31)); }

// 16 warps: warp w reads TMEM lane group (w & 3) (M=64 accumulator rows 16*(w&3) .. +15 in
// lanes 0-15) and column quarter (w >> 2) of every product.
constexpr int GRAD_THREADS = 512;

// kSplit: a work unit is one value head of a (b, key head, chunk) tile (small problems; see
// grad_split): dq^, dk^ of that head leave raw, and a second kernel sums and normalises them.
template <bool kSplit>
__global__ void __launch_bounds__(GRAD_THREADS, 1)
    grad_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                const __grid_constant__ CUtensorMap mdq, const __grid_constant__ CUtensorMap mdk, GradArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t bar_ld, bar_mma, bar_h, bar_h2, bar_h3;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkProblem& P = a.p;
    const int G = P.Hv / P.Hk;
    const int ntiles = P.B * P.Hk * P.NC;  // (b, key head, chunk), chunk fastest
    const int GU = kSplit ? G : 1;         // work units per tile
    const int nunits = ntiles * GU;
    const int lg = warp & 3, qt = warp >> 2;
    const int r = 16 * lg + (lane & 15);
    const bool act = lane < 16;
    int c = 0, hk = 0, b = 0, t0 = 0;  // the current tile
    const int c32 = 32 * qt, c16 = 16 * qt;  // this thread's columns of N=128 / N=64 products

    // k/q and the GF / ZS scratch swap their two 32 KB regions from tile to tile, so the next
    // tile's k/q can land while this tile's norm backward still reads its own
    uint32_t kq = G_KQ, gfz = G_GF;
    float* GF = reinterpret_cast<float*>(sm + gfz);
    float* ZS = reinterpret_cast<float*>(sm + gfz + 16384);
    float* MF = reinterpret_cast<float*>(sm + G_V);
    float* rk = reinterpret_cast<float*>(sm + G_SM);  // [64]
    float* rq = rk + 64;                                // [64]
    float* gam = rq + 64;                               // [64]
    float* bet = gam + 64;                              // [64]
    float* dgp = bet + 64;                              // [4][64] dgamma partials by column quarter
    float* dbp = dgp + 256;                             // [4][64] dbeta partials
    float* sb3 = dbp + 256;                             // [4][64] b_r db_r partials
    float* part = sb3 + 256;                            // [4][64] norm-backward partial dots
    float* dgc = part + 256;                            // [64] column-sum terms of dgamma
    float* red = dgc + 64;                              // [16 + 256] reductions
    float* hdh = red + 272;                             // <dH1, H0>
    float* gst = hdh + 4;                               // [2][64] the next value head's g, beta (cp.async)
    float* stg = reinterpret_cast<float*>(sm + G_STG) + warp * 160;  // this warp's row-store staging

    uint32_t ld_phase = 0, mma_phase = 0, h_phase = 0, h2_phase = 0, h3_phase = 0;
    bool pend_ld = false, pend_h = false, pend_h2 = false, pend_h3 = false;  // issued, not yet waited for (thread 0)
    bool h_open = false, h2_open = false;  // pieces issued before the arriving piece of their barrier (thread 0)
    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_h, 1);
        mbar_init(&bar_h2, 1);
        mbar_init(&bar_h3, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_sh;
    const uint32_t tl = tmem_at(tm, 32 * lg, 0);  // this warp's TMEM lane base

    auto wait_ld = [&](int site) -> bool {
        bool ok = mbar_wait(&bar_ld, ld_phase, &abort_sh, a.status, site);
        ld_phase ^= 1;
        if (ok) pend_ld = false;
        return !__syncthreads_or(!ok);
    };
    auto wait_mma = [&](int site) -> bool {
        bool ok = mbar_wait(&bar_mma, mma_phase, &abort_sh, a.status, site);
        mma_phase ^= 1;
        ok = !__syncthreads_or(!ok);
        tc_fence_after();
        return ok;
    };
    auto sync_for_mma = [&]() {  // make generic smem writes / TMEM stores visible to the next MMAs
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
    };
    auto mma = [&](uint32_t col, uint64_t ad, uint64_t bd, uint32_t id, bool acc) {
        mma_bf16(tm + col, ad, bd, id, acc ? 1u : 0u);
    };
    // 8 bf16 of row `row` of a panelised tile, logical chunk j
    auto ldrow8 = [&](uint32_t tile, int row, int j, int R, float* x) {
        unpack8(ld_shared_v4(sb + tile + sw128_chunk(row, j, R)), x);
    };
    // fp32 rows of a [64 x 128] result tile to global memory: this warp holds rows 16 lg .. + 15 of
    // column quarter qt, lane l (l & 15: the row) the groups c32 + 8 q + 4 (l >> 4) .. + 3 (q < 4).
    // Four rows at a time go through the warp's staging so that each store instruction writes four
    // whole 128-byte row segments (8 lanes each) instead of one 32-byte sector in each of 16 rows,
    // which stalled the warps on the store queue. g0: row 0 of the tile at column c32; rs: floats
    // per row. Rows past the sequence end are not written.
    auto store_rows = [&](float* g0, size_t rs, const float* v) {
        const int hf = lane >> 4, rl = lane & 15, m = lane >> 3, cg = lane & 7;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            if ((rl >> 2) == i) {
#pragma unroll
                for (int q = 0; q < 4; q++)
                    *reinterpret_cast<float4*>(stg + (rl & 3) * 40 + 8 * q + 4 * hf) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
            __syncwarp();
            const int row = 16 * lg + 4 * i + m;
            const float4 x = *reinterpret_cast<const float4*>(stg + m * 40 + 4 * cg);
            if (t0 + row < P.T) *reinterpret_cast<float4*>(g0 + (size_t)row * rs + 4 * cg) = x;
            __syncwarp();
        }
    };
    const uint32_t id64x128_kk = idesc_bf16(64, 128, 0, 0), id64x128_km = idesc_bf16(64, 128, 0, 1),
                   id64x128_mm = idesc_bf16(64, 128, 1, 1), id64x64_kk = idesc_bf16(64, 64, 0, 0);

    // Inputs of value head hv, issued in pieces as their buffers free up (thread 0 only). Those of the
    // first products complete bar_h: piece 0: P, dO   6: W   5: dH1   1: Kbar   2: H0 (issued last:
    // it arrives, so the phase ends when all have landed). T, first read by M4, completes bar_h2
    // (piece 3); its latency stays off the head's start. v and U~ of the head itself follow its M3
    // (load_vu, bar_h3), over the U image and dH1.
    auto load_piece = [&](int bb, int cc, int hv, int piece) {
        const size_t bh = (size_t)bb * P.Hv + hv;
        const size_t idx = bh * P.NC + cc;
        const int tt = cc * kChunk;
        const uint8_t* rec = a.rec + idx * REC_BYTES;
        const uint8_t* rec2 = a.rec2 + idx * REC2_BYTES;
        switch (piece) {
            case 0:
                h_open = true;
                mbar_add_tx(&bar_h, 8192 + 2 * 8192);
                bulk_load(sm + G_P, rec + REC_P, 8192, &bar_h);
                tma_load_4d(sm + G_DO + 0, &mdo, 0, hv, tt, bb, &bar_h);
                tma_load_4d(sm + G_DO + 8192, &mdo, 64, hv, tt, bb, &bar_h);
                break;
            case 6:
                h_open = true;
                mbar_add_tx(&bar_h, 16384);
                bulk_load(sm + G_W, rec2 + REC2_W, 16384, &bar_h);
                break;
            case 1:
                h_open = true;
                mbar_add_tx(&bar_h, 16384);
                bulk_load(sm + G_KB, rec + REC_K, 16384, &bar_h);
                break;
            case 2:
                h_open = false;
                pend_h = true;
                mbar_expect_tx(&bar_h, 32768);
                bulk_load(sm + G_H0, a.hs + idx * STATE_IMG, 32768, &bar_h);
                break;
            case 3:
                h2_open = false;
                pend_h2 = true;
                mbar_expect_tx(&bar_h2, 8192);
                bulk_load(sm + G_T, rec2 + REC2_T, 8192, &bar_h2);
                break;
            default:
                h_open = true;
                mbar_add_tx(&bar_h, 32768);
                bulk_load(sm + G_DH, a.dhs + idx * STATE_IMG, 32768, &bar_h);
                break;
        }
    };

    auto load_vu = [&](int bb, int cc, int hv) {  // v and U~ of value head hv (thread 0)
        const size_t idx = ((size_t)bb * P.Hv + hv) * P.NC + cc;
        mbar_expect_tx(&bar_h3, 2 * 8192 + 16384);
        tma_load_4d(sm + G_V + 0, &mv, 0, hv, cc * kChunk, bb, &bar_h3);
        tma_load_4d(sm + G_V + 8192, &mv, 64, hv, cc * kChunk, bb, &bar_h3);
        bulk_load(sm + G_DH, a.rec + idx * REC_BYTES + REC_U, 16384, &bar_h3);
        pend_h3 = true;
    };
    auto issue_kq = [&](int bb, int cc, int hh, uint32_t dst) {  // k, q of a tile (thread 0)
        mbar_expect_tx(&bar_ld, 4 * 8192);
        tma_load_4d(sm + dst + 0, &mk, 0, hh, cc * kChunk, bb, &bar_ld);
        tma_load_4d(sm + dst + 16384, &mk, 64, hh, cc * kChunk, bb, &bar_ld);
        tma_load_4d(sm + dst + 8192, &mq, 0, hh, cc * kChunk, bb, &bar_ld);
        tma_load_4d(sm + dst + 24576, &mq, 64, hh, cc * kChunk, bb, &bar_ld);
        pend_ld = true;
    };
    auto stage_gb = [&](int bb, int cc, int hv) {  // g, beta of a head's chunk into gst (threads < 64)
        if (tid < 64) {
            const int t = cc * kChunk + tid;
            const bool valid = t < P.T;
            const size_t bt = valid ? ((size_t)bb * P.T + t) * P.Hv + hv : 0;
            cp_async4(gst + tid, a.g + bt, valid);
            cp_async4(gst + 64 + tid, a.beta + bt, valid);
            cp_async_commit();
        }
    };
    // ---------------------------------------------------------------- persistent loop over tiles
    if ((int)blockIdx.x < nunits) {
        const int t = blockIdx.x / GU;
        stage_gb(t / (P.NC * P.Hk), t % P.NC, ((t / P.NC) % P.Hk) * G + (int)blockIdx.x % GU);
    }
    if (tid == 0 && (int)blockIdx.x < nunits) {
        const int t = blockIdx.x / GU;
        const int cc = t % P.NC, hh = (t / P.NC) % P.Hk, bb = t / (P.NC * P.Hk);
        issue_kq(bb, cc, hh, kq);
        for (int piece : {0, 6, 5, 1, 2, 3}) load_piece(bb, cc, hh * G + (int)blockIdx.x % GU, piece);  // first head
    }
    for (int unit = blockIdx.x; unit < nunits; unit += gridDim.x) {
    const int tile = unit / GU;
    c = tile % P.NC;
    hk = (tile / P.NC) % P.Hk;
    b = tile / (P.NC * P.Hk);
    t0 = c * kChunk;
    const int nunit = unit + (int)gridDim.x;  // the next unit of this CTA: its tile and first value head
    const int ntile = nunit / GU;
    const int nc = ntile % P.NC, nhk = (ntile / P.NC) % P.Hk, nb = ntile / (P.NC * P.Hk);
    const int nh0 = nhk * G + nunit % GU;
    const int hv_lo = hk * G + unit % GU, hv_hi = kSplit ? hv_lo + 1 : (hk + 1) * G;  // this unit's heads
    if (tid == 0 && nunit < nunits) {  // its k, q into L2 now: their copy into shared memory, issued at
        for (int h = 0; h < 2; h++) {  // this tile's end, is then served from L2
            tma_prefetch_4d(&mk, 64 * h, nhk, nc * kChunk, nb);
            tma_prefetch_4d(&mq, 64 * h, nhk, nc * kChunk, nb);
        }
    }
    if (!wait_ld(40)) goto teardown;
    {  // norm factors: 4 threads per row, 32 elements each
        const int row = tid >> 2, pp = tid & 3;
        float ss = 0.f;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            float x[8];
            ldrow8(kq, row, 4 * pp + q, 128, x);
#pragma unroll
            for (int e = 0; e < 8; e++) ss += x[e] * x[e];
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if (pp == 0) {
            const float f = P.use_norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
            if (row < 64) rk[row] = f; else rq[row - 64] = f;
        }
    }
    // G = K K^T into TMP1 (M=64, N=64)
    if (tid == 0) {
        tc_fence_after();
        for (int k0 = 0; k0 < kD; k0 += 16)
            mma(TM_T1, desc_kmajor(sb + kq, 128, 0, k0), desc_kmajor(sb + kq, 128, 0, k0), id64x64_kk, k0 > 0);
        mma_commit(&bar_mma);
    }
    if (!wait_mma(41)) goto teardown;
    {
        float v[16];
        tmem_ld16(tl + TM_T1 + c16, v);
        tmem_wait_ld();
        if (act) {
#pragma unroll
            for (int e = 0; e < 16; e++) GF[fsw(r, c16 + e)] = v[e];
        }
        float z[32];
#pragma unroll
        for (int e = 0; e < 32; e++) z[e] = 0.f;
        tmem_st32(tl + 64 * qt, z);  // zero dQ^ / dK^: 16 warps x 32 lanes x 64 columns
        tmem_st32(tl + 64 * qt + 32, z);
        tmem_wait_st();
    }
    sync_for_mma();

    for (int hv = hv_lo; hv < hv_hi; hv++) {
        const size_t bh = (size_t)b * P.Hv + hv;
        const size_t idx = bh * P.NC + c;
        const uint8_t* rec = a.rec + idx * REC_BYTES;
        // the next value head's inputs (the next tile's first head after the last one), fetched
        // piece by piece as their buffers free up
        const bool last_head = hv + 1 == hv_hi;
        const bool more = !last_head || nunit < nunits;
        auto prefetch = [&](int piece) {
            if (!last_head) load_piece(b, c, hv + 1, piece);
            else load_piece(nb, nc, nh0, piece);
        };
        if (tid < 64) {  // gates of this head, staged during the previous one (thread tid: token tid)
            cp_async_wait_all();
            float gv = gst[tid], bv = gst[64 + tid];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, gv, o);
                if (lane >= o) gv += y;
            }
            gam[tid] = gv;
            bet[tid] = bv;
            dgc[tid] = 0.f;
        }
        if (tid < 256) {
            dgp[tid] = 0.f;
            dbp[tid] = 0.f;
            sb3[tid] = 0.f;
        }
        __syncthreads();
        if (tid >= 32 && tid < 64) gam[tid] += gam[31];
        if (more) {  // the next head's gates into gst (read by the same threads above)
            if (!last_head) stage_gb(b, c, hv + 1);
            else stage_gb(nb, nc, nh0);
        }
        {
            bool okh = mbar_wait(&bar_h, h_phase, &abort_sh, a.status, 42);
            h_phase ^= 1;
            if (okh) pend_h = false;
            if (__syncthreads_or(!okh)) goto teardown;
        }
        const float gC = gam[63];

        // ------------------------------------------------------------ M1: W H0, dU
        if (tid == 0) {
            tc_fence_after();
            for (int k0 = 0; k0 < kD; k0 += 16)
                mma(TM_T1, desc_kmajor(sb + G_W, 64, 0, k0), desc_mnmajor(sb + G_H0, 128, 0, k0), id64x128_km,
                    k0 > 0);
            for (int k0 = 0; k0 < kChunk; k0 += 16)
                mma(TM_T2, desc_mnmajor(sb + G_P, 64, 0, k0), desc_mnmajor(sb + G_DO, 64, 0, k0), id64x128_mm,
                    k0 > 0);
            for (int k0 = 0; k0 < kD; k0 += 16)
                mma(TM_T2, desc_kmajor(sb + G_KB, 64, 0, k0), desc_mnmajor(sb + G_DH, 128, 0, k0), id64x128_km,
                    true);
            mma_commit(&bar_mma);
        }
        {  // <dH1, H0> over the two bf16 images (same layout, so elementwise)
            float s = 0.f;
#pragma unroll
            for (int i = tid; i < 2048; i += GRAD_THREADS) {
                float x[8], y[8];
                unpack8(ld_shared_v4(sb + G_H0 + i * 16), x);
                unpack8(ld_shared_v4(sb + G_DH + i * 16), y);
#pragma unroll
                for (int e = 0; e < 8; e++) s += x[e] * y[e];
            }
            s = warp_sum(s);
            if (lane == 0) red[warp] = s;
        }
        uint4 utv[2];  // this lane's half of U~ slice qt (columns c32 + 16 h ..), fetched while M1 runs
#pragma unroll
        for (int q = 0; q < 2; q++)
            utv[q] = *reinterpret_cast<const uint4*>(rec + REC_U + qt * 4096 + sw64_chunk(r, 2 * (lane >> 4) + q));
        if (!wait_mma(43)) goto teardown;
        if (tid == 0) {
            float s = 0.f;
            for (int w = 0; w < 16; w++) s += red[w];
            *hdh = s;
        }
        {  // U = U~ - W H0 -> U image (G_V);  dU -> dU image (G_KB)
            float x[32], w[16];
            const int q0 = 4 * qt + 2 * (lane >> 4);  // this lane's two 8-column chunks
            tmem_ld32(tl + TM_T1 + c32, x);
            tmem_wait_ld();
            split_cols<32>(x, w, lane);
#pragma unroll
            for (int q = 0; q < 2; q++) {
                float ut[8];
                unpack8(utv[q], ut);
#pragma unroll
                for (int e = 0; e < 8; e++) ut[e] -= w[8 * q + e];
                st_chunk(sb + G_V + sw128_chunk(r, q0 + q, 64), ut, 1.f);
            }
            tmem_ld32(tl + TM_T2 + c32, x);
            tmem_wait_ld();
            split_cols<32>(x, w, lane);
#pragma unroll
            for (int q = 0; q < 2; q++) st_chunk(sb + G_KB + sw128_chunk(r, q0 + q, 64), w + 8 * q, 1.f);
        }
        sync_for_mma();

        // ------------------------------------------------------------ M2: dP = dO U^T, X = dO H0^T
        if (tid == 0) {
            tc_fence_after();
            for (int k0 = 0; k0 < kD; k0 += 16) {
                mma(TM_T2, desc_kmajor(sb + G_DO, 64, 0, k0), desc_kmajor(sb + G_V, 64, 0, k0), id64x64_kk, k0 > 0);
                mma(TM_T1, desc_kmajor(sb + G_DO, 64, 0, k0), desc_kmajor(sb + G_H0, 128, 0, k0), id64x128_kk,
                    k0 > 0);
            }
            mma_commit(&bar_mma);
        }
        if (!wait_mma(44)) goto teardown;
        {
            const float gr = gam[r], Gr = expf(gr);
            {  // X: dgamma_r += scale Gamma_r rq_r sum_d Q_rd X_rd; dQ^ += scale Gamma_r X_r
                float x[32], dq[32];
                tmem_ld32(tl + TM_T1 + c32, x);
                tmem_ld32(tl + TM_DQ + c32, dq);
                tmem_wait_ld();
                const float f = P.scale * Gr;
                float dot = 0.f;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float qq[8];
                    ldrow8(kq, 64 + r, 4 * qt + q, 128, qq);
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        dot += qq[e] * x[8 * q + e];
                        dq[8 * q + e] += f * x[8 * q + e];
                    }
                }
                tmem_st32(tl + TM_DQ + c32, dq);
                if (act) dgp[qt * 64 + r] += f * rq[r] * dot;
            }
            {  // dP: Z = dP .* P, dS = scale E .* dP; dSk = dS diag(rk) (G_P), dSq = diag(rq) dS (G_DO)
                float v[16], w[8];
                tmem_ld16(tl + TM_T2 + c16, v);
                tmem_wait_ld();
                split_cols<16>(v, w, lane);
                const int jc = 2 * qt + (lane >> 4);  // this lane's 8-column chunk of the row
                float pr[8];
                ldrow8(G_P, r, jc, 64, pr);
                // gam, rk of the chunk's 8 columns before the first store (see the prep epilogues)
                const float4 ga0 = *reinterpret_cast<const float4*>(gam + 8 * jc);
                const float4 ga1 = *reinterpret_cast<const float4*>(gam + 8 * jc + 4);
                const float4 rk0 = *reinterpret_cast<const float4*>(rk + 8 * jc);
                const float4 rk1 = *reinterpret_cast<const float4*>(rk + 8 * jc + 4);
                const float gj[8] = {ga0.x, ga0.y, ga0.z, ga0.w, ga1.x, ga1.y, ga1.z, ga1.w};
                const float rkj[8] = {rk0.x, rk0.y, rk0.z, rk0.w, rk1.x, rk1.y, rk1.z, rk1.w};
                const float rqr = rq[r];
                float zs = 0.f;
                float sk[8], sq[8];
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int j = 8 * jc + e;
                    const float z = w[e] * pr[e];
                    zs += z;
                    ZS[fsw(r, j)] = z;
                    const float ds = (j <= r) ? P.scale * __expf(gr - gj[e]) * w[e] : 0.f;
                    sk[e] = ds * rkj[e];
                    sq[e] = ds * rqr;
                }
                zs += __shfl_xor_sync(0xffffffffu, zs, 16);
                if (act) dgp[qt * 64 + r] += zs;
                st_chunk(sb + G_P + sw128_chunk(r, jc, 64), sk, 1.f);
                st_chunk(sb + G_DO + sw128_chunk(r, jc, 64), sq, 1.f);
            }
            tmem_wait_st();
        }
        sync_for_mma();
        // ------------------------------------------------------------ M3
        if (tid == 0) {
            tc_fence_after();
            for (int k0 = 0; k0 < kChunk; k0 += 16) {
                // dQ^ += dSk K ;  dK^ += dSq^T Q
                mma(TM_DQ, desc_kmajor(sb + G_P, 64, 0, k0), desc_mnmajor(sb + kq, 128, 0, k0), id64x128_km, true);
                mma(TM_DK, desc_mnmajor(sb + G_DO, 64, 0, k0), desc_mnmajor(sb + kq, 128, 0, 64 + k0), id64x128_mm,
                    true);
            }
            for (int k0 = 0; k0 < kD; k0 += 16) {
                // Y = U dH1^T ;  dWn = dU H0^T
                mma(TM_T1, desc_kmajor(sb + G_V, 64, 0, k0), desc_kmajor(sb + G_DH, 128, 0, k0), id64x128_kk, k0 > 0);
                mma(TM_T2, desc_kmajor(sb + G_KB, 64, 0, k0), desc_kmajor(sb + G_H0, 128, 0, k0), id64x128_kk,
                    k0 > 0);
            }
            mma_commit(&bar_mma);
        }
        if (tid < 256) {  // column sums of Z (while M3 runs): dgamma_j -= sum_r Z_rj (4 threads per column)
            const int j = tid & 63, part4 = tid >> 6;
            float s = 0.f;
#pragma unroll
            for (int i = 16 * part4; i < 16 * part4 + 16; i++) s += ZS[fsw(i, j)];
            red[16 + tid] = s;
        }
        __syncthreads();
        if (tid < 64) dgc[tid] -= red[16 + tid] + red[80 + tid] + red[144 + tid] + red[208 + tid];
        if (!wait_mma(45)) goto teardown;
        if (tid == 0) {  // P and dO of the next head (their buffers are free after M3); v and U~ of this
            if (more) prefetch(0);  // head over the U image and dH1, which M3 was the last to read
            load_vu(b, c, hv);
        }
        {
            const float br = __expf(gC - gam[r]);
            {  // Y: db_r = rk_r sum_d K_rd Y_rd; dK^ += b_r Y_r
                float y[32], dk[32];
                tmem_ld32(tl + TM_T1 + c32, y);
                tmem_ld32(tl + TM_DK + c32, dk);
                tmem_wait_ld();
                float dot = 0.f;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float kk[8];
                    ldrow8(kq, r, 4 * qt + q, 128, kk);
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        dot += kk[e] * y[8 * q + e];
                        dk[8 * q + e] += br * y[8 * q + e];
                    }
                }
                tmem_st32(tl + TM_DK + c32, dk);
                if (act) sb3[qt * 64 + r] = br * rk[r] * dot;
            }
            {  // dW = -dWn -> dW image (G_H0)
                float x[32];
                tmem_ld32(tl + TM_T2 + c32, x);
                tmem_wait_ld();
                if (act) {
#pragma unroll
                    for (int q = 0; q < 4; q++) st_chunk(sb + G_H0 + sw128_chunk(r, 4 * qt + q, 64), x + 8 * q, -1.f);
                }
            }
            tmem_wait_st();
        }
        sync_for_mma();

        // ------------------------------------------------------------ M4: T^T dU, T^T dW
        {  // T of this head
            bool okh = mbar_wait(&bar_h2, h2_phase, &abort_sh, a.status, 50);
            h2_phase ^= 1;
            if (okh) pend_h2 = false;
            if (__syncthreads_or(!okh)) goto teardown;
        }
        if (tid == 0) {
            tc_fence_after();
            for (int k0 = 0; k0 < kChunk; k0 += 16) {
                mma(TM_T2, desc_mnmajor(sb + G_T, 64, 0, k0), desc_mnmajor(sb + G_KB, 64, 0, k0), id64x128_mm, k0 > 0);
                mma(TM_T1, desc_mnmajor(sb + G_T, 64, 0, k0), desc_mnmajor(sb + G_H0, 64, 0, k0), id64x128_mm, k0 > 0);
            }
            mma_commit(&bar_mma);
        }
        if (!wait_mma(46)) goto teardown;
        {  // v and U~ of this head
            bool okh = mbar_wait(&bar_h3, h3_phase, &abort_sh, a.status, 51);
            h3_phase ^= 1;
            if (okh) pend_h3 = false;
            if (__syncthreads_or(!okh)) goto teardown;
        }
        float dvv[16];  // this lane's 16 values of dv: stored once M5 is issued, because the proxy
                        // fence before M5 would otherwise wait for the global stores to complete
        {
            const int hf = lane >> 4;  // this lane's columns of T^T dU: c32 + 8 q + 4 hf + 0..3
            {  // T^T dU: dv = beta T^T dU; dbeta_r += sum_v V_rv (T^T dU)_rv; its image over dU (G_KB)
                float x[32], w[16];
                tmem_ld32(tl + TM_T2 + c32, x);
                tmem_wait_ld();
                split_cols_sector(x, w, lane);
                float dot = 0.f;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float vv[8];
                    ldrow8(G_V, r, 4 * qt + q, 64, vv);
#pragma unroll
                    for (int i = 0; i < 4; i++) dot += (hf ? vv[4 + i] : vv[i]) * w[4 * q + i];
                    const uint32_t addr = sb + G_KB + sw128_chunk(r, 4 * qt + q, 64) + 8 * hf;
                    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr),
                                 "r"(pack_bf16(w[4 * q], w[4 * q + 1])), "r"(pack_bf16(w[4 * q + 2], w[4 * q + 3]))
                                 : "memory");
                }
                dot += __shfl_xor_sync(0xffffffffu, dot, 16);
                if (act) dbp[qt * 64 + r] += dot;
                const float bb = bet[r];
#pragma unroll
                for (int e = 0; e < 16; e++) dvv[e] = bb * w[e];
            }
            {  // T^T dW: dK^ += beta Gamma (T^T dW); dbeta, dgamma from k^ . (T^T dW); its image over dW (G_H0)
                float x[32], dk[32];
                tmem_ld32(tl + TM_T1 + c32, x);
                tmem_ld32(tl + TM_DK + c32, dk);
                tmem_wait_ld();
                const float Gr = __expf(gam[r]), bgr = bet[r] * Gr;
                float dot = 0.f;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float kk[8];
                    ldrow8(kq, r, 4 * qt + q, 128, kk);
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        dot += kk[e] * x[8 * q + e];
                        dk[8 * q + e] += bgr * x[8 * q + e];
                    }
                }
                tmem_st32(tl + TM_DK + c32, dk);
                if (act) {
                    dbp[qt * 64 + r] += Gr * rk[r] * dot;
                    dgp[qt * 64 + r] += bgr * rk[r] * dot;
#pragma unroll
                    for (int q = 0; q < 4; q++) st_chunk(sb + G_H0 + sw128_chunk(r, 4 * qt + q, 64), x + 8 * q, 1.f);
                }
            }
            tmem_wait_st();
        }
        sync_for_mma();

        // ------------------------------------------------------------ M5: T^T dT T^T = (T^T dU) U~^T + (T^T dW) W^T
        if (tid == 0) {
            tc_fence_after();
            for (int k0 = 0; k0 < kD; k0 += 16)
                mma(TM_T1, desc_kmajor(sb + G_KB, 64, 0, k0), desc_kmajor_sw64(sb + G_DH, 64, k0), id64x64_kk, k0 > 0);
            for (int k0 = 0; k0 < kD; k0 += 16)
                mma(TM_T1, desc_kmajor(sb + G_H0, 64, 0, k0), desc_kmajor(sb + G_W, 64, 0, k0), id64x64_kk, true);
            mma_commit(&bar_mma);
        }
        store_rows(a.dv + (((size_t)b * P.T + t0) * P.Hv + hv) * kD + c32, (size_t)P.Hv * kD, dvv);  // dv
        if (!wait_mma(48)) goto teardown;
        if (more && tid == 0) {  // W, dH1, Kbar and H0 of the next head: M5 was the last to read their buffers
            prefetch(6);
            prefetch(5);
            prefetch(1);
            if (kSplit || !last_head) prefetch(2);  // else H0's buffer first stages the tile's dk
        }

        {  // dA = strict_lower(-T^T dT T^T); terms of A_rj = beta_r rk_r rk_j E_rj G_rj
            float v[16], w[8];
            tmem_ld16(tl + TM_T1 + c16, v);
            tmem_wait_ld();
            split_cols<16>(v, w, lane);
            {
                const int jc = 2 * qt + (lane >> 4);
                const float gr = gam[r], br = bet[r], rkr = rk[r];
                // every shared-memory input of the 8 columns before the first store
                const float4 ga0 = *reinterpret_cast<const float4*>(gam + 8 * jc);
                const float4 ga1 = *reinterpret_cast<const float4*>(gam + 8 * jc + 4);
                const float4 rk0 = *reinterpret_cast<const float4*>(rk + 8 * jc);
                const float4 rk1 = *reinterpret_cast<const float4*>(rk + 8 * jc + 4);
                const float gj[8] = {ga0.x, ga0.y, ga0.z, ga0.w, ga1.x, ga1.y, ga1.z, ga1.w};
                const float rkj[8] = {rk0.x, rk0.y, rk0.z, rk0.w, rk1.x, rk1.y, rk1.z, rk1.w};
                float gf[8];
#pragma unroll
                for (int e = 0; e < 8; e++) gf[e] = GF[fsw(r, 8 * jc + e)];
                float db = 0.f, zs = 0.f;
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int j = 8 * jc + e;
                    float m = 0.f, z = 0.f;
                    if (j < r) {
                        const float dA = -w[e];
                        const float E = __expf(gr - gj[e]);
                        const float kk = rkr * rkj[e] * gf[e];
                        db += dA * E * kk;
                        z = dA * br * E * kk;
                        m = dA * br * E;
                    }
                    zs += z;
                    ZS[fsw(r, j)] = z;
                    MF[fsw(r, j)] = m;
                }
                db += __shfl_xor_sync(0xffffffffu, db, 16);
                zs += __shfl_xor_sync(0xffffffffu, zs, 16);
                if (act) {
                    dbp[qt * 64 + r] += db;
                    dgp[qt * 64 + r] += zs;
                }
            }
        }
        __syncthreads();
        {  // N_rj = rk_j (M_rj + M_jr) -> image (G_T: T is no longer read); 8 columns per lane
            const int jc = 2 * qt + (lane >> 4);
            float nrow[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const int j = 8 * jc + e;
                nrow[e] = rk[j] * (MF[fsw(r, j)] + MF[fsw(j, r)]);
            }
            st_chunk(sb + G_T + sw128_chunk(r, jc, 64), nrow, 1.f);
        }
        sync_for_mma();

        // ------------------------------------------------------------ M6: dK^ += N K
        if (tid == 0) {
            tc_fence_after();
            for (int k0 = 0; k0 < kChunk; k0 += 16)
                mma(TM_DK, desc_kmajor(sb + G_T, 64, 0, k0), desc_mnmajor(sb + kq, 128, 0, k0), id64x128_km,
                    true);
            mma_commit(&bar_mma);
        }
        if (tid < 256) {  // column sums of dA-Z (while M6 runs)
            const int j = tid & 63, part4 = tid >> 6;
            float s = 0.f;
#pragma unroll
            for (int i = 16 * part4; i < 16 * part4 + 16; i++) s += ZS[fsw(i, j)];
            red[16 + tid] = s;
        }
        __syncthreads();
        // per-head scalars: dgamma -> dg (reverse cumsum within the chunk), dbeta
        if (tid < 64) {  // two warps; row r = tid
            float s3 = 0.f, dgr = dgc[tid] - (red[16 + tid] + red[80 + tid] + red[144 + tid] + red[208 + tid]);
#pragma unroll
            for (int k = 0; k < 4; k++) {
                s3 += sb3[k * 64 + tid];
                dgr += dgp[k * 64 + tid];
            }
            dgr -= s3;
            const float tot3 = warp_sum(s3);  // per warp; the two halves meet through red[]
            if (lane == 0) red[warp] = tot3;
            // suffix sum within the warp
            float suf = dgr;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += y;
            }
            ZS[tid] = suf;
        }
        __syncthreads();
        if (tid < 64) {
            // rows 0-31 also get the suffix of rows 32-63; every row gets the gamma_C terms
            // (they sit on the last row, which every suffix includes)
            const float last = red[0] + red[1] + expf(gC) * (*hdh);  // sum b db + Gamma_C <dH1,H0>
            float s = ZS[tid] + last + (tid < 32 ? ZS[32] : 0.f);
            if (t0 + tid < P.T) {
                const size_t bt = ((size_t)b * P.T + t0 + tid) * P.Hv + hv;
                a.dg[bt] = s;
                a.dbeta[bt] = dbp[tid] + dbp[64 + tid] + dbp[128 + tid] + dbp[192 + tid];
            }
        }
        if (!wait_mma(49)) goto teardown;
        if (more && tid == 0) prefetch(3);  // T: its buffer held N, read by M6
        if (last_head && tid == 0 && nunit < nunits) issue_kq(nb, nc, nhk, gfz);  // GF / ZS are free now
    }

    // ---------------------------------------------------------------- dq, dk: norm backward
    if (kSplit) {  // this value head's dq^, dk^ as they are (summed and normalised by the next kernel)
        float x[32], w[16];
#pragma unroll 1
        for (int which = 0; which < 2; which++) {
            tmem_ld32(tl + (which == 0 ? TM_DQ : TM_DK) + c32, x);
            tmem_wait_ld();
            split_cols_sector(x, w, lane);
            store_rows((which == 0 ? a.dqh : a.dkh) + (((size_t)b * P.T + t0) * P.Hv + hv_lo) * kD + c32,
                       (size_t)P.Hv * kD, w);
        }
        tc_fence_before();
        __syncthreads();
    } else {  // row r, columns c32 + 8 q + 4 hf + 0..3 (q < 4)
        // dq = rq (dq^ - rq^2 (q . dq^) q), dk likewise, leave by tensor-map stores of four [64 x 32]
        // fp32 boxes each (128-byte swizzle), staged over k/q (dq) and H0's buffer (dk), so no warp
        // waits on its global stores. H0 of the next tile's first head is copied in once they are read.
        const int hf = lane >> 4;
        float w[2][16];
#pragma unroll
        for (int which = 0; which < 2; which++) {  // 0: q, 1: k
            float x[32];
            tmem_ld32(tl + (which == 0 ? TM_DQ : TM_DK) + c32, x);
            tmem_wait_ld();
            split_cols_sector(x, w[which], lane);
            const int krow = which == 0 ? 64 + r : r;
            float dot = 0.f;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                float x8[8];
                ldrow8(kq, krow, 4 * qt + q, 128, x8);
#pragma unroll
                for (int i = 0; i < 4; i++) dot += (hf ? x8[4 + i] : x8[i]) * w[which][4 * q + i];
            }
            dot += __shfl_xor_sync(0xffffffffu, dot, 16);
            if (act) (which == 0 ? part : red + 16)[qt * 64 + r] = dot;
        }
        tc_fence_before();
        __syncthreads();
#pragma unroll
        for (int which = 0; which < 2; which++) {
            const float* pw = which == 0 ? part : red + 16;
            const float rr = (which == 0 ? rq : rk)[r];
            const float full = pw[r] + pw[64 + r] + pw[128 + r] + pw[192 + r];
            const int krow = which == 0 ? 64 + r : r;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                float x8[8];
                ldrow8(kq, krow, 4 * qt + q, 128, x8);
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const float xv = hf ? x8[4 + i] : x8[i];
                    float& o = w[which][4 * q + i];
                    if (P.use_norm) o = rr * (o - rr * xv * rr * full);
                }
            }
        }
        __syncthreads();  // k/q read: its region and H0's buffer take the staging
#pragma unroll
        for (int which = 0; which < 2; which++) {
            uint8_t* box = sm + (which == 0 ? kq : G_H0) + qt * 8192;
#pragma unroll
            for (int q = 0; q < 4; q++)
                *reinterpret_cast<float4*>(box + sw128_chunk(r, 2 * q + hf, 64)) =
                    make_float4(w[which][4 * q], w[which][4 * q + 1], w[which][4 * q + 2], w[which][4 * q + 3]);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            for (int qq = 0; qq < 4; qq++) {
                tma_store_4d(&mdq, sm + kq + qq * 8192, 32 * qq, hk, t0, b);
                tma_store_4d(&mdk, sm + G_H0 + qq * 8192, 32 * qq, hk, t0, b);
            }
            bulk_commit();
            bulk_wait_read_all();  // the staging is read: both regions may be rewritten
            if (nunit < nunits) load_piece(nb, nc, nh0, 2);
        }
    }
    {  // swap the k/q and scratch regions for the next tile
        const uint32_t t = kq;
        kq = gfz;
        gfz = t;
        GF = reinterpret_cast<float*>(sm + gfz);
        ZS = reinterpret_cast<float*>(sm + gfz + 16384);
    }
    }  // units

teardown:
    cp_async_wait_all();  // staged gates still in flight
    if (tid == 0) bulk_wait_all();  // dq, dk stores
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0) {  // let copies still in flight land before the CTA exits
        volatile int never = 0;
        if (pend_ld) mbar_wait(&bar_ld, ld_phase, &never, nullptr, 0);
        if (h_open) {  // pieces in flight without their arrival: arrive, so the phase ends when they land
            mbar_arrive(&bar_h);
            pend_h = true;
        }
        if (h2_open) {
            mbar_arrive(&bar_h2);
            pend_h2 = true;
        }
        if (pend_h) mbar_wait(&bar_h, h_phase, &never, nullptr, 0);
        if (pend_h2) mbar_wait(&bar_h2, h2_phase, &never, nullptr, 0);
        if (pend_h3) mbar_wait(&bar_h3, h3_phase, &never, nullptr, 0);
        mbar_wait(&bar_mma, mma_phase, &never, nullptr, 0);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

cudaError_t launch_chunk_bwd(const ChunkBwdArgs& a, cudaStream_t s) {
    const ChunkProblem& p = a.p;
    const bool saved = a.states != nullptr;
    const uint8_t* keep = static_cast<const uint8_t*>(a.saved);
    const WsLayout w = ws_layout(p, true, saved);
    const SavedLayout l = saved_layout(p);
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    CUtensorMap mq, mk, mv, mdo32, mdo64;
    if (!make_qkv_maps(p, a.q, a.k, a.v, &mq, &mk, &mv)) return cudaErrorInvalidValue;
    if (!make_map_4d_bf16(&mdo32, a.do_, kD, p.Hv, p.T, p.B, 32, kChunk, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_4d_bf16(&mdo64, a.do_, kD, p.Hv, p.T, p.B, 64, kChunk, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    int* status = reinterpret_cast<int*>(ws);
    cudaError_t e = cudaSuccess;
    PrepArgs pa;
    pa.p = p;
    pa.g = a.g;
    pa.beta = a.beta;
    pa.status = status;
    if (keep) {  // the forward kept its operators: no prep, no forward scan
        pa.gam = reinterpret_cast<float*>(const_cast<uint8_t*>(keep + l.gam));
        pa.rec = const_cast<uint8_t*>(keep + l.rec);
        pa.rec2 = const_cast<uint8_t*>(keep + l.rec2);
        pa.ncpad = l.ncpad;
    } else {
        pa.gam = reinterpret_cast<float*>(ws + w.gam);
        pa.rec = ws + w.rec;
        pa.rec2 = ws + w.rec2;
        pa.ncpad = w.ncpad;
        if ((e = p.channel ? launch_prep_ch(pa, mq, mk, mv, s) : launch_prep(pa, mq, mk, mv, s)) != cudaSuccess)
            return e;
    }
    const SavedBwdLayout sl = saved_bwd_layout(p);
    uint8_t* dhs = keep ? ws + sl.dhs : ws + w.dhs;
    ScanArgs sa;
    sa.p = p;
    sa.gam = pa.gam;
    sa.rec = pa.rec;
    sa.hinit = a.h0;
    sa.o = nullptr;
    sa.hfinal = nullptr;
    sa.states = ws + w.hs;
    sa.status = status;
    sa.ncpad = pa.ncpad;
    const uint8_t* hs = keep ? keep + l.hs : saved ? static_cast<const uint8_t*>(a.states) : ws + w.hs;
    if (!keep && !saved && (e = launch_scan(sa, SCAN_FWD_STATES, nullptr, s)) != cudaSuccess) return e;
    sa.hinit = a.dht;
    sa.hfinal = a.dh0;
    sa.states = dhs;
    if ((e = launch_scan(sa, SCAN_BWD, &mdo32, s)) != cudaSuccess) return e;
    if (p.channel) {
        GradChArgs ca;
        ca.p = p;
        ca.q = a.q;
        ca.k = a.k;
        ca.g = a.g;
        ca.beta = a.beta;
        ca.rec = pa.rec;
        ca.rec2 = pa.rec2;
        ca.hs = hs;
        ca.dhs = dhs;
        ca.chx = ws + (keep ? sl.chx : w.chx);
        ca.dqh = reinterpret_cast<float*>(ws + (keep ? sl.dqh : w.dqh));
        ca.dkh = reinterpret_cast<float*>(ws + (keep ? sl.dkh : w.dkh));
        ca.dq = a.dq;
        ca.dk = a.dk;
        ca.dv = a.dv;
        ca.dg = a.dg;
        ca.dbeta = a.dbeta;
        ca.status = status;
        return launch_grad_ch(ca, mv, mdo64, s);
    }
    GradArgs ga;
    ga.p = p;
    ga.g = a.g;
    ga.beta = a.beta;
    ga.rec = pa.rec;
    ga.rec2 = pa.rec2;
    ga.hs = hs;
    ga.dhs = dhs;
    ga.gam = pa.gam;
    ga.dq = a.dq;
    ga.dk = a.dk;
    ga.dv = a.dv;
    ga.dg = a.dg;
    ga.dbeta = a.dbeta;
    ga.status = status;
    const bool split = grad_split(p);
    ga.dqh = split ? reinterpret_cast<float*>(ws + (keep ? sl.dqh : w.dqh)) : nullptr;
    ga.dkh = split ? reinterpret_cast<float*>(ws + (keep ? sl.dkh : w.dkh)) : nullptr;
    const int smem = G_BYTES + 1024;
    if ((e = cudaFuncSetAttribute(grad_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(grad_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
            cudaSuccess)
        return e;
    static int nsm = 0;  // one 222 KB CTA per SM: a persistent grid of one per SM
    if (nsm == 0) {
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    }
    const int nunits = p.B * p.Hk * p.NC * (split ? p.Hv / p.Hk : 1);
    dim3 grid(nunits < nsm ? nunits : nsm);
    CUtensorMap mdq, mdk;  // fp32 [B][T][Hk][Dk] stores of [64 x 32] boxes
    if (!make_map_4d(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dq, kD, p.Hk, p.T, p.B, 32, kChunk,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_4d(&mdk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dk, kD, p.Hk, p.T, p.B, 32, kChunk,
                     CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    trace_begin("chunk_grad", s);
    if (split)
        grad_kernel<true><<<grid, GRAD_THREADS, smem, s>>>(mq, mk, mv, mdo64, mdq, mdk, ga);
    else
        grad_kernel<false><<<grid, GRAD_THREADS, smem, s>>>(mq, mk, mv, mdo64, mdq, mdk, ga);
    trace_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess || !split) return e;
    // the value-head sum and the norm backward of the split gradient
    SeqBwdArgs f{};
    f.B = p.B; f.T = p.T; f.Hk = p.Hk; f.Hv = p.Hv; f.Dk = kD; f.Dv = kD;
    f.use_norm = p.use_norm;
    f.bf16 = 1;
    f.q = a.q; f.k = a.k;
    f.dq = a.dq; f.dk = a.dk;
    f.dqh = ga.dqh; f.dkh = ga.dkh;
    return launch_qk_norm_backward(f, s);
}

}  // namespace gdr
