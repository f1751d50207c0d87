// chunk_fwd.cu - tensor-core chunked gated delta rule (chunks of 64 tokens, Dk = Dv = 128):
//   prep_kernel : persistent, two CTAs per SM; a CTA takes (b, key head, chunk) groups in
//                 turn and, for each, the value heads sharing that key head one after the
//                 other (k, q and their norms loaded once per group; the next head's v is
//                 fetched while the current head finishes). When there are too few groups to
//                 give every SM a CTA, each value head is a unit of its own (prep_kernel<true>). Builds each chunk's operators
//                 (UT/WY transform of the k k^T beta block, output and state operators) on
//                 tcgen05 with TMEM accumulators and writes them as ready-to-use
//                 shared-memory images.
// The chunk-to-chunk scans that consume these operators are in scan.cu.
// The algebra is stated in chunk.h. The chunked prefill and its backward are the
// "chunked case" of "Adding VJP for gated delta net" (MLX PR #4565); the q/k L2 norm is
// applied inside ("fold q/k L2-norm into the gated_delta_rule kernel", eps 1e-6) as an
// fp32 factor on the raw bf16 operands, so normalised q/k are never rounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "chunk.h"
#include "chunk_dev.cuh"
#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace gdr {

// ================================================================== prep kernel
// Shared memory (offsets from a 1024-aligned base), ~97 KB so two CTAs share an SM:
// the record images go straight from registers to global memory, nothing is staged.
constexpr uint32_t PS_KQ = 0;        // k rows 0-63 / q rows 64-127 of a 128-row tile (panels 16 KB)
constexpr uint32_t PS_V = 32768;     // v [64 tok x 128] (panels 8 KB)
constexpr uint32_t PS_A = 49152;     // A fp32 [64][LDA]; then [Tw; Tu] 128 x 64 bf16; then Wbar image
constexpr uint32_t PS_T = 66560;     // T fp32 [64][LDA]; then W image [64 x 128]
constexpr uint32_t PS_P = 83968;     // P image [64 x 64]
constexpr uint32_t PS_SCR = 92160;   // solve scratch: Y_IK blocks [6][16][LDY] fp32
constexpr uint32_t PS_SMALL = PS_SCR + SOLVE_SCRATCH_BYTES;  // per-token factors (8 x 64 fp32)
constexpr uint32_t PS_GST = PS_SMALL + 2048;  // next value head's gates g, beta (2 x 64 fp32), cp.async
constexpr uint32_t PS_BYTES = PS_GST + 512;
constexpr uint32_t PS_TT = PS_A, PS_WBAR = PS_A, PS_W = PS_T;
// After the last products of a value head, A, T, P and the solve scratch are dead: the Mneg and Qc
// images are staged there and leave by two bulk copies (a thread's 16-byte stores into the record
// would touch one 128-byte line each).
constexpr uint32_t PS_STAGE = PS_A, PS_STAGE_Q = PS_STAGE + 32768;
// The intra-chunk decays E_ij = exp(gamma_i - gamma_j) (j <= i) of A and P, kept in the solve scratch
// until the solve: inside the 16 x 16 diagonal blocks directly, ED [4][16][EDS] fp32; below them
// factored through the start s = 16 (i / 16) of row i's block, E_ij = exp(gamma_i - gamma_s) x
// exp(gamma_s - gamma_j), both factors at most 1 for a decay (EA [64] and EB [4][64] fp32). This
// takes 1024 + 160 exponentials per value head instead of 8192.
constexpr int EDS = 20;  // row stride (floats): 16-byte rows, conflict-free float4 reads
constexpr uint32_t PS_ED = PS_SCR, PS_EA = PS_ED + 4 * 16 * EDS * 4, PS_EB = PS_EA + 64 * 4;
static_assert(PS_EB + 4 * 64 * 4 <= PS_SCR + SOLVE_SCRATCH_BYTES, "decay tables in the solve scratch");
static_assert(PS_STAGE_Q + 16384 <= PS_SMALL, "staging below the small arrays");
static_assert(PS_A % 1024 == 0 && PS_T % 1024 == 0 && PS_P % 1024 == 0, "align");
static_assert(PS_A + 64 * LDA * 4 <= PS_T && PS_T + 64 * LDA * 4 <= PS_P, "fp32 tiles");
static_assert(2 * (PS_BYTES + 1024) <= 228 * 1024, "two prep CTAs per SM");

template <bool kSplit>
__global__ void __launch_bounds__(256, 2)
    prep_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                const __grid_constant__ CUtensorMap mv, PrepArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t bar_kq, bar_v, bar_mma;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkProblem& P = a.p;
    const int G = P.Hv / P.Hk;
    const int ngroups = P.B * P.Hk * P.NC;  // (b, key head, chunk); its G value heads run in turn
    // A work unit is a group's value heads, or (kSplit, when the groups alone would leave SMs idle)
    // one of them, each unit then loading the group's k and q itself.
    const int parts = kSplit ? G : 1, hpp = kSplit ? 1 : G, nunits = ngroups * parts;
    float* gam = reinterpret_cast<float*>(sm + PS_SMALL);  // in-chunk cumulative log-decay
    float* bet = gam + 64;
    float* rho = bet + 64;   // [128] rows 0-63: k norm factors, 64-127: q norm factors
    float* fw = rho + 128;   // beta Gamma rho_k     (columns of Tw)
    float* fb = fw + 64;     // exp(gamma_C - gamma) rho_k   (rows of Kbar, Wbar)
    float* fq = fb + 64;     // scale Gamma rho_q     (rows of Qc)
    float* gst = reinterpret_cast<float*>(sm + PS_GST);
    float* ed = reinterpret_cast<float*>(sm + PS_ED);
    float* ea = reinterpret_cast<float*>(sm + PS_EA);
    float* eb = reinterpret_cast<float*>(sm + PS_EB);
    float* Am = reinterpret_cast<float*>(sm + PS_A);
    float* Tm = reinterpret_cast<float*>(sm + PS_T);
    float* Xs = reinterpret_cast<float*>(sm + PS_SCR);
    uint32_t kq_ph = 0, v_ph = 0, mph = 0;  // mbarrier phases
    bool kq_pend = false, v_pend = false;   // copies issued and not yet waited for (thread 0)
    bool ok = true;
    // group g -> (b, hk, c); value head hv = hk * G + hh
    auto issue_kq = [&](int g) {
        const int c = g % P.NC, hk = (g / P.NC) % P.Hk, b = g / (P.NC * P.Hk);
        mbar_expect_tx(&bar_kq, 4 * 8192);
        tma_load_4d(sm + PS_KQ + 0, &mk, 0, hk, c * kChunk, b, &bar_kq);
        tma_load_4d(sm + PS_KQ + 16384, &mk, 64, hk, c * kChunk, b, &bar_kq);
        tma_load_4d(sm + PS_KQ + 8192, &mq, 0, hk, c * kChunk, b, &bar_kq);
        tma_load_4d(sm + PS_KQ + 24576, &mq, 64, hk, c * kChunk, b, &bar_kq);
        kq_pend = true;
    };
    auto issue_v = [&](int g, int hh) {
        const int c = g % P.NC, hk = (g / P.NC) % P.Hk, b = g / (P.NC * P.Hk);
        mbar_expect_tx(&bar_v, 2 * 8192);
        tma_load_4d(sm + PS_V + 0, &mv, 0, hk * G + hh, c * kChunk, b, &bar_v);
        tma_load_4d(sm + PS_V + 8192, &mv, 64, hk * G + hh, c * kChunk, b, &bar_v);
        v_pend = true;
    };
    // threads 0-63 stage token tid's g and beta of (group g, value head hh); each thread later
    // reads only the slots it staged itself. Tokens past T are zero-filled (g = 0, beta = 0).
    auto stage_gb = [&](int g, int hh) {
        const int c = g % P.NC, hk = (g / P.NC) % P.Hk, b = g / (P.NC * P.Hk);
        const int t = c * kChunk + tid;
        const bool in = t < P.T;
        const size_t bt = in ? ((size_t)b * P.T + t) * P.Hv + hk * G + hh : 0;
        cp_async4(gst + tid, a.g + bt, in);
        cp_async4(gst + 64 + tid, a.beta + bt, in);
        cp_async_commit();
    };

    if (tid < 64 && (int)blockIdx.x < nunits) stage_gb(blockIdx.x / parts, (blockIdx.x % parts) * hpp);
    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_kq, 1);
        mbar_init(&bar_v, 1);
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
    if (tid == 0 && (int)blockIdx.x < nunits) {
        issue_kq(blockIdx.x / parts);
        issue_v(blockIdx.x / parts, (blockIdx.x % parts) * hpp);
    }

    for (int unit = blockIdx.x; unit < nunits; unit += gridDim.x) {
        const int grp = unit / parts, hb = (unit % parts) * hpp, he = hb + hpp;  // heads hb .. he - 1
        const int c = grp % P.NC, hk = (grp / P.NC) % P.Hk, b = grp / (P.NC * P.Hk);
        const int nunit = unit + (int)gridDim.x;  // this CTA's next unit: its group and first head
        const int next = nunit < nunits ? nunit / parts : ngroups, nh0 = (nunit % parts) * hpp;
        ok = mbar_wait(&bar_kq, kq_ph, &abort_sh, a.status, 10);
        kq_ph ^= 1;
        if (tid == 0) kq_pend = false;
        if (__syncthreads_or(!ok)) goto teardown;

        for (int hh = hb; hh < he; hh++) {
            const int hv = hk * G + hh;
            const size_t bh = (size_t)b * P.Hv + hv;
            uint8_t* rec = a.rec + (bh * P.NC + c) * REC_BYTES;
            uint8_t* rec2 = a.rec2 ? a.rec2 + (bh * P.NC + c) * REC2_BYTES : nullptr;

            // G = K K^T (rows 0-63) and Q K^T (rows 64-127) in one M=128 product on the raw bf16
            // operands; the norm factors are applied in the epilogue, so they are computed meanwhile
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, 0, 0);
                for (int k0 = 0; k0 < kD; k0 += 16)
                    mma_bf16(tm, desc_kmajor(sb + PS_KQ, 128, 0, k0), desc_kmajor(sb + PS_KQ, 128, 0, k0), id, k0 > 0);
                mma_commit(&bar_mma);
            }
            // gates of the chunk; tokens past T act as g = 0, beta = 0 (state passes unchanged)
            if (tid < 64) {
                cp_async_wait_all();
                float gv = gst[tid];
                const float bv = gst[64 + tid];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, gv, o);
                    if (lane >= o) gv += y;
                }
                gam[tid] = gv;
                bet[tid] = bv;
            }
            if (hh == hb) {  // L2 norm factors of the 64 keys (rows 0-63) and 64 queries (rows 64-127)
                const int row = tid >> 1, half = tid & 1;
                const uint32_t base = sb + PS_KQ + half * 16384 + row * 128;
                float ss = 0.f;
#pragma unroll
                for (int ch = 0; ch < 8; ch++) {  // physical chunk order rotated per thread: a quarter warp
                    float x[8];                   // (4 rows x 2 halves) then reads 8 distinct bank groups
                    unpack8(ld_shared_v4(base + ((ch + 2 * row + half) & 7) * 16), x);
#pragma unroll
                    for (int e = 0; e < 8; e++) ss += x[e] * x[e];
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (half == 0) rho[row] = P.use_norm ? 1.0f / sqrtf(ss + 1e-6f) : 1.0f;
            }
            if (tid == 0) bulk_wait_read_all();  // the previous head's staged images are read (the decay
            __syncthreads();                     // tables below and A / P are written over them)
            if (tid >= 32 && tid < 64) gam[tid] += gam[31];
            __syncthreads();
            if (tid < 64) {
                const float G = expf(gam[tid]);
                fw[tid] = bet[tid] * G * rho[tid];
                fb[tid] = expf(gam[63] - gam[tid]) * rho[tid];
                fq[tid] = P.scale * G * rho[64 + tid];
                ea[tid] = __expf(gam[tid] - gam[tid & ~15]);
            } else if (tid < 160) {  // exp(gamma_s - gamma_j), block starts s = 16, 32, 48 and j < s
                const int u = tid - 64;
                const int kb = u < 16 ? 1 : u < 48 ? 2 : 3, jj = u < 16 ? u : u < 48 ? u - 16 : u - 48;
                eb[kb * 64 + jj] = __expf(gam[16 * kb] - gam[jj]);
            }
#pragma unroll
            for (int e = 0; e < 4; e++) {  // diagonal blocks: entry (block, r, c) = exp(gamma_r - gamma_c), c <= r
                const int idx = tid + 256 * e, bk = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
                ed[(bk * 16 + r) * EDS + cc] = cc <= r ? __expf(gam[16 * bk + r] - gam[16 * bk + cc]) : 0.f;
            }

            ok = mbar_wait(&bar_mma, mph, &abort_sh, a.status, 11);
            mph ^= 1;
            if (__syncthreads_or(!ok)) goto teardown;
            tc_fence_after();
            {  // A = strict_lower(beta_i rho_i rho_j E_ij G_ij) in fp32;  P = scale tril(rho rho E S) in bf16
                const int lg = warp & 3, h = warp >> 2;
                const int r = 32 * lg + lane;
                float v[32];
                tmem_ld32(tmem_at(tm, 32 * lg, 32 * h), v);
                tmem_wait_ld();
                // All loads first, then all stores: stores into the same shared memory in between
                // would keep the compiler from overlapping the loads (it cannot rule out aliasing).
                const bool arow = r < 64;  // warp-uniform
                const int i = r & 63;
                const int lim = arow ? i : i + 1;  // A: j < i (strict), P: j <= i
                const int bi = i >> 4;
                const float ai = ea[i], ci = arow ? bet[i] * rho[i] : P.scale * rho[64 + i];
                const float4* r4 = reinterpret_cast<const float4*>(rho + 32 * h);
                const float4* b4 = reinterpret_cast<const float4*>(eb + bi * 64 + 32 * h);
                const float4* d4 = reinterpret_cast<const float4*>(ed + (bi * 16 + (i & 15)) * EDS);
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    const int j0 = 32 * h + 4 * q, bj = j0 >> 4;  // the 4 columns share a block
                    const float4 rr = r4[q];
                    float4 ee = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (bj < bi) {
                        const float4 bb = b4[q];
                        ee = make_float4(ai * bb.x, ai * bb.y, ai * bb.z, ai * bb.w);
                    } else if (bj == bi) {
                        ee = d4[(j0 & 15) >> 2];
                    }
                    const float rj[4] = {rr.x, rr.y, rr.z, rr.w}, ej[4] = {ee.x, ee.y, ee.z, ee.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int jj = 4 * q + e;
                        v[jj] = (32 * h + jj < lim) ? ci * rj[e] * ej[e] * v[jj] : 0.f;
                    }
                }
                if (arow) {
#pragma unroll
                    for (int q = 0; q < 8; q++)
                        *reinterpret_cast<float4*>(Am + i * LDA + 32 * h + 4 * q) =
                            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const uint4 u = pack8(v + 8 * q, 1.f);
                        const uint32_t off = sw128_chunk(i, 4 * h + q, 64);
                        st_shared_v4(sb + PS_P + off, u.x, u.y, u.z, u.w);
                    }
                    fence_proxy_async_smem();  // the P image leaves by a bulk copy
                }
            }
            tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                bulk_store(rec + REC_P, sm + PS_P, 8192);
                bulk_commit();
            }

            ut_solve(Am, Tm, Xs, tid);  // T = (I + A)^-1
            {  // [Tw; Tu] with Tw = T diag(beta Gamma rho_k), Tu = T diag(beta): K-major A operand (over A).
               // T's blocks above the block diagonal are zero and never stored: masked here.
                const int row = tid >> 1, half = tid & 1;
                const int i = row & 63;
                const bool isw = row < 64;
                const float* trow = Tm + i * LDA + 32 * half;
                const float* fac = (isw ? fw : bet) + 32 * half;
                float t[32], x[32];
#pragma unroll
                for (int q = 0; q < 8; q++) {  // all loads first (see the A/P epilogue)
                    const float4 f = *reinterpret_cast<const float4*>(trow + 4 * q);
                    const float4 w = *reinterpret_cast<const float4*>(fac + 4 * q);
                    const float tv[4] = {f.x, f.y, f.z, f.w}, wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int j = 32 * half + 4 * q + e;
                        t[4 * q + e] = (j >> 4) <= (i >> 4) ? tv[e] : 0.f;
                        x[4 * q + e] = t[4 * q + e] * wv[e];
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; q++) st_chunk(sb + PS_TT + sw128_chunk(row, 4 * half + q, 128), x + 8 * q, 1.f);
            }
            fence_proxy_async_smem();
            __syncthreads();

            // W = Tw K and U~ = Tu V as two M=128 products of [Tw; Tu] (rows 0-63 of the first and
            // rows 64-127 of the second are the wanted ones; an M=64 product would take as long and
            // leave half of every warp idle in the epilogue). B operands: raw k / v tiles, MN-major.
            if (tid == 0) {
                // v of this value head (prefetched while the previous head was finishing)
                if (mbar_wait(&bar_v, v_ph, &abort_sh, a.status, 14)) {
                    v_pend = false;
                    tc_fence_after();
                    const uint32_t id = idesc_bf16(128, 128, 0, 1);
                    for (int k0 = 0; k0 < kChunk; k0 += 16) {
                        mma_bf16(tm + 0, desc_kmajor(sb + PS_TT, 128, 0, k0), desc_mnmajor(sb + PS_KQ, 128, 0, k0), id,
                                 k0 > 0);
                        mma_bf16(tm + 128, desc_kmajor(sb + PS_TT, 128, 0, k0), desc_mnmajor(sb + PS_V, 64, 0, k0), id,
                                 k0 > 0);
                    }
                    mma_commit(&bar_mma);
                    v_ph ^= 1;
                }
            }
            if (rec2 && tid < 128) {  // T itself for the backward, from the fp32 tile (intact until the
                // W/U~ epilogue), stored once the products are issued: the proxy fence before them
                // would otherwise wait for these global stores
                const int i = tid >> 1, half = tid & 1;
                const float* trow = Tm + i * LDA + 32 * half;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    float t[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        const int j = 32 * half + 8 * q + e;
                        t[e] = (j >> 4) <= (i >> 4) ? trow[8 * q + e] : 0.f;
                    }
                    st_global16(rec2 + REC2_T + sw128_chunk(i, 4 * half + q, 64), pack8(t, 1.f));
                }
            }
            ok = mbar_wait(&bar_mma, mph, &abort_sh, a.status, 12);
            mph ^= 1;
            if (__syncthreads_or(!ok)) goto teardown;
            if (tid < 64) {  // the next value head's gates (or the next group's first)
                if (hh + 1 < he) stage_gb(grp, hh + 1);
                else if (next < ngroups) stage_gb(next, nh0);
            }
            tc_fence_after();
            {
                const int lg = warp & 3, h = warp >> 2;
                if (lg < 2) {  // W rows i = 32 lg + lane (first product, columns 64 h ..)
                    const int i = 32 * lg + lane;
                    const float sbar = fb[i];
#pragma unroll 1
                    for (int hh2 = 0; hh2 < 2; hh2++) {  // 32 columns at a time (register budget)
                        float w[32];
                        tmem_ld32(tmem_at(tm, 32 * lg, 64 * h + 32 * hh2), w);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const uint4 u = pack8(w + 8 * q, 1.f);
                            const uint32_t off = sw128_chunk(i, 8 * h + 4 * hh2 + q, 64);
                            st_shared_v4(sb + PS_W + off, u.x, u.y, u.z, u.w);
                            st_chunk(sb + PS_WBAR + off, w + 8 * q, sbar);
                        }
                    }
                } else {  // U~ rows i = 32 lg + lane - 64 (second product)
                    const int i = 32 * lg + lane - 64;
#pragma unroll 1
                    for (int hh2 = 0; hh2 < 2; hh2++) {
                        float u[32];
                        tmem_ld32(tmem_at(tm, 32 * lg, 128 + 64 * h + 32 * hh2), u);
                        tmem_wait_ld();
                        const int col = 64 * h + 32 * hh2;  // one 32-column U~ slice
#pragma unroll
                        for (int q = 0; q < 4; q++)  // the record's slice image, staged over v (read)
                            st_chunk(sb + PS_V + (col >> 5) * 4096 + sw64_chunk(i, q), u + 8 * q, 1.f);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();

            // Mneg = -K^T Wbar (M=128: A = k tile read MN-major) and P W (M=64)
            if (tid == 0) {  // U~ (and W for the backward) to the record, from their images
                bulk_store(rec + REC_U, sm + PS_V, 16384);
                if (rec2) bulk_store(rec2 + REC2_W, sm + PS_W, 16384);
                bulk_commit();
                tc_fence_after();
                const uint32_t idm = idesc_bf16(128, 128, 1, 1);
                for (int k0 = 0; k0 < kChunk; k0 += 16)
                    mma_bf16(tm + 0, desc_mnmajor(sb + PS_KQ, 128, 0, k0), desc_mnmajor(sb + PS_WBAR, 64, 0, k0), idm,
                             k0 > 0);
                const uint32_t idp = idesc_bf16(64, 128, 0, 1);
                for (int k0 = 0; k0 < kChunk; k0 += 16)
                    mma_bf16(tm + 128, desc_kmajor(sb + PS_P, 64, 0, k0), desc_mnmajor(sb + PS_W, 64, 0, k0), idp,
                             k0 > 0);
                mma_commit(&bar_mma);
            }
            {  // Kbar = diag(exp(gamma_C - gamma) rho_k) K, straight to the record once the products are
               // issued (the proxy fence before them would otherwise wait for these global stores)
                uint4 kv[4];
                float fr[4];
#pragma unroll
                for (int n = 0; n < 4; n++) {
                    const int idx = tid + 256 * n, r = idx >> 4, j = idx & 15;
                    kv[n] = ld_shared_v4(sb + PS_KQ + sw128_chunk(r, j, 128));
                    fr[n] = fb[r];
                }
#pragma unroll
                for (int n = 0; n < 4; n++) {
                    const int idx = tid + 256 * n, r = idx >> 4, j = idx & 15;
                    float x[8];
                    unpack8(kv[n], x);
                    st_global16(rec + REC_K + sw128_chunk(r, j, 64), pack8(x, fr[n]));
                }
            }
            ok = mbar_wait(&bar_mma, mph, &abort_sh, a.status, 13);
            mph ^= 1;
            if (tid == 0) {
                bulk_wait_read_all();  // the P, U~ and W images are read: the staging may overwrite them,
                if (hh + 1 < he) issue_v(grp, hh + 1);  // and the next value head's v (or the next
                else if (next < ngroups) issue_v(next, nh0);  // unit's first) may land over U~
            }
            if (__syncthreads_or(!ok)) goto teardown;
            tc_fence_after();
            {
                const int lg = warp & 3, h = warp >> 2;
                {  // Mneg rows d = 32 lg + lane
                    const int d = 32 * lg + lane;
#pragma unroll 1
                    for (int hh2 = 0; hh2 < 2; hh2++) {
                        float m[32];
                        tmem_ld32(tmem_at(tm, 32 * lg, 64 * h + 32 * hh2), m);
                        tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 4; q++)
                        {
                            const uint4 u = pack8(m + 8 * q, -1.f);
                            st_shared_v4(sb + PS_STAGE + sw128_chunk(d, 8 * h + 4 * hh2 + q, 128), u.x, u.y, u.z, u.w);
                        }
                    }
                }
                {  // Qc = scale diag(Gamma rho_q) Q - P W, rows i = 16 lg + lane
                    // M=64 rows live in lanes 0-15; lane l + 16 takes columns 32-63 of lane l's row
                    const int i = 16 * lg + (lane & 15);
                    const int hf = lane >> 4;
                    float pw[32];
                    {
                        float lo[32];
                        tmem_ld32(tmem_at(tm, 32 * lg, 128 + 64 * h), lo);
                        tmem_ld32(tmem_at(tm, 32 * lg, 128 + 64 * h + 32), pw);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; e++) {
                            const float hi = __shfl_sync(0xffffffffu, pw[e], lane & 15);
                            pw[e] = hf ? hi : lo[e];
                        }
                    }
                    const float f = fq[i];
                    uint4 qv[4];
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        qv[q] = ld_shared_v4(sb + PS_KQ + sw128_chunk(64 + i, 8 * h + 4 * hf + q, 128));
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        float x[8];
                        unpack8(qv[q], x);
#pragma unroll
                        for (int e = 0; e < 8; e++) x[e] = f * x[e] - pw[8 * q + e];
                        const uint4 u = pack8(x, 1.f);
                        st_shared_v4(sb + PS_STAGE_Q + sw128_chunk(i, 8 * h + 4 * hf + q, 64), u.x, u.y, u.z, u.w);
                    }
                }
            }
            if (tid == 0) a.gam[bh * a.ncpad + c] = expf(gam[63]);
            fence_proxy_async_smem();  // the staged images leave by bulk copies
            tc_fence_before();
            __syncthreads();  // every buffer of this value head is free again
            tc_fence_after();
            if (tid == 0) {
                // after the unit's last head k, q are no longer read: the next unit's copy goes into
                // the copy engine ahead of this head's record stores
                if (hh + 1 == he && next < ngroups) issue_kq(next);
                bulk_store(rec + REC_M, sm + PS_STAGE, 32768);
                bulk_store(rec + REC_Q, sm + PS_STAGE_Q, 16384);
                bulk_commit();
            }
        }  // value heads of the unit
    }  // units
teardown:
    cp_async_wait_all();
    if (tid == 0) bulk_wait_all();  // record stores complete
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0) {  // let copies still in flight land before the CTA exits
        volatile int never = 0;
        if (kq_pend) mbar_wait(&bar_kq, kq_ph, &never, nullptr, 0);
        if (v_pend) mbar_wait(&bar_v, v_ph, &never, nullptr, 0);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

cudaError_t launch_prep(const PrepArgs& a, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        cudaStream_t s) {
    const int smem = PS_BYTES + 1024;
    cudaError_t e = cudaFuncSetAttribute(prep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    static int nsm = 0;  // 2 CTAs fit an SM (smem, TMEM, registers): a persistent grid of 2 per SM
    if (nsm == 0) {
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    }
    const int ngroups = a.p.B * a.p.Hk * a.p.NC, G = a.p.Hv / a.p.Hk;
    const bool split = (long)ngroups * G <= nsm;  // one value head per unit when each still gets an SM
    const int nunits = split ? ngroups * G : ngroups;
    dim3 grid(nunits < 2 * nsm ? nunits : 2 * nsm);
    trace_begin("chunk_prep", s);
    if (split)
        prep_kernel<true><<<grid, 256, smem, s>>>(mq, mk, mv, a);
    else
        prep_kernel<false><<<grid, 256, smem, s>>>(mq, mk, mv, a);
    trace_end(s);
    return cudaGetLastError();
}

bool make_qkv_maps(const ChunkProblem& p, const void* q, const void* k, const void* v, CUtensorMap* mq,
                   CUtensorMap* mk, CUtensorMap* mv) {
    return make_map_4d_bf16(mq, q, kD, p.Hk, p.T, p.B, 64, kChunk, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map_4d_bf16(mk, k, kD, p.Hk, p.T, p.B, 64, kChunk, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_map_4d_bf16(mv, v, kD, p.Hv, p.T, p.B, 64, kChunk, CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_chunk_fwd(const ChunkFwdArgs& a, cudaStream_t s) {
    const WsLayout w = ws_layout(a.p, false);
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    uint8_t* keep = static_cast<uint8_t*>(a.saved);
    const SavedLayout l = saved_layout(a.p);
    CUtensorMap mq, mk, mv;
    if (!make_qkv_maps(a.p, a.q, a.k, a.v, &mq, &mk, &mv)) return cudaErrorInvalidValue;
    PrepArgs pa;
    pa.p = a.p;
    pa.g = a.g;
    pa.beta = a.beta;
    pa.gam = reinterpret_cast<float*>(keep ? keep + l.gam : ws + w.gam);
    pa.rec = keep ? keep + l.rec : ws + w.rec;
    pa.rec2 = keep ? keep + l.rec2 : nullptr;
    pa.status = reinterpret_cast<int*>(ws);
    pa.ncpad = keep ? l.ncpad : w.ncpad;
    cudaError_t e = a.p.channel ? launch_prep_ch(pa, mq, mk, mv, s) : launch_prep(pa, mq, mk, mv, s);
    if (e != cudaSuccess) return e;
    ScanArgs sa;
    sa.p = a.p;
    sa.gam = pa.gam;
    sa.rec = pa.rec;
    sa.hinit = a.h0;
    sa.o = a.o;
    sa.hfinal = a.ht;
    sa.states = keep ? keep + l.hs : static_cast<uint8_t*>(a.states);
    sa.status = pa.status;
    sa.ncpad = pa.ncpad;
    return launch_scan(sa, SCAN_FWD_OUT, nullptr, s);
}

}  // namespace gdr
