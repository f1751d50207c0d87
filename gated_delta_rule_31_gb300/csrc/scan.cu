// scan.cu - the chunk-to-chunk state scans of the chunked gated delta rule (the sequential
// part of the "chunked case" of "Adding VJP for gated delta net", MLX PR #4565):
//   forward  H1 = Gamma_C H0 + Mneg H0 + Kbar^T U~, writing O = Qc H0 + P U~ for every chunk
//   states   the same recurrence, keeping the state entering every chunk
//   backward dH0 = Gamma_C dH1 + Mneg^T dH1 + Qc^T dO (chunks in reverse order)
// (operators in chunk.h, built per chunk by the prep kernels). Per chunk a scan issues one
// dependent tensor-core product on the bf16 image of the state, with the fp32 state held in
// registers. Two kernels:
//   slice_scan_kernel: one CTA per (b, value head, 32 state columns); the forward's output
//     products (Qc H0 and P U~) run in the same CTA. Used for the states and backward scans
//     and for forwards of a few chunks (short prefills), where it fits two or three CTAs per SM.
//   pair_scan_kernel: forward with outputs over longer sequences. A tcgen05 instruction holds
//     the tensor pipe about 70 cycles whatever its N up to 128, so in one CTA the 12 output
//     instructions per chunk double the pipe time of the 12 state instructions. Here a two-CTA
//     cluster owns 64 state columns: the state CTA runs the recurrence and sends each state
//     image (bf16 [128 x 64], one panel of the saved state image) into the output CTA's shared
//     memory by a bulk copy; the output CTA computes O and releases the slot with a multicast
//     commit that arrives on the state CTA's barrier when its products complete.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "chunk.h"
#include "chunk_dev.cuh"
#include "common.cuh"
#include "kernels.h"

namespace gdr {

namespace {

constexpr int kSlice = 32;  // state columns per slice-scan CTA
constexpr int kSlices = kD / kSlice;

// ------------------------------------------------------------------ slice scan
// One ring stage per chunk. Forward with outputs (2 stages): Mneg 32 KB | Kbar 16 KB | Qc 16 KB |
// P 8 KB | U~ slice 4 KB. States / backward (3 stages): Mneg 32 KB | Kbar or Qc 16 KB | U~ or dO
// slice 4 KB. The third stage lets the next chunk's operators arrive a step earlier. A sequence
// with fewer chunks than stages never wraps the ring: the state tiles follow the stages it uses
// and it launches with that much shared memory (one chunk: 2 CTAs per SM instead of 1).
template <int MODE>
struct SliceLayout {
    static constexpr int NS = MODE == SCAN_FWD_OUT ? 2 : 3;
    static constexpr uint32_t ST_M = 0, ST_K = 32768;  // ST_K: Kbar (forward) or Qc (backward)
    static constexpr uint32_t ST_Q = 49152, ST_P = 65536;  // forward outputs only
    static constexpr uint32_t ST_U = MODE == SCAN_FWD_OUT ? 73728 : 49152;
    static constexpr uint32_t STG = MODE == SCAN_FWD_OUT ? 78848 : 53248;
    static constexpr uint32_t BYTES = NS * STG + 16384;  // + two bf16 [128 x 32] SW64 state tiles
    // offset of the state tiles for NC chunks (the stages that NC chunks occupy)
    __host__ __device__ static constexpr uint32_t ss_h(int NC) { return (NC < 1 ? 1 : NC < NS ? NC : NS) * STG; }
    static_assert(BYTES + 1024 <= 232448, "scan smem");
    static_assert(STG % 1024 == 0, "stage alignment");
};

__device__ __forceinline__ void write_state_tile(uint32_t tile, int d, const float* H) {
#pragma unroll
    for (int q = 0; q < 4; q++)
        st_shared_v4(tile + sw64_chunk(d, q), pack_bf16(H[8 * q], H[8 * q + 1]), pack_bf16(H[8 * q + 2], H[8 * q + 3]),
                     pack_bf16(H[8 * q + 4], H[8 * q + 5]), pack_bf16(H[8 * q + 6], H[8 * q + 7]));
}

template <int MODE>
__global__ void __launch_bounds__(192, 1) slice_scan_kernel(const __grid_constant__ CUtensorMap mdo, ScanArgs a) {
    using LY = SliceLayout<MODE>;
    constexpr int NS = LY::NS;
    constexpr uint32_t ST_M = LY::ST_M, ST_K = LY::ST_K, ST_Q = LY::ST_Q, ST_P = LY::ST_P, ST_U = LY::ST_U;
    constexpr uint32_t STG = LY::STG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t full[3], empty[3], hready, sfull, ofull[2], drain;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = blockIdx.x, hv = blockIdx.y, b = blockIdx.z;
    const ChunkProblem& P = a.p;
    const int NC = P.NC;
    const uint32_t SS_H = LY::ss_h(NC);
    const size_t bh = (size_t)b * P.Hv + hv;
    auto chunk_of = [&](int i) { return MODE == SCAN_BWD ? NC - 1 - i : i; };

    if (tid == 0) {
        abort_sh = 0;
        for (int s = 0; s < NS; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&ofull[0], 1);
        mbar_init(&ofull[1], 1);
        mbar_init(&hready, 1);
        mbar_init(&sfull, 1);
        mbar_init(&drain, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_sh, 128);  // Ds[0..1] cols 0-63, Do[0..1] cols 64-127
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_sh;
    int last_loaded = -1;

    if (warp == 0) {
        if (lane == 0) {  // producer: bulk copies of the chunk records (+ dO slice via TMA)
            for (int i = 0; i < NC; i++) {
                const int c = chunk_of(i), s = i % NS;
                if (i >= NS && !mbar_wait(&empty[s], ((i / NS) + 1) & 1, &abort_sh, a.status, 20)) break;
                uint8_t* st = sm + s * STG;
                const uint8_t* rec = a.rec + (bh * NC + c) * REC_BYTES;
                uint32_t bytes = 32768 + 4096 + 16384;
                if (MODE == SCAN_FWD_OUT) bytes += 16384 + 8192;
                mbar_expect_tx(&full[s], bytes);
                bulk_load(st + ST_M, rec + REC_M, 32768, &full[s]);
                if (MODE != SCAN_BWD) {
                    bulk_load(st + ST_K, rec + REC_K, 16384, &full[s]);
                    bulk_load(st + ST_U, rec + REC_U + j * 4096, 4096, &full[s]);
                }
                if (MODE == SCAN_FWD_OUT) {
                    bulk_load(st + ST_Q, rec + REC_Q, 16384, &full[s]);
                    bulk_load(st + ST_P, rec + REC_P, 8192, &full[s]);
                }
                if (MODE == SCAN_BWD) {
                    bulk_load(st + ST_K, rec + REC_Q, 16384, &full[s]);
                    tma_load_4d(st + ST_U, &mdo, kSlice * j, hv, kChunk * c, b, &full[s]);
                }
                last_loaded = i;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            const uint32_t id_state = MODE == SCAN_BWD ? idesc_bf16(128, 32, 1, 1) : idesc_bf16(128, 32, 0, 1);
            const uint32_t id_pre = idesc_bf16(128, 32, 1, 1);
            const uint32_t id_out = idesc_bf16(64, 32, 0, 1);
            auto issue_pre = [&](int i) {  // state-independent term into Ds[i & 1]
                const uint32_t st = sb + (i % NS) * STG;
                const uint32_t src = st + ST_K;  // Qc^T dO (backward)  or  Kbar^T U~ (forward)
                for (int k0 = 0; k0 < kChunk; k0 += 16)
                    mma_bf16(tm + 32 * (i & 1), desc_mnmajor(src, 64, 0, k0), desc_mnmajor_sw64(st + ST_U, 64, k0),
                             id_pre, k0 > 0);
            };
            for (int i = 0; i < NC; i++) {
                const int s = i % NS, sd = i & 1;  // ring stage, double-buffer index
                const uint32_t st = sb + s * STG;
                if (i == 0) {
                    if (!mbar_wait(&full[0], 0, &abort_sh, a.status, 21)) break;
                    tc_fence_after();
                    issue_pre(0);
                }
                if (!mbar_wait(&hready, i & 1, &abort_sh, a.status, 22)) break;
                tc_fence_after();
                const uint32_t ht = sb + SS_H + (i & 1) * 8192;
                for (int k0 = 0; k0 < kD; k0 += 16) {
                    const uint64_t ad =
                        MODE == SCAN_BWD ? desc_mnmajor(st + ST_M, 128, 0, k0) : desc_kmajor(st + ST_M, 128, 0, k0);
                    mma_bf16(tm + 32 * sd, ad, desc_mnmajor_sw64(ht, 128, k0), id_state, 1);
                }
                mma_commit(&sfull);
                if (MODE == SCAN_FWD_OUT) {
                    for (int k0 = 0; k0 < kD; k0 += 16)
                        mma_bf16(tm + 64 + 32 * sd, desc_kmajor(st + ST_Q, 64, 0, k0), desc_mnmajor_sw64(ht, 128, k0),
                                 id_out, k0 > 0);
                    for (int k0 = 0; k0 < kChunk; k0 += 16)
                        mma_bf16(tm + 64 + 32 * sd, desc_kmajor(st + ST_P, 64, 0, k0),
                                 desc_mnmajor_sw64(st + ST_U, 64, k0), id_out, 1);
                    mma_commit(&ofull[sd]);
                }
                mma_commit(&empty[s]);
                if (i + 1 < NC) {
                    if (!mbar_wait(&full[(i + 1) % NS], ((i + 1) / NS) & 1, &abort_sh, a.status, 23)) break;
                    tc_fence_after();
                    issue_pre(i + 1);
                }
            }
            // every product issued so far has completed before TMEM is released
            mma_commit(&drain);
            volatile int never = 0;
            mbar_wait(&drain, 0, &never, nullptr, 0);
        }
    } else {  // epilogue: 4 warps, thread <-> TMEM lane d = state row (key channel)
        const int et = tid - 64;
        const int lg = warp & 3;
        const int d = 32 * lg + lane;
        float H[32];
#pragma unroll
        for (int n = 0; n < 32; n++)
            H[n] = a.hinit ? a.hinit[(bh * kD + kSlice * j + n) * kD + d] : 0.f;
        write_state_tile(sb + SS_H, d, H);
        fence_proxy_async_smem();
        bool bad = bar_sync_or(1, 128, false);
        if (et == 0) mbar_arrive(&hready);
        // Gamma_C of each chunk: one per head, or one per key channel (this thread's row d)
        const float* gam = P.channel ? a.gam + bh * NC * kD + d : a.gam + bh * a.ncpad;
        const int gstride = P.channel ? kD : 1;
        float gnext = gam[chunk_of(0) * gstride];
        int i = 0;
        for (; i < NC && !bad; i++) {
            const int c = chunk_of(i), s = i & 1;
            const float gC = gnext;
            if (i + 1 < NC) gnext = gam[chunk_of(i + 1) * gstride];
            if (MODE != SCAN_FWD_OUT || a.states) {  // state entering this step, SW128 [128 x 128] image
                uint8_t* img = a.states + (bh * NC + c) * (size_t)STATE_IMG;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    uint4 v = make_uint4(pack_bf16(H[8 * q], H[8 * q + 1]), pack_bf16(H[8 * q + 2], H[8 * q + 3]),
                                         pack_bf16(H[8 * q + 4], H[8 * q + 5]), pack_bf16(H[8 * q + 6], H[8 * q + 7]));
                    *reinterpret_cast<uint4*>(img + sw128_chunk(d, 4 * j + q, 128)) = v;
                }
            }
            bool ok = __all_sync(0xffffffffu, mbar_wait(&sfull, i & 1, &abort_sh, a.status, 30));
            tc_fence_after();
            float D[32], O[32];
            if (ok) tmem_ld32(tmem_at(tm, 32 * lg, 32 * s), D);
            if (MODE == SCAN_FWD_OUT && i > 0 && ok) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&ofull[(i - 1) & 1], ((i - 1) >> 1) & 1, &abort_sh, a.status, 31));
                tc_fence_after();
                if (ok) tmem_ld32(tmem_at(tm, 32 * lg, 64 + 32 * ((i - 1) & 1)), O);
            }
            tmem_wait_ld();
#pragma unroll
            for (int n = 0; n < 32; n++) H[n] = gC * H[n] + D[n];
            if (i + 1 < NC) {
                write_state_tile(sb + SS_H + ((i + 1) & 1) * 8192, d, H);
                fence_proxy_async_smem();
            }
            tc_fence_before();
            bad = bar_sync_or(1, 128, !ok || abort_sh);
            if (bad) break;
            if (i + 1 < NC && et == 0) mbar_arrive(&hready);
            if (MODE == SCAN_FWD_OUT && i > 0 && lane < 16) {  // output rows of chunk c-1
                const int r = 16 * lg + lane, t = kChunk * (c - 1) + r;
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) +
                                                      (((size_t)b * P.T + t) * P.Hv + hv) * kD + kSlice * j);
#pragma unroll
                for (int q = 0; q < 4; q++)
                    dst[q] = make_uint4(pack_bf16(O[8 * q], O[8 * q + 1]), pack_bf16(O[8 * q + 2], O[8 * q + 3]),
                                        pack_bf16(O[8 * q + 4], O[8 * q + 5]), pack_bf16(O[8 * q + 6], O[8 * q + 7]));
            }
        }
        if (!bad && MODE == SCAN_FWD_OUT) {  // outputs of the last chunk
            const int i_last = NC - 1;
            bool ok = __all_sync(0xffffffffu,
                                 mbar_wait(&ofull[i_last & 1], (i_last >> 1) & 1, &abort_sh, a.status, 32));
            tc_fence_after();
            float O[32];
            if (ok) tmem_ld32(tmem_at(tm, 32 * lg, 64 + 32 * (i_last & 1)), O);
            tmem_wait_ld();
            const int r = 16 * lg + lane, t = kChunk * i_last + r;
            if (ok && lane < 16 && t < P.T) {
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) +
                                                      (((size_t)b * P.T + t) * P.Hv + hv) * kD + kSlice * j);
#pragma unroll
                for (int q = 0; q < 4; q++)
                    dst[q] = make_uint4(pack_bf16(O[8 * q], O[8 * q + 1]), pack_bf16(O[8 * q + 2], O[8 * q + 3]),
                                        pack_bf16(O[8 * q + 4], O[8 * q + 5]), pack_bf16(O[8 * q + 6], O[8 * q + 7]));
            }
            bad = !ok;
        }
        if (!bad && a.hfinal) {
#pragma unroll
            for (int n = 0; n < 32; n++) a.hfinal[(bh * kD + kSlice * j + n) * kD + d] = H[n];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0 && last_loaded >= 0) {  // copies still in flight must land first
        volatile int never = 0;
        for (int i = last_loaded >= NS - 1 ? last_loaded - (NS - 1) : 0; i <= last_loaded; i++)
            mbar_wait(&full[i % NS], (i / NS) & 1, &never, nullptr, 0);
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 128);
}

// ------------------------------------------------------------------ pair scan (forward, long sequences)
constexpr int kHalf = 64;  // state columns (value channels) per cluster
constexpr int NSTAGE = 3, NTILE = 3, NSLOT = 2;
constexpr int kPairMinChunks = 4;  // shorter forwards use the slice kernel (more CTAs per SM)
// State CTA ring stage: Mneg 32 KB | Kbar 16 KB | U~ half (two 32-column SW64 slices of the record) 8 KB.
constexpr uint32_t SS_M = 0, SS_K = 32768, SS_U = 49152, SS_STG = 57344;
// Output CTA ring stage: Qc 16 KB | P 8 KB | U~ half 8 KB.
constexpr uint32_t OS_Q = 0, OS_P = 16384, OS_U = 24576, OS_STG = 32768;
constexpr uint32_t TILE = 16384;   // bf16 [128 d x 64 v] SW128 state tile = one panel of a state image
constexpr int PAIR_THREADS = 320;  // producer warp, MMA warp, 8 epilogue warps (4 in the output CTA)

__host__ __device__ constexpr int pair_stages(int NC) { return NC < 1 ? 1 : (NC < NSTAGE ? NC : NSTAGE); }
__host__ __device__ constexpr uint32_t pair_smem(int NC) { return pair_stages(NC) * SS_STG + NTILE * TILE; }
static_assert(NSTAGE * OS_STG + NSLOT * TILE <= NSTAGE * SS_STG + NTILE * TILE, "output CTA layout");
static_assert(NSTAGE * SS_STG + NTILE * TILE + 1024 <= 232448, "pair scan smem");

__global__ void __launch_bounds__(PAIR_THREADS, 1) pair_scan_kernel(ScanArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    __shared__ uint64_t full[NSTAGE], empty[NSTAGE], hready, sfull, drain;
    __shared__ uint64_t slot_empty[NSLOT];              // state CTA: the output CTA released a slot
    __shared__ uint64_t recv[NSLOT], ofull[2], ofree[2];  // output CTA
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool out_role = cluster_ctarank() == 1;
    const int j = blockIdx.x >> 1;  // which 64 state columns
    const int hv = blockIdx.y, b = blockIdx.z;
    const ChunkProblem& P = a.p;
    const int NC = P.NC;
    const int NS = pair_stages(NC);
    const size_t bh = (size_t)b * P.Hv + hv;

    if (tid == 0) {
        abort_sh = 0;
        for (int s = 0; s < NSTAGE; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < NSLOT; s++) {
            mbar_init(&slot_empty[s], 1);
            mbar_init(&recv[s], 1);
        }
        for (int s = 0; s < 2; s++) {
            mbar_init(&ofull[s], 1);
            mbar_init(&ofree[s], 1);
        }
        mbar_init(&hready, 1);
        mbar_init(&sfull, 1);
        mbar_init(&drain, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_sh, 128);  // two 64-column accumulators
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the peer's barriers exist before any remote access
    const uint32_t tm = tmem_sh;
    int last_loaded = -1;

    if (!out_role) {  // ------------------------------------------------ state CTA
        const uint32_t tiles = sb + NS * SS_STG;
        if (warp == 0) {
            if (lane == 0) {  // producer: bulk copies of Mneg, Kbar and this half of U~
                for (int i = 0; i < NC; i++) {
                    const int s = i % NS;
                    if (i >= NS && !mbar_wait(&empty[s], ((i / NS) + 1) & 1, &abort_sh, a.status, 20)) break;
                    uint8_t* st = sm + s * SS_STG;
                    const uint8_t* rec = a.rec + (bh * NC + i) * REC_BYTES;
                    mbar_expect_tx(&full[s], 32768 + 16384 + 8192);
                    bulk_load(st + SS_M, rec + REC_M, 32768, &full[s]);
                    bulk_load(st + SS_K, rec + REC_K, 16384, &full[s]);
                    bulk_load(st + SS_U, rec + REC_U + j * 8192, 8192, &full[s]);
                    last_loaded = i;
                }
            }
        } else if (warp == 1) {
            if (lane == 0) {  // MMA issuer
                const uint32_t id_state = idesc_bf16(128, kHalf, 0, 1);
                const uint32_t id_pre = idesc_bf16(128, kHalf, 1, 1);
                auto issue_pre = [&](int i) {  // Kbar^T U~ (independent of the state) into D[i & 1]
                    const uint32_t st = sb + (i % NS) * SS_STG;
                    for (int k0 = 0; k0 < kChunk; k0 += 16)
                        mma_bf16(tm + kHalf * (i & 1), desc_mnmajor(st + SS_K, 64, 0, k0),
                                 desc_mnmajor_sw64(st + SS_U, 64, k0), id_pre, k0 > 0);
                };
                for (int i = 0; i < NC; i++) {
                    const int s = i % NS;
                    const uint32_t st = sb + s * SS_STG;
                    if (i == 0) {
                        if (!mbar_wait(&full[0], 0, &abort_sh, a.status, 21)) break;
                        tc_fence_after();
                        issue_pre(0);
                    }
                    if (!mbar_wait(&hready, i & 1, &abort_sh, a.status, 22)) break;
                    tc_fence_after();
                    const uint32_t ht = tiles + (i % NTILE) * TILE;
                    for (int k0 = 0; k0 < kD; k0 += 16)
                        mma_bf16(tm + kHalf * (i & 1), desc_kmajor(st + SS_M, 128, 0, k0), desc_mnmajor(ht, 128, 0, k0),
                                 id_state, 1);
                    mma_commit(&sfull);
                    mma_commit(&empty[s]);
                    if (i + 1 < NC) {
                        if (!mbar_wait(&full[(i + 1) % NS], ((i + 1) / NS) & 1, &abort_sh, a.status, 23)) break;
                        tc_fence_after();
                        issue_pre(i + 1);
                    }
                }
                mma_commit(&drain);  // every product issued has completed before TMEM is released
                volatile int never = 0;
                mbar_wait(&drain, 0, &never, nullptr, 0);
            }
        } else {  // epilogue: 8 warps; thread <-> state row d (TMEM lane), 32 of the 64 columns
            const int et = tid - 64;
            const int lg = warp & 3, ch = (warp - 2) >> 2;
            const int d = 32 * lg + lane;
            const int v0 = kHalf * j + 32 * ch;
            float H[32];
#pragma unroll
            for (int n = 0; n < 32; n++) H[n] = a.hinit ? a.hinit[(bh * kD + v0 + n) * kD + d] : 0.f;
            auto write_tile = [&](int k) {
                const uint32_t t = tiles + (k % NTILE) * TILE;
#pragma unroll
                for (int q = 0; q < 4; q++)
                    st_shared_v4(t + sw128_chunk(d, 4 * ch + q, 128), pack_bf16(H[8 * q], H[8 * q + 1]),
                                 pack_bf16(H[8 * q + 2], H[8 * q + 3]), pack_bf16(H[8 * q + 4], H[8 * q + 5]),
                                 pack_bf16(H[8 * q + 6], H[8 * q + 7]));
            };
            // The state entering step k (thread et == 0): into slot k % NSLOT of the output CTA (same
            // shared-memory offsets there), then as panel j of its image for the backward.
            auto publish = [&](int k) {
                const uint32_t t = tiles + (k % NTILE) * TILE;
                bulk_copy_to_cta(mapa_shared(sb + NS * OS_STG + (k % NSLOT) * TILE, 1), t, TILE,
                                 mapa_shared(smem_u32(&recv[k % NSLOT]), 1));
                if (a.states) {
                    bulk_store(a.states + (bh * NC + k) * (size_t)STATE_IMG + j * TILE, sm + (t - sb), TILE);
                    bulk_commit();
                }
            };
            write_tile(0);
            fence_proxy_async_smem();
            bool bad = bar_sync_or(1, 256, false);
            if (et == 0) {
                mbar_arrive(&hready);
                publish(0);
            }
            // Gamma_C of each chunk: one per head, or one per key channel (this thread's row d)
            const float* gam = P.channel ? a.gam + bh * NC * kD + d : a.gam + bh * a.ncpad;
            const int gstride = P.channel ? kD : 1;
            float gnext = gam[0];
            for (int i = 0; i < NC && !bad; i++) {
                const float gC = gnext;
                if (i + 1 < NC) gnext = gam[(i + 1) * gstride];
                bool ok = __all_sync(0xffffffffu, mbar_wait(&sfull, i & 1, &abort_sh, a.status, 30));
                tc_fence_after();
                float D[32];
                if (ok) tmem_ld32(tmem_at(tm, 32 * lg, kHalf * (i & 1) + 32 * ch), D);
                tmem_wait_ld();
#pragma unroll
                for (int n = 0; n < 32; n++) H[n] = gC * H[n] + D[n];
                if (i + 1 < NC) {
                    write_tile(i + 1);
                    fence_proxy_async_smem();
                }
                // Before the next step overwrites the tile of the state entering step i - 1: its image
                // store has read it, and the output CTA has received it and finished the products that
                // read it (which also frees that slot for the state of step i + 1).
                if (et == 0) {
                    if (a.states) bulk_wait_read_but1();
                    if (i >= 1 && !mbar_wait_cluster(&slot_empty[(i - 1) % NSLOT], ((i - 1) / NSLOT) & 1, &abort_sh,
                                                     a.status, 33))
                        ok = false;
                }
                tc_fence_before();
                bad = bar_sync_or(1, 256, !ok || abort_sh);
                if (bad) break;
                if (i + 1 < NC && et == 0) {
                    mbar_arrive(&hready);
                    publish(i + 1);
                }
            }
            if (!bad && a.hfinal) {
#pragma unroll
                for (int n = 0; n < 32; n++) a.hfinal[(bh * kD + v0 + n) * kD + d] = H[n];
            }
            if (et == 0) bulk_wait_all();  // image stores complete before the CTA exits
        }
    } else {  // ------------------------------------------------ output CTA
        const uint32_t slots = sb + NS * OS_STG;
        if (warp == 0) {
            if (lane == 0) {  // producer: Qc, P and the U~ half of each chunk
                for (int i = 0; i < NC; i++) {
                    const int s = i % NS;
                    if (i >= NS && !mbar_wait(&empty[s], ((i / NS) + 1) & 1, &abort_sh, a.status, 24)) break;
                    uint8_t* st = sm + s * OS_STG;
                    const uint8_t* rec = a.rec + (bh * NC + i) * REC_BYTES;
                    mbar_expect_tx(&full[s], 16384 + 8192 + 8192);
                    bulk_load(st + OS_Q, rec + REC_Q, 16384, &full[s]);
                    bulk_load(st + OS_P, rec + REC_P, 8192, &full[s]);
                    bulk_load(st + OS_U, rec + REC_U + j * 8192, 8192, &full[s]);
                    last_loaded = i;
                }
            }
        } else if (warp == 1) {
            if (lane == 0) {  // MMA issuer: O = Qc H0 + P U~ into O[i & 1]
                const uint32_t id_out = idesc_bf16(64, kHalf, 0, 1);
                int armed[NSLOT] = {-1, -1};  // slot uses armed and not yet waited for
                for (int i = 0; i < NC; i++) {
                    const int s = i % NS, sl = i % NSLOT;
                    mbar_expect_tx(&recv[sl], TILE);  // this use of the slot: one arrival and the tile's bytes
                    armed[sl] = i;
                    if (i >= 2 && !mbar_wait(&ofree[i & 1], ((i >> 1) - 1) & 1, &abort_sh, a.status, 25)) break;
                    if (!mbar_wait(&full[s], (i / NS) & 1, &abort_sh, a.status, 26)) break;
                    if (!mbar_wait(&recv[sl], (i / NSLOT) & 1, &abort_sh, a.status, 27)) break;
                    armed[sl] = -1;
                    tc_fence_after();
                    const uint32_t st = sb + s * OS_STG, ht = slots + sl * TILE;
                    for (int k0 = 0; k0 < kD; k0 += 16)
                        mma_bf16(tm + kHalf * (i & 1), desc_kmajor(st + OS_Q, 64, 0, k0), desc_mnmajor(ht, 128, 0, k0),
                                 id_out, k0 > 0);
                    for (int k0 = 0; k0 < kChunk; k0 += 16)
                        mma_bf16(tm + kHalf * (i & 1), desc_kmajor(st + OS_P, 64, 0, k0),
                                 desc_mnmajor_sw64(st + OS_U, 64, k0), id_out, 1);
                    mma_commit(&ofull[i & 1]);
                    mma_commit(&empty[s]);
                    mma_commit_multicast(&slot_empty[sl], 0x1);  // the state CTA may refill this slot
                }
                mma_commit(&drain);
                volatile int never = 0;
                mbar_wait(&drain, 0, &never, nullptr, 0);
                // a slot armed but not received: the state CTA may still be copying into it
                for (int sl = 0; sl < NSLOT; sl++)
                    if (armed[sl] >= 0) mbar_wait(&recv[sl], (armed[sl] / NSLOT) & 1, &never, nullptr, 0);
            }
        } else if (warp < 6) {  // epilogue: 4 warps; M=64 rows 16 lg .. 16 lg + 15 in lanes 0-15
            const int et = tid - 64;
            const int lg = warp & 3;
            for (int i = 0; i < NC; i++) {
                bool ok = __all_sync(0xffffffffu, mbar_wait(&ofull[i & 1], (i >> 1) & 1, &abort_sh, a.status, 34));
                tc_fence_after();
                float x0[32], x1[32];
                if (ok) {
                    tmem_ld32(tmem_at(tm, 32 * lg, kHalf * (i & 1)), x0);
                    tmem_ld32(tmem_at(tm, 32 * lg, kHalf * (i & 1) + 32), x1);
                }
                tmem_wait_ld();
                tc_fence_before();
                if (bar_sync_or(2, 128, !ok || abort_sh)) break;
                if (et == 0) mbar_arrive(&ofree[i & 1]);  // O[i & 1] is read
                // lane l < 16: columns 0-31 of row 16 lg + l; lane l + 16: columns 32-63 of that row
                float w[32];
#pragma unroll
                for (int e = 0; e < 32; e++) {
                    const float hi = __shfl_sync(0xffffffffu, x1[e], lane & 15);
                    w[e] = (lane >> 4) ? hi : x0[e];
                }
                const int r = 16 * lg + (lane & 15), t = kChunk * i + r;
                if (t < P.T) {
                    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) +
                                                          (((size_t)b * P.T + t) * P.Hv + hv) * kD + kHalf * j +
                                                          32 * (lane >> 4));
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        dst[q] = make_uint4(pack_bf16(w[8 * q], w[8 * q + 1]), pack_bf16(w[8 * q + 2], w[8 * q + 3]),
                                            pack_bf16(w[8 * q + 4], w[8 * q + 5]), pack_bf16(w[8 * q + 6], w[8 * q + 7]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0 && last_loaded >= 0) {  // copies still in flight must land first
        volatile int never = 0;
        for (int i = last_loaded >= NS - 1 ? last_loaded - (NS - 1) : 0; i <= last_loaded; i++)
            mbar_wait(&full[i % NS], (i / NS) & 1, &never, nullptr, 0);
    }
    __syncthreads();
    cluster_sync();  // no CTA leaves while its peer may still reach its shared memory
    if (warp == 0) tmem_dealloc(tm, 128);
}

cudaError_t launch_pair_scan(const ScanArgs& a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(pair_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)pair_smem(NSTAGE) + 1024);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(2 * (kD / kHalf), a.p.Hv, a.p.B);  // (state, output) CTA pairs per 64 columns
    cfg.blockDim = dim3(PAIR_THREADS);
    cfg.dynamicSmemBytes = pair_smem(a.p.NC) + 1024;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    trace_begin("chunk_scan_fwd", s);
    e = cudaLaunchKernelEx(&cfg, pair_scan_kernel, a);
    trace_end(s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_slice_scan(const ScanArgs& a, int mode, const CUtensorMap* mdo, cudaStream_t s) {
    // the attribute always allows the full ring; a launch asks for what its chunk count uses
    const int smem_max = (mode == SCAN_FWD_OUT ? SliceLayout<SCAN_FWD_OUT>::BYTES : SliceLayout<SCAN_BWD>::BYTES) + 1024;
    const int smem = (mode == SCAN_FWD_OUT ? SliceLayout<SCAN_FWD_OUT>::ss_h(a.p.NC) : SliceLayout<SCAN_BWD>::ss_h(a.p.NC)) +
                     16384 + 1024;
    dim3 grid(kSlices, a.p.Hv, a.p.B);
    CUtensorMap dummy;
    memset(&dummy, 0, sizeof(dummy));
    const CUtensorMap& m = mdo ? *mdo : dummy;
    cudaError_t e;
    switch (mode) {
        case SCAN_FWD_OUT:
            e = cudaFuncSetAttribute(slice_scan_kernel<SCAN_FWD_OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
            if (e != cudaSuccess) return e;
            trace_begin("chunk_scan_fwd", s);
            slice_scan_kernel<SCAN_FWD_OUT><<<grid, 192, smem, s>>>(m, a);
            trace_end(s);
            break;
        case SCAN_FWD_STATES:
            e = cudaFuncSetAttribute(slice_scan_kernel<SCAN_FWD_STATES>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_max);
            if (e != cudaSuccess) return e;
            trace_begin("chunk_scan_states", s);
            slice_scan_kernel<SCAN_FWD_STATES><<<grid, 192, smem, s>>>(m, a);
            trace_end(s);
            break;
        default:
            e = cudaFuncSetAttribute(slice_scan_kernel<SCAN_BWD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
            if (e != cudaSuccess) return e;
            trace_begin("chunk_scan_bwd", s);
            slice_scan_kernel<SCAN_BWD><<<grid, 192, smem, s>>>(m, a);
            trace_end(s);
            break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, int mode, const CUtensorMap* mdo, cudaStream_t s) {
    if (mode == SCAN_FWD_OUT && a.p.NC >= kPairMinChunks) return launch_pair_scan(a, s);
    return launch_slice_scan(a, mode, mdo, s);
}

}  // namespace gdr
