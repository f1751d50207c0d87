// chunk_f32.cu - the chunked gated delta rule for fp32 q/k/v: the chunk algebra of the
// tensor-core path, computed with fp32 FMA on the CUDA cores, for every gate and Dk, Dv in
// {32, 64, 128}. The tensor cores take bf16 operands, whose rounding (about 4e-3) is far above
// the 1e-4 bound that fp32 inputs are held to, so fp32 problems take this path; it is written
// for exactness, not speed.
//
// Chunk algebra per (b, value head, chunk of C = 64 tokens), with the per-key-channel view of
// the decay (a scalar gate is the same gate on every channel): gamma[r][d] the in-chunk
// cumulative log-decay, E_rj = exp(gamma_r - gamma_j) (elementwise over d, r >= j, never above 1),
// Gamma_r = exp(gamma_r), b_r = exp(gamma_C - gamma_r), k^ = rho_k k, q^ = rho_q q:
//   A_rj = beta_r sum_d k^_rd k^_jd E_rjd (j < r),   T = (I + A)^-1 (unit lower triangular)
//   W = T diag(beta) (Gamma .* K^),   U~ = T diag(beta) V,   P_rj = scale sum_d q^_rd k^_jd E_rjd (j <= r)
//   Kbar = b .* K^,   Qg = scale Gamma .* Q^
// and, for one row v of the state S (S = H^T, o_t = S q^_t):
//   u = U~[:, v] - W s_v,   o[:, v] = Qg s_v + P u,   s_v <- Gamma_C .* s_v + Kbar^T u
// The backward scan runs the adjoint of that map over the chunks in reverse:
//   du = P^T do[:, v] + Kbar ds_v,   ds_v <- Gamma_C .* ds_v + Qg^T do[:, v] - W^T du
// and the chunk-local gradients follow from the chunk-start state H0 and the chunk-end state
// gradient dH1 (the derivation is the reverse mode of the equations above; the per-channel
// decay weights make the contractions with E elementwise in d):
//   U = U~ - W H0,  dU = P^T dO + Kbar dH1,  dPs = scale tril(dO U^T),  X = dO H0^T,  Y = U dH1^T
//   dW = -dU H0^T,  Z = T^T dW,  dT = (dU V^T + dW (Gamma .* K^)^T) diag(beta),  dA = -strict_lower(T^T dT T^T)
//   X1_r = sum_{j<=r} dPs_rj k^_j E_rj,  Y1_r = sum_{j<r} dA_rj k^_j E_rj
//   X2_j = sum_{i>=j} dPs_ij q^_i E_ij + sum_{i>j} dA_ij beta_i k^_i E_ij
//   dq^ = scale Gamma X + X1,   dk^ = b Y + beta Gamma Z + beta Y1 + X2,   dv = beta T^T dU
//   dbeta = rowsum(V .* T^T dU) + rowsum(Gamma K^ Z) + rowsum(K^ Y1)
//   dgamma = scale Gamma Q^ X - b K^ Y + beta Gamma K^ Z + Q^ X1 + beta K^ Y1 - K^ X2  (per channel)
//   dgamma_C += sum_r b K^ Y + Gamma_C <dH1, H0> (per channel);  dg = reverse cumsum of dgamma
// (a scalar gate sums dg over the channels). dq, dk then come from the sum of dq^, dk^ over the
// value heads of each key head and the L2-norm backward, as in the sequential VJP.
#include <cuda_runtime.h>
#include <stdint.h>

#include "chunk.h"
#include "common.cuh"
#include "kernels.h"

namespace gdr {
namespace {

constexpr int C = kChunk;
constexpr int kThreads = 256;
constexpr int kGradCtas = 304;  // persistent grad CTAs, one scratch slot each: two per SM of a GB300

// Record of one (b, value head, chunk), fp32, row-major; offsets in floats.
struct RecOff {
    int W, Kb, Qg, Gm, Ut, P, T, n;
};
__host__ __device__ inline RecOff rec_off(int K, int V) {
    RecOff o;
    o.W = 0;
    o.Kb = C * K;
    o.Qg = 2 * C * K;
    o.Gm = 3 * C * K;   // gamma per channel
    o.Ut = 4 * C * K;
    o.P = 4 * C * K + C * V;
    o.T = o.P + C * C;
    o.n = (o.T + C * C + 63) / 64 * 64;
    return o;
}

// Grad scratch of one CTA, offsets in floats: [C][K] and [C][V] planes, [C][C] matrices.
struct GradOff {
    int Kh, Qh, GK, X, Y, dW, Z, X1, Y1, X2, dgam, V, dO, U, dU, TdU, dPs, dT, M1, dA, n;
};
__host__ __device__ inline GradOff grad_off(int K, int V) {
    GradOff o;
    int at = 0;
    auto take = [&](int n) { const int r = at; at += n; return r; };
    o.Kh = take(C * K); o.Qh = take(C * K); o.GK = take(C * K); o.X = take(C * K); o.Y = take(C * K);
    o.dW = take(C * K); o.Z = take(C * K); o.X1 = take(C * K); o.Y1 = take(C * K); o.X2 = take(C * K);
    o.dgam = take(C * K);
    o.V = take(C * V); o.dO = take(C * V); o.U = take(C * V); o.dU = take(C * V); o.TdU = take(C * V);
    o.dPs = take(C * C); o.dT = take(C * C); o.M1 = take(C * C); o.dA = take(C * C);
    o.n = (at + 63) / 64 * 64;
    return o;
}

// ---------------------------------------------------------------------------------------------
// prep: one CTA per (chunk, value head, b) writes the chunk's record.
__global__ void __launch_bounds__(kThreads) prep32_kernel(Chunk32Args A) {
    extern __shared__ float sm[];
    const int K = A.Dk, V = A.Dv, KS = K + 1, VS = V + 1, CS = C + 1;
    const int c = blockIdx.x, hv = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    const int hk = hv / (A.Hv / A.Hk), t0 = c * C, n = min(C, A.T - t0);
    float* sK = sm;              // [C][KS] k^
    float* sQ = sK + C * KS;     // [C][KS] q^, later beta Gamma k^
    float* sG = sQ + C * KS;     // [C][KS] g, then gamma
    float* sV = sG + C * KS;     // [C][VS]
    float* sA = sV + C * VS;     // [C][CS]
    float* sT = sA + C * CS;     // [C][CS]
    float* sb = sT + C * CS;     // [C] beta
    float* srk = sb + C;         // [C]
    float* srq = srk + C;        // [C]
    const RecOff ro = rec_off(K, V);
    float* rec = A.rec + (((size_t)b * A.Hv + hv) * A.NC + c) * ro.n;

    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, d = i % K;
        const bool in = r < n;
        const size_t tok = (size_t)b * A.T + t0 + r;
        const size_t xi = (tok * A.Hk + hk) * K + d;
        sK[r * KS + d] = in ? A.k[xi] : 0.f;
        sQ[r * KS + d] = in ? A.q[xi] : 0.f;
        sG[r * KS + d] = !in ? 0.f : A.channel ? A.g[(tok * A.Hv + hv) * K + d] : A.g[tok * A.Hv + hv];
    }
    for (int i = tid; i < C * V; i += kThreads) {
        const int r = i / V, d = i % V;
        sV[r * VS + d] = r < n ? A.v[(((size_t)b * A.T + t0 + r) * A.Hv + hv) * V + d] : 0.f;
    }
    if (tid < C) sb[tid] = tid < n ? A.beta[((size_t)b * A.T + t0 + tid) * A.Hv + hv] : 0.f;
    __syncthreads();
    {  // norm factors, one warp per row
        const int warp = tid >> 5, lane = tid & 31;
        for (int r = warp; r < C; r += kThreads / 32) {
            float sk = 0.f, sq = 0.f;
            for (int d = lane; d < K; d += 32) {
                sk += sK[r * KS + d] * sK[r * KS + d];
                sq += sQ[r * KS + d] * sQ[r * KS + d];
            }
            sk = warp_sum(sk);
            sq = warp_sum(sq);
            if (lane == 0) {
                srk[r] = A.use_norm ? 1.0f / sqrtf(sk + 1e-6f) : 1.0f;
                srq[r] = A.use_norm ? 1.0f / sqrtf(sq + 1e-6f) : 1.0f;
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, d = i % K;
        sK[r * KS + d] *= srk[r];
        sQ[r * KS + d] *= srq[r];
    }
    if (tid < K) {  // gamma: in-chunk cumulative sum per channel
        float acc = 0.f;
        for (int r = 0; r < C; r++) {
            acc += sG[r * KS + tid];
            sG[r * KS + tid] = acc;
        }
    }
    __syncthreads();
    // A (strictly lower, into sA) and P (lower with the diagonal, straight to the record)
    for (int i = tid; i < C * C; i += kThreads) {
        const int r = i / C, j = i % C;
        float a = 0.f, p = 0.f;
        if (j <= r) {
            if (A.channel) {
                for (int d = 0; d < K; d++) {
                    const float e = expf(sG[r * KS + d] - sG[j * KS + d]);
                    const float kj = sK[j * KS + d] * e;
                    a += sK[r * KS + d] * kj;
                    p += sQ[r * KS + d] * kj;
                }
            } else {
                for (int d = 0; d < K; d++) {
                    a += sK[r * KS + d] * sK[j * KS + d];
                    p += sQ[r * KS + d] * sK[j * KS + d];
                }
                const float e = expf(sG[r * KS] - sG[j * KS]);
                a *= e;
                p *= e;
            }
        }
        sA[r * CS + j] = j < r ? sb[r] * a : 0.f;
        rec[ro.P + r * C + j] = j <= r ? A.scale * p : 0.f;
    }
    __syncthreads();
    if (tid < C) {  // T = (I + A)^-1 by forward substitution, thread j solves column j
        const int j = tid;
        for (int r = 0; r < C; r++) {
            float x = r == j ? 1.f : 0.f;
            for (int m = 0; m < r; m++)
                if (m >= j) x -= sA[r * CS + m] * sT[m * CS + j];
            sT[r * CS + j] = r < j ? 0.f : x;
        }
    }
    for (int i = tid; i < C * K; i += kThreads) {  // elementwise records; sQ becomes beta Gamma k^
        const int r = i / K, d = i % K;
        const float gr = sG[r * KS + d], gc = sG[(C - 1) * KS + d], Gr = expf(gr);
        rec[ro.Qg + r * K + d] = A.scale * Gr * sQ[r * KS + d];
        rec[ro.Kb + r * K + d] = expf(gc - gr) * sK[r * KS + d];
        rec[ro.Gm + r * K + d] = gr;
        sQ[r * KS + d] = sb[r] * Gr * sK[r * KS + d];
    }
    __syncthreads();
    for (int i = tid; i < C * C; i += kThreads) rec[ro.T + i] = sT[(i / C) * CS + i % C];
    for (int i = tid; i < C * K; i += kThreads) {  // W = T (beta Gamma k^)
        const int r = i / K, d = i % K;
        float w = 0.f;
        for (int j = 0; j <= r; j++) w += sT[r * CS + j] * sQ[j * KS + d];
        rec[ro.W + i] = w;
    }
    for (int i = tid; i < C * V; i += kThreads) {  // U~ = T diag(beta) V
        const int r = i / V, d = i % V;
        float u = 0.f;
        for (int j = 0; j <= r; j++) u += sT[r * CS + j] * sb[j] * sV[j * VS + d];
        rec[ro.Ut + i] = u;
    }
}

// ---------------------------------------------------------------------------------------------
// scans: sequential over the chunks; one CTA per (16 state rows, value head, b), warp w owns
// row v = 16 blockIdx.x + w, lane l its columns l + 32 m.
// MODE 0: forward with o (and the chunk-start states when A.states is set); 1: chunk-start
// states only; 2: reverse (chunk-end state gradients into A.dstates, dh0).
constexpr int kScanThreads = 512;
constexpr int kRowsPerCta = kScanThreads / 32;

template <int MODE>
__global__ void __launch_bounds__(kScanThreads) scan32_kernel(Chunk32Args A) {
    extern __shared__ float sm[];
    const int K = A.Dk, V = A.Dv, KS = K + 1, CS = C + 1, R = kRowsPerCta;
    const int hv = blockIdx.y, b = blockIdx.z, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.x * R, v = v0 + warp;
    const size_t bh = (size_t)b * A.Hv + hv;
    // What a mode does not use takes no room: the reverse scan reads P from the record (L2) and
    // keeps no outputs, so two of its CTAs share an SM and its grid is one wave.
    float* sW = sm;                                // [C][KS]
    float* sKb = sW + C * KS;                      // [C][KS]
    float* sQg = sKb + C * KS;                     // [C][KS] (forward with outputs, reverse)
    float* sP = sQg + (MODE != 1 ? C * KS : 0);    // [C][CS] (forward with outputs)
    float* sX = sP + (MODE == 0 ? C * CS : 0);    // [C][R] U~ (forward) or dO (reverse) columns of the rows
    float* sS = sX + C * R;       // [R][K] state (gradient) rows
    float* sU = sS + R * K;       // [R][C] u or du per row
    float* sO = sU + R * C;       // [C][R] outputs (forward with outputs)
    const RecOff ro = rec_off(K, V);
    const int M = K / 32;
    float s[4];
    const float* init = MODE == 2 ? A.dht : A.h0;
    for (int m = 0; m < M; m++) {
        s[m] = init ? init[(bh * V + v) * K + lane + 32 * m] : 0.f;
        sS[warp * K + lane + 32 * m] = s[m];
    }
    for (int step = 0; step < A.NC; step++) {
        const int c = MODE == 2 ? A.NC - 1 - step : step;
        const int t0 = c * C, n = min(C, A.T - t0);
        const float* rec = A.rec + (bh * A.NC + c) * ro.n;
        if (tid == 0 && step + 1 < A.NC) {  // the next step's record into L2 while this one is read
            const int cn = MODE == 2 ? c - 1 : c + 1;
            const float* nrec = A.rec + (bh * A.NC + cn) * ro.n;
            for (int o = 0; o < 3 * C * K; o += 8192)  // W, Kbar, Qg
                bulk_prefetch_l2(nrec + o, (uint32_t)min(8192, 3 * C * K - o) * 4);
            bulk_prefetch_l2(nrec + ro.Gm + (C - 1) * K, K * 4);
            bulk_prefetch_l2(nrec + ro.Ut, (C * V + C * C) * 4);  // U~ and P
        }
        for (int i4 = tid; i4 < C * K / 4; i4 += kScanThreads) {  // 16-byte loads, padded rows in smem
            const int i = 4 * i4, r = i / K, d = i % K;
            const float4 w = *reinterpret_cast<const float4*>(rec + ro.W + i);
            const float4 kb = *reinterpret_cast<const float4*>(rec + ro.Kb + i);
            float* pw = sW + r * KS + d;
            float* pk = sKb + r * KS + d;
            pw[0] = w.x; pw[1] = w.y; pw[2] = w.z; pw[3] = w.w;
            pk[0] = kb.x; pk[1] = kb.y; pk[2] = kb.z; pk[3] = kb.w;
            if (MODE != 1) {
                const float4 q = *reinterpret_cast<const float4*>(rec + ro.Qg + i);
                float* pq = sQg + r * KS + d;
                pq[0] = q.x; pq[1] = q.y; pq[2] = q.z; pq[3] = q.w;
            }
        }
        if (MODE == 0)
            for (int i4 = tid; i4 < C * C / 4; i4 += kScanThreads) {
                const int i = 4 * i4;
                const float4 x = *reinterpret_cast<const float4*>(rec + ro.P + i);
                float* pp = sP + (i / C) * CS + i % C;
                pp[0] = x.x; pp[1] = x.y; pp[2] = x.z; pp[3] = x.w;
            }
        float gc[4];  // Gamma_C of this lane's state columns
        for (int m = 0; m < M; m++) gc[m] = expf(rec[ro.Gm + (C - 1) * K + lane + 32 * m]);
        for (int i = tid; i < C * R; i += kScanThreads) {
            const int r = i / R, w = i % R;
            if (MODE == 2)
                sX[i] = r < n ? A.do_[(((size_t)b * A.T + t0 + r) * A.Hv + hv) * V + v0 + w] : 0.f;
            else
                sX[i] = rec[ro.Ut + r * V + v0 + w];
        }
        __syncthreads();
        float* keep = MODE == 2 ? A.dstates : A.states;
        if (keep)
            for (int m = 0; m < M; m++) keep[((bh * A.NC + c) * V + v) * K + lane + 32 * m] = s[m];
        const float* srow = sS + warp * K;
        float* urow = sU + warp * C;
        if (MODE != 2) {
            for (int i = lane; i < C; i += 32) {  // u = U~ - W s
                float acc = 0.f;
                for (int d = 0; d < K; d++) acc += sW[i * KS + d] * srow[d];
                urow[i] = sX[i * R + warp] - acc;
            }
            __syncwarp();
            if (MODE == 0)
                for (int i = lane; i < C; i += 32) {  // o = Qg s + P u
                    float acc = 0.f;
                    for (int d = 0; d < K; d++) acc += sQg[i * KS + d] * srow[d];
                    for (int j = 0; j <= i; j++) acc += sP[i * CS + j] * urow[j];
                    sO[i * R + warp] = acc;
                }
            for (int m = 0; m < M; m++) {  // s <- Gamma_C s + Kbar^T u
                const int d = lane + 32 * m;
                float acc = 0.f;
                for (int i = 0; i < C; i++) acc += sKb[i * KS + d] * urow[i];
                s[m] = gc[m] * s[m] + acc;
            }
        } else {
            const float* prec = rec + ro.P;  // P [C][C] row-major: lanes read a row's consecutive entries
            for (int i = lane; i < C; i += 32) {  // du = P^T do + Kbar ds
                float acc = 0.f;
                for (int j = i; j < C; j++) acc += prec[j * C + i] * sX[j * R + warp];
                for (int d = 0; d < K; d++) acc += sKb[i * KS + d] * srow[d];
                urow[i] = acc;
            }
            __syncwarp();
            for (int m = 0; m < M; m++) {  // ds <- Gamma_C ds + Qg^T do - W^T du
                const int d = lane + 32 * m;
                float acc = 0.f;
                for (int i = 0; i < C; i++) acc += sQg[i * KS + d] * sX[i * R + warp] - sW[i * KS + d] * urow[i];
                s[m] = gc[m] * s[m] + acc;
            }
        }
        __syncthreads();
        if (MODE == 0)
            for (int i = tid; i < n * R; i += kScanThreads) {
                const int r = i / R, w = i % R;
                A.o[(((size_t)b * A.T + t0 + r) * A.Hv + hv) * V + v0 + w] = sO[i];
            }
        for (int m = 0; m < M; m++) sS[warp * K + lane + 32 * m] = s[m];
        __syncthreads();
    }
    float* fin = MODE == 2 ? A.dh0 : A.ht;
    if (fin)
        for (int m = 0; m < M; m++) fin[(bh * V + v) * K + lane + 32 * m] = s[m];
}

// ---------------------------------------------------------------------------------------------
// grad: persistent CTAs over the (b, value head, chunk) units, each unit a sequence of block-wide
// products through the CTA's scratch slot (fixed summation order: deterministic).

// out[m][n] = alpha * sum_k a[m*ars + k*acs] * b[k*brs + n*bcs] (+ out when acc) for m < 64,
// n < Nc, over the outputs allowed by tri (0: all, 1: n <= m, 2: n < m; the others are set to
// zero). Tiles of 64 x 64 outputs, 4 x 4 per thread, with 16-deep slices of both operands staged
// in shared memory (each loaded along its contiguous index); the sum over k runs in a fixed
// order, so results are deterministic.
__device__ void bmm(int Nc, int Kd, const float* a, int ars, int acs, const float* bm, int brs, int bcs, float* out,
                    float alpha, bool acc, int tri = 0) {
    __shared__ float sa[16][C + 1], sbm[16][C + 1];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    for (int n0 = 0; n0 < Nc; n0 += C) {
        float r[4][4];
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) r[i][j] = 0.f;
        for (int k0 = 0; k0 < Kd; k0 += 16) {
            __syncthreads();
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const int i = tid + kThreads * e;  // 1024 elements of each 16 x 64 slice
                const int kk = acs == 1 ? i & 15 : i >> 6, m = acs == 1 ? i >> 4 : i & 63;
                sa[kk][m] = a[m * ars + (k0 + kk) * acs];
                const int kb = bcs == 1 ? i >> 6 : i & 15, nn = bcs == 1 ? i & 63 : i >> 4;
                sbm[kb][nn] = n0 + nn < Nc ? bm[(k0 + kb) * brs + (n0 + nn) * bcs] : 0.f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < 16; kk++) {
                float av[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; i++) av[i] = sa[kk][4 * ty + i];
#pragma unroll
                for (int j = 0; j < 4; j++) bv[j] = sbm[kk][tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int j = 0; j < 4; j++) r[i][j] += av[i] * bv[j];
            }
        }
#pragma unroll
        for (int i = 0; i < 4; i++)
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int m = 4 * ty + i, nn = n0 + tx + 16 * j;
                if (nn >= Nc) continue;
                const bool live = tri == 0 || (tri == 1 ? nn <= m : nn < m);
                const float v = live ? alpha * r[i][j] : 0.f;
                out[m * Nc + nn] = acc ? out[m * Nc + nn] + v : v;
            }
    }
}

__global__ void __launch_bounds__(kThreads) grad32_kernel(Chunk32Args A) {
    __shared__ float sb[C], srk[C], srq[C];
    const int K = A.Dk, V = A.Dv, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const RecOff ro = rec_off(K, V);
    const GradOff go = grad_off(K, V);
    float* w = A.scratch + (size_t)blockIdx.x * go.n;
    float *Kh = w + go.Kh, *Qh = w + go.Qh, *GK = w + go.GK, *X = w + go.X, *Y = w + go.Y, *dW = w + go.dW;
    float *Z = w + go.Z, *X1 = w + go.X1, *Y1 = w + go.Y1, *X2 = w + go.X2, *dgam = w + go.dgam;
    float *Vm = w + go.V, *dO = w + go.dO, *U = w + go.U, *dU = w + go.dU, *TdU = w + go.TdU;
    float *dPs = w + go.dPs, *dT = w + go.dT, *M1 = w + go.M1, *dA = w + go.dA;
    const int units = A.B * A.Hv * A.NC;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const int c = u % A.NC, hv = (u / A.NC) % A.Hv, b = u / (A.NC * A.Hv);
        const int hk = hv / (A.Hv / A.Hk), t0 = c * C, n = min(C, A.T - t0);
        const size_t bh = (size_t)b * A.Hv + hv;
        const float* rec = A.rec + (bh * A.NC + c) * ro.n;
        const float* H0 = A.states + (bh * A.NC + c) * (size_t)V * K;   // [V][K]
        const float* dH1 = A.dstates + (bh * A.NC + c) * (size_t)V * K; // [V][K]
        const float *W = rec + ro.W, *Kb = rec + ro.Kb, *Gm = rec + ro.Gm, *Ut = rec + ro.Ut;
        const float *P = rec + ro.P, *Tm = rec + ro.T;
        auto tok = [&](int r) { return (size_t)b * A.T + t0 + r; };
        // inputs of the unit (zero beyond the last token)
        for (int i = tid; i < C * K; i += kThreads) {
            const int r = i / K, d = i % K;
            const size_t xi = (tok(r) * A.Hk + hk) * K + d;
            Kh[i] = r < n ? A.k[xi] : 0.f;
            Qh[i] = r < n ? A.q[xi] : 0.f;
        }
        for (int i = tid; i < C * V; i += kThreads) {
            const int r = i / V, d = i % V;
            const size_t xi = (tok(r) * A.Hv + hv) * V + d;
            Vm[i] = r < n ? A.v[xi] : 0.f;
            dO[i] = r < n ? A.do_[xi] : 0.f;
        }
        if (tid < C) sb[tid] = tid < n ? A.beta[tok(tid) * A.Hv + hv] : 0.f;
        __syncthreads();
        for (int r = warp; r < C; r += kThreads / 32) {
            float sk = 0.f, sq = 0.f;
            for (int d = lane; d < K; d += 32) {
                sk += Kh[r * K + d] * Kh[r * K + d];
                sq += Qh[r * K + d] * Qh[r * K + d];
            }
            sk = warp_sum(sk);
            sq = warp_sum(sq);
            if (lane == 0) {
                srk[r] = A.use_norm ? 1.0f / sqrtf(sk + 1e-6f) : 1.0f;
                srq[r] = A.use_norm ? 1.0f / sqrtf(sq + 1e-6f) : 1.0f;
            }
        }
        __syncthreads();
        for (int i = tid; i < C * K; i += kThreads) {
            const int r = i / K;
            Kh[i] *= srk[r];
            Qh[i] *= srq[r];
            GK[i] = expf(Gm[i]) * Kh[i];
        }
        __syncthreads();
        // U = U~ - W H0;  dU = P^T dO + Kbar dH1;  X = dO H0
        bmm(V, K, W, K, 1, H0, 1, K, U, -1.f, false);
        bmm(V, C, P, 1, C, dO, V, 1, dU, 1.f, false);
        bmm(K, V, dO, V, 1, H0, K, 1, X, 1.f, false);
        __syncthreads();
        for (int i = tid; i < C * V; i += kThreads) U[i] += Ut[i];
        bmm(V, K, Kb, K, 1, dH1, 1, K, dU, 1.f, true);
        __syncthreads();
        // Y = U dH1;  dW = -dU H0;  dPs = scale tril(dO U^T);  T^T dU
        bmm(K, V, U, V, 1, dH1, K, 1, Y, 1.f, false);
        bmm(K, V, dU, V, 1, H0, K, 1, dW, -1.f, false);
        bmm(C, V, dO, V, 1, U, 1, V, dPs, A.scale, false, 1);
        bmm(V, C, Tm, 1, C, dU, V, 1, TdU, 1.f, false);
        __syncthreads();
        // Z = T^T dW;  dT = dU V^T + dW (Gamma k^)^T  (columns scaled by beta below)
        bmm(K, C, Tm, 1, C, dW, K, 1, Z, 1.f, false);
        bmm(C, V, dU, V, 1, Vm, 1, V, dT, 1.f, false);
        __syncthreads();
        bmm(C, K, dW, K, 1, GK, 1, K, dT, 1.f, true);
        __syncthreads();
        for (int i = tid; i < C * C; i += kThreads) dT[i] *= sb[i % C];
        __syncthreads();
        bmm(C, C, Tm, 1, C, dT, C, 1, M1, 1.f, false);  // T^T dT
        __syncthreads();
        bmm(C, C, M1, C, 1, Tm, 1, C, dA, -1.f, false, 2);  // -strict_lower(T^T dT T^T)
        __syncthreads();
        // the decay-weighted contractions (E elementwise per channel)
        for (int i = tid; i < C * K; i += kThreads) {
            const int r = i / K, d = i % K;
            const float gr = Gm[i];
            float x1 = 0.f, y1 = 0.f, x2 = 0.f;
            for (int j = 0; j <= r; j++) {  // row side: j <= r
                const float ke = Kh[j * K + d] * expf(gr - Gm[j * K + d]);
                x1 += dPs[r * C + j] * ke;
                y1 += dA[r * C + j] * ke;
            }
            for (int ii = r; ii < C; ii++) {  // column side: rows ii >= r of column r
                const float e = expf(Gm[ii * K + d] - gr);
                x2 += (dPs[ii * C + r] * Qh[ii * K + d] + dA[ii * C + r] * sb[ii] * Kh[ii * K + d]) * e;
            }
            X1[i] = x1;
            Y1[i] = y1;
            X2[i] = x2;
        }
        __syncthreads();
        for (int i = tid; i < C * K; i += kThreads) {
            const int r = i / K, d = i % K;
            const float Gr = expf(Gm[i]), bd = expf(Gm[(C - 1) * K + d] - Gm[i]), be = sb[r];
            const float dq = A.scale * Gr * X[i] + X1[i];
            const float dk = bd * Y[i] + be * Gr * Z[i] + be * Y1[i] + X2[i];
            dgam[i] = A.scale * Gr * Qh[i] * X[i] - bd * Kh[i] * Y[i] + be * Gr * Kh[i] * Z[i] + Qh[i] * X1[i] +
                      be * Kh[i] * Y1[i] - Kh[i] * X2[i];
            if (r < n) {
                const size_t xi = (tok(r) * A.Hv + hv) * K + d;
                A.dqh[xi] = dq;
                A.dkh[xi] = dk;
            }
        }
        for (int i = tid; i < n * V; i += kThreads) A.dv[(tok(i / V) * A.Hv + hv) * V + i % V] = sb[i / V] * TdU[i];
        __syncthreads();
        for (int d = tid; d < K; d += kThreads) {  // dgamma_C, then dg = reverse cumsum + dgamma_C
            const float GC = expf(Gm[(C - 1) * K + d]);
            float gc = 0.f, hd = 0.f;
            for (int r = 0; r < C; r++) gc += expf(Gm[(C - 1) * K + d] - Gm[r * K + d]) * Kh[r * K + d] * Y[r * K + d];
            for (int vv = 0; vv < V; vv++) hd += dH1[vv * K + d] * H0[vv * K + d];
            gc += GC * hd;
            float acc = 0.f;
            for (int r = C - 1; r >= 0; r--) {
                acc += dgam[r * K + d];
                dgam[r * K + d] = acc + gc;
            }
        }
        __syncthreads();
        for (int r = warp; r < n; r += kThreads / 32) {  // dbeta, and dg of a scalar gate
            float db = 0.f, dg = 0.f;
            for (int d = lane; d < V; d += 32) db += Vm[r * V + d] * TdU[r * V + d];
            for (int d = lane; d < K; d += 32) {
                db += (expf(Gm[r * K + d]) * Z[r * K + d] + Y1[r * K + d]) * Kh[r * K + d];
                dg += dgam[r * K + d];
            }
            db = warp_sum(db);
            dg = warp_sum(dg);
            const size_t ti = tok(r) * A.Hv + hv;
            if (lane == 0) {
                A.dbeta[ti] = db;
                if (!A.channel) A.dg[ti] = dg;
            }
            if (A.channel)
                for (int d = lane; d < K; d += 32) A.dg[ti * K + d] = dgam[r * K + d];
        }
        __syncthreads();
    }
}

size_t rec_bytes(int B, int Hv, int NC, int Dk, int Dv) {
    return (size_t)B * Hv * NC * rec_off(Dk, Dv).n * sizeof(float);
}

}  // namespace

Chunk32Layout chunk32_layout(int B, int T, int Hv, int Dk, int Dv, bool bwd, bool own_rec, bool own_states) {
    Chunk32Layout l;
    const int NC = (T + C - 1) / C;
    const size_t plane = (size_t)B * Hv * NC * Dv * Dk * sizeof(float);
    const size_t per_tok = (size_t)B * T * Hv * Dk * sizeof(float);
    size_t at = 256;  // status word
    auto take = [&](size_t bytes) {
        const size_t r = at;
        at = round_up(at + bytes, 256);
        return r;
    };
    l.rec = l.states = l.dstates = l.dqh = l.dkh = l.scratch = 0;
    l.nscratch = 0;
    if (own_rec) l.rec = take(rec_bytes(B, Hv, NC, Dk, Dv));
    if (bwd) {
        if (own_states) l.states = take(plane);
        l.dstates = take(plane);
        l.dqh = take(per_tok);
        l.dkh = take(per_tok);
        const long units = (long)B * Hv * NC;
        l.nscratch = (int)(units < kGradCtas ? units : kGradCtas);
        l.scratch = take((size_t)l.nscratch * grad_off(Dk, Dv).n * sizeof(float));
    }
    l.total = at;
    return l;
}

size_t chunk32_states_bytes(int B, int T, int Hv, int Dk, int Dv) {
    const int NC = (T + C - 1) / C;
    return (size_t)B * Hv * NC * Dv * Dk * sizeof(float);
}

// The forward's saved buffer on this path: the records, then the chunk-start states.
size_t chunk32_saved_states_offset(int B, int T, int Hv, int Dk, int Dv) {
    return round_up(rec_bytes(B, Hv, (T + C - 1) / C, Dk, Dv), 256);
}
size_t chunk32_saved_bytes(int B, int T, int Hv, int Dk, int Dv) {
    return chunk32_saved_states_offset(B, T, Hv, Dk, Dv) + chunk32_states_bytes(B, T, Hv, Dk, Dv);
}

namespace {
size_t prep_smem(int K, int V) { return (size_t)(3 * C * (K + 1) + C * (V + 1) + 2 * C * (C + 1) + 3 * C) * 4; }
size_t scan_smem(int K, int mode) {  // the carve-up of scan32_kernel<mode>
    const int R = kRowsPerCta;
    const int ops = (mode == 1 ? 2 : 3) * C * (K + 1) + (mode == 0 ? C * (C + 1) : 0);
    return (size_t)(ops + C * R + R * K + R * C + (mode == 0 ? C * R : 0)) * 4;
}
cudaError_t run_prep(const Chunk32Args& a, cudaStream_t s) {
    const size_t smem = prep_smem(a.Dk, a.Dv);
    cudaError_t e = cudaFuncSetAttribute(prep32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin("chunk32_prep", s);
    prep32_kernel<<<dim3(a.NC, a.Hv, a.B), kThreads, smem, s>>>(a);
    trace_end(s);
    return cudaGetLastError();
}
template <int MODE>
cudaError_t run_scan(const Chunk32Args& a, cudaStream_t s) {
    const size_t smem = scan_smem(a.Dk, MODE);
    cudaError_t e = cudaFuncSetAttribute(scan32_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin(MODE == 0 ? "chunk32_scan_fwd" : MODE == 1 ? "chunk32_scan_states" : "chunk32_scan_bwd", s);
    scan32_kernel<MODE><<<dim3(a.Dv / kRowsPerCta, a.Hv, a.B), kScanThreads, smem, s>>>(a);  // Dv in {32, 64, 128}
    trace_end(s);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_chunk32_fwd(const Chunk32Args& a, bool prep, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (prep && (e = run_prep(a, s)) != cudaSuccess) return e;
    return run_scan<0>(a, s);
}

cudaError_t launch_chunk32_bwd(const Chunk32Args& a, bool prep, bool states_scan, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (prep && (e = run_prep(a, s)) != cudaSuccess) return e;
    if (states_scan && (e = run_scan<1>(a, s)) != cudaSuccess) return e;
    if ((e = run_scan<2>(a, s)) != cudaSuccess) return e;
    trace_begin("chunk32_grad", s);
    grad32_kernel<<<a.nscratch, kThreads, 0, s>>>(a);
    trace_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    SeqBwdArgs f;
    f.B = a.B; f.T = a.T; f.Hk = a.Hk; f.Hv = a.Hv; f.Dk = a.Dk; f.Dv = a.Dv;
    f.channel = a.channel; f.use_norm = a.use_norm; f.bf16 = 0; f.scale = a.scale;
    f.q = a.q; f.k = a.k; f.v = a.v; f.do_ = a.do_; f.g = a.g; f.beta = a.beta; f.h0 = a.h0; f.dht = a.dht;
    f.dq = a.dq; f.dk = a.dk; f.dv = a.dv; f.dg = a.dg; f.dbeta = a.dbeta; f.dh0 = a.dh0;
    f.ckpt = f.segs = f.dah = nullptr;
    f.dqh = a.dqh; f.dkh = a.dkh;
    return launch_head_sum_norm_backward(f, s);
}

}  // namespace gdr
