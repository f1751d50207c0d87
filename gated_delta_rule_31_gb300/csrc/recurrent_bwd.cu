// recurrent_bwd.cu - sequential (token-by-token) VJP of the gated delta rule, the "sequential
// case" of "Adding VJP for gated delta net" (MLX PR #4565): the reverse-mode recurrence on
// the CUDA cores, for every dtype, gate (scalar or per key channel) and Dk, Dv in {32, 64, 128}.
//
// Rows of the state evolve independently: per row v, p = S_v . (a .* k^), delta = beta (v_v - p),
// S_v <- a .* S_v + delta k^. So one CTA per (b, hv) gives each warp 8 rows; lane l holds columns
// l + 32 c. Reverse mode per token t, row v, with Gb = dL/dS_t (rows of the adjoint):
//   Gb_v += scale do_v q^;  dq^ += scale do_v S_t,v;  dd = Gb_v . k^;  dk^ += delta_v Gb_v
//   dbeta += dd (v_v - p_v);  dv_v = beta dd;  dp = -beta dd;  Gd = Gb_v + dp k^
//   dk^ += dp a .* S_(t-1),v;  da += Gd .* S_(t-1),v;  Gb_v <- Gd .* a;   dg = a .* da
// (scalar gate: dg = a sum_k da_k). The terms summed over rows (dq^, dk^, da, dbeta) go through
// shared memory once per token in a fixed order (deterministic). S_(t-1) comes from a forward
// pass that checkpoints the state every 64 tokens and, per 64-token segment in reverse,
// recomputes the segment's states into workspace. A second kernel sums dq^, dk^ over the value
// heads of each key head and applies the norm backward dx = rho (dx^ - x^ (x^ . dx^)).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace gdr {
namespace {

constexpr int kSeg = 64;   // tokens per checkpoint segment
constexpr int kRows = 8;   // state rows per warp

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <int DK, typename TIn>
struct TokenIn {  // this lane's columns of the token's key-side vectors
    static constexpr int CPL = DK / 32;
    float k[CPL], q[CPL], a[CPL], ak[CPL];
    float beta, ga;  // ga: the scalar gate's a (channel gate: unused)
};

// Raw inputs of token t (this lane's columns of k, q, g; beta): loaded one token ahead.
template <int DK>
struct TokenRaw {
    float k[DK / 32], q[DK / 32], g[DK / 32], beta;
};
template <int DK, typename TIn>
__device__ __forceinline__ void load_raw(const SeqBwdArgs& A, int b, int hk, int hv, int t, int lane,
                                         TokenRaw<DK>& r, bool need_q) {
    constexpr int CPL = DK / 32;
    const TIn* kp = static_cast<const TIn*>(A.k) + (((size_t)b * A.T + t) * A.Hk + hk) * DK;
    const TIn* qp = static_cast<const TIn*>(A.q) + (((size_t)b * A.T + t) * A.Hk + hk) * DK;
    const size_t bt = ((size_t)b * A.T + t) * A.Hv + hv;
#pragma unroll
    for (int c = 0; c < CPL; c++) {
        r.k[c] = ldf(kp + lane + 32 * c);
        r.q[c] = need_q ? ldf(qp + lane + 32 * c) : 0.f;
        r.g[c] = A.channel ? A.g[bt * DK + lane + 32 * c] : (c == 0 ? A.g[bt] : 0.f);
    }
    r.beta = A.beta[bt];
}

// k^, q^ (normalised when asked), a = exp(g) and beta of a token from its raw inputs.
template <int DK, typename TIn>
__device__ __forceinline__ void load_token(const SeqBwdArgs& A, const TokenRaw<DK>& r, TokenIn<DK, TIn>& x,
                                           bool need_q) {
    constexpr int CPL = DK / 32;
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; c++) {
        x.k[c] = r.k[c];
        sk += x.k[c] * x.k[c];
        if (need_q) {
            x.q[c] = r.q[c];
            sq += x.q[c] * x.q[c];
        }
    }
    if (A.use_norm) {
        const float rk = 1.0f / sqrtf(warp_sum(sk) + 1e-6f);
#pragma unroll
        for (int c = 0; c < CPL; c++) x.k[c] *= rk;
        if (need_q) {
            const float rq = 1.0f / sqrtf(warp_sum(sq) + 1e-6f);
#pragma unroll
            for (int c = 0; c < CPL; c++) x.q[c] *= rq;
        }
    }
    if (A.channel) {
#pragma unroll
        for (int c = 0; c < CPL; c++) x.a[c] = expf(r.g[c]);
        x.ga = 0.f;
    } else {
        x.ga = expf(r.g[0]);
#pragma unroll
        for (int c = 0; c < CPL; c++) x.a[c] = x.ga;
    }
#pragma unroll
    for (int c = 0; c < CPL; c++) x.ak[c] = x.a[c] * x.k[c];
    x.beta = r.beta;
}

template <int DK, typename TIn>
__global__ void __launch_bounds__(512) seq_bwd_kernel(SeqBwdArgs A) {
    constexpr int CPL = DK / 32;
    constexpr int NRED = 3 * DK + 1;  // per warp and token: dq^, dk^, da (per column), dbeta
    extern __shared__ float red[];     // [2][nwarps][NRED]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nw = blockDim.x >> 5;
    const int bh = blockIdx.x, b = bh / A.Hv, hv = bh % A.Hv, hk = hv / (A.Hv / A.Hk);
    const int row0 = warp * kRows;
    const int Dv = A.Dv, T = A.T;
    const int nseg = (T + kSeg - 1) / kSeg;
    const size_t plane = (size_t)Dv * DK;  // one state, fp32
    float* ckpt = A.ckpt + (size_t)bh * nseg * plane;
    float* segs = A.segs + (size_t)bh * kSeg * plane;
    const TIn* vp = static_cast<const TIn*>(A.v);
    const TIn* dop = static_cast<const TIn*>(A.do_);

    float S[kRows][CPL], Gb[kRows][CPL];
#pragma unroll
    for (int r = 0; r < kRows; r++)
#pragma unroll
        for (int c = 0; c < CPL; c++)
            S[r][c] = A.h0 ? A.h0[(size_t)bh * plane + (size_t)(row0 + r) * DK + lane + 32 * c] : 0.f;

    auto step = [&](const TokenIn<DK, TIn>& x, int t, float* Srow_store) {
        // forward step of this warp's rows; optionally stores the state entering the token
#pragma unroll
        for (int r = 0; r < kRows; r++) {
            float pp = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; c++) {
                if (Srow_store) Srow_store[(size_t)(row0 + r) * DK + lane + 32 * c] = S[r][c];
                pp += S[r][c] * x.ak[c];
            }
            const float p = warp_sum(pp);
            const float vv = ldf(vp + (((size_t)b * T + t) * A.Hv + hv) * Dv + row0 + r);
            const float delta = x.beta * (vv - p);
#pragma unroll
            for (int c = 0; c < CPL; c++) S[r][c] = x.a[c] * S[r][c] + delta * x.k[c];
        }
    };

    // ---- forward pass: checkpoint the state entering every segment
    TokenRaw<DK> cur, nxt;
    load_raw<DK, TIn>(A, b, hk, hv, 0, lane, cur, false);
    for (int t = 0; t < T; t++) {
        if (t + 1 < T) load_raw<DK, TIn>(A, b, hk, hv, t + 1, lane, nxt, false);
        TokenIn<DK, TIn> x;
        load_token<DK, TIn>(A, cur, x, false);
        step(x, t, (t % kSeg) == 0 ? ckpt + (size_t)(t / kSeg) * plane : nullptr);
        cur = nxt;
    }

    // ---- reverse pass
#pragma unroll
    for (int r = 0; r < kRows; r++)
#pragma unroll
        for (int c = 0; c < CPL; c++)
            Gb[r][c] = A.dht ? A.dht[(size_t)bh * plane + (size_t)(row0 + r) * DK + lane + 32 * c] : 0.f;
    for (int sg = nseg - 1; sg >= 0; sg--) {
        const int t0 = sg * kSeg, t1 = min(T, t0 + kSeg);
        // recompute the segment, keeping the state entering each token
#pragma unroll
        for (int r = 0; r < kRows; r++)
#pragma unroll
            for (int c = 0; c < CPL; c++)
                S[r][c] = ckpt[(size_t)sg * plane + (size_t)(row0 + r) * DK + lane + 32 * c];
        load_raw<DK, TIn>(A, b, hk, hv, t0, lane, cur, false);
        for (int t = t0; t < t1; t++) {
            if (t + 1 < t1) load_raw<DK, TIn>(A, b, hk, hv, t + 1, lane, nxt, false);
            TokenIn<DK, TIn> x;
            load_token<DK, TIn>(A, cur, x, false);
            step(x, t, segs + (size_t)(t - t0) * plane);
            cur = nxt;
        }
        load_raw<DK, TIn>(A, b, hk, hv, t1 - 1, lane, cur, true);
        for (int t = t1 - 1; t >= t0; t--) {
            if (t - 1 >= t0) load_raw<DK, TIn>(A, b, hk, hv, t - 1, lane, nxt, true);
            TokenIn<DK, TIn> x;
            load_token<DK, TIn>(A, cur, x, true);
            const float* Sp_all = segs + (size_t)(t - t0) * plane;
            float dq[CPL], dk[CPL], da[CPL], dbeta = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; c++) dq[c] = dk[c] = da[c] = 0.f;
            const size_t vt = (((size_t)b * T + t) * A.Hv + hv) * Dv + row0;
#pragma unroll
            for (int r = 0; r < kRows; r++) {
                float Sp[CPL], pp = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; c++) {
                    Sp[c] = Sp_all[(size_t)(row0 + r) * DK + lane + 32 * c];
                    pp += Sp[c] * x.ak[c];
                }
                const float p = warp_sum(pp);
                const float vv = ldf(vp + vt + r), dov = ldf(dop + vt + r);
                const float delta = x.beta * (vv - p);
                float gk = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; c++) {
                    const float Sc = x.a[c] * Sp[c] + delta * x.k[c];
                    Gb[r][c] += A.scale * dov * x.q[c];
                    dq[c] += A.scale * dov * Sc;
                    gk += Gb[r][c] * x.k[c];
                }
                const float dd = warp_sum(gk);
                dbeta += dd * (vv - p);
                if (lane == 0) A.dv[vt + r] = x.beta * dd;
                const float dp = -x.beta * dd;
#pragma unroll
                for (int c = 0; c < CPL; c++) {
                    const float Gd = Gb[r][c] + dp * x.k[c];
                    dk[c] += delta * Gb[r][c] + dp * x.a[c] * Sp[c];
                    da[c] += Gd * Sp[c];
                    Gb[r][c] = Gd * x.a[c];
                }
            }
            // sums over the CTA's rows, in a fixed order
            float* rw = red + ((size_t)(t & 1) * nw + warp) * NRED;
#pragma unroll
            for (int c = 0; c < CPL; c++) {
                rw[lane + 32 * c] = dq[c];
                rw[DK + lane + 32 * c] = dk[c];
                rw[2 * DK + lane + 32 * c] = da[c];
            }
            if (lane == 0) rw[3 * DK] = dbeta;
            __syncthreads();
            const float* rr = red + (size_t)(t & 1) * nw * NRED;
            const size_t bt = ((size_t)b * T + t) * A.Hv + hv;
            if (tid < DK) {  // dq^, dk^ of this value head (summed over the group later), dg
                float sq = 0.f, sk = 0.f, sa = 0.f;
                for (int w = 0; w < nw; w++) {
                    sq += rr[w * NRED + tid];
                    sk += rr[w * NRED + DK + tid];
                    sa += rr[w * NRED + 2 * DK + tid];
                }
                A.dqh[(bt * DK) + tid] = sq;
                A.dkh[(bt * DK) + tid] = sk;
                if (A.channel) A.dg[bt * DK + tid] = expf(A.g[bt * DK + tid]) * sa;
                else A.dah[bt * DK + tid] = sa;
            } else if (tid == DK) {
                float s = 0.f;
                for (int w = 0; w < nw; w++) s += rr[w * NRED + 3 * DK];
                A.dbeta[bt] = s;
            }
            cur = nxt;
        }
    }
#pragma unroll
    for (int r = 0; r < kRows; r++)
#pragma unroll
        for (int c = 0; c < CPL; c++)
            if (A.dh0) A.dh0[(size_t)bh * plane + (size_t)(row0 + r) * DK + lane + 32 * c] = Gb[r][c];
}

// dq, dk: sum dq^, dk^ over the value heads of each key head, then the norm backward.
// Scalar gate: dg = a sum_k da_k. One block of DK threads per (b, t, hk).
template <int DK, typename TIn>
__global__ void __launch_bounds__(128) seq_bwd_finish_kernel(SeqBwdArgs A) {
    __shared__ float part[2][4];
    const int col = threadIdx.x, warp = col >> 5, lane = col & 31;
    const int hk = blockIdx.x % A.Hk, bt = blockIdx.x / A.Hk;  // bt = b * T + t
    const int G = A.Hv / A.Hk;
    float dqh = 0.f, dkh = 0.f;
    for (int h = 0; h < G; h++) {
        const size_t i = ((size_t)bt * A.Hv + hk * G + h) * DK + col;
        dqh += A.dqh[i];
        dkh += A.dkh[i];
    }
    const size_t xi = ((size_t)bt * A.Hk + hk) * DK + col;
    const float qv = ldf(static_cast<const TIn*>(A.q) + xi), kv = ldf(static_cast<const TIn*>(A.k) + xi);
    // per-block sums: |q|^2, |k|^2, then q . dq^, k . dk^
    auto block_sum2 = [&](float x, float y, float& sx, float& sy) {
        x = warp_sum(x);
        y = warp_sum(y);
        __syncthreads();
        if (lane == 0) {
            part[0][warp] = x;
            part[1][warp] = y;
        }
        __syncthreads();
        sx = sy = 0.f;
        for (int w = 0; w < DK / 32; w++) {
            sx += part[0][w];
            sy += part[1][w];
        }
    };
    float ssq, ssk;
    block_sum2(qv * qv, kv * kv, ssq, ssk);
    float dq = dqh, dk = dkh;
    if (A.use_norm) {
        const float rq = 1.0f / sqrtf(ssq + 1e-6f), rk = 1.0f / sqrtf(ssk + 1e-6f);
        const float qh = rq * qv, kh = rk * kv;
        float dotq, dotk;
        block_sum2(qh * dqh, kh * dkh, dotq, dotk);
        dq = rq * (dqh - qh * dotq);
        dk = rk * (dkh - kh * dotk);
    }
    A.dq[xi] = dq;
    A.dk[xi] = dk;
    if (!A.channel) {  // dg of the group's value heads at this token: a sum_k da_k
        for (int h = 0; h < G; h++) {
            const size_t i = (size_t)bt * A.Hv + hk * G + h;
            float s = A.dah[i * DK + col];
            float tot, dummy;
            block_sum2(s, 0.f, tot, dummy);
            if (col == 0) A.dg[i] = expf(A.g[i]) * tot;
        }
    }
}

template <int DK, typename TIn>
cudaError_t launch_seq_bwd_t(const SeqBwdArgs& a, cudaStream_t s) {
    const int threads = a.Dv / kRows * 32;
    const int nw = threads / 32;
    const size_t smem = 2 * (size_t)nw * (3 * DK + 1) * sizeof(float);
    cudaError_t e =
        cudaFuncSetAttribute(seq_bwd_kernel<DK, TIn>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    trace_begin("seq_bwd", s);
    seq_bwd_kernel<DK, TIn><<<a.B * a.Hv, threads, smem, s>>>(a);
    trace_end(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_begin("seq_bwd_finish", s);
    seq_bwd_finish_kernel<DK, TIn><<<a.B * a.T * a.Hk, DK, 0, s>>>(a);
    trace_end(s);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_seq_bwd_d(const SeqBwdArgs& a, cudaStream_t s) {
    switch (a.Dk) {
        case 32: return launch_seq_bwd_t<32, TIn>(a, s);
        case 64: return launch_seq_bwd_t<64, TIn>(a, s);
        default: return launch_seq_bwd_t<128, TIn>(a, s);
    }
}

// The same sum and norm backward for bf16 q, k with Dk = 128, one warp per (b, t, key head):
// lane l owns channels 4l .. 4l + 3 (128-bit loads of dq^, dk^, 64-bit loads of q, k), and the
// four sums are warp reductions, so a block of 8 warps handles 8 rows without a barrier.
__global__ void __launch_bounds__(256) qk_norm_bwd_warp_kernel(SeqBwdArgs A) {
    const int lane = threadIdx.x & 31;
    const size_t row = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // (b * T + t) * Hk + hk
    if (row >= (size_t)A.B * A.T * A.Hk) return;
    const int G = A.Hv / A.Hk;
    const size_t bt = row / A.Hk;
    const int hk = (int)(row % A.Hk);
    float4 dq = make_float4(0.f, 0.f, 0.f, 0.f), dk = dq;
    for (int h = 0; h < G; h++) {
        const size_t i = (bt * A.Hv + (size_t)hk * G + h) * 128 + 4 * lane;
        const float4 x = *reinterpret_cast<const float4*>(A.dqh + i), y = *reinterpret_cast<const float4*>(A.dkh + i);
        dq.x += x.x; dq.y += x.y; dq.z += x.z; dq.w += x.w;
        dk.x += y.x; dk.y += y.y; dk.z += y.z; dk.w += y.w;
    }
    const size_t xi = row * 128 + 4 * lane;
    const uint2 qu = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(A.q) + xi);
    const uint2 ku = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(A.k) + xi);
    const float q[4] = {bf16lo(qu.x), bf16hi(qu.x), bf16lo(qu.y), bf16hi(qu.y)};
    const float k[4] = {bf16lo(ku.x), bf16hi(ku.x), bf16lo(ku.y), bf16hi(ku.y)};
    float oq[4] = {dq.x, dq.y, dq.z, dq.w}, ok[4] = {dk.x, dk.y, dk.z, dk.w};
    if (A.use_norm) {
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            sq += q[e] * q[e];
            sk += k[e] * k[e];
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float rq = 1.0f / sqrtf(sq + 1e-6f), rk = 1.0f / sqrtf(sk + 1e-6f);
        float tq = 0.f, tk = 0.f;  // q^ . dq^, k^ . dk^
#pragma unroll
        for (int e = 0; e < 4; e++) {
            tq += rq * q[e] * oq[e];
            tk += rk * k[e] * ok[e];
        }
        tq = warp_sum(tq);
        tk = warp_sum(tk);
#pragma unroll
        for (int e = 0; e < 4; e++) {
            oq[e] = rq * (oq[e] - rq * q[e] * tq);
            ok[e] = rk * (ok[e] - rk * k[e] * tk);
        }
    }
    *reinterpret_cast<float4*>(A.dq + xi) = make_float4(oq[0], oq[1], oq[2], oq[3]);
    *reinterpret_cast<float4*>(A.dk + xi) = make_float4(ok[0], ok[1], ok[2], ok[3]);
}

}  // namespace

cudaError_t launch_qk_norm_backward(const SeqBwdArgs& a, cudaStream_t s) {
    if (a.Dk != 128 || !a.bf16) return cudaErrorInvalidValue;
    const size_t rows = (size_t)a.B * a.T * a.Hk;
    trace_begin("qk_norm_backward", s);
    qk_norm_bwd_warp_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a);
    trace_end(s);
    return cudaGetLastError();
}

cudaError_t launch_head_sum_norm_backward(SeqBwdArgs a, cudaStream_t s) {
    a.channel = 1;  // the finish kernel's scalar-gate dg step is the sequential VJP's own
    const unsigned blocks = (unsigned)((size_t)a.B * a.T * a.Hk);
    trace_begin("head_sum_norm_backward", s);
    switch (a.Dk * 2 + a.bf16) {
        case 64: seq_bwd_finish_kernel<32, float><<<blocks, 32, 0, s>>>(a); break;
        case 65: seq_bwd_finish_kernel<32, __nv_bfloat16><<<blocks, 32, 0, s>>>(a); break;
        case 128: seq_bwd_finish_kernel<64, float><<<blocks, 64, 0, s>>>(a); break;
        case 129: seq_bwd_finish_kernel<64, __nv_bfloat16><<<blocks, 64, 0, s>>>(a); break;
        case 256: seq_bwd_finish_kernel<128, float><<<blocks, 128, 0, s>>>(a); break;
        case 257: seq_bwd_finish_kernel<128, __nv_bfloat16><<<blocks, 128, 0, s>>>(a); break;
        default: trace_end(s); return cudaErrorInvalidValue;
    }
    trace_end(s);
    return cudaGetLastError();
}

size_t seq_bwd_workspace(int B, int T, int Hv, int Dk, int Dv) {
    const size_t nh = (size_t)B * Hv, plane = (size_t)Dv * Dk * sizeof(float);
    const size_t nseg = (T + kSeg - 1) / kSeg;
    const size_t per_tok = (size_t)B * T * Hv * Dk * sizeof(float);
    return 256 + nh * nseg * plane + nh * kSeg * plane + 3 * per_tok;
}

cudaError_t launch_seq_bwd(SeqBwdArgs a, void* ws, cudaStream_t s) {
    uint8_t* w = static_cast<uint8_t*>(ws) + 256;
    const size_t nh = (size_t)a.B * a.Hv, plane = (size_t)a.Dv * a.Dk * sizeof(float);
    const size_t nseg = (a.T + kSeg - 1) / kSeg;
    const size_t per_tok = (size_t)a.B * a.T * a.Hv * a.Dk * sizeof(float);
    a.ckpt = reinterpret_cast<float*>(w);
    w += nh * nseg * plane;
    a.segs = reinterpret_cast<float*>(w);
    w += nh * kSeg * plane;
    a.dqh = reinterpret_cast<float*>(w);
    a.dkh = reinterpret_cast<float*>(w + per_tok);
    a.dah = reinterpret_cast<float*>(w + 2 * per_tok);
    return a.bf16 ? launch_seq_bwd_d<__nv_bfloat16>(a, s) : launch_seq_bwd_d<float>(a, s);
}

}  // namespace gdr
