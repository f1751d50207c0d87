// recurrent.cu - token-by-token gated delta rule on CUDA cores: the sequential forward
// (gdr_fwd_sequential) and the single-token decode step (gdr_decode_step).
//
// Every row v of the state S [Dv x Dk] evolves on its own given the token's k^, q^, a,
// beta and v_t[v]:   S[v,:] <- a (.) S[v,:] + beta (v_t[v] - <S[v,:], a (.) k^>) k^.
// So a warp owns whole state rows (Dk/32 consecutive fp32 per lane, one 128-bit load
// per row at Dk = 128) and runs two traversals of each row per token, as in "Two-pass
// optimization for channelwise gated delta rule kernel" (Summary): the first forms the
// prediction <S, a (.) k^> with the decay folded in, the second applies decay plus the
// rank-one update while accumulating the output <S', q^>. The state is read from HBM
// once and written once per call; the q/k L2 norm (eps 1e-6, "fold q/k L2-norm into the
// gated_delta_rule kernel", What) is computed in fp32 registers with warp shuffles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace gdr {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

template <int EL>
__device__ __forceinline__ void ld_row(const float* p, float* x) {
    if constexpr (EL == 4) {
        float4 t = *reinterpret_cast<const float4*>(p);
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else if constexpr (EL == 2) {
        float2 t = *reinterpret_cast<const float2*>(p);
        x[0] = t.x; x[1] = t.y;
    } else {
        x[0] = *p;
    }
}
template <int EL>
__device__ __forceinline__ void st_row(float* p, const float* x) {
    if constexpr (EL == 4) {
        *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else if constexpr (EL == 2) {
        *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    } else {
        *p = x[0];
    }
}

// grid (ceil(Dv / (WARPS*ROWS)), Hv, B), block WARPS*32. Each warp owns ROWS state rows.
template <int DK, typename TIn, int ROWS, int WARPS>
__global__ void __launch_bounds__(WARPS * 32) recurrent_rows_kernel(RecurrentArgs a) {
    constexpr int EL = DK / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = blockIdx.z, hv = blockIdx.y;
    const int hk = hv / (a.Hv / a.Hk);
    const int r0 = (blockIdx.x * WARPS + warp) * ROWS;
    if (r0 >= a.Dv) return;
    const int c0 = lane * EL;
    const size_t st_base = ((size_t)b * a.Hv + hv) * (size_t)a.Dv * DK;

    float S[ROWS][EL];
#pragma unroll
    for (int i = 0; i < ROWS; i++) {
        if (r0 + i < a.Dv && a.h0) {
            ld_row<EL>(a.h0 + st_base + (size_t)(r0 + i) * DK + c0, S[i]);
        } else {
#pragma unroll
            for (int e = 0; e < EL; e++) S[i][e] = 0.f;
        }
    }
    const TIn* q = reinterpret_cast<const TIn*>(a.q);
    const TIn* k = reinterpret_cast<const TIn*>(a.k);
    const TIn* v = reinterpret_cast<const TIn*>(a.v);
    TIn* o = reinterpret_cast<TIn*>(a.o);

    // the raw inputs of token t + 1 are loaded while token t is processed
    struct Raw {
        float k[EL], q[EL], g[EL], beta, v[ROWS];
    };
    auto load_raw = [&](int t, Raw& x) {
        const size_t qk_off = (((size_t)b * a.T + t) * a.Hk + hk) * DK + c0;
        const size_t bt = ((size_t)b * a.T + t) * a.Hv + hv;
#pragma unroll
        for (int e = 0; e < EL; e++) {
            x.k[e] = to_f(k[qk_off + e]);
            x.q[e] = to_f(q[qk_off + e]);
            x.g[e] = a.channel ? a.g[bt * DK + c0 + e] : (e == 0 ? a.g[bt] : 0.f);
        }
        x.beta = a.beta[bt];
#pragma unroll
        for (int i = 0; i < ROWS; i++) x.v[i] = (r0 + i < a.Dv) ? to_f(v[bt * (size_t)a.Dv + r0 + i]) : 0.f;
    };
    Raw cur, nxt;
    if (a.T > 0) load_raw(0, cur);
    for (int t = 0; t < a.T; t++) {
        if (t + 1 < a.T) load_raw(t + 1, nxt);
        const size_t bt = ((size_t)b * a.T + t) * a.Hv + hv;
        float kh[EL], qh[EL], dec[EL];
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int e = 0; e < EL; e++) {
            kh[e] = cur.k[e];
            qh[e] = cur.q[e];
            sk += kh[e] * kh[e];
            sq += qh[e] * qh[e];
        }
        if (a.use_norm) {
            sk = warp_sum(sk);
            sq = warp_sum(sq);
            const float rk = 1.0f / sqrtf(sk + 1e-6f), rq = 1.0f / sqrtf(sq + 1e-6f);
#pragma unroll
            for (int e = 0; e < EL; e++) {
                kh[e] *= rk;
                qh[e] *= rq;
            }
        }
        if (a.channel) {
#pragma unroll
            for (int e = 0; e < EL; e++) dec[e] = expf(cur.g[e]);
        } else {
            const float s = expf(cur.g[0]);
#pragma unroll
            for (int e = 0; e < EL; e++) dec[e] = s;
        }
        const float beta = cur.beta;
        const size_t vo = bt * (size_t)a.Dv + r0;
        // pass 1: prediction with the decay folded in
        float p[ROWS];
#pragma unroll
        for (int i = 0; i < ROWS; i++) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EL; e++) acc += S[i][e] * (dec[e] * kh[e]);
            p[i] = acc;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int i = 0; i < ROWS; i++) p[i] += __shfl_xor_sync(0xffffffffu, p[i], off);
        // pass 2: decay + rank-one update, output accumulated on the fly
        float out[ROWS];
#pragma unroll
        for (int i = 0; i < ROWS; i++) {
            const float d = beta * (cur.v[i] - p[i]);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EL; e++) {
                S[i][e] = dec[e] * S[i][e] + d * kh[e];
                acc += S[i][e] * qh[e];
            }
            out[i] = acc;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int i = 0; i < ROWS; i++) out[i] += __shfl_xor_sync(0xffffffffu, out[i], off);
#pragma unroll
        for (int i = 0; i < ROWS; i++)
            if (lane == i && r0 + i < a.Dv) o[vo + i] = from_f<TIn>(a.scale * out[i]);
        cur = nxt;
    }
    if (a.ht) {
#pragma unroll
        for (int i = 0; i < ROWS; i++)
            if (r0 + i < a.Dv) st_row<EL>(a.ht + st_base + (size_t)(r0 + i) * DK + c0, S[i]);
    }
}

// Decode: one CTA of 4 warps per (b, hv); warp w streams state rows [w*Dv/4, (w+1)*Dv/4) in
// groups of 4 rows, loading group g+1 while it reduces and writes group g, so each lane
// keeps four to eight 128-bit loads in flight for the whole CTA life. With one wave of
// CTAs (B*Hv of them) the grid has no tail. The step is launched as a programmatic dependent
// of the kernel before it on the stream: it lets the next launch begin at once
// (griddepcontrol.launch_dependents), loads q, k, v, g, beta and forms the norms, and only then
// waits for the previous kernel to complete (griddepcontrol.wait) before it reads the state or
// writes anything. Back-to-back steps so overlap one step's start with the previous one's end.
#ifndef GDR_DECODE_GROUP
#define GDR_DECODE_GROUP 4
#endif
template <int DK, typename TIn>
__global__ void __launch_bounds__(128) decode_kernel(RecurrentArgs a) {
    constexpr int EL = DK / 32;
    constexpr int G = GDR_DECODE_GROUP;  // rows per group
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hv = blockIdx.x, b = blockIdx.y;
    const int hk = hv / (a.Hv / a.Hk);
    const int rows_per_warp = a.Dv / 4;
    const int ngroups = rows_per_warp / G;
    const int r0 = warp * rows_per_warp;
    const int c0 = lane * EL;
    const size_t bh = (size_t)b * a.Hv + hv;
    const float* Sin = a.h0 + bh * (size_t)a.Dv * DK;
    float* Sout = a.ht + bh * (size_t)a.Dv * DK;

    float cur[G][EL], nxt[G][EL];

    const TIn* q = reinterpret_cast<const TIn*>(a.q);
    const TIn* k = reinterpret_cast<const TIn*>(a.k);
    const TIn* v = reinterpret_cast<const TIn*>(a.v);
    TIn* o = reinterpret_cast<TIn*>(a.o);
    const size_t qk_off = ((size_t)b * a.Hk + hk) * DK + c0;
    float kh[EL], qh[EL], dec[EL];
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int e = 0; e < EL; e++) {
        kh[e] = to_f(k[qk_off + e]);
        qh[e] = to_f(q[qk_off + e]);
        sk += kh[e] * kh[e];
        sq += qh[e] * qh[e];
    }
    if (a.use_norm) {
        sk = warp_sum(sk);
        sq = warp_sum(sq);
        const float rk = 1.0f / sqrtf(sk + 1e-6f), rq = 1.0f / sqrtf(sq + 1e-6f);
#pragma unroll
        for (int e = 0; e < EL; e++) {
            kh[e] *= rk;
            qh[e] *= rq;
        }
    }
    if (a.channel) {
#pragma unroll
        for (int e = 0; e < EL; e++) dec[e] = expf(a.g[bh * DK + c0 + e]);
    } else {
        const float sg = expf(a.g[bh]);
#pragma unroll
        for (int e = 0; e < EL; e++) dec[e] = sg;
    }
    float ak[EL];
#pragma unroll
    for (int e = 0; e < EL; e++) ak[e] = dec[e] * kh[e];
    const float beta = a.beta[bh];
    const size_t vo = bh * (size_t)a.Dv;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernel's writes are complete
#pragma unroll
    for (int i = 0; i < G; i++) ld_row<EL>(Sin + (size_t)(r0 + i) * DK + c0, cur[i]);

    for (int gi = 0; gi < ngroups; gi++) {
        const int rg = r0 + gi * G;
        if (gi + 1 < ngroups) {
#pragma unroll
            for (int i = 0; i < G; i++) ld_row<EL>(Sin + (size_t)(rg + G + i) * DK + c0, nxt[i]);
        }
        // pass 1: prediction with the decay folded in
        float p[G];
#pragma unroll
        for (int i = 0; i < G; i++) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EL; e++) acc += cur[i][e] * ak[e];
            p[i] = acc;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int i = 0; i < G; i++) p[i] += __shfl_xor_sync(0xffffffffu, p[i], off);
        // pass 2: decay + rank-one update, output accumulated on the fly
        float out[G];
#pragma unroll
        for (int i = 0; i < G; i++) {
            const float d = beta * (to_f(v[vo + rg + i]) - p[i]);
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < EL; e++) {
                cur[i][e] = dec[e] * cur[i][e] + d * kh[e];
                acc += cur[i][e] * qh[e];
            }
            out[i] = acc;
            st_row<EL>(Sout + (size_t)(rg + i) * DK + c0, cur[i]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int i = 0; i < G; i++) out[i] += __shfl_xor_sync(0xffffffffu, out[i], off);
#pragma unroll
        for (int i = 0; i < G; i++)
            if (lane == i) o[vo + rg + i] = from_f<TIn>(a.scale * out[i]);
#pragma unroll
        for (int i = 0; i < G; i++)
#pragma unroll
            for (int e = 0; e < EL; e++) cur[i][e] = nxt[i][e];
    }
}

template <int DK, typename TIn>
static cudaError_t launch_decode(const RecurrentArgs& a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.Hv, a.B);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see decode_kernel
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    trace_begin("decode_step", s);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<DK, TIn>, a);
    trace_end(s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int DK, typename TIn, int ROWS, int WARPS>
static cudaError_t launch_rows(const RecurrentArgs& a, cudaStream_t s) {
    dim3 grid((a.Dv + WARPS * ROWS - 1) / (WARPS * ROWS), a.Hv, a.B);
    trace_begin("recurrent_fwd", s);
    recurrent_rows_kernel<DK, TIn, ROWS, WARPS><<<grid, WARPS * 32, 0, s>>>(a);
    trace_end(s);
    return cudaGetLastError();
}

template <typename TIn, int ROWS, int WARPS>
static cudaError_t launch_dk(const RecurrentArgs& a, cudaStream_t s) {
    switch (a.Dk) {
        case 32: return launch_rows<32, TIn, ROWS, WARPS>(a, s);
        case 64: return launch_rows<64, TIn, ROWS, WARPS>(a, s);
        case 128: return launch_rows<128, TIn, ROWS, WARPS>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename TIn>
static cudaError_t launch_decode_dk(const RecurrentArgs& a, cudaStream_t s) {
    switch (a.Dk) {
        case 32: return launch_decode<32, TIn>(a, s);
        case 64: return launch_decode<64, TIn>(a, s);
        case 128: return launch_decode<128, TIn>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_recurrent(const RecurrentArgs& a, bool decode, cudaStream_t s) {
    if (decode) return a.bf16 ? launch_decode_dk<__nv_bfloat16>(a, s) : launch_decode_dk<float>(a, s);
    // Few rows in flight (small B * Hv): 2 rows per warp, the most warps. Many rows: 8 rows per
    // warp, so the grid stays near one wave and each warp overlaps 8 rows' reductions.
    const long long rows = (long long)a.B * a.Hv * a.Dv;
    if (rows > 16384)
        return a.bf16 ? launch_dk<__nv_bfloat16, 8, 4>(a, s) : launch_dk<float, 8, 4>(a, s);
    return a.bf16 ? launch_dk<__nv_bfloat16, 2, 4>(a, s) : launch_dk<float, 2, 4>(a, s);
}

}  // namespace gdr
