// kernels.h - internal launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdr {

struct RecurrentArgs {
    int B, T, Hk, Hv, Dk, Dv;
    int channel, use_norm, bf16;
    float scale;
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    void* o;
    float* ht;
};
cudaError_t launch_recurrent(const RecurrentArgs& a, bool decode, cudaStream_t s);

// Sequential VJP (recurrent_bwd.cu).
struct SeqBwdArgs {
    int B, T, Hk, Hv, Dk, Dv;
    int channel, use_norm, bf16;
    float scale;
    const void *q, *k, *v, *do_;
    const float *g, *beta, *h0, *dht;
    float *dq, *dk, *dv, *dg, *dbeta, *dh0;
    float *ckpt, *segs, *dqh, *dkh, *dah;  // workspace pieces, set by launch_seq_bwd
};
size_t seq_bwd_workspace(int B, int T, int Hv, int Dk, int Dv);
cudaError_t launch_seq_bwd(SeqBwdArgs a, void* ws, cudaStream_t s);
// dq, dk from per-value-head dq^, dk^ (fp32 [B][T][Hv][Dk] in dqh / dkh): the sum over the
// value heads of each key head, then the L2-norm backward (bf16 q, k; Dk = 128; dg untouched).
cudaError_t launch_qk_norm_backward(const SeqBwdArgs& a, cudaStream_t s);

// Staging copies (pad.cu): [outer][rs][cs] -> [outer][rd][cd] with zero fill (pad), or the
// [outer][rd][cd] corner of an [outer][rs][cs] tensor (crop); elements of 2 or 4 bytes.
cudaError_t launch_pad(const void* src, void* dst, int elem_bytes, size_t outer, int rs, int cs, int rd, int cd,
                       cudaStream_t s);
cudaError_t launch_crop(const void* src, void* dst, int elem_bytes, size_t outer, int rs, int cs, int rd, int cd,
                        cudaStream_t s);

// Launch tracing (api.cu): no-ops unless gdr_trace_enable(1) was called.
void trace_begin(const char* name, cudaStream_t s);
void trace_end(cudaStream_t s);

}  // namespace gdr
