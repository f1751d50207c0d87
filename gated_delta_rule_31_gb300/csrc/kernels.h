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

// dq, dk from per-value-head dq^, dk^ (fp32 [B][T][Hv][Dk] in dqh / dkh) for every dtype and
// head size: the value-head sum and the L2-norm backward; dg untouched.
cudaError_t launch_head_sum_norm_backward(SeqBwdArgs a, cudaStream_t s);

// fp32 chunked path (chunk_f32.cu): the chunk algebra with fp32 FMA on the CUDA cores.
struct Chunk32Args {
    int B, T, Hk, Hv, Dk, Dv, NC;
    int channel, use_norm;
    float scale;
    const float *q, *k, *v, *g, *beta, *h0, *do_, *dht;
    float *o, *ht, *dq, *dk, *dv, *dg, *dbeta, *dh0;
    float* rec;       // per-(b, hv, chunk) records
    float* states;    // chunk-start states [B*Hv][NC][Dv][Dk] (forward: optional)
    float* dstates;   // chunk-end state gradients [B*Hv][NC][Dv][Dk] (backward)
    float *dqh, *dkh; // dq^, dk^ per value head [B][T][Hv][Dk] (backward)
    float* scratch;   // backward: one slot per grad CTA
    int nscratch;     // grad CTAs
};
// Workspace of a call on this path (byte offsets; 0 where absent): the status word, then the
// records unless the caller keeps them, and for the backward the chunk-start states unless the
// caller keeps them, the chunk-end state gradients, dq^, dk^ and the grad scratch.
struct Chunk32Layout {
    size_t rec, states, dstates, dqh, dkh, scratch, total;
    int nscratch;
};
Chunk32Layout chunk32_layout(int B, int T, int Hv, int Dk, int Dv, bool bwd, bool own_rec, bool own_states);
size_t chunk32_states_bytes(int B, int T, int Hv, int Dk, int Dv);
size_t chunk32_saved_states_offset(int B, int T, int Hv, int Dk, int Dv);
size_t chunk32_saved_bytes(int B, int T, int Hv, int Dk, int Dv);
// Forward: records (when prep), then o, ht and, with a.states set, the chunk-start states.
cudaError_t launch_chunk32_fwd(const Chunk32Args& a, bool prep, cudaStream_t s);
// Backward: records (when prep), chunk-start states (when states_scan), the reverse scan, the
// chunk-local gradients and the value-head sum with the norm backward.
cudaError_t launch_chunk32_bwd(const Chunk32Args& a, bool prep, bool states_scan, cudaStream_t s);

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
