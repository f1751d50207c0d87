// chunk.h - chunked (C = 64) gated delta rule on the tensor cores: launch interfaces and
// the workspace layout shared by the forward and backward launches.
//
// Chunk algebra (derived from the recurrence; H = S^T is the Dk x Dv state, rows r of a
// chunk are its tokens, gamma_r the in-chunk cumulative log-decay, E_rj = exp(gamma_r -
// gamma_j), Gamma_r = exp(gamma_r), b_r = exp(gamma_C - gamma_r), k^ = rho_k k):
//   A  = strict_lower(diag(beta) (E .* K^K^T)),   T = (I + A)^-1
//   W  = T diag(beta Gamma) K^,   U~ = T diag(beta) V,   P = scale tril(E .* Q^K^T)
//   U  = U~ - W H0;   O = scale diag(Gamma) Q^ H0 + P U;   H1 = Gamma_C H0 + K^T diag(b) U
// Folding W into the per-chunk operators removes one dependent product from the scan:
//   H1 = Gamma_C H0 + Mneg H0 + Kbar^T U~      with Mneg = -Kbar^T W, Kbar = diag(b) K^
//   O  = Qc H0 + P U~                          with Qc = scale diag(Gamma) Q^ - P W
//   dH0 = Gamma_C dH1 + Mneg^T dH1 + Qc^T dO   (the backward scan)
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdr {

constexpr int kChunk = 64;
constexpr int kD = 128;        // Dk = Dv handled by the tensor-core path

// Per-(b, hv, chunk) record written by the prep kernel, as shared-memory images
// (panelised SW128 tiles unless noted) so the scans fetch them with plain bulk copies.
constexpr uint32_t REC_M = 0;            // Mneg  [128 d  x 128 d']  32 KB
constexpr uint32_t REC_K = 32768;        // Kbar  [64 tok x 128 d]   16 KB
constexpr uint32_t REC_Q = 49152;        // Qc    [64 tok x 128 d]   16 KB
constexpr uint32_t REC_P = 65536;        // P     [64 tok x 64 tok]   8 KB
constexpr uint32_t REC_U = 73728;        // U~    4 x [64 tok x 32] SW64 slices, 4 KB each (a 64-column
                                         //       half is two consecutive slices: N=64 operand, LBO 4 KB)
constexpr uint32_t REC_BYTES = 90112;
constexpr uint32_t STATE_IMG = 32768;    // one bf16 [128 d x 128 v] SW128 state image
// Extra per-chunk record kept for the backward: T = (I + A)^-1 [64 x 64] and W [64 x 128].
constexpr uint32_t REC2_T = 0, REC2_W = 8192, REC2_BYTES = 24576;
// Per-channel backward: the tensor-core pass exports, per (b, hv, chunk), fp32 [64][128]
// X = dO H0^T, Y = U dH1^T, Z = T^T dW; fp32 [64][64] dPs = scale tril(dO U^T) and
// dA = -strict_lower(T^T dT T^T); per state row d <dH1, H0>_d; per token V . (T^T dU).
constexpr uint32_t CHX_X = 0, CHX_Y = 32768, CHX_Z = 65536, CHX_DP = 98304, CHX_DA = 114688;
constexpr uint32_t CHX_HDH = 131072, CHX_DB = 131584, CHX_BYTES = 131840;

struct ChunkProblem {
    int B, T, Hk, Hv, NC;
    float scale;
    int use_norm;
    int channel;  // per-channel gate g [B,T,Hv,Dk]; else one gate per head
};

struct WsLayout {
    size_t gam;      // float [B*Hv][ncpad]: Gamma_C per chunk ([B*Hv][NC][Dk] per channel)
    size_t rec;      // records [B*Hv][NC]
    size_t rec2;     // bwd: T and W per chunk [B*Hv][NC]
    size_t hs;       // bwd: chunk-start states [B*Hv][NC] images
    size_t dhs;      // bwd: chunk-end state gradients [B*Hv][NC] images
    size_t chx;      // bwd, per-channel gate: tensor-core exports [B*Hv][NC]
    size_t dqh, dkh; // bwd, per-channel gate or split gradient: dq^, dk^ per value head, fp32 [B][T][Hv][Dk]
    size_t total;
    int ncpad;
};

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Scalar-gate backward of a small problem: when its (b, key head, chunk) tiles times the value heads
// per key head number at most this, the gradient kernel takes one value head per CTA (so every head
// has an SM) and writes dq^, dk^ per value head; a second kernel sums them over the key head's
// value heads and applies the norm backward. The workspace then holds those two planes.
constexpr int kGradSplitUnits = 128;
inline bool grad_split(const ChunkProblem& p) {
    return !p.channel && (long)p.B * p.Hk * p.NC * (p.Hv / p.Hk) <= kGradSplitUnits;
}

// bwd_states: a backward that reads saved chunk-start states (no states region of its own).
inline WsLayout ws_layout(const ChunkProblem& p, bool bwd, bool bwd_states = false) {
    WsLayout w;
    w.ncpad = (int)round_up((size_t)p.NC, 4);
    size_t nh = (size_t)p.B * p.Hv;
    w.gam = 256;
    const size_t ngam = p.channel ? (size_t)p.NC * kD : (size_t)w.ncpad;
    w.rec = round_up(w.gam + nh * ngam * sizeof(float), 1024);
    size_t end = w.rec + nh * p.NC * (size_t)REC_BYTES;
    w.rec2 = w.hs = w.dhs = w.chx = w.dqh = w.dkh = 0;
    if (bwd) {
        w.rec2 = end;
        end = w.rec2 + nh * p.NC * (size_t)REC2_BYTES;
        w.hs = end;
        if (!bwd_states) end += nh * p.NC * (size_t)STATE_IMG;
        w.dhs = end;
        end = w.dhs + nh * p.NC * (size_t)STATE_IMG;
        if (p.channel) {
            w.chx = end;
            end = w.chx + nh * p.NC * (size_t)CHX_BYTES;
        }
        if (p.channel || grad_split(p)) {
            const size_t plane = round_up((size_t)p.B * p.T * p.Hv * kD * sizeof(float), 1024);
            w.dqh = end;
            w.dkh = end + plane;
            end += 2 * plane;
        }
    }
    w.total = end;
    return w;
}
inline size_t chunk_fwd_workspace(const ChunkProblem& p) { return ws_layout(p, false).total; }
inline size_t chunk_bwd_workspace(const ChunkProblem& p) { return ws_layout(p, true).total; }
inline size_t chunk_bwd_states_workspace(const ChunkProblem& p) { return ws_layout(p, true, true).total; }
inline size_t chunk_states_bytes(const ChunkProblem& p) { return (size_t)p.B * p.Hv * p.NC * STATE_IMG; }

// Everything the forward can keep for the backward (the caller's "saved" buffer): Gamma_C per
// chunk, the operator records, T and W per chunk, and the chunk-start state images. With it
// the backward runs neither prep nor the forward states scan. Its own workspace then holds
// the status word and the chunk-end state gradients.
struct SavedLayout {
    size_t gam, rec, rec2, hs, total;
    int ncpad;
};
inline SavedLayout saved_layout(const ChunkProblem& p) {
    SavedLayout l;
    l.ncpad = (int)round_up((size_t)p.NC, 4);
    const size_t nh = (size_t)p.B * p.Hv;
    const size_t ngam = p.channel ? (size_t)p.NC * kD : (size_t)l.ncpad;  // Gamma_C per chunk (per channel)
    l.gam = 0;
    l.rec = round_up(nh * ngam * sizeof(float), 1024);
    l.rec2 = l.rec + nh * p.NC * (size_t)REC_BYTES;
    l.hs = l.rec2 + nh * p.NC * (size_t)REC2_BYTES;
    l.total = l.hs + nh * p.NC * (size_t)STATE_IMG;
    return l;
}
inline size_t chunk_saved_bytes(const ChunkProblem& p) { return saved_layout(p).total; }
constexpr size_t kSavedFwdWorkspace = 256;  // status word only
// The backward's own workspace next to a saved buffer: the status word, the chunk-end state
// gradients and, with a per-channel gate, the exports and per-value-head dq^, dk^ (also for a
// split gradient).
struct SavedBwdLayout {
    size_t dhs, chx, dqh, dkh, total;
};
inline SavedBwdLayout saved_bwd_layout(const ChunkProblem& p) {
    SavedBwdLayout l;
    const size_t nh = (size_t)p.B * p.Hv;
    l.dhs = 1024;
    l.total = l.dhs + nh * p.NC * (size_t)STATE_IMG;
    l.chx = l.dqh = l.dkh = 0;
    if (p.channel) {
        l.chx = l.total;
        l.total = l.chx + nh * p.NC * (size_t)CHX_BYTES;
    }
    if (p.channel || grad_split(p)) {
        const size_t plane = round_up((size_t)p.B * p.T * p.Hv * kD * sizeof(float), 1024);
        l.dqh = l.total;
        l.dkh = l.dqh + plane;
        l.total = l.dkh + plane;
    }
    return l;
}
inline size_t chunk_bwd_saved_workspace(const ChunkProblem& p) { return saved_bwd_layout(p).total; }

struct ChunkFwdArgs {
    ChunkProblem p;
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    void* o;
    float* ht;
    void* states;  // optional: chunk-start states kept for the backward
    void* saved;   // optional: the whole saved buffer (saved_layout); then ws is the status word only
    void* ws;
};
struct ChunkBwdArgs {
    ChunkProblem p;
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    const void* do_;
    const float* dht;
    float *dq, *dk, *dv, *dg, *dbeta, *dh0;
    const void* states;  // optional: chunk-start states saved by the forward
    const void* saved;   // optional: the forward's saved buffer (saved_layout)
    void* ws;
};

cudaError_t launch_chunk_fwd(const ChunkFwdArgs& a, cudaStream_t s);
cudaError_t launch_chunk_bwd(const ChunkBwdArgs& a, cudaStream_t s);

// Pieces shared by the forward and backward launches (chunk_fwd.cu).
struct PrepArgs {
    ChunkProblem p;
    const float *g, *beta;
    float* gam;
    uint8_t* rec;
    uint8_t* rec2;  // null in the forward
    int* status;
    int ncpad;
};
cudaError_t launch_prep(const PrepArgs& a, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                        cudaStream_t s);
// Per-channel gate (chunk_fwd_ch.cu): same record, Gamma_C as [B*Hv][NC][Dk].
cudaError_t launch_prep_ch(const PrepArgs& a, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           cudaStream_t s);
// Per-channel gate backward after the scans (chunk_bwd_ch.cu): the tensor-core pass, the
// CUDA-core pass and the value-head sum with the norm backward.
struct GradChArgs {
    ChunkProblem p;
    const void *q, *k;
    const float *g, *beta;
    const uint8_t *rec, *rec2, *hs, *dhs;
    uint8_t* chx;
    float *dqh, *dkh;
    float *dq, *dk, *dv, *dg, *dbeta;
    int* status;
};
cudaError_t launch_grad_ch(const GradChArgs& a, const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s);

enum ScanMode : int { SCAN_FWD_OUT = 0, SCAN_FWD_STATES = 1, SCAN_BWD = 2 };
struct ScanArgs {
    ChunkProblem p;
    const float* gam;
    const uint8_t* rec;
    const float* hinit;   // h0 (forward) or dht (backward); may be null
    void* o;              // forward output
    float* hfinal;        // ht (forward) or dh0 (backward); may be null
    uint8_t* states;      // per-chunk state images (SCAN_FWD_STATES / SCAN_BWD)
    int* status;
    int ncpad;
};
cudaError_t launch_scan(const ScanArgs& a, int mode, const CUtensorMap* mdo, cudaStream_t s);

bool make_qkv_maps(const ChunkProblem& p, const void* q, const void* k, const void* v, CUtensorMap* mq,
                   CUtensorMap* mk, CUtensorMap* mv);

}  // namespace gdr
