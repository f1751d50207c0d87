/*
 * gdr.h - C ABI of the GB300 (sm_103a) gated delta rule library (libgdr.so).
 *
 * The operation (Gated DeltaNet recurrence). Per batch b and value head hv, with key
 * head hk = hv / (Hv / Hk), a state S in R^{Dv x Dk} evolves over tokens t:
 *
 *     k^ = n(k_t),  q^ = n(q_t),   n(x) = x * (sum x^2 + 1e-6)^(-1/2)  (if use_qk_l2norm)
 *     S_t = S_{t-1} diag(a_t) (I - beta_t k^ k^T) + beta_t v_t k^T,   a_t = exp(g_t)
 *     o_t = scale * S_t q^
 *
 * a_t is one value per (b,t,hv) (scalar gate) or a vector over the Dk key channels
 * (channel gate). Sources: "perf(gated_delta_net): fold q/k L2-norm into the
 * gated_delta_rule kernel" (Megatron-LM PR #5396), What/Why: the kernel owns the q/k
 * L2 norm of the last dimension with eps 1e-6; "Two-pass optimization for channelwise
 * gated delta rule kernel" (ExecuTorch PR #21020), Summary: per-channel decay, decode
 * in two state traversals with the decay folded into the prediction; "Adding VJP for
 * gated delta net" (MLX PR #4565), description and Performance: a chunked and a
 * sequential backward over B in {1,4,8}, T 8..4096, Hk=16, Hv=32, Dk=Dv=128.
 *
 * Layouts: dense row-major, innermost last.
 *   q, k        [B, T, Hk, Dk]   dtype (fp32 or bf16)
 *   v, o, do    [B, T, Hv, Dv]   dtype
 *   g           [B, T, Hv] (scalar gate) or [B, T, Hv, Dk] (channel gate), fp32, log-decay
 *   beta        [B, T, Hv]       fp32 (already in (0,1); the gradient is w.r.t. beta)
 *   h0, ht, dht, dh0, state      [B, Hv, Dv, Dk] fp32 (row v of S is contiguous)
 *   dq, dk      [B, T, Hk, Dk]   fp32 (summed over the value heads sharing a key head)
 *   dv          [B, T, Hv, Dv]   fp32;  dg like g, dbeta like beta, fp32
 * Decode uses the same layouts with the T axis removed.
 *
 * Ownership: every pointer is device memory owned by the caller (for example torch
 * tensors). The library keeps no allocation between calls and allocates nothing in
 * the compute calls; launches are asynchronous on the given stream and no call
 * synchronises. Outputs may not alias inputs (except decode's in-place state).
 *
 * Errors: arguments are validated before anything is launched. A bad argument returns
 * GDR_ERR_INVALID_ARG, a combination this build does not implement returns
 * GDR_ERR_UNSUPPORTED, a short workspace GDR_ERR_WORKSPACE, all with nothing launched.
 * A failed launch returns GDR_ERR_CUDA. The chunked kernels bound every wait; if a
 * wait expires the kernel stops and records GDR_ERR_TIMEOUT in the workspace's
 * status word, which gdr_workspace_status() reads back.
 */
#ifndef GDR_H_
#define GDR_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gdr_stream_t; /* same type as cudaStream_t; NULL = default stream */

typedef enum {
    GDR_OK = 0,
    GDR_ERR_INVALID_ARG = 1, /* null required pointer, bad size, misaligned pointer, ... */
    GDR_ERR_UNSUPPORTED = 2, /* valid, but not implemented by this build (see each call) */
    GDR_ERR_WORKSPACE = 3,   /* ws_bytes smaller than the matching *_workspace() query */
    GDR_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed */
    GDR_ERR_TIMEOUT = 5      /* a bounded device-side wait expired (read from the workspace) */
} gdr_status;

typedef enum { GDR_F32 = 0, GDR_BF16 = 1 } gdr_dtype;             /* of q, k, v, o, do */
typedef enum { GDR_GATE_SCALAR = 0, GDR_GATE_CHANNEL = 1 } gdr_gate;

typedef struct {
    int B, T, Hk, Hv, Dk, Dv; /* Hv % Hk == 0; T >= 0 (T == 1 for decode) */
    gdr_dtype dtype;
    gdr_gate gate;
    float scale;              /* applied to o = scale * S q^ (commonly Dk^-1/2) */
    int use_qk_l2norm;        /* 1: normalise q and k inside, eps 1e-6; 0: use as given */
} gdr_problem;

/* Human-readable name of a status code (static storage). */
const char* gdr_status_string(gdr_status s);

/* Bytes of device workspace gdr_fwd_chunked / gdr_bwd_chunked need for this problem
 * (0 if the problem is invalid). The workspace is scratch owned by the caller; its
 * first 256 bytes hold the status word. */
size_t gdr_fwd_chunked_workspace(const gdr_problem* p);
size_t gdr_bwd_chunked_workspace(const gdr_problem* p);

/* Chunked prefill forward (chunks of 64 tokens): o and, if ht != NULL, the final state.
 * h0 may be NULL (zero initial state). Implemented for both dtypes with Dk, Dv in {32, 64, 128},
 * with the scalar gate or the per-channel gate (g [B,T,Hv,Dk], the channelwise variant of
 * "Two-pass optimization for channelwise gated delta rule kernel", ExecuTorch PR #21020).
 * BF16: tensor-core kernels on 128 key and value channels; for Dk or Dv below 128 the call
 * stages zero-padded 128-wide copies of its inputs in the workspace (which the size query
 * includes) and crops the results; the zero channels contribute nothing, so results are those
 * of the original sizes. F32: the same chunk algebra with fp32 FMA on the CUDA cores (bf16
 * tensor-core operands cannot meet fp32 accuracy), every head size in place; o is fp32.
 * Pointers 16-byte aligned.
 * Work: per chunk a 64x64 unit-lower-triangular (UT/WY) transform of the k k^T beta
 * block, then one sequential scan over chunks per (b, hv, Dv slice) with the fp32 state held
 * on chip. Clears and then sets the workspace status word. */
gdr_status gdr_fwd_chunked(const gdr_problem* p, const void* q, const void* k, const void* v,
                           const float* g, const float* beta, const float* h0, void* o, float* ht,
                           void* ws, size_t ws_bytes, gdr_stream_t stream);

/* Token-by-token forward (no workspace): o and, if ht != NULL, the final state. For every
 * dtype, gate and Dk, Dv in {32, 64, 128}. */
gdr_status gdr_fwd_sequential(const gdr_problem* p, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const float* h0, void* o,
                              float* ht, gdr_stream_t stream);

/* Chunked backward (VJP) of gdr_fwd_chunked for the loss <do, o> + <dht, ht>: writes dq, dk,
 * dv, dg, dbeta and, if dh0 != NULL, dh0. h0 and dht may be NULL (zero). Recomputes the
 * chunk-local terms and the chunk-start states instead of reading saved activations;
 * the normalisation backward is done inside. Same support matrix as gdr_fwd_chunked; with the
 * per-channel gate dg is [B,T,Hv,Dk] (one gradient per key channel); its decay-weighted
 * intra-chunk contractions run by 16-token blocks, below the block diagonal on the tensor
 * cores with operands scaled by products of per-token factors, inside the diagonal blocks
 * with running products on the CUDA cores (no decay can overflow).
 * Deterministic: no floating-point atomics. */
gdr_status gdr_bwd_chunked(const gdr_problem* p, const void* q, const void* k, const void* v,
                           const float* g, const float* beta, const float* h0, const void* do_,
                           const float* dht, float* dq, float* dk, float* dv, float* dg,
                           float* dbeta, float* dh0, void* ws, size_t ws_bytes,
                           gdr_stream_t stream);

/* Sequential (token-by-token) VJP of gdr_fwd_sequential for the loss <do, o> + <dht, ht>:
 * the "sequential case" of "Adding VJP for gated delta net" (MLX PR #4565). Every dtype, gate
 * (scalar or per channel) and Dk, Dv in {32, 64, 128}. Arguments, layouts and outputs as gdr_bwd_chunked (gradients fp32; dg has g's shape). The forward is
 * re-run with a checkpoint every 64 tokens (B*Hv*ceil(T/64) fp32 states in the workspace)
 * and each 64-token segment is recomputed in reverse. Deterministic (fixed-order sums, no
 * atomics). Workspace: gdr_bwd_sequential_workspace() bytes, 256-byte aligned. */
size_t gdr_bwd_sequential_workspace(const gdr_problem* p);
gdr_status gdr_bwd_sequential(const gdr_problem* p, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const float* h0, const void* do_,
                              const float* dht, float* dq, float* dk, float* dv, float* dg,
                              float* dbeta, float* dh0, void* ws, size_t ws_bytes,
                              gdr_stream_t stream);

/* Saved-state handoff from the forward to the backward. The forward can keep the state
 * entering every chunk (opaque layout, gdr_chunk_states_bytes() bytes: B*Hv*ceil(T/64)*32 KB
 * of bf16 images for BF16, B*Hv*ceil(T/64)*Dv*Dk*4 of fp32 states for F32; caller-owned,
 * 256-byte aligned); the backward then reads them
 * instead of re-running the forward scan. Chunk-local operators are still recomputed by
 * the backward. Same support matrix as gdr_bwd_chunked (scalar or per-channel gate); 0 if
 * the problem is invalid. */
size_t gdr_chunk_states_bytes(const gdr_problem* p);
size_t gdr_bwd_chunked_states_workspace(const gdr_problem* p);

/* gdr_fwd_chunked that also writes the chunk-start states into `states`. */
gdr_status gdr_fwd_chunked_states(const gdr_problem* p, const void* q, const void* k, const void* v,
                                  const float* g, const float* beta, const float* h0, void* o, float* ht,
                                  void* states, size_t states_bytes, void* ws, size_t ws_bytes,
                                  gdr_stream_t stream);

/* gdr_bwd_chunked for the same inputs, reading the chunk-start states written by
 * gdr_fwd_chunked_states (h0 is then not needed). Workspace:
 * gdr_bwd_chunked_states_workspace() bytes. */
gdr_status gdr_bwd_chunked_states(const gdr_problem* p, const void* q, const void* k, const void* v,
                                  const float* g, const float* beta, const void* states, size_t states_bytes,
                                  const void* do_, const float* dht, float* dq, float* dk, float* dv, float* dg,
                                  float* dbeta, float* dh0, void* ws, size_t ws_bytes, gdr_stream_t stream);

/* Saved-operator handoff: the forward keeps everything the backward would recompute — the
 * per-chunk decay, the chunk operator records (88 KB), the UT inverse T and W (24 KB) and the
 * chunk-start states (32 KB), i.e. 144 KB per (b, hv, chunk) plus a small header, in one
 * caller-owned, 256-byte-aligned buffer of gdr_chunk_saved_bytes() bytes (opaque layout;
 * 2.4 GB at B=1, T=32768, Hv=32). The backward then runs only the reverse scan and the
 * chunk-local gradient kernel. This trades memory for the backward's recomputation, which
 * the chunked VJP of "Adding VJP for gated delta net" (MLX PR #4565) performs; results are
 * bitwise identical to gdr_fwd_chunked / gdr_bwd_chunked. The buffer must not be modified
 * between the two calls, and the backward must get the same q, k, v, g, beta and problem.
 * Workspaces: gdr_fwd_chunked_saved_workspace() (the status word only) and
 * gdr_bwd_chunked_saved_workspace(). Same support matrix as gdr_bwd_chunked (bf16: 144 KB per
 * (b, hv, chunk) with either gate, plus the per-chunk Gamma_C header; for F32 the buffer holds fp32 records of W, Kbar, scale Gamma Q^, gamma, U~, P and T, then
 * the fp32 chunk-start states: 256 KB per (b, hv, chunk) at Dk = Dv = 128);
 * the size queries return 0 for an invalid or unsupported problem. Errors as gdr_fwd_chunked, plus
 * GDR_ERR_WORKSPACE if `saved` is NULL or smaller than required. */
size_t gdr_chunk_saved_bytes(const gdr_problem* p);
size_t gdr_fwd_chunked_saved_workspace(const gdr_problem* p);
size_t gdr_bwd_chunked_saved_workspace(const gdr_problem* p);

/* gdr_fwd_chunked that also fills `saved`. */
gdr_status gdr_fwd_chunked_saved(const gdr_problem* p, const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, const float* h0, void* o, float* ht,
                                 void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                                 gdr_stream_t stream);

/* gdr_bwd_chunked for the same inputs, reading `saved` from gdr_fwd_chunked_saved (h0 is
 * then not needed; dh0 is still written if non-NULL). */
gdr_status gdr_bwd_chunked_saved(const gdr_problem* p, const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, const void* saved, size_t saved_bytes,
                                 const void* do_, const float* dht, float* dq, float* dk, float* dv, float* dg,
                                 float* dbeta, float* dh0, void* ws, size_t ws_bytes, gdr_stream_t stream);

/* One decode step (p->T must be 1) on the state in place: per state row, one pass forms
 * the prediction with the decay folded in, a second applies decay plus the rank-one
 * update while accumulating the output, so the state is read once and written once.
 * Layouts as above without the T axis. Every dtype, gate and Dk, Dv in {32, 64, 128}.
 * The step is launched as a programmatic dependent launch: it may read q, k, v, g and beta
 * while the kernel enqueued before it on `stream` is still running if that kernel is itself a
 * decode step, and reads the state and writes `o` only once that kernel has completed. So the
 * `o` of one step must not alias the q, k, v, g or beta of the step enqueued right after it. */
gdr_status gdr_decode_step(const gdr_problem* p, const void* q, const void* k, const void* v,
                           const float* g, const float* beta, float* state, void* o,
                           gdr_stream_t stream);

/* Reads (synchronising on `stream`) and clears the workspace status word written by the
 * chunked kernels: GDR_OK, or GDR_ERR_TIMEOUT if a bounded wait expired. */
gdr_status gdr_workspace_status(void* ws, size_t ws_bytes, gdr_stream_t stream);

/* Check of the library's own failure handling (not an operation of the gated delta rule):
 * launches one CTA whose wait on an mbarrier phase that nothing completes gives up after
 * about one second, records GDR_ERR_TIMEOUT in the status word of `ws` (first 256 bytes,
 * 256-byte aligned) and returns, so the context stays usable. Asynchronous on `stream`;
 * gdr_workspace_status then reports GDR_ERR_TIMEOUT. */
gdr_status gdr_selftest_wait_expiry(void* ws, size_t ws_bytes, gdr_stream_t stream);

/* Bytes of the scratch array built into the library for gdr_fwd_chunked_noalloc. */
#define GDR_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* gdr_fwd_chunked without a workspace argument, for callers that cannot allocate device
 * memory: for example a host application whose device memory is entirely owned by
 * another allocator, or a deployment that forbids device allocation once it has started.
 * (The pages on the gated delta rule have no counterpart to this call.) Instead of a
 * caller workspace it uses a scratch array of GDR_NOALLOC_SCRATCH_BYTES (64 MiB) that the
 * library keeps on every GPU where it is loaded, for the life of the process. The call
 * itself allocates nothing, but with lazy module loading (the CUDA default) the driver
 * reserves that 64 MiB on a device when the first call on it looks up the scratch address:
 * make the first call on each device at start-up (a problem with B = 0 is enough), and
 * before any stream capture. Problems whose gdr_fwd_chunked_workspace() exceeds the
 * scratch return GDR_ERR_WORKSPACE with nothing launched (about 740 chunk records: for
 * example B=1, Hv=32, T <= 1472). `stream` must belong to the current device
 * (GDR_ERR_INVALID_ARG otherwise). Inputs, outputs and the support matrix are those of
 * gdr_fwd_chunked. All calls share the one array and it keeps the last call's contents
 * (the call clears the status word it needs at zero): calls that can overlap on the GPU
 * (different streams, or different host threads) race on it, so serialise them. A
 * bounded-wait expiry is recorded in the scratch's status word: read it with
 * gdr_noalloc_status before the next call clears it. */
gdr_status gdr_fwd_chunked_noalloc(const gdr_problem* p, const void* q, const void* k, const void* v,
                                   const float* g, const float* beta, const float* h0, void* o, float* ht,
                                   gdr_stream_t stream);

/* gdr_workspace_status for the scratch of gdr_fwd_chunked_noalloc on the current device:
 * synchronises on `stream` (which must belong to the current device), then returns GDR_OK,
 * or GDR_ERR_TIMEOUT if a wait of the last call expired, and clears the word. GDR_OK if no
 * call has run on this device. */
gdr_status gdr_noalloc_status(gdr_stream_t stream);

/* Launch tracing for profiling. While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on its own stream (host-side events only; no
 * device memory). gdr_trace_collect() waits for the recorded events, writes up to `max`
 * (kernel name, milliseconds) pairs in launch order, clears the list and returns the
 * number of launches recorded since the last collect (which may exceed `max`). Names
 * point to static strings. Not thread-safe: trace from one host thread at a time. */
gdr_status gdr_trace_enable(int on);
int gdr_trace_collect(const char** names, float* ms, int max);

#ifdef __cplusplus
}
#endif
#endif /* GDR_H_ */
