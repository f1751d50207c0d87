// api.cu - the C ABI (include/gdr.h): argument validation, workspace layout and launches.
// Nothing here allocates device memory; every launch goes to the caller's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "gdr.h"
#include "chunk.h"
#include "common.cuh"
#include "kernels.h"

using namespace gdr;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One CTA waits on an mbarrier phase that nothing completes: the bounded wait gives up after
// about a second, records the expiry in the status word and the kernel returns.
__global__ void wait_expiry_kernel(int* status) {
    __shared__ uint64_t bar;
    __shared__ int abort_sh;
    if (threadIdx.x == 0) {
        abort_sh = 0;
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    mbar_wait(&bar, 0, &abort_sh, status, 99);
    __syncthreads();
}
bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

gdr_status check_problem(const gdr_problem* p, bool decode) {
    if (!p) return GDR_ERR_INVALID_ARG;
    if (p->B < 0 || p->T < 0 || p->Hk <= 0 || p->Hv <= 0 || p->Dk <= 0 || p->Dv <= 0) return GDR_ERR_INVALID_ARG;
    if (p->Hv % p->Hk != 0) return GDR_ERR_INVALID_ARG;
    if (decode && p->T != 1) return GDR_ERR_INVALID_ARG;
    if (p->dtype != GDR_F32 && p->dtype != GDR_BF16) return GDR_ERR_INVALID_ARG;
    if (p->gate != GDR_GATE_SCALAR && p->gate != GDR_GATE_CHANNEL) return GDR_ERR_INVALID_ARG;
    if (p->use_qk_l2norm != 0 && p->use_qk_l2norm != 1) return GDR_ERR_INVALID_ARG;
    if (!isfinite(p->scale)) return GDR_ERR_INVALID_ARG;
    if (!dim_ok(p->Dk) || !dim_ok(p->Dv)) return GDR_ERR_UNSUPPORTED;
    if (p->B > 65535 || p->Hv > 65535) return GDR_ERR_UNSUPPORTED;  // grid y/z limits
    return GDR_OK;
}

// `required` pointers may be null only when the problem has no token (B * T == 0: empty
// tensors have no storage); every non-null pointer must be 16-byte aligned.
gdr_status check_ptrs(const gdr_problem* p, std::initializer_list<const void*> required,
                      std::initializer_list<const void*> optional) {
    const bool empty = p->B == 0 || p->T == 0;
    for (const void* x : required)
        if (!x && !empty) return GDR_ERR_INVALID_ARG;
    for (const void* x : required)
        if (x && !aligned16(x)) return GDR_ERR_INVALID_ARG;
    for (const void* x : optional)
        if (x && !aligned16(x)) return GDR_ERR_INVALID_ARG;
    return GDR_OK;
}

// The chunked calls take every problem check_problem accepts: bf16 q/k/v run on the tensor
// cores, fp32 q/k/v on the CUDA-core fp32 path (chunk_f32.cu).
bool f32(const gdr_problem* p) { return p->dtype == GDR_F32; }

Chunk32Layout layout32(const gdr_problem* p, bool bwd, bool own_rec, bool own_states) {
    return chunk32_layout(p->B, p->T, p->Hv, p->Dk, p->Dv, bwd, own_rec, own_states);
}

// Head sizes below 128 on the chunked path: the kernels work on 128 key and value channels, so
// the inputs are copied into zero-padded 128-wide buffers in the workspace (after the padded
// problem's own workspace) and the results cropped back into the caller's tensors. Zero channels
// and zero state rows / columns contribute nothing, so the original channels are exact.
bool narrow(const gdr_problem* p) { return !f32(p) && (p->Dk != 128 || p->Dv != 128); }

struct Staging {
    size_t q, k, v, g, h0, o, ht, do_, dht, dq, dk, dv, dg, dh0, total;
};
Staging staging(const gdr_problem* p, bool bwd, size_t base) {
    Staging s;
    memset(&s, 0, sizeof(s));
    const size_t tk = (size_t)p->B * p->T * p->Hk * 128, tv = (size_t)p->B * p->T * p->Hv * 128;
    const size_t st = (size_t)p->B * p->Hv * 128 * 128;
    const bool ch = p->gate == GDR_GATE_CHANNEL;
    size_t off = round_up(base, 256);
    auto take = [&](size_t bytes) {
        const size_t r = off;
        off = round_up(off + bytes, 256);
        return r;
    };
    s.q = take(tk * 2);
    s.k = take(tk * 2);
    s.v = take(tv * 2);
    if (ch) s.g = take(tv * 4);
    s.h0 = take(st * 4);
    if (bwd) {
        s.do_ = take(tv * 2);
        s.dht = take(st * 4);
        s.dq = take(tk * 4);
        s.dk = take(tk * 4);
        s.dv = take(tv * 4);
        if (ch) s.dg = take(tv * 4);
        s.dh0 = take(st * 4);
    } else {
        s.o = take(tv * 2);
        s.ht = take(st * 4);
    }
    s.total = off;
    return s;
}
// Workspace bytes of a chunked call whose padded problem needs `core`.
size_t with_staging(const gdr_problem* p, bool bwd, size_t core) {
    return narrow(p) ? staging(p, bwd, core).total : core;
}

RecurrentArgs recurrent_args(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                             const float* beta, const float* h0, void* o, float* ht) {
    RecurrentArgs a;
    a.B = p->B; a.T = p->T; a.Hk = p->Hk; a.Hv = p->Hv; a.Dk = p->Dk; a.Dv = p->Dv;
    a.channel = p->gate == GDR_GATE_CHANNEL;
    a.use_norm = p->use_qk_l2norm;
    a.bf16 = p->dtype == GDR_BF16;
    a.scale = p->scale;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.o = o; a.ht = ht;
    return a;
}

ChunkProblem chunk_problem(const gdr_problem* p) {
    ChunkProblem c;
    c.B = p->B; c.T = p->T; c.Hk = p->Hk; c.Hv = p->Hv;
    c.NC = (p->T + kChunk - 1) / kChunk;
    c.scale = p->scale;
    c.use_norm = p->use_qk_l2norm;
    c.channel = p->gate == GDR_GATE_CHANNEL;
    return c;
}

Chunk32Args args32(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                   const float* beta, const float* h0) {
    Chunk32Args a;
    memset(&a, 0, sizeof(a));
    a.B = p->B; a.T = p->T; a.Hk = p->Hk; a.Hv = p->Hv; a.Dk = p->Dk; a.Dv = p->Dv;
    a.NC = (p->T + kChunk - 1) / kChunk;
    a.channel = p->gate == GDR_GATE_CHANNEL;
    a.use_norm = p->use_qk_l2norm;
    a.scale = p->scale;
    a.q = static_cast<const float*>(q); a.k = static_cast<const float*>(k); a.v = static_cast<const float*>(v);
    a.g = g; a.beta = beta; a.h0 = h0;
    return a;
}

// Bytes of the caller's chunk-start states / saved buffer for this problem.
size_t states_bytes(const gdr_problem* p) {
    return f32(p) ? chunk32_states_bytes(p->B, p->T, p->Hv, p->Dk, p->Dv) : chunk_states_bytes(chunk_problem(p));
}
size_t saved_bytes(const gdr_problem* p) {
    return f32(p) ? chunk32_saved_bytes(p->B, p->T, p->Hv, p->Dk, p->Dv) : chunk_saved_bytes(chunk_problem(p));
}

struct TraceRec {
    const char* name;
    cudaEvent_t start, stop;
};
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

}  // namespace

namespace gdr {
void trace_begin(const char* name, cudaStream_t s) {
    if (!g_trace_on) return;
    TraceRec r{name, pooled_event(), pooled_event()};
    cudaEventRecord(r.start, s);
    g_trace.push_back(r);
}
void trace_end(cudaStream_t s) {
    if (!g_trace_on || g_trace.empty()) return;
    cudaEventRecord(g_trace.back().stop, s);
}
}  // namespace gdr

extern "C" {

gdr_status gdr_trace_enable(int on) {
    g_trace_on = on != 0;
    return GDR_OK;
}

int gdr_trace_collect(const char** names, float* ms, int max) {
    const int n = (int)g_trace.size();
    for (int i = 0; i < n; i++) {
        TraceRec& r = g_trace[i];
        float t = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess)
            t = -1.f;
        if (i < max) {
            if (names) names[i] = r.name;
            if (ms) ms[i] = t;
        }
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_trace.clear();
    return n;
}


const char* gdr_status_string(gdr_status s) {
    switch (s) {
        case GDR_OK: return "GDR_OK";
        case GDR_ERR_INVALID_ARG: return "GDR_ERR_INVALID_ARG: invalid argument";
        case GDR_ERR_UNSUPPORTED: return "GDR_ERR_UNSUPPORTED: combination not implemented";
        case GDR_ERR_WORKSPACE: return "GDR_ERR_WORKSPACE: workspace too small";
        case GDR_ERR_CUDA: return "GDR_ERR_CUDA: CUDA launch or runtime error";
        case GDR_ERR_TIMEOUT: return "GDR_ERR_TIMEOUT: a bounded device wait expired";
        default: return "unknown gdr_status";
    }
}

size_t gdr_fwd_chunked_workspace(const gdr_problem* p) {
    if (check_problem(p, false) != GDR_OK) return 0;
    if (f32(p)) return layout32(p, false, true, false).total;
    return with_staging(p, false, chunk_fwd_workspace(chunk_problem(p)));
}

size_t gdr_bwd_chunked_workspace(const gdr_problem* p) {
    if (check_problem(p, false) != GDR_OK) return 0;
    if (f32(p)) return layout32(p, true, true, true).total;
    return with_staging(p, true, chunk_bwd_workspace(chunk_problem(p)));
}

gdr_status gdr_fwd_sequential(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                              const float* beta, const float* h0, void* o, float* ht, gdr_stream_t stream) {
    gdr_status s = check_problem(p, false);
    if (s != GDR_OK) return s;
    if ((s = check_ptrs(p, {q, k, v, g, beta, o}, {h0, ht})) != GDR_OK) return s;
    if (p->B == 0) return GDR_OK;
    RecurrentArgs a = recurrent_args(p, q, k, v, g, beta, h0, o, ht);
    return launch_recurrent(a, false, (cudaStream_t)stream) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status gdr_decode_step(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float* state, void* o, gdr_stream_t stream) {
    gdr_status s = check_problem(p, true);
    if (s != GDR_OK) return s;
    if ((s = check_ptrs(p, {q, k, v, g, beta, state, o}, {})) != GDR_OK) return s;
    if (p->B == 0) return GDR_OK;
    RecurrentArgs a = recurrent_args(p, q, k, v, g, beta, state, o, state);
    return launch_recurrent(a, true, (cudaStream_t)stream) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

size_t gdr_chunk_states_bytes(const gdr_problem* p) {
    if (check_problem(p, false) != GDR_OK) return 0;
    if (f32(p)) return states_bytes(p);
    return chunk_states_bytes(chunk_problem(p));
}

size_t gdr_bwd_chunked_states_workspace(const gdr_problem* p) {
    if (check_problem(p, false) != GDR_OK) return 0;
    if (f32(p)) return layout32(p, true, true, false).total;
    return with_staging(p, true, chunk_bwd_states_workspace(chunk_problem(p)));
}

static gdr_status fwd_chunked_impl(const gdr_problem* p, const void* q, const void* k, const void* v,
                                   const float* g, const float* beta, const float* h0, void* o, float* ht,
                                   void* states, void* saved, void* ws, size_t ws_bytes, gdr_stream_t stream);

gdr_status gdr_fwd_chunked_states(const gdr_problem* p, const void* q, const void* k, const void* v,
                                  const float* g, const float* beta, const float* h0, void* o, float* ht,
                                  void* states, size_t states_bytes, void* ws, size_t ws_bytes,
                                  gdr_stream_t stream) {
    gdr_status s = check_problem(p, false);
    if (s != GDR_OK) return s;
    const size_t need = ::states_bytes(p);
    if (need && (!states || states_bytes < need)) return GDR_ERR_WORKSPACE;
    if (states && (reinterpret_cast<uintptr_t>(states) & 255u) != 0) return GDR_ERR_INVALID_ARG;
    return fwd_chunked_impl(p, q, k, v, g, beta, h0, o, ht, states, nullptr, ws, ws_bytes, stream);
}

gdr_status gdr_fwd_chunked(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                           const float* beta, const float* h0, void* o, float* ht, void* ws, size_t ws_bytes,
                           gdr_stream_t stream) {
    return fwd_chunked_impl(p, q, k, v, g, beta, h0, o, ht, nullptr, nullptr, ws, ws_bytes, stream);
}

size_t gdr_chunk_saved_bytes(const gdr_problem* p) {
    if (check_problem(p, false) != GDR_OK) return 0;
    return saved_bytes(p);
}

size_t gdr_fwd_chunked_saved_workspace(const gdr_problem* p) {
    if (check_problem(p, false) != GDR_OK) return 0;
    if (f32(p)) return layout32(p, false, false, false).total;
    return with_staging(p, false, kSavedFwdWorkspace);
}

size_t gdr_bwd_chunked_saved_workspace(const gdr_problem* p) {
    if (check_problem(p, false) != GDR_OK) return 0;
    if (f32(p)) return layout32(p, true, false, false).total;
    return with_staging(p, true, chunk_bwd_saved_workspace(chunk_problem(p)));
}

gdr_status gdr_fwd_chunked_saved(const gdr_problem* p, const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, const float* h0, void* o, float* ht,
                                 void* saved, size_t saved_bytes, void* ws, size_t ws_bytes, gdr_stream_t stream) {
    gdr_status s = check_problem(p, false);
    if (s != GDR_OK) return s;
    const size_t need = ::saved_bytes(p);
    if (need && (!saved || saved_bytes < need)) return GDR_ERR_WORKSPACE;
    if (saved && (reinterpret_cast<uintptr_t>(saved) & 255u) != 0) return GDR_ERR_INVALID_ARG;
    return fwd_chunked_impl(p, q, k, v, g, beta, h0, o, ht, nullptr, saved, ws, ws_bytes, stream);
}

static gdr_status fwd_chunked_impl(const gdr_problem* p, const void* q, const void* k, const void* v,
                                   const float* g, const float* beta, const float* h0, void* o, float* ht,
                                   void* states, void* saved, void* ws, size_t ws_bytes, gdr_stream_t stream) {
    gdr_status s = check_problem(p, false);
    if (s != GDR_OK) return s;
    if ((s = check_ptrs(p, {q, k, v, g, beta, o}, {h0, ht})) != GDR_OK) return s;
    const size_t core = f32(p)  ? layout32(p, false, !saved, false).total
                        : saved ? kSavedFwdWorkspace
                                : chunk_fwd_workspace(chunk_problem(p));
    const size_t need = with_staging(p, false, core);
    if (!ws || ws_bytes < need) return GDR_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GDR_ERR_INVALID_ARG;
    if (p->B == 0) return GDR_OK;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return GDR_ERR_CUDA;
    if (p->T == 0) {  // no token: ht = h0 (or zero)
        if (!ht) return GDR_OK;
        RecurrentArgs a = recurrent_args(p, q, k, v, g, beta, h0, o, ht);
        return launch_recurrent(a, false, st) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    }
    if (f32(p)) {
        Chunk32Args a = args32(p, q, k, v, g, beta, h0);
        a.o = static_cast<float*>(o);
        a.ht = ht;
        uint8_t* w = static_cast<uint8_t*>(ws);
        const Chunk32Layout l = layout32(p, false, !saved, false);
        uint8_t* sv = static_cast<uint8_t*>(saved);
        a.rec = reinterpret_cast<float*>(saved ? sv : w + l.rec);
        a.states = reinterpret_cast<float*>(
            saved ? sv + chunk32_saved_states_offset(p->B, p->T, p->Hv, p->Dk, p->Dv) : states);
        return launch_chunk32_fwd(a, true, st) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    }
    ChunkFwdArgs a;
    a.p = chunk_problem(p);
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.o = o; a.ht = ht;
    a.states = states;
    a.saved = saved;
    a.ws = ws;
    if (!narrow(p)) return launch_chunk_fwd(a, st) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    // head sizes below 128: zero-padded copies in, cropped results out
    const Staging sg = staging(p, false, core);
    uint8_t* w = static_cast<uint8_t*>(ws);
    const size_t tk = (size_t)p->B * p->T * p->Hk, tv = (size_t)p->B * p->T * p->Hv, bh = (size_t)p->B * p->Hv;
    const bool ch = p->gate == GDR_GATE_CHANNEL;
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    ok(launch_pad(q, w + sg.q, 2, tk, 1, p->Dk, 1, 128, st));
    ok(launch_pad(k, w + sg.k, 2, tk, 1, p->Dk, 1, 128, st));
    ok(launch_pad(v, w + sg.v, 2, tv, 1, p->Dv, 1, 128, st));
    if (ch) ok(launch_pad(g, w + sg.g, 4, tv, 1, p->Dk, 1, 128, st));
    if (h0) ok(launch_pad(h0, w + sg.h0, 4, bh, p->Dv, p->Dk, 128, 128, st));
    if (e != cudaSuccess) return GDR_ERR_CUDA;
    a.q = w + sg.q; a.k = w + sg.k; a.v = w + sg.v;
    a.g = ch ? reinterpret_cast<const float*>(w + sg.g) : g;
    a.h0 = h0 ? reinterpret_cast<const float*>(w + sg.h0) : nullptr;
    a.o = w + sg.o;
    a.ht = ht ? reinterpret_cast<float*>(w + sg.ht) : nullptr;
    if (launch_chunk_fwd(a, st) != cudaSuccess) return GDR_ERR_CUDA;
    ok(launch_crop(w + sg.o, o, 2, tv, 1, 128, 1, p->Dv, st));
    if (ht) ok(launch_crop(w + sg.ht, ht, 4, bh, 128, 128, p->Dv, p->Dk, st));
    return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

static gdr_status bwd_chunked_impl(const gdr_problem* p, const void* q, const void* k, const void* v,
                                   const float* g, const float* beta, const float* h0, const void* states,
                                   const void* saved, const void* do_, const float* dht, float* dq, float* dk,
                                   float* dv, float* dg, float* dbeta, float* dh0, void* ws, size_t ws_bytes,
                                   gdr_stream_t stream);

gdr_status gdr_bwd_chunked(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                           const float* beta, const float* h0, const void* do_, const float* dht, float* dq,
                           float* dk, float* dv, float* dg, float* dbeta, float* dh0, void* ws, size_t ws_bytes,
                           gdr_stream_t stream) {
    return bwd_chunked_impl(p, q, k, v, g, beta, h0, nullptr, nullptr, do_, dht, dq, dk, dv, dg, dbeta, dh0, ws,
                            ws_bytes, stream);
}

gdr_status gdr_bwd_chunked_states(const gdr_problem* p, const void* q, const void* k, const void* v,
                                  const float* g, const float* beta, const void* states, size_t states_bytes,
                                  const void* do_, const float* dht, float* dq, float* dk, float* dv, float* dg,
                                  float* dbeta, float* dh0, void* ws, size_t ws_bytes, gdr_stream_t stream) {
    gdr_status s = check_problem(p, false);
    if (s != GDR_OK) return s;
    const size_t need = ::states_bytes(p);
    if (need && (!states || states_bytes < need)) return GDR_ERR_WORKSPACE;
    if (states && (reinterpret_cast<uintptr_t>(states) & 255u) != 0) return GDR_ERR_INVALID_ARG;
    return bwd_chunked_impl(p, q, k, v, g, beta, nullptr, states, nullptr, do_, dht, dq, dk, dv, dg, dbeta,
                            dh0, ws, ws_bytes, stream);
}

gdr_status gdr_bwd_chunked_saved(const gdr_problem* p, const void* q, const void* k, const void* v,
                                 const float* g, const float* beta, const void* saved, size_t saved_bytes,
                                 const void* do_, const float* dht, float* dq, float* dk, float* dv, float* dg,
                                 float* dbeta, float* dh0, void* ws, size_t ws_bytes, gdr_stream_t stream) {
    gdr_status s = check_problem(p, false);
    if (s != GDR_OK) return s;
    const size_t need = ::saved_bytes(p);
    if (need && (!saved || saved_bytes < need)) return GDR_ERR_WORKSPACE;
    if (saved && (reinterpret_cast<uintptr_t>(saved) & 255u) != 0) return GDR_ERR_INVALID_ARG;
    return bwd_chunked_impl(p, q, k, v, g, beta, nullptr, nullptr, saved, do_, dht, dq, dk, dv, dg, dbeta, dh0,
                            ws, ws_bytes, stream);
}

static gdr_status bwd_chunked_impl(const gdr_problem* p, const void* q, const void* k, const void* v,
                                   const float* g, const float* beta, const float* h0, const void* states,
                                   const void* saved, const void* do_, const float* dht, float* dq, float* dk,
                                   float* dv, float* dg, float* dbeta, float* dh0, void* ws, size_t ws_bytes,
                                   gdr_stream_t stream) {
    gdr_status s = check_problem(p, false);
    if (s != GDR_OK) return s;
    if ((s = check_ptrs(p, {q, k, v, g, beta, do_, dq, dk, dv, dg, dbeta}, {h0, dht, dh0})) != GDR_OK) return s;
    const ChunkProblem cp = chunk_problem(p);
    const size_t core = f32(p)   ? layout32(p, true, !saved, !saved && !states).total
                        : saved  ? chunk_bwd_saved_workspace(cp)
                        : states ? chunk_bwd_states_workspace(cp)
                                 : chunk_bwd_workspace(cp);
    const size_t need = with_staging(p, true, core);
    if (!ws || ws_bytes < need) return GDR_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GDR_ERR_INVALID_ARG;
    if (p->B == 0) return GDR_OK;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return GDR_ERR_CUDA;
    if (p->T == 0) {  // no token: dh0 = dht (or zero)
        if (!dh0) return GDR_OK;
        const size_t bytes = (size_t)p->B * p->Hv * p->Dv * p->Dk * sizeof(float);
        cudaError_t e = dht ? cudaMemcpyAsync(dh0, dht, bytes, cudaMemcpyDeviceToDevice, st)
                            : cudaMemsetAsync(dh0, 0, bytes, st);
        return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    }
    if (f32(p)) {
        Chunk32Args a = args32(p, q, k, v, g, beta, h0);
        a.do_ = static_cast<const float*>(do_);
        a.dht = dht;
        a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
        uint8_t* w = static_cast<uint8_t*>(ws);
        const Chunk32Layout l = layout32(p, true, !saved, !saved && !states);
        const uint8_t* sv = static_cast<const uint8_t*>(saved);
        const float* hs = saved  ? reinterpret_cast<const float*>(
                                       sv + chunk32_saved_states_offset(p->B, p->T, p->Hv, p->Dk, p->Dv))
                          : states ? static_cast<const float*>(states)
                                   : reinterpret_cast<const float*>(w + l.states);
        a.rec = saved ? reinterpret_cast<float*>(const_cast<uint8_t*>(sv)) : reinterpret_cast<float*>(w + l.rec);
        a.states = const_cast<float*>(hs);
        a.dstates = reinterpret_cast<float*>(w + l.dstates);
        a.dqh = reinterpret_cast<float*>(w + l.dqh);
        a.dkh = reinterpret_cast<float*>(w + l.dkh);
        a.scratch = reinterpret_cast<float*>(w + l.scratch);
        a.nscratch = l.nscratch;
        return launch_chunk32_bwd(a, !saved, !saved && !states, st) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    }
    ChunkBwdArgs a;
    a.p = chunk_problem(p);
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.do_ = do_; a.dht = dht;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
    a.states = states;
    a.saved = saved;
    a.ws = ws;
    if (!narrow(p)) return launch_chunk_bwd(a, st) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    // head sizes below 128: zero-padded copies in, cropped gradients out
    const Staging sg = staging(p, true, core);
    uint8_t* w = static_cast<uint8_t*>(ws);
    const size_t tk = (size_t)p->B * p->T * p->Hk, tv = (size_t)p->B * p->T * p->Hv, bh = (size_t)p->B * p->Hv;
    const bool ch = p->gate == GDR_GATE_CHANNEL;
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
    ok(launch_pad(q, w + sg.q, 2, tk, 1, p->Dk, 1, 128, st));
    ok(launch_pad(k, w + sg.k, 2, tk, 1, p->Dk, 1, 128, st));
    ok(launch_pad(v, w + sg.v, 2, tv, 1, p->Dv, 1, 128, st));
    ok(launch_pad(do_, w + sg.do_, 2, tv, 1, p->Dv, 1, 128, st));
    if (ch) ok(launch_pad(g, w + sg.g, 4, tv, 1, p->Dk, 1, 128, st));
    if (h0) ok(launch_pad(h0, w + sg.h0, 4, bh, p->Dv, p->Dk, 128, 128, st));
    if (dht) ok(launch_pad(dht, w + sg.dht, 4, bh, p->Dv, p->Dk, 128, 128, st));
    if (e != cudaSuccess) return GDR_ERR_CUDA;
    a.q = w + sg.q; a.k = w + sg.k; a.v = w + sg.v; a.do_ = w + sg.do_;
    a.g = ch ? reinterpret_cast<const float*>(w + sg.g) : g;
    a.h0 = h0 ? reinterpret_cast<const float*>(w + sg.h0) : nullptr;
    a.dht = dht ? reinterpret_cast<const float*>(w + sg.dht) : nullptr;
    a.dq = reinterpret_cast<float*>(w + sg.dq);
    a.dk = reinterpret_cast<float*>(w + sg.dk);
    a.dv = reinterpret_cast<float*>(w + sg.dv);
    a.dg = ch ? reinterpret_cast<float*>(w + sg.dg) : dg;
    a.dh0 = dh0 ? reinterpret_cast<float*>(w + sg.dh0) : nullptr;
    if (launch_chunk_bwd(a, st) != cudaSuccess) return GDR_ERR_CUDA;
    ok(launch_crop(w + sg.dq, dq, 4, tk, 1, 128, 1, p->Dk, st));
    ok(launch_crop(w + sg.dk, dk, 4, tk, 1, 128, 1, p->Dk, st));
    ok(launch_crop(w + sg.dv, dv, 4, tv, 1, 128, 1, p->Dv, st));
    if (ch) ok(launch_crop(w + sg.dg, dg, 4, tv, 1, 128, 1, p->Dk, st));
    if (dh0) ok(launch_crop(w + sg.dh0, dh0, 4, bh, 128, 128, p->Dv, p->Dk, st));
    return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

size_t gdr_bwd_sequential_workspace(const gdr_problem* p) {
    if (check_problem(p, false) != GDR_OK) return 0;
    return seq_bwd_workspace(p->B, p->T, p->Hv, p->Dk, p->Dv);
}

gdr_status gdr_bwd_sequential(const gdr_problem* p, const void* q, const void* k, const void* v, const float* g,
                              const float* beta, const float* h0, const void* do_, const float* dht, float* dq,
                              float* dk, float* dv, float* dg, float* dbeta, float* dh0, void* ws, size_t ws_bytes,
                              gdr_stream_t stream) {
    gdr_status s = check_problem(p, false);
    if (s != GDR_OK) return s;
    if ((s = check_ptrs(p, {q, k, v, g, beta, do_, dq, dk, dv, dg, dbeta}, {h0, dht, dh0})) != GDR_OK) return s;
    const size_t need = seq_bwd_workspace(p->B, p->T, p->Hv, p->Dk, p->Dv);
    if (!ws || ws_bytes < need) return GDR_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GDR_ERR_INVALID_ARG;
    if (p->B == 0) return GDR_OK;
    cudaStream_t st = (cudaStream_t)stream;
    if (p->T == 0) {  // no token: dh0 = dht (or zero)
        if (!dh0) return GDR_OK;
        const size_t bytes = (size_t)p->B * p->Hv * p->Dv * p->Dk * sizeof(float);
        cudaError_t e = dht ? cudaMemcpyAsync(dh0, dht, bytes, cudaMemcpyDeviceToDevice, st)
                            : cudaMemsetAsync(dh0, 0, bytes, st);
        return e == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
    }
    SeqBwdArgs a;
    a.B = p->B; a.T = p->T; a.Hk = p->Hk; a.Hv = p->Hv; a.Dk = p->Dk; a.Dv = p->Dv;
    a.channel = p->gate == GDR_GATE_CHANNEL;
    a.use_norm = p->use_qk_l2norm;
    a.bf16 = p->dtype == GDR_BF16;
    a.scale = p->scale;
    a.q = q; a.k = k; a.v = v; a.do_ = do_; a.g = g; a.beta = beta; a.h0 = h0; a.dht = dht;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
    return launch_seq_bwd(a, ws, st) == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status gdr_workspace_status(void* ws, size_t ws_bytes, gdr_stream_t stream) {
    if (!ws || ws_bytes < 256) return GDR_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int word[4] = {0, 0, 0, 0};
    if (cudaMemcpyAsync(word, ws, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess) return GDR_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDR_ERR_CUDA;
    if (word[0] == 0) return GDR_OK;
    if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
        return GDR_ERR_CUDA;
    return word[0] == GDR_ERR_TIMEOUT ? GDR_ERR_TIMEOUT : GDR_ERR_CUDA;
}

gdr_status gdr_selftest_wait_expiry(void* ws, size_t ws_bytes, gdr_stream_t stream) {
    if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return GDR_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return GDR_ERR_CUDA;
    wait_expiry_kernel<<<1, 32, 0, st>>>(static_cast<int*>(ws));
    return cudaGetLastError() == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // extern "C"
