/*
 * Gated delta rule: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or load this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg do. It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the definition, written out step by step, no blocking or
 * reordering beyond it):
 *
 *   Per batch b and value head hv, with key/query head hk = hv / (Hv / Hk)
 *   (grouped-query sharing: consecutive value heads read the same key head), a state
 *   S in R^{Dv x Dk} starts at h0 (zero if absent) and for t = 0 .. T-1:
 *
 *     k^ = n(k_t), q^ = n(q_t),  n(x) = x * (sum x^2 + 1e-6)^(-1/2)  if the flag is set
 *     a  = exp(g_t)              (a scalar per head, or one value per key channel)
 *     S  = a S (I - beta_t k^ k^T) + beta_t v_t k^T        (decay folded into the state)
 *     o_t = scale * S q^
 *
 *   The update is evaluated in the expanded order   Sd = S diag(a);  p = Sd k^;
 *   S = Sd + beta (v - p) k^T,  which is the same matrix as the product form above.
 *
 * Sources (pages on the gated delta rule):
 *   - "perf(gated_delta_net): fold q/k L2-norm into the gated_delta_rule kernel"
 *     (Megatron-LM PR #5396), "What"/"Why" sections: the kernel owns the q/k L2
 *     normalisation of the last dimension, eps = 1e-6.
 *   - "Two-pass optimization for channelwise gated delta rule kernel" (ExecuTorch
 *     PR #21020), Summary: a per-channel decay vector; the prediction uses the
 *     decayed state ("folding in decay").
 *   - "Adding VJP for gated delta net" (MLX PR #4565): the backward (VJP) with
 *     respect to q, k, v, g, beta and the initial state.
 *   The recurrence itself is the Gated DeltaNet recurrence those pages refer to.
 *
 * The backward is hand-derived reverse mode of exactly the steps above (fp64), with
 * the state checkpointed every SEG steps and recomputed inside a segment.
 *
 * Layouts (dense, row-major): q,k [B,T,Hk,Dk]; v,o,do [B,T,Hv,Dv]; g [B,T,Hv]
 * (scalar gate) or [B,T,Hv,Dk] (channel gate); beta [B,T,Hv]; states [B,Hv,Dv,Dk].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define NORM_EPS 1e-6
#define SEG 64

typedef struct {
    int B, T, Hk, Hv, Dk, Dv;
    int channel_gate; /* 0: g is one log-decay per (b,t,hv); 1: one per key channel */
    int use_l2norm;   /* 1: normalise q and k inside (eps 1e-6) */
    double scale;
} dims_t;

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* x^ = x * (sum x^2 + eps)^(-1/2); returns the factor rho so that x^ = rho * x. */
static double l2n(const double* x, int n, int on, double* out) {
    double rho = 1.0;
    if (on) {
        double ss = 0.0;
        for (int i = 0; i < n; i++) ss += x[i] * x[i];
        rho = 1.0 / sqrt(ss + NORM_EPS);
    }
    for (int i = 0; i < n; i++) out[i] = x[i] * rho;
    return rho;
}

static size_t qk_off(const dims_t* d, int b, int t, int hk) {
    return (((size_t)b * d->T + t) * d->Hk + hk) * d->Dk;
}
static size_t vo_off(const dims_t* d, int b, int t, int hv) {
    return (((size_t)b * d->T + t) * d->Hv + hv) * d->Dv;
}
static size_t bt_off(const dims_t* d, int b, int t, int hv) {
    return ((size_t)b * d->T + t) * d->Hv + hv;
}
static size_t st_off(const dims_t* d, int b, int hv) {
    return ((size_t)b * d->Hv + hv) * d->Dv * d->Dk;
}

/* decay vector a (length Dk) for token t of head hv */
static void gate_vec(const dims_t* d, const double* g, int b, int t, int hv, double* a) {
    if (d->channel_gate) {
        const double* gp = g + bt_off(d, b, t, hv) * d->Dk;
        for (int i = 0; i < d->Dk; i++) a[i] = exp(gp[i]);
    } else {
        double s = exp(g[bt_off(d, b, t, hv)]);
        for (int i = 0; i < d->Dk; i++) a[i] = s;
    }
}

/* One step of the recurrence on one head's state S [Dv x Dk].
 * kh, qh: normalised key/query; a: decay; writes the prediction p and the
 * residual delta = beta (v - p) (both length Dv) and o (length Dv). */
static void step(int Dk, int Dv, double* S, const double* kh, const double* qh, const double* a,
                 double beta, const double* v, double scale, double* p, double* delta, double* o) {
    for (int i = 0; i < Dv; i++) {
        double* Si = S + (size_t)i * Dk;
        double acc = 0.0;
        for (int c = 0; c < Dk; c++) {
            Si[c] *= a[c];          /* Sd = S diag(a) */
            acc += Si[c] * kh[c];   /* p = Sd k^ */
        }
        p[i] = acc;
        delta[i] = beta * (v[i] - acc);
        double out = 0.0;
        for (int c = 0; c < Dk; c++) {
            Si[c] += delta[i] * kh[c];  /* S = Sd + delta k^T */
            out += Si[c] * qh[c];
        }
        o[i] = scale * out;
    }
}

int oracle_forward(int B, int T, int Hk, int Hv, int Dk, int Dv, int channel_gate, double scale,
                   int use_l2norm, const double* q, const double* k, const double* v,
                   const double* g, const double* beta, const double* h0, double* o, double* ht) {
    if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0 || Hv % Hk != 0) return 1;
    dims_t d = {B, T, Hk, Hv, Dk, Dv, channel_gate, use_l2norm, scale};
    int group = Hv / Hk;
    long nh = (long)B * Hv;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bh = 0; bh < nh; bh++) {
        int b = (int)(bh / Hv), hv = (int)(bh % Hv), hk = hv / group;
        double* S = (double*)malloc(sizeof(double) * Dv * Dk);
        double* kh = (double*)malloc(sizeof(double) * Dk);
        double* qh = (double*)malloc(sizeof(double) * Dk);
        double* a = (double*)malloc(sizeof(double) * Dk);
        double* p = (double*)malloc(sizeof(double) * Dv);
        double* dl = (double*)malloc(sizeof(double) * Dv);
        if (h0) memcpy(S, h0 + st_off(&d, b, hv), sizeof(double) * Dv * Dk);
        else memset(S, 0, sizeof(double) * Dv * Dk);
        for (int t = 0; t < T; t++) {
            l2n(k + qk_off(&d, b, t, hk), Dk, use_l2norm, kh);
            l2n(q + qk_off(&d, b, t, hk), Dk, use_l2norm, qh);
            gate_vec(&d, g, b, t, hv, a);
            step(Dk, Dv, S, kh, qh, a, beta[bt_off(&d, b, t, hv)], v + vo_off(&d, b, t, hv), scale,
                 p, dl, o + vo_off(&d, b, t, hv));
        }
        if (ht) memcpy(ht + st_off(&d, b, hv), S, sizeof(double) * Dv * Dk);
        free(S); free(kh); free(qh); free(a); free(p); free(dl);
    }
    return 0;
}

/* One single-token step on a state held in place: the decode operation.
 * q,k [B,Hk,Dk]; v,o [B,Hv,Dv]; g [B,Hv] or [B,Hv,Dk]; beta [B,Hv]; state [B,Hv,Dv,Dk]. */
int oracle_decode_step(int B, int Hk, int Hv, int Dk, int Dv, int channel_gate, double scale,
                       int use_l2norm, const double* q, const double* k, const double* v,
                       const double* g, const double* beta, double* state, double* o) {
    return oracle_forward(B, 1, Hk, Hv, Dk, Dv, channel_gate, scale, use_l2norm, q, k, v, g, beta,
                          state, o, state);
}

/*
 * Reverse mode of oracle_forward for the loss  L = <do, o> + <dht, ht>.
 * Outputs (all overwritten): dq, dk [B,T,Hk,Dk] (summed over the value heads that
 * share a key head); dv [B,T,Hv,Dv]; dg like g; dbeta [B,T,Hv]; dh0 [B,Hv,Dv,Dk]
 * (may be NULL). h0 and dht may be NULL (zero).
 *
 * Per step, in reverse, with G the adjoint of the state after the step:
 *   G += scale do q^T;            dq^ = scale S^T do
 *   ddelta = G k^;                dk^ += G^T delta
 *   dbeta = ddelta . (v - p);     dv = beta ddelta;      dp = -beta ddelta
 *   Gd = G + dp k^T               (adjoint of Sd = S_prev diag(a))
 *   dk^ += Sd^T dp;               da_c = sum_i Gd[i,c] S_prev[i,c]
 *   G  = Gd diag(a);              dg = a * da  (scalar gate: summed over channels)
 *   norm:  dx = rho (dx^ - x^ (x^ . dx^))
 */
int oracle_backward(int B, int T, int Hk, int Hv, int Dk, int Dv, int channel_gate, double scale,
                    int use_l2norm, const double* q, const double* k, const double* v,
                    const double* g, const double* beta, const double* h0, const double* dout,
                    const double* dht, double* dq, double* dk, double* dv, double* dg,
                    double* dbeta, double* dh0) {
    if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || Dk <= 0 || Dv <= 0 || Hv % Hk != 0) return 1;
    dims_t d = {B, T, Hk, Hv, Dk, Dv, channel_gate, use_l2norm, scale};
    int group = Hv / Hk;
    size_t SS = (size_t)Dv * Dk;
    memset(dq, 0, sizeof(double) * (size_t)B * T * Hk * Dk);
    memset(dk, 0, sizeof(double) * (size_t)B * T * Hk * Dk);
    long ngroups = (long)B * Hk;
#pragma omp parallel for schedule(dynamic, 1)
    for (long bg = 0; bg < ngroups; bg++) {
        int b = (int)(bg / Hk), hk = (int)(bg % Hk);
        int nseg = (T + SEG - 1) / SEG;
        double* ckpt = (double*)malloc(sizeof(double) * SS * (size_t)(nseg > 0 ? nseg : 1));
        double* Sseg = (double*)malloc(sizeof(double) * SS * (SEG + 1)); /* states in a segment */
        double* KH = (double*)malloc(sizeof(double) * Dk * SEG);
        double* QH = (double*)malloc(sizeof(double) * Dk * SEG);
        double* RK = (double*)malloc(sizeof(double) * SEG);
        double* RQ = (double*)malloc(sizeof(double) * SEG);
        double* AA = (double*)malloc(sizeof(double) * Dk * SEG);
        double* PP = (double*)malloc(sizeof(double) * Dv * SEG);
        double* DL = (double*)malloc(sizeof(double) * Dv * SEG);
        double* G = (double*)malloc(sizeof(double) * SS);
        double* Gd = (double*)malloc(sizeof(double) * SS);
        double* tmp_o = (double*)malloc(sizeof(double) * Dv);
        double* dqh = (double*)malloc(sizeof(double) * Dk);
        double* dkh = (double*)malloc(sizeof(double) * Dk);
        double* dd = (double*)malloc(sizeof(double) * Dv);
        double* dp = (double*)malloc(sizeof(double) * Dv);
        double* da = (double*)malloc(sizeof(double) * Dk);
        for (int hv = hk * group; hv < (hk + 1) * group; hv++) {
            /* forward pass storing a checkpoint at the start of every segment */
            double* S = Sseg;
            if (h0) memcpy(S, h0 + st_off(&d, b, hv), sizeof(double) * SS);
            else memset(S, 0, sizeof(double) * SS);
            for (int t = 0; t < T; t++) {
                if (t % SEG == 0) memcpy(ckpt + SS * (t / SEG), S, sizeof(double) * SS);
                l2n(k + qk_off(&d, b, t, hk), Dk, use_l2norm, KH);
                l2n(q + qk_off(&d, b, t, hk), Dk, use_l2norm, QH);
                gate_vec(&d, g, b, t, hv, AA);
                step(Dk, Dv, S, KH, QH, AA, beta[bt_off(&d, b, t, hv)], v + vo_off(&d, b, t, hv),
                     scale, PP, DL, tmp_o);
            }
            if (dht) memcpy(G, dht + st_off(&d, b, hv), sizeof(double) * SS);
            else memset(G, 0, sizeof(double) * SS);
            for (int sg = nseg - 1; sg >= 0; sg--) {
                int t0 = sg * SEG, t1 = t0 + SEG < T ? t0 + SEG : T, L = t1 - t0;
                /* recompute the segment: Sseg[j] is the state before step t0+j */
                memcpy(Sseg, ckpt + SS * sg, sizeof(double) * SS);
                for (int j = 0; j < L; j++) {
                    int t = t0 + j;
                    memcpy(Sseg + SS * (j + 1), Sseg + SS * j, sizeof(double) * SS);
                    RK[j] = l2n(k + qk_off(&d, b, t, hk), Dk, use_l2norm, KH + (size_t)j * Dk);
                    RQ[j] = l2n(q + qk_off(&d, b, t, hk), Dk, use_l2norm, QH + (size_t)j * Dk);
                    gate_vec(&d, g, b, t, hv, AA + (size_t)j * Dk);
                    step(Dk, Dv, Sseg + SS * (j + 1), KH + (size_t)j * Dk, QH + (size_t)j * Dk,
                         AA + (size_t)j * Dk, beta[bt_off(&d, b, t, hv)], v + vo_off(&d, b, t, hv),
                         scale, PP + (size_t)j * Dv, DL + (size_t)j * Dv, tmp_o);
                }
                for (int j = L - 1; j >= 0; j--) {
                    int t = t0 + j;
                    const double* Sprev = Sseg + SS * j;
                    const double* Scur = Sseg + SS * (j + 1);
                    const double* kh = KH + (size_t)j * Dk;
                    const double* qh = QH + (size_t)j * Dk;
                    const double* a = AA + (size_t)j * Dk;
                    const double* p = PP + (size_t)j * Dv;
                    const double* dl = DL + (size_t)j * Dv;
                    const double* dot = dout + vo_off(&d, b, t, hv);
                    const double* vt = v + vo_off(&d, b, t, hv);
                    double bt = beta[bt_off(&d, b, t, hv)];
                    /* output o = scale S q^ */
                    for (int c = 0; c < Dk; c++) dqh[c] = 0.0;
                    for (int i = 0; i < Dv; i++) {
                        for (int c = 0; c < Dk; c++) {
                            G[(size_t)i * Dk + c] += scale * dot[i] * qh[c];
                            dqh[c] += scale * Scur[(size_t)i * Dk + c] * dot[i];
                        }
                    }
                    /* S = Sd + delta k^T */
                    for (int c = 0; c < Dk; c++) dkh[c] = 0.0;
                    double dbt = 0.0;
                    for (int i = 0; i < Dv; i++) {
                        double acc = 0.0;
                        for (int c = 0; c < Dk; c++) {
                            acc += G[(size_t)i * Dk + c] * kh[c];
                            dkh[c] += G[(size_t)i * Dk + c] * dl[i];
                        }
                        dd[i] = acc;
                        /* delta = beta (v - p) */
                        dbt += acc * (vt[i] - p[i]);
                        dv[vo_off(&d, b, t, hv) + i] = bt * acc;
                        dp[i] = -bt * acc;
                    }
                    dbeta[bt_off(&d, b, t, hv)] = dbt;
                    /* p = Sd k^ with Sd = S_prev diag(a) */
                    for (int c = 0; c < Dk; c++) da[c] = 0.0;
                    for (int i = 0; i < Dv; i++) {
                        for (int c = 0; c < Dk; c++) {
                            size_t ic = (size_t)i * Dk + c;
                            Gd[ic] = G[ic] + dp[i] * kh[c];
                            dkh[c] += Sprev[ic] * a[c] * dp[i];
                            da[c] += Gd[ic] * Sprev[ic];
                        }
                    }
                    for (int i = 0; i < Dv; i++)
                        for (int c = 0; c < Dk; c++) G[(size_t)i * Dk + c] = Gd[(size_t)i * Dk + c] * a[c];
                    if (channel_gate) {
                        double* dgp = dg + bt_off(&d, b, t, hv) * Dk;
                        for (int c = 0; c < Dk; c++) dgp[c] = a[c] * da[c];
                    } else {
                        double s = 0.0;
                        for (int c = 0; c < Dk; c++) s += da[c];
                        dg[bt_off(&d, b, t, hv)] = a[0] * s;
                    }
                    /* normalisation backward, then sum into the shared key head */
                    double* dqo = dq + qk_off(&d, b, t, hk);
                    double* dko = dk + qk_off(&d, b, t, hk);
                    if (use_l2norm) {
                        double sq = 0.0, sk = 0.0;
                        for (int c = 0; c < Dk; c++) { sq += qh[c] * dqh[c]; sk += kh[c] * dkh[c]; }
                        for (int c = 0; c < Dk; c++) {
                            dqo[c] += RQ[j] * (dqh[c] - qh[c] * sq);
                            dko[c] += RK[j] * (dkh[c] - kh[c] * sk);
                        }
                    } else {
                        for (int c = 0; c < Dk; c++) { dqo[c] += dqh[c]; dko[c] += dkh[c]; }
                    }
                }
            }
            if (dh0) memcpy(dh0 + st_off(&d, b, hv), G, sizeof(double) * SS);
        }
        free(ckpt); free(Sseg); free(KH); free(QH); free(RK); free(RQ); free(AA); free(PP);
        free(DL); free(G); free(Gd); free(tmp_o); free(dqh); free(dkh); free(dd); free(dp); free(da);
    }
    return 0;
}
