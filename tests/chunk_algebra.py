"""The chunked form of the gated delta rule in plain numpy fp64, written the way the CUDA
kernels organise it (same per-chunk operators, same folding of the L2-norm factors and
decays into raw q/k operands). It is not the oracle and does not feed any stored value:
tests check it against the oracle (sequential recurrence) to ~1e-12, which pins the
chunk algebra the kernels implement, forward and backward, independently of CUDA.

Per chunk (rows r = tokens, chunk length C), with K, Q raw keys/queries, rk/rq their
norm factors, gamma the in-chunk cumulative log-decay, Gamma = exp(gamma),
b = exp(gamma_C - gamma), E_rj = exp(gamma_r - gamma_j):
    A   = strict_lower(beta_r rk_r rk_j E_rj (K K^T)_rj),  T = (I + A)^-1
    W   = T diag(beta Gamma rk) K,    U~ = T diag(beta) V
    P   = scale * tril(rq_r rk_j E_rj (Q K^T)_rj)
    Kbar = diag(b rk) K,  Mneg = -Kbar^T W,  Qc = scale diag(Gamma rq) Q - P W
    H1 = Gamma_C H0 + Mneg H0 + Kbar^T U~,   O = Qc H0 + P U~
Backward scan: dH0 = Gamma_C dH1 + Mneg^T dH1 + Qc^T dO.
"""
import numpy as np


def _norm_factor(x, on):
    if not on:
        return np.ones(x.shape[:-1])
    return 1.0 / np.sqrt(np.sum(x * x, axis=-1) + 1e-6)


def chunk_ops(K, Q, V, g, beta, scale, rk, rq):
    C = K.shape[0]
    gam = np.cumsum(g)
    Gam = np.exp(gam)
    b = np.exp(gam[-1] - gam)
    diff = gam[:, None] - gam[None, :]
    low = np.tril(np.ones((C, C)), -1)
    lowi = np.tril(np.ones((C, C)))
    E = np.where(lowi > 0, np.exp(np.where(lowi > 0, diff, 0.0)), 0.0)
    A = low * (beta * rk)[:, None] * rk[None, :] * E * (K @ K.T)
    T = np.linalg.inv(np.eye(C) + A)
    W = T @ ((beta * Gam * rk)[:, None] * K)
    Ut = T @ (beta[:, None] * V)
    P = scale * lowi * rq[:, None] * rk[None, :] * E * (Q @ K.T)
    Kbar = (b * rk)[:, None] * K
    Mneg = -Kbar.T @ W
    Qc = scale * (Gam * rq)[:, None] * Q - P @ W
    return dict(gam=gam, Gam=Gam, b=b, E=E, A=A, T=T, W=W, Ut=Ut, P=P, Kbar=Kbar, Mneg=Mneg, Qc=Qc)


def _chunks(T, C):
    return [(s, min(s + C, T)) for s in range(0, T, C)]


def _pad(x, n):
    if x.shape[0] == n:
        return x
    out = np.zeros((n,) + x.shape[1:])
    out[: x.shape[0]] = x
    return out


def forward(q, k, v, g, beta, h0, scale, norm=True, C=64):
    """Scalar gate. Shapes as the oracle; returns o, ht and the per-chunk start states."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2:]
    grp = Hv // Hk
    o = np.zeros((B, T, Hv, Dv))
    ht = np.zeros((B, Hv, Dv, Dk))
    states = {}
    for b_ in range(B):
        for hv in range(Hv):
            hk = hv // grp
            H = np.zeros((Dk, Dv)) if h0 is None else h0[b_, hv].T.copy()
            for ci, (s, e) in enumerate(_chunks(T, C)):
                K = _pad(k[b_, s:e, hk], C)
                Q = _pad(q[b_, s:e, hk], C)
                V = _pad(v[b_, s:e, hv], C)
                gg = _pad(g[b_, s:e, hv], C)
                bb = _pad(beta[b_, s:e, hv], C)
                ops = chunk_ops(K, Q, V, gg, bb, scale, _norm_factor(K, norm), _norm_factor(Q, norm))
                states[(b_, hv, ci)] = H.copy()
                O = ops["Qc"] @ H + ops["P"] @ ops["Ut"]
                H = np.exp(ops["gam"][-1]) * H + ops["Mneg"] @ H + ops["Kbar"].T @ ops["Ut"]
                o[b_, s:e, hv] = O[: e - s]
            ht[b_, hv] = H.T
    return o, ht, states


def backward(q, k, v, g, beta, h0, do, dht, scale, norm=True, C=64):
    """Gradients of <do, o> + <dht, ht> by chunks: recompute the chunk-start states, run the
    reverse scan for the chunk-end state gradients, then chunk-local gradients."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2:]
    grp = Hv // Hk
    _, _, states = forward(q, k, v, g, beta, h0, scale, norm, C)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dg = np.zeros_like(g)
    dbeta = np.zeros_like(beta)
    dh0 = np.zeros((B, Hv, Dv, Dk))
    chunks = _chunks(T, C)
    for b_ in range(B):
        for hk in range(Hk):
            dQh = {ci: np.zeros((C, Dk)) for ci in range(len(chunks))}
            dKh = {ci: np.zeros((C, Dk)) for ci in range(len(chunks))}
            for hv in range(hk * grp, (hk + 1) * grp):
                dH = np.zeros((Dk, Dv)) if dht is None else dht[b_, hv].T.copy()
                for ci in reversed(range(len(chunks))):
                    s, e = chunks[ci]
                    K = _pad(k[b_, s:e, hk], C)
                    Q = _pad(q[b_, s:e, hk], C)
                    V = _pad(v[b_, s:e, hv], C)
                    gg = _pad(g[b_, s:e, hv], C)
                    bb = _pad(beta[b_, s:e, hv], C)
                    dO = _pad(do[b_, s:e, hv], C)
                    rk, rq = _norm_factor(K, norm), _norm_factor(Q, norm)
                    ops = chunk_ops(K, Q, V, gg, bb, scale, rk, rq)
                    H0 = states[(b_, hv, ci)]
                    dH1 = dH
                    g_, Gam, bv, E, A, Tm, W, Ut, P = (ops[n] for n in ("gam", "Gam", "b", "E", "A", "T", "W", "Ut", "P"))
                    Kh, Qh = rk[:, None] * K, rq[:, None] * Q
                    U = Ut - W @ H0
                    dU = P.T @ dO + (bv * rk)[:, None] * (K @ dH1)
                    dP = np.tril(dO @ U.T)
                    dgam = np.zeros(C)
                    # O = scale diag(Gamma) Q^ H0 + P U
                    X = dO @ H0.T
                    dQ = scale * Gam[:, None] * X
                    dgam += scale * Gam * np.sum(Qh * X, axis=1)
                    dS = scale * E * dP
                    dQ += dS @ Kh
                    dK = dS.T @ Qh
                    Z = dP * P
                    dgam += Z.sum(1) - Z.sum(0)
                    # H1 = Gamma_C H0 + K^^T diag(b) U
                    Y = U @ dH1.T
                    dK += bv[:, None] * Y
                    db = np.sum(Kh * Y, axis=1)
                    dgam -= bv * db
                    dgam[-1] += np.sum(bv * db) + np.exp(g_[-1]) * np.sum(dH1 * H0)
                    # U = U~ - W H0, U~ = T diag(beta) V, W = T diag(beta Gamma) K^
                    dW = -dU @ H0.T
                    dT = dU @ (bb[:, None] * V).T + dW @ ((bb * Gam)[:, None] * Kh).T
                    TdU = Tm.T @ dU
                    TdW = Tm.T @ dW
                    dV = bb[:, None] * TdU
                    dbt = np.sum(V * TdU, axis=1) + Gam * np.sum(Kh * TdW, axis=1)
                    dK += (bb * Gam)[:, None] * TdW
                    dgam += bb * Gam * np.sum(Kh * TdW, axis=1)
                    # T = (I + A)^-1, A = strict_lower(beta_r E k^_r . k^_j)
                    dA = np.tril(-Tm.T @ dT @ Tm.T, -1)
                    M = dA * bb[:, None] * E
                    dbt += np.sum(dA * E * (Kh @ Kh.T), axis=1)
                    Z = dA * A
                    dgam += Z.sum(1) - Z.sum(0)
                    dK += M @ Kh + M.T @ Kh
                    # gamma = cumsum(g) within the chunk
                    dgg = np.cumsum(dgam[::-1])[::-1]
                    n = e - s
                    dv[b_, s:e, hv] = dV[:n]
                    dbeta[b_, s:e, hv] = dbt[:n]
                    dg[b_, s:e, hv] = dgg[:n]
                    dQh[ci] += dQ
                    dKh[ci] += dK
                    dH = np.exp(g_[-1]) * dH1 + ops["Mneg"].T @ dH1 + ops["Qc"].T @ dO
                dh0[b_, hv] = dH.T
            for ci, (s, e) in enumerate(chunks):
                n = e - s
                for name, X, Dst, raw in (("q", dQh[ci], dq, q), ("k", dKh[ci], dk, k)):
                    x = raw[b_, s:e, hk]
                    r = _norm_factor(x, norm)
                    xh = r[:, None] * x
                    Xn = X[:n]
                    if norm:
                        Dst[b_, s:e, hk] = r[:, None] * (Xn - xh * np.sum(xh * Xn, axis=1, keepdims=True))
                    else:
                        Dst[b_, s:e, hk] = Xn
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dh0=dh0)


def chunk_ops_channel(K, Q, V, g, beta, scale, rk, rq):
    """Per-channel gate g [C, Dk], written as the per-channel kernel forms it: every decay is a
    product of per-token factors a_t = exp(g_t) <= 1 (E_rj = prod_{j<t<=r} a_t per channel,
    Gamma_r = prod_{t<=r} a_t, Kbar's factor prod_{t>r} a_t), never an exp of a difference."""
    C, Dk = K.shape
    a = np.exp(g)
    Gam = np.cumprod(a, axis=0)                                   # [C, Dk]
    suf = np.ones_like(a)                                         # prod_{t>r} a_t
    for r in range(C - 2, -1, -1):
        suf[r] = suf[r + 1] * a[r + 1]
    E = np.zeros((C, C, Dk))                                      # E[r, j, :] for j <= r
    for j in range(C):
        e = np.ones(Dk)
        for r in range(j, C):
            if r > j:
                e = e * a[r]
            E[r, j] = e
    Kh, Qh = rk[:, None] * K, rq[:, None] * Q
    A = np.zeros((C, C))
    P = np.zeros((C, C))
    for r in range(C):
        for j in range(r + 1):
            if j < r:
                A[r, j] = beta[r] * np.sum(Kh[r] * Kh[j] * E[r, j])
            P[r, j] = scale * np.sum(Qh[r] * Kh[j] * E[r, j])
    T = np.linalg.inv(np.eye(C) + A)
    W = T @ (beta[:, None] * (Kh * Gam))
    Ut = T @ (beta[:, None] * V)
    Kbar = Kh * suf
    Mneg = -Kbar.T @ W
    Qc = scale * Qh * Gam - P @ W
    return dict(GamC=Gam[-1], W=W, Ut=Ut, P=P, Kbar=Kbar, Mneg=Mneg, Qc=Qc, T=T, a=a, Gam=Gam, suf=suf)


def forward_channel(q, k, v, g, beta, h0, scale, norm=True, C=64, states=None):
    """Per-channel gate: o, ht with H1 = diag(Gamma_C) H0 + Mneg H0 + Kbar^T U~ per chunk
    (chunk-start states into `states[(b, hv, chunk)]` when a dict is given)."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2:]
    grp = Hv // Hk
    o = np.zeros((B, T, Hv, Dv))
    ht = np.zeros((B, Hv, Dv, Dk))
    for b_ in range(B):
        for hv in range(Hv):
            hk = hv // grp
            H = np.zeros((Dk, Dv)) if h0 is None else h0[b_, hv].T.copy()
            for s, e in _chunks(T, C):
                K = _pad(k[b_, s:e, hk], C)
                Q = _pad(q[b_, s:e, hk], C)
                ops = chunk_ops_channel(K, Q, _pad(v[b_, s:e, hv], C), _pad(g[b_, s:e, hv], C),
                                        _pad(beta[b_, s:e, hv], C), scale, _norm_factor(K, norm), _norm_factor(Q, norm))
                if states is not None:
                    states[(b_, hv, s // C)] = H.copy()
                O = ops["Qc"] @ H + ops["P"] @ ops["Ut"]
                H = ops["GamC"][:, None] * H + ops["Mneg"] @ H + ops["Kbar"].T @ ops["Ut"]
                o[b_, s:e, hv] = O[: e - s]
            ht[b_, hv] = H.T
    return o, ht


def _blocked_contractions(dPs, dA, Kh, Qh, beta, a, bs):
    """The four decay-weighted contractions of the per-channel VJP, organised as the kernel
    does: by bs-row blocks, the parts below the block diagonal as products of operands scaled
    by products of per-token factors (the decay factored through the block boundary), the
    diagonal blocks with running products. Returns X1, Y1 (row side) and X2 (column side):
        X1[r] = sum_{j<=r} dPs_rj k^_j E_rj,   Y1[r] = sum_{j<r} dA_rj k^_j E_rj
        X2[j] = sum_{i>=j} dPs_ij q^_i E_ij + sum_{i>j} dA_ij beta_i k^_i E_ij"""
    C, Dk = Kh.shape
    X1, Y1, X2 = np.zeros((C, Dk)), np.zeros((C, Dk)), np.zeros((C, Dk))
    nb = C // bs
    for I in range(nb):
        rows = range(bs * I, bs * I + bs)
        # row side, j in earlier blocks: E_rj = [prod_{bs I<=t<=r} a_t] [prod_{j<t<bs I} a_t]
        if I > 0:
            R = np.zeros((bs * I, Dk))
            sfx = np.ones(Dk)
            for j in range(bs * I - 1, -1, -1):
                R[j] = Kh[j] * sfx
                sfx = sfx * a[j]
            DX = dPs[bs * I:bs * I + bs, :bs * I] @ R
            DY = dA[bs * I:bs * I + bs, :bs * I] @ R
            c = np.ones(Dk)
            for i, r in enumerate(rows):
                c = c * a[r]
                X1[r] += c * DX[i]
                Y1[r] += c * DY[i]
        # row side inside the diagonal block: running decay
        for r in rows:
            e = np.ones(Dk)
            for j in range(r, bs * I - 1, -1):
                if j < r:
                    e = e * a[j + 1]
                X1[r] += dPs[r, j] * Kh[j] * e
                Y1[r] += dA[r, j] * Kh[j] * e
        # column side, i in later blocks: E_ij = [prod_{j<t<=bs I+bs-1} a_t] [prod_{bs I+bs<=t<=i} a_t]
        if I < nb - 1:
            i0 = bs * I + bs
            Qs = np.zeros((C - i0, Dk))
            Ks = np.zeros((C - i0, Dk))
            pr = np.ones(Dk)
            for i in range(i0, C):
                pr = pr * a[i]
                Qs[i - i0] = Qh[i] * pr
                Ks[i - i0] = beta[i] * Kh[i] * pr
            DC = dPs[i0:, bs * I:bs * I + bs].T @ Qs + dA[i0:, bs * I:bs * I + bs].T @ Ks
            f = np.ones(Dk)
            for jj in range(bs - 1, -1, -1):
                j = bs * I + jj
                X2[j] += f * DC[jj]
                f = f * a[j]
        # column side inside the diagonal block
        for j in rows:
            e = np.ones(Dk)
            for i in range(j, bs * I + bs):
                if i > j:
                    e = e * a[i]
                X2[j] += (dPs[i, j] * Qh[i] + dA[i, j] * beta[i] * Kh[i]) * e
    return X1, Y1, X2


def backward_channel(q, k, v, g, beta, h0, do, dht, scale, norm=True, C=64, bs=16):
    """Per-channel gate VJP of <do, o> + <dht, ht> as the chunked kernels organise it: the
    forward states, the reverse scan dH0 = diag(Gamma_C) dH1 + Mneg^T dH1 + Qc^T dO, the dense
    products X = dO H0^T, Y = U dH1^T, Z = T^T dW, dP, dT, dA, and the decay-weighted
    contractions by bs-row blocks (_blocked_contractions); dgamma per key channel, dg its
    in-chunk reverse cumulative sum plus the Gamma_C terms on every token."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2:]
    grp = Hv // Hk
    states = {}
    forward_channel(q, k, v, g, beta, h0, scale, norm, C, states=states)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dg, dbeta = np.zeros_like(g), np.zeros_like(beta)
    dh0 = np.zeros((B, Hv, Dv, Dk))
    chunks = _chunks(T, C)
    for b_ in range(B):
        for hk in range(Hk):
            dQh = {ci: np.zeros((C, Dk)) for ci in range(len(chunks))}
            dKh = {ci: np.zeros((C, Dk)) for ci in range(len(chunks))}
            for hv in range(hk * grp, (hk + 1) * grp):
                dH = np.zeros((Dk, Dv)) if dht is None else dht[b_, hv].T.copy()
                for ci in reversed(range(len(chunks))):
                    s, e = chunks[ci]
                    K, Q = _pad(k[b_, s:e, hk], C), _pad(q[b_, s:e, hk], C)
                    V, gg = _pad(v[b_, s:e, hv], C), _pad(g[b_, s:e, hv], C)
                    bb, dO = _pad(beta[b_, s:e, hv], C), _pad(do[b_, s:e, hv], C)
                    rk, rq = _norm_factor(K, norm), _norm_factor(Q, norm)
                    ops = chunk_ops_channel(K, Q, V, gg, bb, scale, rk, rq)
                    Kh, Qh = rk[:, None] * K, rq[:, None] * Q
                    H0, dH1 = states[(b_, hv, ci)], dH
                    Tm, W, Ut, P, Kbar = ops["T"], ops["W"], ops["Ut"], ops["P"], ops["Kbar"]
                    a, Gam, bdec, GamC = ops["a"], ops["Gam"], ops["suf"], ops["GamC"]
                    U = Ut - W @ H0
                    dU = P.T @ dO + Kbar @ dH1
                    dPs = scale * np.tril(dO @ U.T)
                    X, Y = dO @ H0.T, U @ dH1.T
                    dW = -dU @ H0.T
                    Z = Tm.T @ dW
                    dT = dU @ (bb[:, None] * V).T + dW @ (bb[:, None] * Kh * Gam).T
                    TdU = Tm.T @ dU
                    dA = np.tril(-Tm.T @ dT @ Tm.T, -1)
                    X1, Y1, X2 = _blocked_contractions(dPs, dA, Kh, Qh, bb, a, bs)
                    dQ = scale * Gam * X + X1
                    dK = bdec * Y + bb[:, None] * Gam * Z + bb[:, None] * Y1 + X2
                    dgam = (scale * Gam * Qh * X - bdec * Kh * Y + bb[:, None] * Gam * Kh * Z
                            + Qh * X1 + bb[:, None] * Kh * Y1 - Kh * X2)
                    dgamC = np.sum(bdec * Kh * Y, axis=0) + GamC * np.sum(dH1 * H0, axis=1)
                    dgg = np.cumsum(dgam[::-1], axis=0)[::-1] + dgamC[None, :]
                    n = e - s
                    dv[b_, s:e, hv] = (bb[:, None] * TdU)[:n]
                    dbeta[b_, s:e, hv] = (np.sum(V * TdU, axis=1) + np.sum(Gam * Kh * Z, axis=1)
                                          + np.sum(Kh * Y1, axis=1))[:n]
                    dg[b_, s:e, hv] = dgg[:n]
                    dQh[ci] += dQ
                    dKh[ci] += dK
                    dH = GamC[:, None] * dH1 + ops["Mneg"].T @ dH1 + ops["Qc"].T @ dO
                dh0[b_, hv] = dH.T
            for ci, (s, e) in enumerate(chunks):
                n = e - s
                for X_, Dst, raw in ((dQh[ci], dq, q), (dKh[ci], dk, k)):
                    x = raw[b_, s:e, hk]
                    r = _norm_factor(x, norm)
                    xh = r[:, None] * x
                    Xn = X_[:n]
                    if norm:
                        Dst[b_, s:e, hk] = r[:, None] * (Xn - xh * np.sum(xh * Xn, axis=1, keepdims=True))
                    else:
                        Dst[b_, s:e, hk] = Xn
    return dict(dq=dq, dk=dk, dv=dv, dg=dg, dbeta=dbeta, dh0=dh0)
