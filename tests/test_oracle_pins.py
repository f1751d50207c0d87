"""Pins of the fp64 oracle against facts the gated delta rule itself fixes.

None of these compares the oracle with itself: each check is a closed form, a brute
force of the recurrence in its product form, an invariant of the mathematics, or
finite differences. A plausible slip in the oracle (a dropped term, a wrong sign, a
transposed state, decay applied after the prediction, a wrong head map, the wrong
eps) fails at least one of them.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def rand_inputs(B=1, T=6, Hk=1, Hv=2, Dk=4, Dv=3, channel=False, h0=True, seed=0, gate_scale=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, Hk, Dk))
    k = r.standard_normal((B, T, Hk, Dk))
    v = r.standard_normal((B, T, Hv, Dv))
    gs = (B, T, Hv, Dk) if channel else (B, T, Hv)
    g = -np.log1p(np.exp(r.standard_normal(gs))) * gate_scale
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, Hv))))
    hh = r.standard_normal((B, Hv, Dv, Dk)) * 0.5 if h0 else None
    return q, k, v, g, beta, hh


def product_form(q, k, v, g, beta, h0, scale, norm):
    """The recurrence exactly as printed in product form,
    S_t = S_{t-1} diag(a_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = scale S_t q_t,
    evaluated with dense matrix products (a different order from the oracle's)."""
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2:]
    o = np.zeros((B, T, Hv, Dv))
    ht = np.zeros((B, Hv, Dv, Dk))
    for b in range(B):
        for hv in range(Hv):
            hk = (hv * Hk) // Hv  # value heads hk*G .. hk*G+G-1 share key head hk
            S = np.zeros((Dv, Dk)) if h0 is None else h0[b, hv].copy()
            for t in range(T):
                kk, qq = k[b, t, hk], q[b, t, hk]
                if norm:
                    kk = kk / np.linalg.norm(np.append(kk, 1e-3))  # sqrt(|k|^2 + 1e-6)
                    qq = qq / np.linalg.norm(np.append(qq, 1e-3))
                a = np.exp(g[b, t, hv]) * np.ones(Dk)
                Dg = np.diag(a)
                I = np.eye(Dk)
                S = S @ Dg @ (I - beta[b, t, hv] * np.outer(kk, kk)) + beta[b, t, hv] * np.outer(v[b, t, hv], kk)
                o[b, t, hv] = scale * S @ qq
            ht[b, hv] = S
    return o, ht


@pytest.mark.parametrize("channel", [False, True])
@pytest.mark.parametrize("norm", [False, True])
def test_matches_product_form(channel, norm):
    q, k, v, g, beta, h0 = rand_inputs(B=2, T=9, Hk=2, Hv=4, Dk=5, Dv=3, channel=channel, seed=1)
    o, ht = oracle.forward(q, k, v, g, beta, h0, scale=0.37, use_qk_l2norm=norm)
    o2, ht2 = product_form(q, k, v, g, beta, h0, 0.37, norm)
    assert np.max(np.abs(o - o2)) <= 1e-12 * max(1, np.max(np.abs(o2)))
    assert np.max(np.abs(ht - ht2)) <= 1e-12 * max(1, np.max(np.abs(ht2)))


def test_pure_decay_closed_form():
    """beta = 0: nothing is written, so S_t = (prod_{s<=t} a_s) S_0 and
    o_t = scale (prod_{s<=t} a_s) S_0 q_t."""
    q, k, v, g, beta, h0 = rand_inputs(B=1, T=12, Hk=1, Hv=2, Dk=6, Dv=4, seed=2, gate_scale=0.1)
    beta[:] = 0.0
    o, ht = oracle.forward(q, k, v, g, beta, h0, scale=1.5, use_qk_l2norm=False)
    for hv in range(2):
        decay = np.exp(np.cumsum(g[0, :, hv]))
        want = 1.5 * decay[:, None] * (q[0, :, 0] @ h0[0, hv].T)
        assert np.allclose(o[0, :, hv], want, rtol=1e-13, atol=1e-14)
        assert np.allclose(ht[0, hv], decay[-1] * h0[0, hv], rtol=1e-13, atol=1e-14)


def test_pure_decay_channel_closed_form():
    """beta = 0 with a per-channel gate: column c of S decays by prod a_{s,c}."""
    q, k, v, g, beta, h0 = rand_inputs(B=1, T=10, Hk=1, Hv=1, Dk=5, Dv=3, channel=True, seed=3,
                                       gate_scale=0.1)
    beta[:] = 0.0
    o, ht = oracle.forward(q, k, v, g, beta, h0, scale=1.0, use_qk_l2norm=False)
    decay = np.exp(np.cumsum(g[0, :, 0], axis=0))  # [T, Dk]
    assert np.allclose(ht[0, 0], h0[0, 0] * decay[-1][None, :], rtol=1e-13)
    want = np.einsum("vc,tc,tc->tv", h0[0, 0], decay, q[0, :, 0])
    assert np.allclose(o[0, :, 0], want, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("with_h0", [False, True])
def test_orthonormal_keys_retrieve_values(with_h0):
    """a = 1, beta = 1, keys orthonormal: each write replaces the memory along its
    key, so S_T k_i = v_i exactly; querying with q_t = k_t reads o_t = scale v_t."""
    T, D, Dv = 6, 8, 5
    Qm, _ = np.linalg.qr(RNG.standard_normal((D, D)))
    keys = Qm[:T]
    q = keys[None, :, None, :].copy()
    k = keys[None, :, None, :].copy()
    v = RNG.standard_normal((1, T, 1, Dv))
    g = np.zeros((1, T, 1))
    beta = np.ones((1, T, 1))
    h0 = RNG.standard_normal((1, 1, Dv, D)) if with_h0 else None
    o, ht = oracle.forward(q, k, v, g, beta, h0, scale=2.0, use_qk_l2norm=False)
    S = ht[0, 0]
    for i in range(T):
        assert np.allclose(S @ keys[i], v[0, i, 0], atol=1e-12)
        assert np.allclose(o[0, i, 0], 2.0 * v[0, i, 0], atol=1e-12)


def test_norm_eps_value():
    """With one channel, x^ = x / sqrt(x^2 + eps). At x = 1e-3 and eps = 1e-6 this is
    exactly 1/sqrt(2), so one write (beta = 1, v = 1, S_0 = 0) and a read with
    scale 1 give o = k^ q^ = 1/2. Any other eps gives a different value."""
    one = np.ones((1, 1, 1, 1))
    o, ht = oracle.forward(one * 1e-3, one * 1e-3, one, np.zeros((1, 1, 1)), np.ones((1, 1, 1)),
                           None, scale=1.0, use_qk_l2norm=True)
    assert abs(o[0, 0, 0, 0] - 0.5) < 1e-12
    assert abs(ht[0, 0, 0, 0] - 2 ** -0.5) < 1e-12


def test_in_kernel_norm_equals_caller_norm():
    """Normalising inside (flag on) equals normalising q and k before the call."""
    q, k, v, g, beta, h0 = rand_inputs(B=1, T=8, Hk=2, Hv=4, Dk=6, Dv=3, seed=5)

    def caller_norm(x):
        return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + 1e-6)

    o1, h1 = oracle.forward(q, k, v, g, beta, h0, use_qk_l2norm=True)
    o2, h2 = oracle.forward(caller_norm(q), caller_norm(k), v, g, beta, h0, use_qk_l2norm=False)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-13)
    assert np.allclose(h1, h2, rtol=1e-12, atol=1e-13)


def test_norm_scale_invariance_and_zero_vectors():
    q, k, v, g, beta, h0 = rand_inputs(B=1, T=8, Hk=1, Hv=2, Dk=6, Dv=3, seed=6)
    o1, h1 = oracle.forward(q, k, v, g, beta, h0, use_qk_l2norm=True)
    o2, h2 = oracle.forward(q * 3.7, k * 0.6, v, g, beta, h0, use_qk_l2norm=True)
    assert np.allclose(o1, o2, rtol=1e-6, atol=1e-8)
    q[0, 3] = 0.0
    k[0, 5] = 0.0
    o3, h3 = oracle.forward(q, k, v, g, beta, h0, use_qk_l2norm=True)
    assert np.all(np.isfinite(o3)) and np.all(np.isfinite(h3))
    assert np.all(o3[0, 3] == 0.0)  # a zero query reads nothing


def test_split_sequence_equals_whole():
    q, k, v, g, beta, h0 = rand_inputs(B=2, T=13, Hk=1, Hv=2, Dk=4, Dv=3, seed=7)
    o, ht = oracle.forward(q, k, v, g, beta, h0)
    oa, ha = oracle.forward(q[:, :5], k[:, :5], v[:, :5], g[:, :5], beta[:, :5], h0)
    ob, hb = oracle.forward(q[:, 5:], k[:, 5:], v[:, 5:], g[:, 5:], beta[:, 5:], ha)
    assert np.allclose(np.concatenate([oa, ob], axis=1), o, rtol=1e-13, atol=1e-14)
    assert np.allclose(hb, ht, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("channel", [False, True])
def test_decode_steps_equal_forward(channel):
    q, k, v, g, beta, h0 = rand_inputs(B=2, T=5, Hk=2, Hv=4, Dk=4, Dv=3, channel=channel, seed=8)
    o, ht = oracle.forward(q, k, v, g, beta, h0)
    st = h0
    for t in range(5):
        ot, st = oracle.decode_step(q[:, t], k[:, t], v[:, t], g[:, t], beta[:, t], st)
        assert np.allclose(ot, o[:, t], rtol=1e-13, atol=1e-14)
    assert np.allclose(st, ht, rtol=1e-13, atol=1e-14)


def test_channel_gate_with_equal_channels_equals_scalar_gate():
    q, k, v, g, beta, h0 = rand_inputs(B=1, T=9, Hk=1, Hv=2, Dk=5, Dv=3, seed=9)
    gc = np.repeat(g[..., None], 5, axis=-1)
    o1, h1 = oracle.forward(q, k, v, g, beta, h0)
    o2, h2 = oracle.forward(q, k, v, gc, beta, h0)
    assert np.allclose(o1, o2, rtol=1e-13) and np.allclose(h1, h2, rtol=1e-13)
    do = RNG.standard_normal(o1.shape)
    g1 = oracle.backward(q, k, v, g, beta, h0, do)
    g2 = oracle.backward(q, k, v, gc, beta, h0, do)
    assert np.allclose(g1["dg"], g2["dg"].sum(-1), rtol=1e-11, atol=1e-13)
    for name in ("dq", "dk", "dv", "dbeta", "dh0"):
        assert np.allclose(g1[name], g2[name], rtol=1e-11, atol=1e-13), name


def test_gqa_equals_repeated_heads():
    """Hk=2 key heads shared by Hv=6 value heads (group 3) equals Hk=Hv=6 with each key
    and query head repeated 3 times; the shared-head gradient is the group sum."""
    q, k, v, g, beta, h0 = rand_inputs(B=1, T=7, Hk=2, Hv=6, Dk=4, Dv=3, seed=10)
    qr, kr = np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2)
    o1, h1 = oracle.forward(q, k, v, g, beta, h0)
    o2, h2 = oracle.forward(qr, kr, v, g, beta, h0)
    assert np.allclose(o1, o2, rtol=1e-13) and np.allclose(h1, h2, rtol=1e-13)
    do = RNG.standard_normal(o1.shape)
    g1 = oracle.backward(q, k, v, g, beta, h0, do)
    g2 = oracle.backward(qr, kr, v, g, beta, h0, do)
    assert np.allclose(g1["dq"], g2["dq"].reshape(1, 7, 2, 3, 4).sum(3), rtol=1e-11, atol=1e-13)
    assert np.allclose(g1["dk"], g2["dk"].reshape(1, 7, 2, 3, 4).sum(3), rtol=1e-11, atol=1e-13)
    for name in ("dv", "dg", "dbeta", "dh0"):
        assert np.allclose(g1[name], g2[name], rtol=1e-11, atol=1e-13), name


def _loss(q, k, v, g, beta, h0, do, dht, norm, scale):
    o, ht = oracle.forward(q, k, v, g, beta, h0, scale=scale, use_qk_l2norm=norm)
    return float(np.sum(o * do) + np.sum(ht * dht))


@pytest.mark.parametrize("channel,norm,T", [(False, True, 6), (True, True, 5), (False, False, 6),
                                            (False, True, 70)])
def test_backward_matches_finite_differences(channel, norm, T):
    """Central differences in fp64 (h = 1e-6 max(1,|x|)) of L = <do,o> + <dht,ht> agree
    with every gradient to 1e-6 relative. T=70 crosses the oracle's 64-step
    checkpoint segment."""
    Dk = 3 if T > 10 else 4
    q, k, v, g, beta, h0 = rand_inputs(B=1, T=T, Hk=1, Hv=2, Dk=Dk, Dv=3, channel=channel, seed=11)
    r = np.random.default_rng(12)
    do = r.standard_normal((1, T, 2, 3))
    dht = r.standard_normal((1, 2, 3, Dk))
    scale = 0.8
    grads = oracle.backward(q, k, v, g, beta, h0, do, dht, scale=scale, use_qk_l2norm=norm)
    inputs = dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    stride = 7 if T > 10 else 1
    for name, x in inputs.items():
        an = grads[names[name]]
        flat = x.reshape(-1)
        idx = range(0, flat.size, stride)
        fd = []
        for i in idx:
            h = 1e-6 * max(1.0, abs(flat[i]))
            old = flat[i]
            flat[i] = old + h
            lp = _loss(**inputs, do=do, dht=dht, norm=norm, scale=scale)
            flat[i] = old - h
            lm = _loss(**inputs, do=do, dht=dht, norm=norm, scale=scale)
            flat[i] = old
            fd.append((lp - lm) / (2 * h))
        fd = np.array(fd)
        ref = an.reshape(-1)[list(idx)]
        err = np.max(np.abs(fd - ref)) / max(1.0, np.max(np.abs(ref)))
        assert err < 1e-6, (name, err)


def test_euler_identity_and_norm_orthogonality():
    """o and ht are jointly linear in (v, h0), so L = sum v dv + sum h0 dh0 exactly; with
    the in-kernel norm, L does not change when one q_t or k_t is scaled, so
    q_t . dq_t = k_t . dk_t = 0 (up to the eps term)."""
    q, k, v, g, beta, h0 = rand_inputs(B=2, T=11, Hk=1, Hv=3, Dk=5, Dv=4, seed=13)
    q, k = q * 4.0, k * 4.0  # |x|^2 ~ 80 so eps / |x|^2 ~ 1e-8
    r = np.random.default_rng(14)
    do = r.standard_normal(v.shape)
    dht = r.standard_normal((2, 3, 4, 5))
    L = _loss(q, k, v, g, beta, h0, do, dht, True, 0.5)
    gr = oracle.backward(q, k, v, g, beta, h0, do, dht, scale=0.5, use_qk_l2norm=True)
    euler = np.sum(v * gr["dv"]) + np.sum(h0 * gr["dh0"])
    assert abs(euler - L) <= 1e-11 * max(1.0, abs(L))
    qd = np.einsum("bthd,bthd->bth", q, gr["dq"])
    kd = np.einsum("bthd,bthd->bth", k, gr["dk"])
    gscale = max(np.max(np.abs(gr["dq"])), np.max(np.abs(gr["dk"])))
    assert np.max(np.abs(qd)) < 1e-6 * gscale and np.max(np.abs(kd)) < 1e-6 * gscale


def test_empty_sequence():
    q, k, v, g, beta, h0 = rand_inputs(B=1, T=0, Hk=1, Hv=2, Dk=4, Dv=3, seed=15)
    o, ht = oracle.forward(q, k, v, g, beta, h0)
    assert o.shape == (1, 0, 2, 3)
    assert np.array_equal(ht, h0)
    gr = oracle.backward(q, k, v, g, beta, h0, np.zeros((1, 0, 2, 3)), np.ones((1, 2, 3, 4)))
    assert np.array_equal(gr["dh0"], np.ones((1, 2, 3, 4)))
