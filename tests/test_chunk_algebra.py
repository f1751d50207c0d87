"""The chunk algebra the CUDA kernels implement (tests/chunk_algebra.py, numpy fp64)
equals the sequential oracle to rounding, forward and backward, including ragged last
chunks, GQA sharing, no-norm, zero initial state and several chunk lengths."""
import numpy as np
import pytest

import oracle
from tests import chunk_algebra as ca
from tests.test_oracle_pins import rand_inputs


@pytest.mark.parametrize("C,T,Hk,Hv,norm,h0", [(4, 11, 1, 2, True, True), (8, 16, 2, 4, True, False),
                                              (64, 70, 1, 1, True, True), (5, 5, 1, 2, False, True),
                                              (16, 3, 1, 1, True, True)])
def test_chunk_forward_and_backward_equal_oracle(C, T, Hk, Hv, norm, h0):
    q, k, v, g, beta, hh = rand_inputs(B=2, T=T, Hk=Hk, Hv=Hv, Dk=6, Dv=5, seed=C + T, h0=h0)
    r = np.random.default_rng(7)
    do = r.standard_normal(v.shape)
    dht = r.standard_normal((2, Hv, 5, 6))
    scale = 0.7
    o, ht = oracle.forward(q, k, v, g, beta, hh, scale=scale, use_qk_l2norm=norm)
    o2, ht2, _ = ca.forward(q, k, v, g, beta, hh, scale, norm, C)
    assert np.max(np.abs(o - o2)) < 1e-11 and np.max(np.abs(ht - ht2)) < 1e-11
    ref = oracle.backward(q, k, v, g, beta, hh, do, dht, scale=scale, use_qk_l2norm=norm)
    got = ca.backward(q, k, v, g, beta, hh, do, dht, scale, norm, C)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        err = np.max(np.abs(ref[name] - got[name])) / max(1.0, np.max(np.abs(ref[name])))
        assert err < 1e-10, (name, err)


@pytest.mark.parametrize("C,T,Hk,Hv,norm,h0,gs", [(4, 11, 1, 2, True, True, 1.0), (8, 16, 2, 4, True, False, 1.0),
                                                  (5, 5, 1, 2, False, True, 1.0), (16, 21, 1, 1, True, True, 8.0),
                                              (64, 150, 1, 2, True, True, 8.0)])
def test_channel_chunk_forward_equals_oracle(C, T, Hk, Hv, norm, h0, gs):
    """The per-channel chunk algebra (decays as products of per-token factors, diag(Gamma_C)
    in the state update) equals the sequential oracle; gs = 8 makes per-token factors as small
    as e^-40, where a factorised form exp(gamma_r) exp(-gamma_j) would overflow."""
    q, k, v, g, beta, hh = rand_inputs(B=2, T=T, Hk=Hk, Hv=Hv, Dk=6, Dv=5, channel=True, seed=3 * C + T, h0=h0,
                                       gate_scale=gs)
    o, ht = oracle.forward(q, k, v, g, beta, hh, scale=0.7, use_qk_l2norm=norm)
    o2, ht2 = ca.forward_channel(q, k, v, g, beta, hh, 0.7, norm, C)
    assert np.max(np.abs(o - o2)) < 1e-11 * max(1.0, np.max(np.abs(o)))
    assert np.max(np.abs(ht - ht2)) < 1e-11 * max(1.0, np.max(np.abs(ht)))


@pytest.mark.parametrize("C,bs,T,Hk,Hv,norm,h0,gs", [(8, 2, 19, 1, 2, True, True, 1.0), (16, 4, 16, 2, 4, True, False, 1.0),
                                                     (8, 4, 5, 1, 1, False, True, 1.0), (16, 4, 37, 1, 2, True, True, 8.0),
                                                     (64, 16, 150, 1, 2, True, True, 8.0),   # the kernels' blocking
                                                     (64, 16, 64, 2, 4, True, False, 0.3)])
def test_channel_chunk_backward_equals_oracle(C, bs, T, Hk, Hv, norm, h0, gs):
    """The per-channel VJP as the chunked kernels organise it (dense products; the decay-weighted
    contractions by blocks, factored through the block boundaries below the block diagonal;
    dgamma per channel) equals the oracle's hand-derived reverse mode; gs = 8 takes per-token
    factors down to e^-40."""
    q, k, v, g, beta, hh = rand_inputs(B=2, T=T, Hk=Hk, Hv=Hv, Dk=6, Dv=5, channel=True, seed=5 * C + T, h0=h0,
                                       gate_scale=gs)
    r = np.random.default_rng(11)
    do = r.standard_normal(v.shape)
    dht = r.standard_normal((2, Hv, 5, 6))
    ref = oracle.backward(q, k, v, g, beta, hh, do, dht, scale=0.7, use_qk_l2norm=norm)
    got = ca.backward_channel(q, k, v, g, beta, hh, do, dht, 0.7, norm, C, bs)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        err = np.max(np.abs(ref[name] - got[name])) / max(1.0, np.max(np.abs(ref[name])))
        assert err < 1e-10, (name, err)


@pytest.mark.parametrize("channel", [False, True])
def test_degenerate_tokens_forward_and_backward_equal_oracle(channel):
    """Tokens with beta = 0 (no write), g = 0 (no decay), beta = 1 (full replacement), and zero
    key or query vectors under the in-kernel norm (k^ = 0 writes nothing, q^ = 0 reads nothing,
    and the norm backward scales by 1/sqrt(eps) = 1000) inside a sequence of several chunks: the
    chunk algebra as the kernels organise it still equals the oracle."""
    q, k, v, g, beta, hh = rand_inputs(B=1, T=40, Hk=1, Hv=2, Dk=6, Dv=5, channel=channel, seed=21)
    beta[0, 3:6] = 0.0
    beta[0, 20] = 1.0
    g[0, 8:12] = 0.0
    g[0, 30:] = 0.0
    k[0, 7] = 0.0
    k[0, 17] = 0.0
    q[0, 9] = 0.0
    q[0, 33] = 0.0
    r = np.random.default_rng(22)
    do = r.standard_normal(v.shape)
    dht = r.standard_normal((1, 2, 5, 6))
    o, ht = oracle.forward(q, k, v, g, beta, hh, scale=0.7, use_qk_l2norm=True)
    assert np.all(o[0, 9] == 0.0) and np.all(o[0, 33] == 0.0)
    if channel:
        o2, ht2 = ca.forward_channel(q, k, v, g, beta, hh, 0.7, True, 16)
        got = ca.backward_channel(q, k, v, g, beta, hh, do, dht, 0.7, True, 16, 4)
    else:
        o2, ht2, _ = ca.forward(q, k, v, g, beta, hh, 0.7, True, 16)
        got = ca.backward(q, k, v, g, beta, hh, do, dht, 0.7, True, 16)
    assert np.max(np.abs(o - o2)) < 1e-11 and np.max(np.abs(ht - ht2)) < 1e-11
    ref = oracle.backward(q, k, v, g, beta, hh, do, dht, scale=0.7, use_qk_l2norm=True)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        err = np.max(np.abs(ref[name] - got[name])) / max(1.0, np.max(np.abs(ref[name])))
        assert err < 1e-10, (name, err)
    # a zero key still receives a gradient, scaled by 1/sqrt(eps) through the norm backward
    assert np.max(np.abs(ref["dk"][0, 7])) > 10 * np.max(np.abs(ref["dk"][0, [6, 8]]))
