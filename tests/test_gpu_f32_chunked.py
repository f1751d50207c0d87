"""The chunked forward and VJP for fp32 q/k/v (CUDA-core fp32 kernels of the chunk algebra)
against the fp64 oracle at the fp32 bound max|gpu - oracle| / max|oracle| <= 1e-4.

Cases: the tiny fp32 configuration (B=1, T=64, Hk=Hv=2, Dk=Dv=32, h0=0) through the chunked
calls, then several chunks with a ragged tail, shared key heads, both gates, every head size,
unequal Dk and Dv, no in-kernel norm, sequences shorter than one chunk and strong decays. The
saved-state and saved-operator handoffs must give the recompute path's gradients bit for bit.
"""
import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.synth import Shape, make_inputs
from tests.util import F32_TOL, cuda_device, rel_err, to_dev

pytestmark = pytest.mark.gpu
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def test_tiny_fp32_config_through_the_chunked_calls():
    dev = cuda_device()
    x = make_inputs(Shape(1, 64, 2, 2, 32, 32), dtype=torch.float32, seed=0, h0_std=None, grads=True,
                    dht_std=None)
    d = to_dev(x, dev)
    o, ht = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, scale=32 ** -0.5)
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], None, scale=32 ** -0.5)
    assert o.dtype == torch.float32 and tuple(o.shape) == (1, 64, 2, 32) and tuple(ht.shape) == (1, 2, 32, 32)
    assert rel_err(o, ro) <= F32_TOL and rel_err(ht, rht) <= F32_TOL
    gr = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], None, scale=32 ** -0.5)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["do"], None, scale=32 ** -0.5)
    errs = {n: rel_err(gr[n], ref[n]) for n in NAMES}
    assert all(e <= F32_TOL for e in errs.values()), errs


CASES = [  # B, T, Hk, Hv, Dk, Dv, gate, norm, h0, gate_scale
    (2, 150, 2, 4, 128, 128, "scalar", True, True, 1.0),
    (1, 200, 1, 2, 64, 32, "channel", True, True, 1.0),
    (2, 64, 2, 2, 32, 64, "channel", False, False, 0.3),
    (1, 129, 2, 4, 128, 64, "scalar", True, True, 8.0),
    (3, 5, 1, 1, 32, 32, "scalar", True, True, 1.0),
    (1, 300, 2, 2, 128, 128, "channel", True, True, 8.0),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}T{c[1]}H{c[2]}-{c[3]}D{c[4]}-{c[5]}-{c[6]}"
                                             f"{'' if c[7] else '-nonorm'}-gs{c[9]}" for c in CASES])
def test_fp32_chunked_forward_and_vjp(case):
    B, T, Hk, Hv, Dk, Dv, gate, norm, h0, gs = case
    dev = cuda_device()
    x = make_inputs(Shape(B, T, Hk, Hv, Dk, Dv), dtype=torch.float32, seed=T + Dk + Dv, gate=gate,
                    h0_std=0.02 if h0 else None, grads=True, gate_scale=gs)
    d = to_dev(x, dev)
    kw = dict(use_qk_l2norm=norm)
    o, ht = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], **kw)
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], use_qk_l2norm=norm)
    assert rel_err(o, ro) <= F32_TOL and rel_err(ht, rht) <= F32_TOL
    gr = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"], **kw)
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"],
                          use_qk_l2norm=norm)
    errs = {n: rel_err(gr[n], ref[n]) for n in NAMES}
    assert all(e <= F32_TOL for e in errs.values()), errs
    # the handoffs: chunk-start states, and records + states, kept by the forward
    o2, h2, states = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_states=True, **kw)
    assert torch.equal(o, o2) and torch.equal(ht, h2)
    gs_ = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], states=states, **kw)
    o3, h3, saved = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_all=True, **kw)
    assert torch.equal(o, o3) and torch.equal(ht, h3)
    gv = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], saved=saved, **kw)
    for n in NAMES:
        assert torch.equal(gs_[n], gr[n]) and torch.equal(gv[n], gr[n]), n


def test_fp32_chunked_is_deterministic_and_matches_sequential():
    """Two runs give the same bits; the chunked and token-by-token fp32 paths agree with each
    other at the fp32 bound (both against the oracle too) on 1024 tokens of 4 value heads."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 1024, 2, 4, 128, 128), dtype=torch.float32, seed=77, grads=True)
    d = to_dev(x, dev)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o, ht = gdr.fwd_chunked(*args)
    o_, ht_ = gdr.fwd_chunked(*args)
    assert torch.equal(o, o_) and torch.equal(ht, ht_)
    so, sht = gdr.fwd_sequential(*args)
    assert rel_err(o, so.cpu()) <= F32_TOL and rel_err(ht, sht.cpu()) <= F32_TOL
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert rel_err(o, ro) <= F32_TOL and rel_err(ht, rht) <= F32_TOL
    gr = gdr.bwd_chunked(*args, d["do"], d["dht"])
    gr2 = gdr.bwd_chunked(*args, d["do"], d["dht"])
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"])
    for n in NAMES:
        assert torch.equal(gr[n], gr2[n]), n
        assert rel_err(gr[n], ref[n]) <= F32_TOL, (n, rel_err(gr[n], ref[n]))
