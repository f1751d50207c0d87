"""Chunked forward and VJP for head sizes 32 and 64 (bf16), against the fp64 oracle.

The tensor-core kernels work on 128 key and value channels; a call with Dk or Dv below 128
stages zero-padded 128-wide copies of its inputs in the workspace and crops the results, so
these cases check the staging (layouts, strides, the per-channel gate's Dk axis, the state's
Dv x Dk shape) as well as the chunked path on them.
"""
import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.autograd import gated_delta_rule
from gated_delta_rule_31_gb300.synth import Shape, make_inputs
from tests.util import BF16_TOL, cuda_device, rel_err, to_dev

pytestmark = pytest.mark.gpu
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
CASES = [(32, 32, "scalar"), (64, 64, "channel"), (64, 128, "scalar"), (128, 32, "channel"), (32, 64, "scalar"),
         (64, 64, "scalar")]


@pytest.mark.parametrize("dk,dv,gate", CASES, ids=[f"Dk{a}Dv{b}-{c}" for a, b, c in CASES])
def test_narrow_chunked_forward_and_vjp(dk, dv, gate):
    dev = cuda_device()
    x = make_inputs(Shape(2, 150, 2, 4, dk, dv), dtype=torch.bfloat16, seed=dk + 3 * dv, gate=gate, grads=True,
                    gate_scale=0.2)
    d = to_dev(x, dev)
    o, ht = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert tuple(o.shape) == (2, 150, 4, dv) and tuple(ht.shape) == (2, 4, dv, dk)
    assert rel_err(o, ro) <= BF16_TOL and rel_err(ht, rht) <= BF16_TOL
    gr = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"])
    errs = {n: rel_err(gr[n], ref[n]) for n in NAMES}
    assert all(e <= BF16_TOL for e in errs.values()), errs
    # the saved-state handoff in the padded layout
    o2, h2, states = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_states=True)
    assert torch.equal(o, o2) and torch.equal(ht, h2)
    gs = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], states=states)
    for n in NAMES:
        assert torch.equal(gs[n], gr[n]), n


def test_narrow_layer_uses_the_chunked_path():
    """The autograd function takes bf16 heads of 64 through the chunked kernels (the saved-state
    handoff), with gradients matching the oracle."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 130, 1, 2, 64, 64), dtype=torch.bfloat16, seed=64, grads=True, gate_scale=0.3)
    d = to_dev(x, dev)
    leaves = {n: d[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "beta", "h0")}
    o, ht = gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"], leaves["h0"])
    torch.autograd.backward([o, ht], [d["do"], d["dht"]])
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"])
    for n, leaf in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), ("q", "k", "v", "g", "beta", "h0")):
        assert rel_err(leaves[leaf].grad.float(), ref[n]) <= BF16_TOL, n
