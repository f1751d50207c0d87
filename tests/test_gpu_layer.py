"""Layer-level parity through torch.autograd (bf16, no model weights).

The validation of "fold q/k L2-norm into the gated_delta_rule kernel" (Megatron-LM PR #5396)
compares a caller-side L2 norm followed by the kernel without its norm against the kernel
that owns the norm, on outputs and on input gradients. Here both routes run through
``gated_delta_rule`` (the autograd.Function over the C ABI): the caller-side route normalises
q and k with torch (fp32 math, eps 1e-6, rounded to bf16 as a caller would store them) and
differentiates through that; the in-kernel route passes raw q and k. Bounds: both routes
within 2e-2 (max-abs / max|ref|) of each other and of the fp64 oracle.
"""
import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.autograd import gated_delta_rule
from gated_delta_rule_31_gb300.synth import Shape, make_inputs
from tests.util import BF16_TOL, cuda_device, rel_err

pytestmark = pytest.mark.gpu
INPUTS = ("q", "k", "v", "g", "beta", "h0")


def caller_l2norm(x):
    xf = x.float()
    return (xf * torch.rsqrt((xf * xf).sum(-1, keepdim=True) + 1e-6)).to(x.dtype)


def leaves(x, dev):
    return {n: x[n].to(dev).requires_grad_(True) for n in INPUTS}


def run_route(x, dev, in_kernel):
    t = leaves(x, dev)
    q, k = (t["q"], t["k"]) if in_kernel else (caller_l2norm(t["q"]), caller_l2norm(t["k"]))
    o, ht = gated_delta_rule(q, k, t["v"], t["g"], t["beta"], t["h0"], use_qk_l2norm=in_kernel)
    loss = (o.float() * x["do"].to(dev).float()).sum() + (ht * x["dht"].to(dev)).sum()
    loss.backward()
    grads = {"d" + n: t[n].grad for n in INPUTS}
    return o.detach(), ht.detach(), grads


@pytest.mark.parametrize("shape", [Shape(1, 200, 2, 4, 128, 128), Shape(2, 64, 1, 2, 128, 128)])
def test_in_kernel_norm_matches_caller_side_norm(shape):
    dev = cuda_device()
    x = make_inputs(shape, dtype=torch.bfloat16, seed=500 + shape.T, grads=True, gate_scale=0.1)
    o_in, ht_in, g_in = run_route(x, dev, in_kernel=True)
    o_cs, ht_cs, g_cs = run_route(x, dev, in_kernel=False)
    assert rel_err(o_in, o_cs) <= BF16_TOL and rel_err(ht_in, ht_cs) <= BF16_TOL
    errs = {n: rel_err(g_in[n], g_cs[n]) for n in g_in}
    assert all(e <= BF16_TOL for e in errs.values()), errs
    # and both against the oracle (norm inside, fp64)
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"])
    for o, ht, gr in ((o_in, ht_in, g_in), (o_cs, ht_cs, g_cs)):
        assert rel_err(o, ro) <= BF16_TOL and rel_err(ht, rht) <= BF16_TOL
        errs = {n: rel_err(gr[n], ref[n]) for n in gr}
        assert all(e <= BF16_TOL for e in errs.values()), errs


def test_autograd_equals_direct_calls():
    """The autograd path returns exactly what the C ABI calls return (q/k/v gradients after
    their cast to bf16)."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 130, 2, 4, 128, 128), dtype=torch.bfloat16, seed=17, grads=True)
    o, ht, gr = run_route(x, dev, in_kernel=True)
    d = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o2, ht2 = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    ref = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    assert torch.equal(o, o2) and torch.equal(ht, ht2)
    for n in ("dq", "dk", "dv"):
        assert torch.equal(gr[n], ref[n].to(torch.bfloat16)), n
    for n in ("dg", "dbeta", "dh0"):
        assert torch.equal(gr[n], ref[n]), n


def test_keep_operators_is_bitwise_identical():
    dev = cuda_device()
    x = make_inputs(Shape(1, 150, 2, 4, 128, 128), dtype=torch.bfloat16, seed=31, grads=True)
    res = []
    for keep in (False, True):
        t = leaves(x, dev)
        o, ht = gated_delta_rule(t["q"], t["k"], t["v"], t["g"], t["beta"], t["h0"], keep_operators=keep)
        ((o.float() * x["do"].to(dev).float()).sum() + (ht * x["dht"].to(dev)).sum()).backward()
        res.append([o.detach(), ht.detach()] + [t[n].grad for n in INPUTS])
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_unused_outputs_and_no_grad():
    dev = cuda_device()
    x = make_inputs(Shape(1, 70, 1, 2, 128, 128), dtype=torch.bfloat16, seed=23, grads=True, h0_std=None)
    t = leaves({**x, "h0": torch.zeros(1, 2, 128, 128)}, dev)
    o, ht = gated_delta_rule(t["q"], t["k"], t["v"], t["g"], t["beta"], None)
    (o.float() * x["do"].to(dev).float()).sum().backward()  # ht unused: dht = None
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], None, x["do"], None)
    for n in ("q", "k", "v", "g", "beta"):
        assert rel_err(t[n].grad, ref["d" + n]) <= BF16_TOL, n
    with torch.no_grad():
        o3, _ = gated_delta_rule(t["q"], t["k"], t["v"], t["g"], t["beta"], None)
    assert torch.equal(o3, o.detach())


@pytest.mark.parametrize("dtype,D,gate,tol", [(torch.float32, 64, "scalar", 1e-4),
                                              (torch.float32, 32, "channel", 1e-4)],
                         ids=["fp32-D64-scalar", "fp32-D32-channel"])
@pytest.mark.parametrize("keep_operators", [False, True])
def test_autograd_fp32_runs_the_fp32_chunked_path(dtype, D, gate, tol, keep_operators):
    """fp32 problems run the CUDA-core fp32 chunked kernels under autograd, both handoffs."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 100, 1, 2, D, D), dtype=dtype, seed=41, gate=gate, grads=True, gate_scale=0.3)
    t = leaves(x, dev)
    with gdr.trace() as tr:
        o, ht = gated_delta_rule(t["q"], t["k"], t["v"], t["g"], t["beta"], t["h0"], keep_operators=keep_operators)
        ((o.float() * x["do"].to(dev).float()).sum() + (ht * x["dht"].to(dev)).sum()).backward()
        torch.cuda.synchronize()
    names = {n for n, _ in tr.records}
    assert {"chunk32_scan_fwd", "chunk32_scan_bwd", "chunk32_grad"} <= names, names
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"])
    assert rel_err(o.detach(), ro) <= tol and rel_err(ht.detach(), rht) <= tol
    errs = {n: rel_err(t[n].grad, ref["d" + n]) for n in INPUTS}
    assert all(e <= tol for e in errs.values()), errs
