"""GPU parity of the sequential VJP (gdr_bwd_sequential) against the fp64 oracle's reverse
mode: every dtype, gate (scalar / per channel) and head size. Bounds: max|gpu - oracle| /
max|oracle| <= 1e-4 for fp32 inputs and <= 2e-2 for bf16 inputs, per gradient tensor."""
import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.synth import TINY_SEQ, Shape, make_inputs
from tests.util import BF16_TOL, F32_TOL, cuda_device, rel_err, to_dev

pytestmark = pytest.mark.gpu
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def run(x, dev, norm=True):
    d = to_dev(x, dev)
    return gdr.bwd_sequential(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"],
                              use_qk_l2norm=norm)


def check(gr, x, tol, norm=True):
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"], use_qk_l2norm=norm)
    errs = {n: rel_err(gr[n], ref[n]) for n in NAMES}
    assert all(e <= tol for e in errs.values()), errs


def test_tiny_config_fp32():
    """B=1, T=64, Hk=Hv=2, Dk=Dv=32, fp32, h0 = 0, in-kernel norm."""
    dev = cuda_device()
    x = make_inputs(TINY_SEQ, dtype=torch.float32, seed=1000, grads=True, h0_std=None)
    check(run(x, dev), x, F32_TOL)


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_sequential_backward_matrix(D, dtype, gate):
    dev = cuda_device()
    x = make_inputs(Shape(2, 37, 2, 4, D, D), dtype=dtype, seed=D + 7, gate=gate, grads=True)
    check(run(x, dev), x, F32_TOL if dtype == torch.float32 else BF16_TOL)


@pytest.mark.parametrize("case", [(1, 130, 1, 2, False, 0.01), (1, 1, 1, 1, True, 1.0), (2, 64, 2, 2, True, 3.0)],
                         ids=["T130-nonorm-mild", "T1", "T64-strong"])
def test_sequential_backward_segments_and_edges(case):
    """Crossing checkpoint segments with a ragged end, a single token, strong decay; h0 and
    dht absent in the first case."""
    dev = cuda_device()
    B, T, Hk, Hv, norm, gs = case
    x = make_inputs(Shape(B, T, Hk, Hv, 64, 64), dtype=torch.float32, seed=T, gate="channel", grads=True,
                    h0_std=None if not norm else 0.02, dht_std=None if not norm else 0.01, gate_scale=gs,
                    qk_std=1.0 if norm else 64 ** -0.5)
    check(run(x, dev, norm), x, F32_TOL, norm)


def test_channel_gate_layer_bf16():
    """The per-channel gate end to end at D=128, bf16: chunked forward, sequential VJP."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 300, 2, 4, 128, 128), dtype=torch.bfloat16, seed=21, gate="channel", grads=True,
                    gate_scale=0.3)
    d = to_dev(x, dev)
    o, ht = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert rel_err(o, ro) <= BF16_TOL and rel_err(ht, rht) <= BF16_TOL
    check(run(x, dev), x, BF16_TOL)


def test_sequential_equals_chunked_backward():
    dev = cuda_device()
    x = make_inputs(Shape(1, 200, 2, 4, 128, 128), dtype=torch.bfloat16, seed=5, grads=True, gate_scale=0.1)
    d = to_dev(x, dev)
    a = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    b = run(x, dev)
    for n in NAMES:
        assert rel_err(b[n], a[n]) <= BF16_TOL, n


def test_sequential_backward_deterministic_and_empty():
    dev = cuda_device()
    x = make_inputs(Shape(1, 70, 1, 2, 64, 64), dtype=torch.float32, seed=3, gate="channel", grads=True)
    a, b = run(x, dev), run(x, dev)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n
    x0 = make_inputs(Shape(1, 0, 1, 2, 64, 64), dtype=torch.float32, seed=1, grads=True)
    assert torch.equal(run(x0, dev)["dh0"].cpu(), x0["dht"])
