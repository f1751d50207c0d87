"""The seeded input recipe (gated_delta_rule_31_gb300/synth.py) that both the CUDA tests and the
oracle consume: deterministic per seed, the stated shapes and dtypes, g <= 0 (a = exp(g) in
(0, 1]), beta in (0, 1), and the stated scales. No method arithmetic is involved."""
import torch

from gated_delta_rule_31_gb300.synth import LONG_TRAIN, PREFILL, Shape, make_decode_inputs, make_inputs


def test_same_seed_same_inputs_other_seed_other_inputs():
    s = Shape(2, 33, 2, 4, 32, 16)
    a = make_inputs(s, seed=5, grads=True)
    b = make_inputs(s, seed=5, grads=True)
    c = make_inputs(s, seed=6, grads=True)
    for n in a:
        assert torch.equal(a[n], b[n]), n
    assert not torch.equal(a["q"], c["q"])


def test_shapes_dtypes_and_ranges():
    s = Shape(2, 50, 2, 4, 32, 16)
    x = make_inputs(s, dtype=torch.bfloat16, seed=1, grads=True)
    assert x["q"].shape == (2, 50, 2, 32) and x["k"].shape == (2, 50, 2, 32) and x["q"].dtype == torch.bfloat16
    assert x["v"].shape == (2, 50, 4, 16) and x["do"].shape == (2, 50, 4, 16) and x["do"].dtype == torch.bfloat16
    assert x["g"].shape == (2, 50, 4) and x["g"].dtype == torch.float32 and bool((x["g"] <= 0).all())
    assert x["beta"].shape == (2, 50, 4) and bool(((x["beta"] > 0) & (x["beta"] < 1)).all())
    assert x["h0"].shape == (2, 4, 16, 32) and x["dht"].shape == (2, 4, 16, 32)
    xc = make_inputs(s, seed=1, gate="channel")
    assert xc["g"].shape == (2, 50, 4, 32) and bool((xc["g"] <= 0).all())
    xn = make_inputs(s, seed=1, h0_std=None, dht_std=None, grads=True)
    assert xn["h0"] is None and xn["dht"] is None


def test_stated_scales():
    x = make_inputs(Shape(1, 256, 2, 4, 64, 64), dtype=torch.float32, seed=2, grads=True)
    assert abs(x["q"].std().item() - 1.0) < 0.05 and abs(x["v"].std().item() - 1.0) < 0.05
    assert abs(x["h0"].std().item() - 0.02) < 0.002 and abs(x["dht"].std().item() - 0.01) < 0.001
    # E[-softplus(N(0,1))] = -0.806 and E[sigmoid(N(0,1))] = 1/2 (symmetry)
    assert abs(x["g"].mean().item() + 0.806) < 0.05 and abs(x["beta"].mean().item() - 0.5) < 0.05
    mild = make_inputs(Shape(1, 256, 2, 4, 64, 64), seed=2, gate_scale=0.01)
    assert torch.allclose(mild["g"], x["g"] * 0.01)


def test_decode_inputs():
    d = make_decode_inputs(3, 2, 4, 32, 16, steps=5, seed=4)
    assert d["q"].shape == (5, 3, 2, 32) and d["v"].shape == (5, 3, 4, 16)
    assert d["g"].shape == (5, 3, 4, 32) and bool((d["g"] <= 0).all())
    assert d["state0"].shape == (3, 4, 16, 32) and d["state0"].dtype == torch.float32


def test_named_workloads():
    assert (LONG_TRAIN.B, LONG_TRAIN.T, LONG_TRAIN.Hk, LONG_TRAIN.Hv, LONG_TRAIN.Dk) == (1, 32768, 16, 32, 128)
    assert (PREFILL.T, PREFILL.Hk, PREFILL.Hv, PREFILL.Dv) == (4096, 16, 32, 128)
