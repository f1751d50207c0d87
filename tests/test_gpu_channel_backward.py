"""GPU parity of the chunked VJP with a per-channel gate (g [B,T,Hv,Dk]: the channelwise
variant of "Two-pass optimization for channelwise gated delta rule kernel", ExecuTorch PR
#21020, in the chunked reverse mode of "Adding VJP for gated delta net", MLX PR #4565) against
the fp64 oracle's reverse mode. Loss <do, o> + <dht, ht>; gradients dq, dk, dv, dg (one per key
channel), dbeta, dh0. Bound: max|gpu - oracle| / max|oracle| <= 2e-2 per tensor (bf16 inputs,
fp32 state and gradients)."""
import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.autograd import gated_delta_rule
from gated_delta_rule_31_gb300.synth import PREFILL, Shape, make_inputs
from tests.test_gpu_backward import NAMES, check, gpu_bwd, sliced, sliced_out
from tests.util import BF16_TOL, cuda_device, rel_err, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # (B, T, Hk, Hv, h0 and dht, norm, gate_scale)
    (1, 1, 1, 1, True, True, 1.0),
    (1, 63, 1, 1, False, True, 1.0),
    (1, 64, 1, 2, True, True, 1.0),
    (1, 100, 1, 2, True, True, 1.0),     # ragged last chunk
    (2, 130, 2, 4, True, False, 0.3),    # no norm, B=2, two value heads per key head
    (1, 300, 2, 4, True, True, 5.0),     # strong decay: per-token factors down to ~e^-20
    (1, 257, 1, 4, True, True, 0.01),    # mild decay: the state lives across many chunks
    (3, 65, 1, 8, True, True, 1.0),      # eight value heads per key head, odd batch
    (2, 40, 2, 32, True, True, 1.0),     # one chunk, 256 scan CTAs: two or three share an SM
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}T{c[1]}H{c[2]}x{c[3]}g{c[6]}" for c in CASES])
def test_channel_chunked_backward_small(case):
    dev = cuda_device()
    B, T, Hk, Hv, st, norm, gs = case
    x = make_inputs(Shape(B, T, Hk, Hv, 128, 128), dtype=torch.bfloat16, seed=17 * T + Hv, gate="channel",
                    grads=True, h0_std=0.02 if st else None, dht_std=0.01 if st else None, gate_scale=gs,
                    qk_std=1.0 if norm else 128 ** -0.5)
    gr = gpu_bwd(x, dev, norm)
    assert tuple(gr["dg"].shape) == (B, T, Hv, 128)
    check(gr, x, norm)


def test_channel_chunked_backward_extreme_decay_is_finite():
    """Per-token decays as small as e^-60: the running products underflow to zero, never overflow."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 200, 1, 2, 128, 128), dtype=torch.bfloat16, seed=9, gate="channel", grads=True,
                    gate_scale=30.0)
    gr = gpu_bwd(x, dev)
    for n in NAMES:
        assert torch.isfinite(gr[n]).all(), n
    check(gr, x)


def test_channel_chunked_backward_prefill_config():
    """B=1, T=4096, Hk=16, Hv=32, D=128 with a per-channel gate; key heads 0 and 15 (value heads
    0, 1 and 30, 31) checked against the oracle on the sliced inputs (groups do not interact)."""
    dev = cuda_device()
    x = make_inputs(PREFILL, dtype=torch.bfloat16, seed=2001, gate="channel", grads=True)
    gr = {n: t.cpu() for n, t in gpu_bwd(x, dev).items()}
    for hk in (0, 15):
        check(sliced_out(gr, 0, hk, 2), sliced(x, 0, hk, 2))


def test_channel_chunked_equals_sequential_backward_on_gpu():
    """The chunked and the token-by-token VJP (two unrelated kernels) agree within the bound."""
    dev = cuda_device()
    x = make_inputs(Shape(2, 333, 2, 4, 128, 128), dtype=torch.bfloat16, seed=11, gate="channel", grads=True,
                    gate_scale=0.3)
    d = to_dev(x, dev)
    ga = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    gs = gdr.bwd_sequential(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    errs = {n: rel_err(ga[n], gs[n]) for n in NAMES}
    assert all(e <= BF16_TOL for e in errs.values()), errs


def test_equal_channels_backward_matches_the_scalar_gate():
    """A per-channel gate with every channel equal to a scalar gate: the two chunked VJPs (different
    kernels) agree, and the scalar dg is the sum of the per-channel dg over the channels."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 257, 2, 4, 128, 128), dtype=torch.bfloat16, seed=13, grads=True)
    d = to_dev(x, dev)
    gch = d["g"][..., None].expand(*d["g"].shape, 128).contiguous()
    gsc = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    gc1 = gdr.bwd_chunked(d["q"], d["k"], d["v"], gch, d["beta"], d["h0"], d["do"], d["dht"])
    gc2 = gdr.bwd_chunked(d["q"], d["k"], d["v"], gch, d["beta"], d["h0"], d["do"], d["dht"])
    for n in NAMES:
        assert torch.equal(gc1[n], gc2[n]), n  # deterministic
        ref = gsc[n] if n != "dg" else gsc["dg"]
        got = gc1[n] if n != "dg" else gc1["dg"].sum(-1)
        assert rel_err(got, ref) <= BF16_TOL, n


@pytest.mark.parametrize("shape", [Shape(1, 300, 2, 4, 128, 128), Shape(2, 129, 1, 2, 128, 128)])
def test_channel_state_handoff_matches_recompute(shape):
    """The forward keeps the chunk-start states; the backward that reads them is bitwise the
    backward that recomputes them."""
    dev = cuda_device()
    x = make_inputs(shape, dtype=torch.bfloat16, seed=shape.T, gate="channel", grads=True, gate_scale=0.5)
    d = to_dev(x, dev)
    o1, h1 = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o2, h2, states = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_states=True)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    ga = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    gb = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], states=states)
    for n in NAMES:
        assert torch.equal(ga[n], gb[n]), n
    check(gb, x)


@pytest.mark.parametrize("shape", [Shape(1, 300, 2, 4, 128, 128), Shape(2, 129, 1, 2, 128, 128)])
def test_channel_saved_operator_handoff_matches_recompute(shape):
    """The forward can keep every chunk operator (with K^ .* Gamma for dT) and state: outputs and all
    gradients are bitwise those of the recompute path."""
    dev = cuda_device()
    x = make_inputs(shape, dtype=torch.bfloat16, seed=shape.T + 1, gate="channel", grads=True, gate_scale=0.5)
    d = to_dev(x, dev)
    o1, h1 = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o2, h2, saved = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_all=True)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    ga = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    gb = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], saved=saved)
    for n in NAMES:
        assert torch.equal(ga[n], gb[n]), n
    check(gb, x)


def test_channel_autograd_runs_the_chunked_vjp():
    """gated_delta_rule with a per-channel gate: gradients through the chunked VJP (the launch
    trace names its kernels) match the oracle."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 150, 1, 2, 128, 128), dtype=torch.bfloat16, seed=41, gate="channel", grads=True,
                    gate_scale=0.3)
    t = {n: (None if v is None else v.to(dev).requires_grad_(n in ("q", "k", "v", "g", "beta", "h0")))
         for n, v in x.items() if n not in ("do", "dht")}
    with gdr.trace() as tr:
        o, ht = gated_delta_rule(t["q"], t["k"], t["v"], t["g"], t["beta"], t["h0"])
        ((o.float() * x["do"].to(dev).float()).sum() + (ht * x["dht"].to(dev)).sum()).backward()
        torch.cuda.synchronize()
    names = {n for n, _ in tr.records}
    assert "chunk_grad_channel_mma" in names and "chunk_grad_channel_contract" in names, names
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"])
    for n in ("q", "k", "v", "g", "beta", "h0"):
        assert rel_err(t[n].grad, ref["d" + n]) <= BF16_TOL, n


def test_channel_autograd_keep_operators_matches_the_state_handoff():
    """keep_operators=True (the operator handoff) and the default state handoff give the same
    gradients with a per-channel gate."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 90, 1, 2, 128, 128), dtype=torch.bfloat16, seed=43, gate="channel", grads=True,
                    gate_scale=0.3)
    grads = []
    for keep in (False, True):
        t = {n: (None if v is None else v.to(dev).requires_grad_(True))
             for n, v in x.items() if n not in ("do", "dht")}
        o, ht = gated_delta_rule(t["q"], t["k"], t["v"], t["g"], t["beta"], t["h0"], keep_operators=keep)
        ((o.float() * x["do"].to(dev).float()).sum() + (ht * x["dht"].to(dev)).sum()).backward()
        grads.append({n: t[n].grad for n in ("q", "k", "v", "g", "beta", "h0")})
    for n in grads[0]:
        assert torch.equal(grads[0][n], grads[1][n]), n
