"""GPU parity of the chunked forward with a per-channel gate (g [B,T,Hv,Dk], one decay per key
channel: the channelwise variant of "Two-pass optimization for channelwise gated delta rule
kernel", ExecuTorch PR #21020) against the fp64 oracle. Bound: max|gpu - oracle| / max|oracle|
<= 2e-2 (bf16 inputs, fp32 state and accumulation)."""
import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.synth import PREFILL, Shape, make_inputs
from tests.util import BF16_TOL, cuda_device, rel_err, to_dev

pytestmark = pytest.mark.gpu


def gpu_fwd(x, dev, norm=True):
    d = to_dev(x, dev)
    return gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], use_qk_l2norm=norm)


def check(o, ht, x, norm=True):
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], use_qk_l2norm=norm)
    eo, eh = rel_err(o, ro), rel_err(ht, rht)
    assert eo <= BF16_TOL and eh <= BF16_TOL, (eo, eh)


CASES = [
    # (B, T, Hk, Hv, h0, norm, gate_scale)
    (1, 1, 1, 1, True, True, 1.0),
    (1, 63, 2, 2, False, True, 1.0),
    (1, 64, 1, 1, True, True, 1.0),
    (2, 65, 2, 4, True, True, 1.0),
    (1, 130, 1, 2, True, False, 0.01),
    (1, 300, 2, 4, True, True, 5.0),     # strong decay: per-token factors down to ~e^-20
    (2, 512, 2, 4, True, True, 0.01),    # mild decay: the state lives across many chunks
    (3, 50, 4, 16, True, True, 1.0),     # one chunk, 192 scan CTAs: two share an SM
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}T{c[1]}H{c[2]}x{c[3]}g{c[6]}" for c in CASES])
def test_channel_chunked_forward_small(case):
    dev = cuda_device()
    B, T, Hk, Hv, h0, norm, gs = case
    x = make_inputs(Shape(B, T, Hk, Hv, 128, 128), dtype=torch.bfloat16, seed=7 * T + Hv, gate="channel",
                    h0_std=0.02 if h0 else None, gate_scale=gs, qk_std=1.0 if norm else 128 ** -0.5)
    o, ht = gpu_fwd(x, dev, norm)
    assert tuple(o.shape) == tuple(x["v"].shape) and tuple(ht.shape) == (B, Hv, 128, 128)
    check(o, ht, x, norm)


def test_channel_chunked_extreme_decay_is_finite():
    """Per-token decays as small as e^-60 underflow to zero in the products, never overflow."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 200, 1, 2, 128, 128), dtype=torch.bfloat16, seed=9, gate="channel", gate_scale=30.0)
    o, ht = gpu_fwd(x, dev)
    assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
    check(o, ht, x)


def test_channel_chunked_prefill_config():
    """B=1, T=4096, Hk=16, Hv=32, D=128 with a per-channel gate; key heads 0 and 15 checked
    (value heads 0, 1 and 30, 31): heads do not interact, so the oracle on the sliced inputs
    gives those outputs exactly."""
    dev = cuda_device()
    x = make_inputs(PREFILL, dtype=torch.bfloat16, seed=1001, gate="channel")
    o, ht = gpu_fwd(x, dev)
    o, ht = o.cpu(), ht.cpu()
    for hk in (0, 15):
        sl = {n: (None if t is None else t[:, :, hk:hk + 1] if n in ("q", "k") else
                  t[:, 2 * hk:2 * hk + 2] if n == "h0" else t[:, :, 2 * hk:2 * hk + 2]) for n, t in x.items()}
        check(o[:, :, 2 * hk:2 * hk + 2], ht[:, 2 * hk:2 * hk + 2], sl)


def test_channel_chunked_equals_sequential_on_gpu():
    dev = cuda_device()
    x = make_inputs(Shape(2, 333, 2, 4, 128, 128), dtype=torch.bfloat16, seed=11, gate="channel", gate_scale=0.3)
    d = to_dev(x, dev)
    o1, h1 = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o2, h2 = gdr.fwd_sequential(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    assert rel_err(o1, o2) <= BF16_TOL and rel_err(h1, h2) <= BF16_TOL


def test_equal_channels_match_the_scalar_gate():
    """A per-channel gate with all channels equal is the scalar gate: the two chunked kernels
    (different decay arithmetic) agree within the bound, and the channel one is deterministic."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 257, 2, 4, 128, 128), dtype=torch.bfloat16, seed=13)
    d = to_dev(x, dev)
    gch = d["g"][..., None].expand(*d["g"].shape, 128).contiguous()
    o1, h1 = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o2, h2 = gdr.fwd_chunked(d["q"], d["k"], d["v"], gch, d["beta"], d["h0"])
    o3, h3 = gdr.fwd_chunked(d["q"], d["k"], d["v"], gch, d["beta"], d["h0"])
    assert rel_err(o2, o1) <= BF16_TOL and rel_err(h2, h1) <= BF16_TOL
    assert torch.equal(o2, o3) and torch.equal(h2, h3)
