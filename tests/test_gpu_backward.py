"""GPU parity of the chunked backward (VJP) against the fp64 oracle's reverse mode.

Loss <do, o> + <dht, ht>; gradients dq, dk, dv, dg, dbeta, dh0. Bound: max|gpu - oracle| /
max|oracle| <= 2e-2 per tensor (bf16 inputs, fp32 state and gradients). At the full
sizes of the VJP sweep and of the long-context training step the oracle checks sampled
(batch, key-head) groups: groups do not interact, so the oracle run on the sliced inputs
gives those outputs exactly.
"""
import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.synth import LONG_TRAIN, VJP_SWEEP, Shape, make_inputs
from tests.util import BF16_TOL, cuda_device, rel_err, to_dev

pytestmark = pytest.mark.gpu
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def gpu_bwd(x, dev, norm=True):
    d = to_dev(x, dev)
    return gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"],
                           use_qk_l2norm=norm)


def sliced(x, b, hk, G):
    """Inputs of one (batch, key head) group."""
    s = {}
    for n, t in x.items():
        if t is None:
            s[n] = None
        elif n in ("q", "k"):
            s[n] = t[b:b + 1, :, hk:hk + 1]
        elif n in ("v", "do", "g", "beta"):
            s[n] = t[b:b + 1, :, hk * G:(hk + 1) * G]
        else:  # h0, dht [B, Hv, Dv, Dk]
            s[n] = t[b:b + 1, hk * G:(hk + 1) * G]
    return s


def sliced_out(gr, b, hk, G):
    out = {}
    for n, t in gr.items():
        if n in ("dq", "dk"):
            out[n] = t[b:b + 1, :, hk:hk + 1]
        elif n == "dh0":
            out[n] = t[b:b + 1, hk * G:(hk + 1) * G]
        else:
            out[n] = t[b:b + 1, :, hk * G:(hk + 1) * G]
    return out


def check(gr, x, norm=True, tol=BF16_TOL):
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"],
                          use_qk_l2norm=norm)
    errs = {n: rel_err(gr[n], ref[n]) for n in NAMES}
    assert all(e <= tol for e in errs.values()), errs
    return errs


BWD_CASES = [
    # (B, T, Hk, Hv, h0, dht, norm, gate_scale)
    (1, 1, 1, 1, True, True, True, 1.0),
    (1, 8, 1, 2, True, True, True, 1.0),
    (1, 63, 2, 2, False, True, True, 1.0),
    (1, 64, 1, 1, True, False, True, 0.01),
    (2, 65, 2, 4, True, True, True, 1.0),
    (1, 130, 1, 2, True, True, False, 0.01),
    (1, 300, 2, 4, False, False, True, 0.01),
    (2, 512, 2, 4, True, True, True, 1.0),
    (3, 64, 4, 16, True, True, True, 1.0),  # one chunk, 192 scan CTAs: two or three share an SM
]


@pytest.mark.parametrize("case", BWD_CASES, ids=[f"B{c[0]}T{c[1]}H{c[2]}x{c[3]}" for c in BWD_CASES])
def test_chunked_backward_small(case):
    dev = cuda_device()
    B, T, Hk, Hv, h0, dht, norm, gs = case
    x = make_inputs(Shape(B, T, Hk, Hv, 128, 128), dtype=torch.bfloat16, seed=3 * T + Hv, grads=True,
                    h0_std=0.02 if h0 else None, dht_std=0.01 if dht else None, gate_scale=gs,
                    qk_std=1.0 if norm else 128 ** -0.5)
    gr = gpu_bwd(x, dev, norm)
    for n in NAMES:
        assert tuple(gr[n].shape) == tuple((x["q"] if n in ("dq", "dk") else x["v"] if n == "dv" else x["g"]
                                            if n == "dg" else x["beta"]).shape) or n == "dh0"
    check(gr, x, norm)


@pytest.mark.parametrize("idx", range(12))
def test_vjp_sweep_point(idx):
    """Every point of the B in {1,4,8} x T in {8,64,512,4096} sweep (Hk=16, Hv=32, D=128), with
    do ~ N(0,1) bf16 and dht ~ N(0, 0.01); groups (b, hk) = (0, 0) and (B-1, 15) checked."""
    dev = cuda_device()
    shape = VJP_SWEEP[idx]
    x = make_inputs(shape, dtype=torch.bfloat16, seed=1200 + idx, grads=True)
    gr = {k: v.cpu() for k, v in gpu_bwd(x, dev).items()}
    for b, hk in ((0, 0), (shape.B - 1, 15)):
        check(sliced_out(gr, b, hk, 2), sliced(x, b, hk, 2))


def sliced_heads(x, heads, G):
    """Inputs of the key heads `heads` (and their value heads) of batch 0."""
    vh = [hk * G + j for hk in heads for j in range(G)]
    s = {}
    for n, t in x.items():
        if t is None:
            s[n] = None
        elif n in ("q", "k"):
            s[n] = t[:1, :, heads].contiguous()
        elif n in ("h0", "dht"):
            s[n] = t[:1, vh].contiguous()
        else:
            s[n] = t[:1, :, vh].contiguous()
    return s, vh


def test_long_context_training_step_backward():
    """B=1, T=32768, h0 = 0, dht = 0, do ~ N(0,1): four key heads spread over the 16 (0, 5, 10,
    15, i.e. value heads 0-1, 10-11, 20-21, 30-31) checked against the oracle."""
    dev = cuda_device()
    x = make_inputs(LONG_TRAIN, dtype=torch.bfloat16, seed=1004, grads=True, h0_std=None, dht_std=None)
    gr = {k: v.cpu() for k, v in gpu_bwd(x, dev).items()}
    heads = [0, 5, 10, 15]
    xs, vh = sliced_heads(x, heads, 2)
    out = {n: (t[:1, :, heads] if n in ("dq", "dk") else t[:1, vh] if n == "dh0" else t[:1, :, vh])
           for n, t in gr.items()}
    check(out, xs)


def test_backward_mild_decay_long_range():
    """Mild decay keeps the state alive over 4096 tokens, exercising the reverse scan."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 4096, 2, 4, 128, 128), dtype=torch.bfloat16, seed=77, grads=True, gate_scale=0.01)
    check(gpu_bwd(x, dev), x)


def test_backward_ragged_many_tiles():
    """A ragged last chunk on the per-tile grad path (more than 128 value-head units: every tile's
    value heads in one CTA, dq / dk / dv leaving by tensor-map stores that must skip the rows past
    T), also run twice for bitwise determinism."""
    dev = cuda_device()
    x = make_inputs(Shape(1, 2000, 4, 8, 128, 128), dtype=torch.bfloat16, seed=41, grads=True, gate_scale=0.05)
    a, b = gpu_bwd(x, dev), gpu_bwd(x, dev)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n
    check(a, x)


def test_backward_deterministic():
    dev = cuda_device()
    x = make_inputs(Shape(1, 333, 2, 4, 128, 128), dtype=torch.bfloat16, seed=5, grads=True)
    a, b = gpu_bwd(x, dev), gpu_bwd(x, dev)
    for n in NAMES:
        assert torch.equal(a[n], b[n]), n


def test_backward_empty_sequence():
    dev = cuda_device()
    x = make_inputs(Shape(1, 0, 1, 2, 128, 128), dtype=torch.bfloat16, seed=1, grads=True)
    gr = gpu_bwd(x, dev)
    assert torch.equal(gr["dh0"].cpu(), x["dht"])


@pytest.mark.parametrize("shape", [Shape(1, 300, 2, 4, 128, 128), Shape(2, 129, 1, 2, 128, 128)])
def test_saved_state_handoff_matches_recompute(shape):
    """The forward can keep its chunk-start states for the backward: same outputs bit for bit,
    and the backward that reads them equals the one that re-runs the forward scan bit for bit
    (and therefore the oracle)."""
    dev = cuda_device()
    x = make_inputs(shape, dtype=torch.bfloat16, seed=shape.T, grads=True, gate_scale=0.1)
    d = to_dev(x, dev)
    o1, h1 = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o2, h2, states = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_states=True)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    ga = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    gb = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], states=states)
    for n in NAMES:
        assert torch.equal(ga[n], gb[n]), n
    check(gb, x)


@pytest.mark.parametrize("shape", [Shape(1, 300, 2, 4, 128, 128), Shape(2, 129, 1, 2, 128, 128),
                                   Shape(1, 64, 1, 1, 128, 128)])
def test_saved_operator_handoff_matches_recompute(shape):
    """The forward can keep every chunk operator and state for the backward: outputs and all
    gradients are bitwise those of the recompute path (and therefore match the oracle)."""
    dev = cuda_device()
    x = make_inputs(shape, dtype=torch.bfloat16, seed=shape.T + 7, grads=True, gate_scale=0.1)
    d = to_dev(x, dev)
    o1, h1 = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    o2, h2, saved = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_all=True)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)
    ga = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    gb = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], saved=saved)
    for n in NAMES:
        assert torch.equal(ga[n], gb[n]), n
    check(gb, x)


def test_saved_operator_handoff_empty_sequence():
    dev = cuda_device()
    x = make_inputs(Shape(1, 0, 1, 2, 128, 128), dtype=torch.bfloat16, seed=1, grads=True)
    d = to_dev(x, dev)
    o, ht, saved = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_all=True)
    assert torch.equal(ht.cpu(), x["h0"])
    gr = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], saved=saved)
    assert torch.equal(gr["dh0"].cpu(), x["dht"])


@pytest.mark.parametrize("shape", [Shape(1, 200, 1, 4, 128, 128), Shape(3, 100, 2, 16, 128, 128),
                                   Shape(1, 130, 1, 8, 128, 128)], ids=["G4", "B3-G8", "G8-ragged"])
def test_wider_head_groups(shape):
    """Value-head groups of 4, 8 and 16 per key head (the persistent prep and grad kernels loop
    over a group's heads and fetch the next one while finishing the current one), an odd batch
    count and ragged last chunks: forward and backward against the oracle."""
    dev = cuda_device()
    x = make_inputs(shape, dtype=torch.bfloat16, seed=shape.Hv + shape.T, grads=True, gate_scale=0.2)
    d = to_dev(x, dev)
    o, ht = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert rel_err(o, ro) <= BF16_TOL and rel_err(ht, rht) <= BF16_TOL
    check(gpu_bwd(x, dev), x)
