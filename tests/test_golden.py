"""The oracle against hand-worked examples (tests/golden/worked_examples.json): tiny cases with
Dk = Dv = 2 whose outputs, final states and gradients were derived by hand from the two-pass
token update ("Two-pass optimization for channelwise gated delta rule kernel", ExecuTorch PR
#21020, Summary), the in-kernel norm (Megatron-LM PR #5396, What/Why) and the loss
<do, o> + <dht, ht> ("Adding VJP for gated delta net", MLX PR #4565). The fixture holds the
derivations; the values in it come from none of this repository's code."""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
with open(os.path.join(HERE, "golden", "worked_examples.json")) as f:
    CASES = json.load(f)["cases"]


def arr(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def inputs(c):
    return [arr(c[n]) for n in ("q", "k", "v", "g", "beta", "h0")]


@pytest.mark.parametrize("c", CASES, ids=[c["name"] for c in CASES])
def test_forward_matches_worked_example(c):
    o, ht = oracle.forward(*inputs(c), scale=c["scale"], use_qk_l2norm=c["use_qk_l2norm"])
    np.testing.assert_allclose(o, arr(c["o"]), rtol=c["tol"], atol=c["tol"])
    np.testing.assert_allclose(ht, arr(c["ht"]), rtol=c["tol"], atol=c["tol"])


@pytest.mark.parametrize("c", [c for c in CASES if len(c["q"][0]) == 1], ids=lambda c: c["name"])
def test_decode_step_matches_worked_example(c):
    """One-token cases through the oracle's decode step (the token axis removed)."""
    q, k, v, g, beta, h0 = inputs(c)
    B, _, Hv, Dv = v.shape
    state = h0 if h0 is not None else np.zeros((B, Hv, Dv, k.shape[-1]))
    o, st = oracle.decode_step(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], state, scale=c["scale"],
                               use_qk_l2norm=c["use_qk_l2norm"])
    np.testing.assert_allclose(o, arr(c["o"])[:, 0], rtol=c["tol"], atol=c["tol"])
    np.testing.assert_allclose(st, arr(c["ht"]), rtol=c["tol"], atol=c["tol"])


@pytest.mark.parametrize("c", [c for c in CASES if "grads" in c], ids=lambda c: c["name"])
def test_backward_matches_worked_example(c):
    got = oracle.backward(*inputs(c), arr(c["do"]), arr(c["dht"]), scale=c["scale"],
                          use_qk_l2norm=c["use_qk_l2norm"])
    for name, want in c["grads"].items():
        np.testing.assert_allclose(got[name], arr(want), rtol=c["tol"], atol=c["tol"], err_msg=name)
