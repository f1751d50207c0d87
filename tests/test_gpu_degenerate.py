"""GPU parity on the method's degenerate tokens, through every CUDA entry point.

Tokens of a seeded sequence are overwritten with the special cases of the recurrence
S_t = S_{t-1} diag(a_t)(I - beta_t k^ k^T) + beta_t v_t k^T: beta = 0 (the token writes
and erases nothing), beta = 1 (the key's old value is replaced exactly), g = 0 (no decay,
a = 1), and all-zero keys and/or queries under the in-kernel L2 norm (k^ = 0, q^ = 0; the
norm factor (0 + 1e-6)^(-1/2) = 1000 of "fold q/k L2-norm into the gated_delta_rule kernel",
What/Why, multiplies their gradients). The chunked forward and VJP (scalar and per-channel
gate; bf16 on the tensor cores, fp32 on the CUDA cores), the token-by-token forward and VJP
(fp32 and bf16) and the decode step are compared with the fp64 oracle on the same inputs. Rows of dq / dk at zero queries / keys carry the
1000x factor, so they are checked apart from the other rows (one shared maximum would hide
errors in either group).
"""
import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.synth import Shape, make_inputs
from tests.util import BF16_TOL, F32_TOL, cuda_device, rel_err, to_dev

pytestmark = pytest.mark.gpu
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
KINDS = ("beta0", "beta1", "g0", "k0", "q0", "qk0")
# positions cover the first and last token of a chunk, both sides of chunk boundaries and the
# ragged tail; kinds are assigned in turn
POSITIONS = (0, 5, 31, 63, 64, 65, 100, 127, 128, 129, 150, 191, 192, 199)


def make_degenerate(shape, dtype, seed, gate="scalar", gate_scale=0.3, grads=False):
    x = make_inputs(shape, dtype=dtype, seed=seed, gate=gate, grads=grads, gate_scale=gate_scale)
    zk, zq = [], []
    for i, t in enumerate(p for p in POSITIONS if p < shape.T):
        kind = KINDS[i % len(KINDS)]
        if kind == "beta0":
            x["beta"][:, t] = 0.0
        elif kind == "beta1":
            x["beta"][:, t] = 1.0
        elif kind == "g0":
            x["g"][:, t] = 0.0
        if kind in ("k0", "qk0"):
            x["k"][:, t] = 0
            zk.append(t)
        if kind in ("q0", "qk0"):
            x["q"][:, t] = 0
            zq.append(t)
    return x, zk, zq


def check_grads(gr, ref, zk, zq, tol):
    """Each gradient within tol of the oracle; dq / dk rows at zero queries / keys apart."""
    for n in NAMES:
        got, want = gr[n].cpu(), torch.from_numpy(ref[n])
        zero = zq if n == "dq" else zk if n == "dk" else []
        if zero:
            m = torch.zeros(got.shape[1], dtype=torch.bool)
            m[zero] = True
            e_zero = rel_err(got[:, m], want[:, m])
            e_rest = rel_err(got[:, ~m], want[:, ~m])
            assert e_zero <= tol and e_rest <= tol, (n, e_zero, e_rest)
            # the norm factor at a zero vector: |dx| = 1000 |dx^|, far above the other rows
            assert float(want[:, m].abs().max()) > 10 * float(want[:, ~m].abs().max()), n
        else:
            assert rel_err(got, want) <= tol, (n, rel_err(got, want))


def oracle_bwd(x):
    return oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], x["do"], x["dht"])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_chunked_forward_and_vjp_degenerate_tokens(gate, dtype):
    dev = cuda_device()
    x, zk, zq = make_degenerate(Shape(2, 200, 2, 4, 128, 128), dtype, seed=501, gate=gate, grads=True)
    d = to_dev(x, dev)
    tol = F32_TOL if dtype == torch.float32 else BF16_TOL
    o, ht = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert torch.isfinite(o.float()).all() and torch.isfinite(ht).all()
    assert rel_err(o, ro) <= tol and rel_err(ht, rht) <= tol
    # a zero query reads nothing: its outputs are exactly zero on the GPU too
    assert torch.count_nonzero(o[:, zq].float()) == 0
    gr = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    for n in NAMES:
        assert torch.isfinite(gr[n]).all(), n
    check_grads(gr, oracle_bwd(x), zk, zq, tol)
    # the saved-state handoff sees the same tokens
    o2, h2, states = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], save_states=True)
    assert torch.equal(o, o2) and torch.equal(ht, h2)
    gs = gdr.bwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], None, d["do"], d["dht"], states=states)
    for n in NAMES:
        assert torch.equal(gs[n], gr[n]), n


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("gate", ["scalar", "channel"])
@pytest.mark.parametrize("D", [64, 128])
def test_sequential_forward_and_vjp_degenerate_tokens(dtype, gate, D):
    dev = cuda_device()
    x, zk, zq = make_degenerate(Shape(1, 150, 2, 4, D, D), dtype, seed=502 + D, gate=gate, grads=True)
    d = to_dev(x, dev)
    tol = F32_TOL if dtype == torch.float32 else BF16_TOL
    o, ht = gdr.fwd_sequential(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
    ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert rel_err(o, ro) <= tol and rel_err(ht, rht) <= tol
    gr = gdr.bwd_sequential(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"])
    for n in NAMES:
        assert torch.isfinite(gr[n]).all(), n
    check_grads(gr, oracle_bwd(x), zk, zq, tol)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_decode_degenerate_tokens(dtype, gate):
    """Decode steps over a sequence with every degenerate kind, against the oracle's decode
    step each token (outputs) and at the end (state)."""
    dev = cuda_device()
    T = 12
    x, zk, zq = make_degenerate(Shape(4, T, 2, 4, 128, 128), dtype, seed=503, gate=gate)
    # place every kind inside the 12 steps
    for i, t in enumerate(range(0, T, 2)):
        kind = KINDS[i]
        if kind == "beta0":
            x["beta"][:, t] = 0.0
        elif kind == "beta1":
            x["beta"][:, t] = 1.0
        elif kind == "g0":
            x["g"][:, t] = 0.0
        if kind in ("k0", "qk0"):
            x["k"][:, t] = 0
        if kind in ("q0", "qk0"):
            x["q"][:, t] = 0
    d = to_dev(x, dev)
    tol = F32_TOL if dtype == torch.float32 else BF16_TOL
    st = d["h0"].clone()
    ref = x["h0"].double().numpy()
    for t in range(T):
        sl = lambda n: x[n][:, t].contiguous()
        o = gdr.decode_step(d["q"][:, t].contiguous(), d["k"][:, t].contiguous(), d["v"][:, t].contiguous(),
                            d["g"][:, t].contiguous(), d["beta"][:, t].contiguous(), st)
        ro, ref = oracle.decode_step(sl("q"), sl("k"), sl("v"), sl("g"), sl("beta"), ref)
        assert torch.isfinite(o.float()).all()
        assert rel_err(o, ro) <= tol, t
    assert rel_err(st, ref) <= tol
