"""The chunk-algebra tests catch plausible mistakes in the derivation the kernels implement.
Each case plants one slip in a copy of tests/chunk_algebra.py (a wrong triangle, a decay
dropped or shifted by one token, a sign, a missing term of the reverse scan or of the
per-channel block contractions) and runs a subset of tests/test_chunk_algebra.py against
it: at least one case must fail. The unaltered model passes them all."""
import os
import types

import pytest

from tests import test_chunk_algebra as tca

SRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "chunk_algebra.py")

# (name, text in chunk_algebra.py, replacement); each text occurs exactly once
MUTANTS = [
    # scalar gate, forward operators
    ("A with its diagonal", "A = low * (beta * rk)", "A = lowi * (beta * rk)"),
    ("P strictly lower", "P = scale * lowi * rq", "P = scale * low * rq"),
    ("W without Gamma", "W = T @ ((beta * Gam * rk)[:, None] * K)", "W = T @ ((beta * rk)[:, None] * K)"),
    ("Kbar without the decay to the chunk end", "Kbar = (b * rk)[:, None] * K", "Kbar = rk[:, None] * K"),
    ("Mneg sign", "    Kbar = (b * rk)[:, None] * K\n    Mneg = -Kbar.T @ W",
     "    Kbar = (b * rk)[:, None] * K\n    Mneg = Kbar.T @ W"),
    ("Qc without -P W", "Qc = scale * (Gam * rq)[:, None] * Q - P @ W", "Qc = scale * (Gam * rq)[:, None] * Q"),
    ("E transposed", "diff = gam[:, None] - gam[None, :]", "diff = gam[None, :] - gam[:, None]"),
    ("state not decayed across the chunk", 'H = np.exp(ops["gam"][-1]) * H + ', "H = H + "),
    ("(I - A)^-1 for (I + A)^-1", "T = np.linalg.inv(np.eye(C) + A)\n    W = T @ ((beta * Gam * rk)",
     "T = np.linalg.inv(np.eye(C) - A)\n    W = T @ ((beta * Gam * rk)"),
    # scalar gate, VJP
    ("dU without P^T dO", "dU = P.T @ dO + (bv * rk)[:, None] * (K @ dH1)", "dU = (bv * rk)[:, None] * (K @ dH1)"),
    ("dgamma_C without <dH1, H0>", " + np.exp(g_[-1]) * np.sum(dH1 * H0)", ""),
    ("dW sign", "                    dW = -dU @ H0.T\n                    dT = dU @ (bb[:, None] * V).T + dW @ ((bb * Gam)",
     "                    dW = dU @ H0.T\n                    dT = dU @ (bb[:, None] * V).T + dW @ ((bb * Gam)"),
    ("dP from U~ without the state correction", "dP = np.tril(dO @ U.T)", "dP = np.tril(dO @ Ut.T)"),
    ("dA with its diagonal", "                    dA = np.tril(-Tm.T @ dT @ Tm.T, -1)\n                    M = dA",
     "                    dA = np.tril(-Tm.T @ dT @ Tm.T, 0)\n                    M = dA"),
    ("reverse scan without Qc^T dO", 'dH = np.exp(g_[-1]) * dH1 + ops["Mneg"].T @ dH1 + ops["Qc"].T @ dO',
     'dH = np.exp(g_[-1]) * dH1 + ops["Mneg"].T @ dH1'),
    ("dg as a forward cumulative sum", "dgg = np.cumsum(dgam[::-1])[::-1]", "dgg = np.cumsum(dgam)"),
    # per-channel gate
    ("E_jj carries a_j", "            if r > j:\n                e = e * a[r]", "            e = e * a[r]"),
    ("Kbar's suffix product includes its own token", "        suf[r] = suf[r + 1] * a[r + 1]",
     "        suf[r] = suf[r + 1] * a[r]"),
    ("channel Qc without Gamma", "Qc = scale * Qh * Gam - P @ W", "Qc = scale * Qh - P @ W"),
    ("row side below the diagonal without the block's factor",
     "                c = c * a[r]\n                X1[r] += c * DX[i]", "                X1[r] += c * DX[i]"),
    ("column side factor applied one token early",
     "                X2[j] += f * DC[jj]\n                f = f * a[j]", "                f = f * a[j]\n                X2[j] += f * DC[jj]"),
    ("diagonal-block running decay shifted by one token", "                if j < r:\n                    e = e * a[j + 1]",
     "                if j < r:\n                    e = e * a[j]"),
    ("channel dgamma_C without <dH1, H0>", " + GamC * np.sum(dH1 * H0, axis=1)", ""),
    ("channel dbeta without the Y1 term", "\n                                          + np.sum(Kh * Y1, axis=1))[:n]", ")[:n]"),
]

CHECKS = [
    ("scalar C=4 T=11", lambda: tca.test_chunk_forward_and_backward_equal_oracle(4, 11, 1, 2, True, True)),
    ("scalar C=8 T=16 GQA", lambda: tca.test_chunk_forward_and_backward_equal_oracle(8, 16, 2, 4, True, False)),
    ("scalar C=64 T=70", lambda: tca.test_chunk_forward_and_backward_equal_oracle(64, 70, 1, 1, True, True)),
    ("channel forward C=4", lambda: tca.test_channel_chunk_forward_equals_oracle(4, 11, 1, 2, True, True, 1.0)),
    ("channel forward C=16 strong decay",
     lambda: tca.test_channel_chunk_forward_equals_oracle(16, 21, 1, 1, True, True, 8.0)),
    ("channel VJP C=8 bs=2", lambda: tca.test_channel_chunk_backward_equals_oracle(8, 2, 19, 1, 2, True, True, 1.0)),
    ("channel VJP C=16 bs=4 strong decay",
     lambda: tca.test_channel_chunk_backward_equals_oracle(16, 4, 37, 1, 2, True, True, 8.0)),
]


def load_variant(text):
    mod = types.ModuleType("chunk_algebra_variant")
    exec(compile(text, SRC, "exec"), mod.__dict__)
    return mod


def run_checks(monkeypatch, mod):
    monkeypatch.setattr(tca, "ca", mod)
    failed = []
    for name, fn in CHECKS:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_unaltered_model_passes_every_check(monkeypatch):
    with open(SRC) as f:
        assert run_checks(monkeypatch, load_variant(f.read())) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_slip_is_caught(monkeypatch, name, old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, name
    assert run_checks(monkeypatch, load_variant(text.replace(old, new))), f"no check fails with: {name}"
