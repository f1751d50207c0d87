"""The oracle's pins catch plausible mistakes. Each case below plants one slip in a copy of
oracle.c (a dropped or misplaced decay, a wrong sign, a dropped factor, the wrong operand, the
wrong head map, the wrong eps, a missing term of the reverse mode), compiles it on the CPU and
runs the golden worked examples and the oracle pins against it: at least one must fail. The
unaltered source, compiled the same way, passes all of them. Every planted slip keeps each
memory access in bounds. Only the oracle is altered; nothing here touches the CUDA path."""
import ctypes
import os
import subprocess

import pytest

import oracle
from tests import test_golden as golden
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement); each text occurs exactly once
MUTANTS = [
    ("prediction from the undecayed state",
     "            Si[c] *= a[c];          /* Sd = S diag(a) */\n            acc += Si[c] * kh[c];   /* p = Sd k^ */",
     "            acc += Si[c] * kh[c];\n            Si[c] *= a[c];"),
    ("residual sign", "delta[i] = beta * (v[i] - acc);", "delta[i] = beta * (v[i] + acc);"),
    ("beta dropped from the residual", "delta[i] = beta * (v[i] - acc);", "delta[i] = (v[i] - acc);"),
    ("output read before the update",
     "            Si[c] += delta[i] * kh[c];  /* S = Sd + delta k^T */\n            out += Si[c] * qh[c];",
     "            out += Si[c] * qh[c];\n            Si[c] += delta[i] * kh[c];"),
    ("key read in place of the query", "l2n(q + qk_off(&d, b, t, hk), Dk, use_l2norm, qh);",
     "l2n(k + qk_off(&d, b, t, hk), Dk, use_l2norm, qh);"),
    ("norm eps", "#define NORM_EPS 1e-6", "#define NORM_EPS 1e-5"),
    ("scalar decay sign", "double s = exp(g[bt_off(d, b, t, hv)]);", "double s = exp(-g[bt_off(d, b, t, hv)]);"),
    ("channel decays reversed", "for (int i = 0; i < d->Dk; i++) a[i] = exp(gp[i]);",
     "for (int i = 0; i < d->Dk; i++) a[i] = exp(gp[d->Dk - 1 - i]);"),
    ("key head map", "int b = (int)(bh / Hv), hv = (int)(bh % Hv), hk = hv / group;",
     "int b = (int)(bh / Hv), hv = (int)(bh % Hv), hk = hv % Hk;"),
    ("initial state ignored", "if (h0) memcpy(S, h0 + st_off(&d, b, hv), sizeof(double) * Dv * Dk);",
     "if (0) memcpy(S, h0 + st_off(&d, b, hv), sizeof(double) * Dv * Dk);"),
    ("dbeta sign", "dbt += acc * (vt[i] - p[i]);", "dbt += acc * (vt[i] + p[i]);"),
    ("dk without the prediction path", "dkh[c] += Sprev[ic] * a[c] * dp[i];", ";"),
    ("state adjoint not decayed", "G[(size_t)i * Dk + c] = Gd[(size_t)i * Dk + c] * a[c];",
     "G[(size_t)i * Dk + c] = Gd[(size_t)i * Dk + c];"),
    ("channel dg without the factor a", "dgp[c] = a[c] * da[c];", "dgp[c] = da[c];"),
    ("scalar dg without the factor a", "dg[bt_off(&d, b, t, hv)] = a[0] * s;", "dg[bt_off(&d, b, t, hv)] = s;"),
    ("norm backward sign", "dqo[c] += RQ[j] * (dqh[c] - qh[c] * sq);", "dqo[c] += RQ[j] * (dqh[c] + qh[c] * sq);"),
    ("dk from the update with p in place of delta", "dkh[c] += G[(size_t)i * Dk + c] * dl[i];",
     "dkh[c] += G[(size_t)i * Dk + c] * p[i];"),
    ("dv without beta", "dv[vo_off(&d, b, t, hv) + i] = bt * acc;", "dv[vo_off(&d, b, t, hv) + i] = acc;"),
    ("dq from the state before the update", "dqh[c] += scale * Scur[(size_t)i * Dk + c] * dot[i];",
     "dqh[c] += scale * Sprev[(size_t)i * Dk + c] * dot[i];"),
    ("dht not seeded into the state adjoint", "if (dht) memcpy(G, dht + st_off(&d, b, hv), sizeof(double) * SS);",
     "if (0) memcpy(G, dht + st_off(&d, b, hv), sizeof(double) * SS);"),
]


def checks():
    """(name, callable) for every golden example and a set of pins; each raises on failure."""
    out = []
    for c in golden.CASES:
        out.append((f"golden forward: {c['name']}", lambda c=c: golden.test_forward_matches_worked_example(c)))
        if "grads" in c:
            out.append((f"golden backward: {c['name']}", lambda c=c: golden.test_backward_matches_worked_example(c)))
    for ch in (False, True):
        for nm in (False, True):
            out.append((f"product form (channel={ch}, norm={nm})",
                        lambda ch=ch, nm=nm: pins.test_matches_product_form(ch, nm)))
    out += [
        ("eps value", pins.test_norm_eps_value),
        ("orthonormal keys", lambda: pins.test_orthonormal_keys_retrieve_values(True)),
        ("equal channels = scalar gate", pins.test_channel_gate_with_equal_channels_equals_scalar_gate),
        ("GQA = repeated heads", pins.test_gqa_equals_repeated_heads),
        ("Euler identity", pins.test_euler_identity_and_norm_orthogonality),
        ("finite differences (scalar, norm)", lambda: pins.test_backward_matches_finite_differences(False, True, 6)),
        ("finite differences (channel, norm)", lambda: pins.test_backward_matches_finite_differences(True, True, 5)),
    ]
    return out


def compile_variant(tmp_path, source, tag):
    src = tmp_path / f"oracle_{tag}.c"
    lib = tmp_path / f"liboracle_{tag}.so"
    src.write_text(source)
    subprocess.run(["gcc", "-O1", "-std=c99", "-fopenmp", "-fPIC", "-shared", str(src), "-o", str(lib), "-lm"],
                   check=True)
    return oracle._bind(ctypes.CDLL(str(lib)))


def run_checks(monkeypatch, lib):
    """Names of the checks that fail with `lib` as the oracle."""
    monkeypatch.setattr(oracle, "_lib", lib)
    failed = []
    for name, fn in checks():
        try:
            fn()
        except (AssertionError, ValueError):
            failed.append(name)
    return failed


def test_unaltered_source_passes_every_check(tmp_path, monkeypatch):
    with open(SRC) as f:
        lib = compile_variant(tmp_path, f.read(), "plain")
    assert run_checks(monkeypatch, lib) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_slip_is_caught(tmp_path, monkeypatch, name, old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == 1, name
    lib = compile_variant(tmp_path, text.replace(old, new), "mutant")
    failed = run_checks(monkeypatch, lib)
    assert failed, f"no check fails when the oracle has this slip: {name}"
