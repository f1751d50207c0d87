"""Host-side checks of the C ABI: the library loads and exports every declared entry
point, and argument validation returns the documented status codes with nothing
launched (so these run without a GPU: invalid calls never reach the CUDA runtime)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
from gated_delta_rule_31_gb300 import Problem

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA, TIMEOUT = range(6)
FAKE = ctypes.c_void_p(0x100000)      # never dereferenced: validation fails first
MISALIGNED = ctypes.c_void_p(0x100004)


@pytest.fixture(scope="module")
def L():
    gdr.build()
    return gdr.lib()  # the binding declares argtypes for every entry point


def declared_functions():
    hdr = open(os.path.join(ROOT, "include", "gdr.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\*]+\s+\**(gdr_\w+)\s*\(", hdr, re.M)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert {"gdr_fwd_chunked", "gdr_bwd_chunked", "gdr_decode_step", "gdr_fwd_sequential"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(6):
        s = L.gdr_status_string(code).decode()
        assert s.startswith("GDR_")
    assert b"unknown" in L.gdr_status_string(99)


def prob(**kw):
    base = dict(B=1, T=64, Hk=2, Hv=4, Dk=128, Dv=128, dtype=1, gate=0, scale=0.088, use_qk_l2norm=1)
    base.update(kw)
    return Problem(*[base[f] for f, _ in Problem._fields_])


def fwd_seq(L, p, ptrs=None):
    ptrs = ptrs or [FAKE] * 8
    return L.gdr_fwd_sequential(ctypes.byref(p) if p is not None else None, *ptrs, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Hv=3), INVALID), (dict(Hk=0), INVALID), (dict(T=-1), INVALID), (dict(B=-2), INVALID),
    (dict(dtype=7), INVALID), (dict(gate=5), INVALID), (dict(use_qk_l2norm=2), INVALID),
    (dict(scale=float("nan")), INVALID), (dict(Dk=96), UNSUPPORTED), (dict(Dv=256), UNSUPPORTED),
    (dict(Dk=0), INVALID),
])
def test_problem_validation(L, kw, code):
    assert fwd_seq(L, prob(**kw)) == code


def test_null_and_misaligned_pointers(L):
    assert fwd_seq(L, None) == INVALID
    p = prob()
    for i in range(6):  # q, k, v, g, beta (h0 optional), o
        ptrs = [FAKE] * 8
        idx = i if i < 5 else 6
        ptrs[idx] = None
        assert fwd_seq(L, p, ptrs) == INVALID, idx
    ptrs = [FAKE] * 8
    ptrs[5] = MISALIGNED  # optional h0, misaligned
    assert fwd_seq(L, p, ptrs) == INVALID


def test_decode_requires_single_token(L):
    p = prob(T=2)
    assert L.gdr_decode_step(ctypes.byref(p), *[FAKE] * 7, None) == INVALID
    p = prob(T=1)
    assert L.gdr_decode_step(ctypes.byref(p), *([FAKE] * 6 + [None]), None) == INVALID


def test_chunked_support_matrix_and_workspace(L):
    # fp32 q/k/v: the CUDA-core fp32 chunked path, every head size in place (no staging). Its
    # forward workspace is the status word and one fp32 record per (b, hv, chunk): W, Kbar, Qg,
    # gamma [64 x Dk] each, U~ [64 x Dv], P and T [64 x 64], padded to 64 floats
    for dk, dv in ((128, 128), (64, 64), (32, 128), (128, 32)):
        p = prob(dtype=0, Dk=dk, Dv=dv)
        rec = (4 * 64 * dk + 64 * dv + 2 * 4096 + 63) // 64 * 64 * 4
        need = L.gdr_fwd_chunked_workspace(ctypes.byref(p))
        assert need == 256 + 4 * rec, (dk, dv)
        need_b = L.gdr_bwd_chunked_workspace(ctypes.byref(p))
        assert need_b > need
        assert L.gdr_fwd_chunked(ctypes.byref(p), *[FAKE] * 8, FAKE, need - 1, None) == WORKSPACE
        assert L.gdr_bwd_chunked(ctypes.byref(p), *[FAKE] * 14, FAKE, need_b - 1, None) == WORKSPACE
        states = 4 * dv * dk * 4  # B * Hv * chunks fp32 Dv x Dk chunk-start states
        assert L.gdr_chunk_states_bytes(ctypes.byref(p)) == states
        assert L.gdr_chunk_saved_bytes(ctypes.byref(p)) == 4 * rec + states
        assert L.gdr_fwd_chunked_saved_workspace(ctypes.byref(p)) == 256
        assert 0 < L.gdr_bwd_chunked_saved_workspace(ctypes.byref(p)) < L.gdr_bwd_chunked_states_workspace(
            ctypes.byref(p)) < need_b
    # bf16 head sizes 32 and 64: the workspace adds the zero-padded 128-wide copies of the inputs and
    # outputs; the saved-state and saved-operator buffers keep the 128-wide layout
    wide = prob()
    for dk, dv in ((32, 32), (64, 64), (64, 128), (128, 32)):
        p = prob(Dk=dk, Dv=dv)
        for q in ("gdr_fwd_chunked_workspace", "gdr_bwd_chunked_workspace", "gdr_bwd_chunked_states_workspace",
                  "gdr_fwd_chunked_saved_workspace", "gdr_bwd_chunked_saved_workspace"):
            assert getattr(L, q)(ctypes.byref(p)) > getattr(L, q)(ctypes.byref(wide)), (dk, dv, q)
        assert L.gdr_chunk_states_bytes(ctypes.byref(p)) == L.gdr_chunk_states_bytes(ctypes.byref(wide))
        assert L.gdr_chunk_saved_bytes(ctypes.byref(p)) == L.gdr_chunk_saved_bytes(ctypes.byref(wide))
        # a workspace one byte short is refused before any launch
        need = L.gdr_fwd_chunked_workspace(ctypes.byref(p))
        assert L.gdr_fwd_chunked(ctypes.byref(p), *[FAKE] * 8, FAKE, need - 1, None) == WORKSPACE
    # per-channel gate: chunked forward, both handoffs and the VJP (Gamma_C per key channel and the
    # backward's per-channel exports: larger buffers; the same T/W record per chunk)
    pc, ps = prob(gate=1), prob()
    assert L.gdr_fwd_chunked_workspace(ctypes.byref(pc)) > L.gdr_fwd_chunked_workspace(ctypes.byref(ps))
    assert L.gdr_bwd_chunked_workspace(ctypes.byref(pc)) > L.gdr_bwd_chunked_workspace(ctypes.byref(ps))
    assert L.gdr_bwd_chunked_states_workspace(ctypes.byref(pc)) > L.gdr_bwd_chunked_states_workspace(ctypes.byref(ps))
    assert L.gdr_chunk_states_bytes(ctypes.byref(pc)) == L.gdr_chunk_states_bytes(ctypes.byref(ps)) > 0
    sbc, sbs = L.gdr_chunk_saved_bytes(ctypes.byref(pc)), L.gdr_chunk_saved_bytes(ctypes.byref(ps))
    # header (Gamma_C per chunk and key channel) + (88 KB record + 24 KB T/W + 32 KB state)
    assert sbc == 2048 + 4 * (90112 + 24576 + 32768) and sbs == 1024 + 4 * (90112 + 24576 + 32768)
    assert L.gdr_bwd_chunked_saved_workspace(ctypes.byref(pc)) > L.gdr_bwd_chunked_saved_workspace(ctypes.byref(ps))
    assert L.gdr_fwd_chunked_saved(ctypes.byref(pc), *[FAKE] * 8, FAKE, sbc - 1, FAKE, 256, None) == WORKSPACE
    nb = L.gdr_bwd_chunked_workspace(ctypes.byref(pc))
    assert L.gdr_bwd_chunked(ctypes.byref(pc), *[FAKE] * 14, FAKE, nb - 1, None) == WORKSPACE
    p = prob()
    need = L.gdr_fwd_chunked_workspace(ctypes.byref(p))
    need_b = L.gdr_bwd_chunked_workspace(ctypes.byref(p))
    assert need > 0 and need_b > need
    assert L.gdr_fwd_chunked(ctypes.byref(p), *[FAKE] * 8, FAKE, need - 1, None) == WORKSPACE
    assert L.gdr_fwd_chunked(ctypes.byref(p), *[FAKE] * 8, None, need, None) == WORKSPACE
    assert L.gdr_bwd_chunked(ctypes.byref(p), *[FAKE] * 14, FAKE, need_b - 1, None) == WORKSPACE
    # dq (a required output) missing
    ptrs = [FAKE] * 14
    ptrs[8] = None
    assert L.gdr_bwd_chunked(ctypes.byref(p), *ptrs, FAKE, need_b, None) == INVALID


def test_workspace_grows_linearly_with_tokens(L):
    a = L.gdr_fwd_chunked_workspace(ctypes.byref(prob(T=64)))
    b = L.gdr_fwd_chunked_workspace(ctypes.byref(prob(T=128)))
    c = L.gdr_fwd_chunked_workspace(ctypes.byref(prob(T=65)))
    assert b > a and c == b  # a ragged chunk costs a whole chunk record


def test_binding_rejects_cpu_tensors():
    q = torch.zeros(1, 4, 1, 32)
    with pytest.raises(ValueError):
        gdr.fwd_sequential(q, q, torch.zeros(1, 4, 1, 32), torch.zeros(1, 4, 1), torch.zeros(1, 4, 1))


def test_saved_state_handoff_validation(L):
    p = prob()
    sb = L.gdr_chunk_states_bytes(ctypes.byref(p))
    wsb = L.gdr_bwd_chunked_states_workspace(ctypes.byref(p))
    assert sb == 1 * 4 * 1 * 32768  # B * Hv * chunks * one 128 x 128 bf16 image
    assert 0 < wsb < L.gdr_bwd_chunked_workspace(ctypes.byref(p))
    need_f = L.gdr_fwd_chunked_workspace(ctypes.byref(p))
    assert L.gdr_fwd_chunked_states(ctypes.byref(p), *[FAKE] * 8, FAKE, sb - 1, FAKE, need_f, None) == WORKSPACE
    assert L.gdr_fwd_chunked_states(ctypes.byref(p), *[FAKE] * 8, None, sb, FAKE, need_f, None) == WORKSPACE
    assert L.gdr_fwd_chunked_states(ctypes.byref(p), *[FAKE] * 8, MISALIGNED, sb, FAKE, need_f, None) == INVALID
    args = [FAKE] * 5 + [FAKE, sb] + [FAKE] * 8
    assert L.gdr_bwd_chunked_states(ctypes.byref(p), *args, FAKE, wsb - 1, None) == WORKSPACE
    args = [FAKE] * 5 + [FAKE, sb - 16] + [FAKE] * 8
    assert L.gdr_bwd_chunked_states(ctypes.byref(p), *args, FAKE, wsb, None) == WORKSPACE
    # fp32 keeps fp32 states (64 KB per chunk and value head here), so the bf16 size is short
    q = prob(dtype=0)
    assert L.gdr_chunk_states_bytes(ctypes.byref(q)) == 2 * sb
    need_q = L.gdr_fwd_chunked_workspace(ctypes.byref(q))
    assert L.gdr_fwd_chunked_states(ctypes.byref(q), *[FAKE] * 8, FAKE, sb, FAKE, need_q, None) == WORKSPACE


def test_autograd_function_has_no_cpu_path():
    from gated_delta_rule_31_gb300.autograd import gated_delta_rule

    q = torch.randn(1, 8, 1, 128, dtype=torch.bfloat16, requires_grad=True)
    v = torch.randn(1, 8, 2, 128, dtype=torch.bfloat16, requires_grad=True)
    g, beta = torch.zeros(1, 8, 2), torch.full((1, 8, 2), 0.5)
    with pytest.raises(ValueError, match="CUDA"):
        gated_delta_rule(q, q, v, g, beta)


def test_saved_operator_handoff_validation(L):
    p = prob()
    sb = L.gdr_chunk_saved_bytes(ctypes.byref(p))
    # header (per-chunk decay, padded) + (88 KB record + 24 KB T/W + 32 KB state) per (b, hv, chunk)
    assert sb == 1024 + 4 * 1 * (90112 + 24576 + 32768)
    fw = L.gdr_fwd_chunked_saved_workspace(ctypes.byref(p))
    bw = L.gdr_bwd_chunked_saved_workspace(ctypes.byref(p))
    # status word + chunk-end state gradients; a problem this small (4 value-head units) also gets
    # the split gradient's dq^ and dk^ per value head (fp32 [B][T][Hv][128] each)
    assert fw == 256 and bw == 1024 + 4 * 32768 + 2 * (64 * 4 * 128 * 4)
    big = prob(T=32768, Hk=16, Hv=32)  # 16384 units: one CTA per key-head tile, no such planes
    assert L.gdr_bwd_chunked_saved_workspace(ctypes.byref(big)) == 1024 + 32 * 512 * 32768
    assert L.gdr_fwd_chunked_saved(ctypes.byref(p), *[FAKE] * 8, FAKE, sb - 1, FAKE, fw, None) == WORKSPACE
    assert L.gdr_fwd_chunked_saved(ctypes.byref(p), *[FAKE] * 8, None, sb, FAKE, fw, None) == WORKSPACE
    assert L.gdr_fwd_chunked_saved(ctypes.byref(p), *[FAKE] * 8, FAKE, sb, FAKE, fw - 1, None) == WORKSPACE
    assert L.gdr_fwd_chunked_saved(ctypes.byref(p), *[FAKE] * 8, MISALIGNED, sb, FAKE, fw, None) == INVALID
    args = [FAKE] * 5 + [FAKE, sb] + [FAKE] * 8
    assert L.gdr_bwd_chunked_saved(ctypes.byref(p), *args, FAKE, bw - 1, None) == WORKSPACE
    args = [FAKE] * 5 + [FAKE, sb - 16] + [FAKE] * 8
    assert L.gdr_bwd_chunked_saved(ctypes.byref(p), *args, FAKE, bw, None) == WORKSPACE
    q = prob(dtype=0)
    sq = L.gdr_chunk_saved_bytes(ctypes.byref(q))
    assert sq > sb
    assert L.gdr_fwd_chunked_saved(ctypes.byref(q), *[FAKE] * 8, FAKE, sq - 1, FAKE, fw, None) == WORKSPACE


def test_sequential_backward_validation(L):
    p = prob(dtype=0, gate=1, Dk=64, Dv=64)  # fp32, per-channel gate, D=64: all supported here
    need = L.gdr_bwd_sequential_workspace(ctypes.byref(p))
    assert need > 0
    assert L.gdr_bwd_sequential(ctypes.byref(p), *[FAKE] * 14, FAKE, need - 1, None) == WORKSPACE
    ptrs = [FAKE] * 14
    ptrs[5] = None  # h0 optional
    ptrs[7] = None  # dht optional
    ptrs[13] = None  # dh0 optional
    assert L.gdr_bwd_sequential(ctypes.byref(p), *ptrs, FAKE, need - 1, None) == WORKSPACE
    ptrs = [FAKE] * 14
    ptrs[6] = None  # do required
    assert L.gdr_bwd_sequential(ctypes.byref(p), *ptrs, FAKE, need, None) == INVALID
    assert L.gdr_bwd_sequential_workspace(ctypes.byref(prob(Dk=96))) == 0


def test_wait_expiry_selftest_validation(L):
    """The expiry self-test checks its workspace before any launch (null, too small, misaligned)."""
    for ptr, n in ((None, 256), (FAKE, 255), (MISALIGNED, 256)):
        assert L.gdr_selftest_wait_expiry(ptr, n, None) == INVALID
    assert L.gdr_workspace_status(None, 256, None) == INVALID


def test_binding_workspace_checks(L):
    """The binding's workspace step: a size query of 0 raises the given status, and a caller's
    workspace must be a CUDA tensor on the problem's device, contiguous and large enough (all
    checked on the host before any launch)."""
    from gated_delta_rule_31_gb300 import _workspace
    with pytest.raises(gdr.GdrError) as e:
        _workspace(L.gdr_fwd_chunked_workspace, prob(Dk=96), torch.device("cuda", 0), None)
    assert e.value.code == UNSUPPORTED
    with pytest.raises(gdr.GdrError) as e:
        _workspace(L.gdr_bwd_sequential_workspace, prob(Dk=96), torch.device("cuda", 0), None, missing=INVALID)
    assert e.value.code == INVALID
    with pytest.raises(ValueError, match="CUDA tensor"):
        _workspace(L.gdr_fwd_chunked_workspace, prob(), torch.device("cuda", 0), torch.empty(1 << 20, dtype=torch.uint8))


def test_noalloc_forward_validation(L):
    """gdr_fwd_chunked_noalloc reports invalid and unsupported problems as gdr_fwd_chunked does,
    and problems beyond its built-in 64 MiB scratch as GDR_ERR_WORKSPACE, all before any launch."""
    P = ctypes.c_void_p
    L.gdr_fwd_chunked_noalloc.argtypes = [ctypes.POINTER(Problem)] + [P] * 8 + [P]
    L.gdr_fwd_chunked_noalloc.restype = ctypes.c_int
    for kw, code in ((dict(Hv=3), INVALID), (dict(Dk=96), UNSUPPORTED), (dict(dtype=0, T=4096, Hk=16, Hv=32), WORKSPACE),
                     (dict(T=4096, Hk=16, Hv=32), WORKSPACE), (dict(T=2048, Hk=16, Hv=32, Dk=64), WORKSPACE)):
        assert L.gdr_fwd_chunked_noalloc(ctypes.byref(prob(**kw)), *[FAKE] * 8, None) == code, kw
    assert L.gdr_fwd_chunked_workspace(ctypes.byref(prob(T=4096, Hk=16, Hv=32))) > 64 * 1024 * 1024
    assert L.gdr_fwd_chunked_noalloc(None, *[FAKE] * 8, None) == INVALID


def test_trace_with_nothing_launched(L):
    """Tracing on and off with no launch in between records nothing (no CUDA call is made)."""
    assert L.gdr_trace_enable(1) == OK
    assert L.gdr_trace_collect(None, None, 0) == 0
    assert L.gdr_trace_enable(0) == OK
    assert L.gdr_trace_collect(None, None, 0) == 0


def test_plain_c_program_links_and_calls_the_library(L, tmp_path):
    """include/gdr.h compiles as C99 and a C program links libgdr.so and calls the host-side
    entry points (workspace query, argument validation, status strings): no C++ or Python
    is needed to use the library."""
    src = tmp_path / "use_gdr.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "gdr.h"
int main(void) {
    gdr_problem p;
    memset(&p, 0, sizeof p);
    p.B = 1; p.T = 64; p.Hk = 1; p.Hv = 2; p.Dk = 128; p.Dv = 128;
    p.dtype = GDR_BF16; p.gate = GDR_GATE_SCALAR; p.scale = 0.088f; p.use_qk_l2norm = 1;
    size_t ws = gdr_fwd_chunked_workspace(&p);
    gdr_status s = gdr_fwd_chunked(&p, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0);
    printf("%zu %d %s\n", ws, (int)s, gdr_status_string(s));
    return (ws > 0 && s == GDR_ERR_INVALID_ARG) ? 0 : 1;
}
''')
    exe = tmp_path / "use_gdr"
    libdir = os.path.dirname(gdr.lib()._name)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-lgdr", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "GDR_ERR_INVALID_ARG" in out.stdout
