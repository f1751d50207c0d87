"""gdr_fwd_chunked_noalloc: the chunked forward for callers that cannot allocate device
memory (their device memory belongs to another allocator, or allocation is forbidden once
they have started), so they cannot hand the library a workspace. It runs on a scratch
array built into the library instead. This test calls it through the C ABI, twice in a row
on each problem (so a leftover of an earlier call would show), with the scalar and the
per-channel gate: it must equal gdr_fwd_chunked (which runs the same kernels on a caller
workspace) bit for bit, match the fp64 oracle within the bf16 bound, and leave a clean
status word (read with gdr_noalloc_status). Kept in its own file, collected last."""
import ctypes

import pytest
import torch

import gated_delta_rule_31_gb300 as gdr
import oracle
from gated_delta_rule_31_gb300.synth import Shape, make_inputs
from tests.util import BF16_TOL, cuda_device, rel_err

pytestmark = pytest.mark.gpu
WORKSPACE_ERR = 3


def _lib():
    gdr.build()
    L = gdr.lib()
    P = ctypes.c_void_p
    L.gdr_fwd_chunked_noalloc.argtypes = [ctypes.POINTER(gdr.Problem)] + [P] * 8 + [P]
    L.gdr_fwd_chunked_noalloc.restype = ctypes.c_int
    L.gdr_noalloc_status.argtypes = [P]
    L.gdr_noalloc_status.restype = ctypes.c_int
    return L


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc_forward(L, d, p, stream):
    o = torch.empty(d["v"].shape, dtype=d["v"].dtype, device=d["v"].device)
    ht = torch.empty((p.B, p.Hv, p.Dv, p.Dk), dtype=torch.float32, device=d["v"].device)
    rc = L.gdr_fwd_chunked_noalloc(ctypes.byref(p), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["g"]),
                                   _ptr(d["beta"]), _ptr(d["h0"]), _ptr(o), _ptr(ht), stream)
    assert rc == 0, L.gdr_status_string(rc)
    return o, ht


CASES = [(21, Shape(1, 200, 2, 4, 128, 128), "scalar"), (22, Shape(2, 130, 1, 2, 128, 128), "scalar"),
         (23, Shape(1, 150, 1, 2, 128, 128), "channel")]


def test_noalloc_forward_matches_workspace_forward_twice():
    dev = cuda_device()
    L = _lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for seed, shape, gate in CASES:
        x = make_inputs(shape, dtype=torch.bfloat16, seed=seed, gate=gate)
        d = {k: v.to(dev) for k, v in x.items()}
        p = gdr._problem(d["q"], d["v"], d["g"], None, True)
        ro, rht = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
        o2, h2 = gdr.fwd_chunked(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"])
        for _ in range(2):
            o1, h1 = _noalloc_forward(L, d, p, stream)
            assert L.gdr_noalloc_status(stream) == 0
            assert torch.equal(o1, o2) and torch.equal(h1, h2), (shape, gate)
            assert rel_err(o1, ro) <= BF16_TOL and rel_err(h1, rht) <= BF16_TOL, (shape, gate)


def test_noalloc_rejects_problems_beyond_its_scratch():
    cuda_device()
    L = _lib()
    p = gdr.Problem(1, 1473, 16, 32, 128, 128, gdr.GDR_BF16, gdr.GDR_GATE_SCALAR, 128 ** -0.5, 1)
    fake = ctypes.c_void_p(0x100000)  # never touched: the size check comes first
    rc = L.gdr_fwd_chunked_noalloc(ctypes.byref(p), *[fake] * 8, None)
    assert rc == WORKSPACE_ERR
