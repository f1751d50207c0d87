"""fp64 CPU oracle of the gated delta rule (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. It wraps ``oracle.c`` (plain C, fp64, OpenMP over heads)
through ctypes and shares no code with the CUDA library.

What it computes is stated in ``oracle.c``: the sequential Gated DeltaNet recurrence
with in-kernel q/k L2 normalisation (eps 1e-6, "fold q/k L2-norm into the
gated_delta_rule kernel", What/Why), scalar or per-channel decay ("Two-pass
optimization for channelwise gated delta rule kernel", Summary), GQA head sharing,
and its hand-derived reverse mode ("Adding VJP for gated delta net").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (portable C, no target flags)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declares the C signatures on a loaded oracle library (also used by the mutation tests,
    which load deliberately altered copies of oracle.c)."""
    i, d, p = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
    lib.oracle_forward.argtypes = [i] * 7 + [d, i] + [p] * 8
    lib.oracle_forward.restype = i
    lib.oracle_backward.argtypes = [i] * 7 + [d, i] + [p] * 14
    lib.oracle_backward.restype = i
    lib.oracle_decode_step.argtypes = [i] * 6 + [d, i] + [p] * 7
    lib.oracle_decode_step.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor on the CPU
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def _dims(q, v, g):
    B, T, Hk, Dk = q.shape
    Hv, Dv = v.shape[2], v.shape[3]
    channel = g.ndim == 4
    return B, T, Hk, Hv, Dk, Dv, channel


def forward(q, k, v, g, beta, h0=None, scale=None, use_qk_l2norm=True):
    """o [B,T,Hv,Dv], ht [B,Hv,Dv,Dk] in fp64. g: [B,T,Hv] (scalar) or [B,T,Hv,Dk]."""
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    B, T, Hk, Hv, Dk, Dv, channel = _dims(q, v, g)
    if scale is None:
        scale = Dk ** -0.5
    o = np.zeros((B, T, Hv, Dv))
    ht = np.zeros((B, Hv, Dv, Dk))
    rc = _load().oracle_forward(B, T, Hk, Hv, Dk, Dv, int(channel), float(scale), int(use_qk_l2norm),
                                _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(ht))
    if rc != 0:
        raise ValueError("oracle_forward: bad dimensions")
    return o, ht


def backward(q, k, v, g, beta, h0, do, dht=None, scale=None, use_qk_l2norm=True):
    """Gradients of <do,o> + <dht,ht>: dict with dq, dk, dv, dg, dbeta, dh0 (fp64)."""
    q, k, v, g, beta, h0, do, dht = map(_f64, (q, k, v, g, beta, h0, do, dht))
    B, T, Hk, Hv, Dk, Dv, channel = _dims(q, v, g)
    if scale is None:
        scale = Dk ** -0.5
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v), dg=np.zeros_like(g),
               dbeta=np.zeros_like(beta), dh0=np.zeros((B, Hv, Dv, Dk)))
    rc = _load().oracle_backward(B, T, Hk, Hv, Dk, Dv, int(channel), float(scale), int(use_qk_l2norm),
                                 _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(do),
                                 _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                                 _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["dh0"]))
    if rc != 0:
        raise ValueError("oracle_backward: bad dimensions")
    return out


def decode_step(q, k, v, g, beta, state, scale=None, use_qk_l2norm=True):
    """One token: q,k [B,Hk,Dk]; v [B,Hv,Dv]; g [B,Hv] or [B,Hv,Dk]; beta [B,Hv];
    state [B,Hv,Dv,Dk]. Returns (o [B,Hv,Dv], new_state) in fp64."""
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    st = _f64(state).copy()
    B, Hk, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[2]
    channel = g.ndim == 3
    if scale is None:
        scale = Dk ** -0.5
    o = np.zeros((B, Hv, Dv))
    rc = _load().oracle_decode_step(B, Hk, Hv, Dk, Dv, int(channel), float(scale), int(use_qk_l2norm),
                                    _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(st), _ptr(o))
    if rc != 0:
        raise ValueError("oracle_decode_step: bad dimensions")
    return o, st
