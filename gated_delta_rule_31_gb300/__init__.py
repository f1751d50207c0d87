"""GB300 (sm_103a) gated delta rule: thin Python binding of the C ABI in ``include/gdr.h``.

Every step of the computation runs in ``libgdr.so``'s CUDA kernels; this module only
checks tensors, allocates outputs and workspace with torch, and passes raw device
pointers and the current CUDA stream through ctypes. There is no CPU fallback: if the
library is missing or a tensor is not on a CUDA device, the calls raise.

Operation (Gated DeltaNet recurrence, per batch and value head, key head hv // (Hv/Hk)):
    k^ = k (|k|^2 + 1e-6)^-1/2,  q^ likewise      (when use_qk_l2norm)
    S_t = S_{t-1} diag(exp g_t) (I - beta_t k^ k^T) + beta_t v_t k^T,   o_t = scale S_t q^
Layouts: q,k [B,T,Hk,Dk]; v,o [B,T,Hv,Dv]; g [B,T,Hv] or [B,T,Hv,Dk] fp32; beta [B,T,Hv]
fp32; states [B,Hv,Dv,Dk] fp32.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB as _LIB_PATH
from ._build import build

__all__ = ["build", "fwd_chunked", "bwd_chunked", "fwd_sequential", "bwd_sequential", "decode_step", "GdrError",
           "fwd_workspace_bytes", "bwd_workspace_bytes", "lib", "Problem", "workspace_status", "selftest_wait_expiry", "trace"]

GDR_F32, GDR_BF16 = 0, 1
GDR_GATE_SCALAR, GDR_GATE_CHANNEL = 0, 1
GDR_ERR_INVALID_ARG, GDR_ERR_UNSUPPORTED = 1, 2


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("Hk", ctypes.c_int), ("Hv", ctypes.c_int),
                ("Dk", ctypes.c_int), ("Dv", ctypes.c_int), ("dtype", ctypes.c_int), ("gate", ctypes.c_int),
                ("scale", ctypes.c_float), ("use_qk_l2norm", ctypes.c_int)]


class GdrError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(msg)
        self.code = code


_lib = None


def lib():
    """The loaded libgdr.so (ctypes handle). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it first (gated_delta_rule_31_gb300.build())")
        L = ctypes.CDLL(_LIB_PATH)
        P, PP, sz, st = ctypes.c_void_p, ctypes.POINTER(Problem), ctypes.c_size_t, ctypes.c_void_p
        L.gdr_status_string.argtypes = [ctypes.c_int]
        L.gdr_status_string.restype = ctypes.c_char_p
        L.gdr_fwd_chunked_workspace.argtypes = [PP]
        L.gdr_fwd_chunked_workspace.restype = sz
        L.gdr_bwd_chunked_workspace.argtypes = [PP]
        L.gdr_bwd_chunked_workspace.restype = sz
        L.gdr_fwd_chunked.argtypes = [PP] + [P] * 8 + [P, sz, st]
        L.gdr_fwd_chunked.restype = ctypes.c_int
        L.gdr_fwd_sequential.argtypes = [PP] + [P] * 8 + [st]
        L.gdr_fwd_sequential.restype = ctypes.c_int
        L.gdr_bwd_chunked.argtypes = [PP] + [P] * 14 + [P, sz, st]
        L.gdr_bwd_sequential_workspace.argtypes = [PP]
        L.gdr_bwd_sequential_workspace.restype = sz
        L.gdr_bwd_sequential.argtypes = [PP] + [P] * 14 + [P, sz, st]
        L.gdr_bwd_sequential.restype = ctypes.c_int
        L.gdr_bwd_chunked.restype = ctypes.c_int
        L.gdr_decode_step.argtypes = [PP] + [P] * 7 + [st]
        L.gdr_decode_step.restype = ctypes.c_int
        L.gdr_chunk_states_bytes.argtypes = [PP]
        L.gdr_chunk_states_bytes.restype = sz
        L.gdr_bwd_chunked_states_workspace.argtypes = [PP]
        L.gdr_bwd_chunked_states_workspace.restype = sz
        L.gdr_fwd_chunked_states.argtypes = [PP] + [P] * 8 + [P, sz, P, sz, st]
        L.gdr_fwd_chunked_states.restype = ctypes.c_int
        L.gdr_bwd_chunked_states.argtypes = [PP] + [P] * 5 + [P, sz] + [P] * 8 + [P, sz, st]
        L.gdr_bwd_chunked_states.restype = ctypes.c_int
        for name in ("gdr_chunk_saved_bytes", "gdr_fwd_chunked_saved_workspace", "gdr_bwd_chunked_saved_workspace"):
            getattr(L, name).argtypes = [PP]
            getattr(L, name).restype = sz
        L.gdr_fwd_chunked_saved.argtypes = [PP] + [P] * 8 + [P, sz, P, sz, st]
        L.gdr_fwd_chunked_saved.restype = ctypes.c_int
        L.gdr_bwd_chunked_saved.argtypes = [PP] + [P] * 5 + [P, sz] + [P] * 8 + [P, sz, st]
        L.gdr_bwd_chunked_saved.restype = ctypes.c_int
        L.gdr_workspace_status.argtypes = [P, sz, st]
        L.gdr_workspace_status.restype = ctypes.c_int
        L.gdr_selftest_wait_expiry.argtypes = [P, sz, st]
        L.gdr_selftest_wait_expiry.restype = ctypes.c_int
        L.gdr_trace_enable.argtypes = [ctypes.c_int]
        L.gdr_trace_enable.restype = ctypes.c_int
        L.gdr_trace_collect.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float),
                                        ctypes.c_int]
        L.gdr_trace_collect.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(code: int):
    if code != 0:
        raise GdrError(code, lib().gdr_status_string(code).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype=None, device=None, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _problem(q, v, g, scale, use_qk_l2norm, T=None):
    if q.dim() == 4:
        B, T_, Hk, Dk = q.shape
    else:  # decode: [B, Hk, Dk]
        B, Hk, Dk = q.shape
        T_ = 1
    Hv, Dv = v.shape[-2], v.shape[-1]
    channel = g.dim() == (4 if q.dim() == 4 else 3)
    dtype = {torch.float32: GDR_F32, torch.bfloat16: GDR_BF16}.get(q.dtype)
    if dtype is None:
        raise ValueError(f"q/k/v dtype must be float32 or bfloat16, got {q.dtype}")
    if scale is None:
        scale = Dk ** -0.5
    return Problem(B, T_ if T is None else T, Hk, Hv, Dk, Dv, dtype,
                   GDR_GATE_CHANNEL if channel else GDR_GATE_SCALAR, float(scale), int(bool(use_qk_l2norm)))


def _check_inputs(q, k, v, g, beta, h0=None):
    dev = q.device
    _need(q, "q", device=dev)
    _need(k, "k", dtype=q.dtype, device=dev, shape=q.shape)
    _need(v, "v", dtype=q.dtype, device=dev)
    _need(g, "g", dtype=torch.float32, device=dev)
    _need(beta, "beta", dtype=torch.float32, device=dev)
    lead = tuple(q.shape[:-2])
    Hv, Dv, Dk = v.shape[-2], v.shape[-1], q.shape[-1]
    if tuple(v.shape[:-2]) != lead:
        raise ValueError("v leading dims must match q")
    if tuple(beta.shape) != lead + (Hv,):
        raise ValueError(f"beta must be {lead + (Hv,)}")
    if tuple(g.shape) not in (lead + (Hv,), lead + (Hv, Dk)):
        raise ValueError(f"g must be {lead + (Hv,)} or {lead + (Hv, Dk)}")
    if h0 is not None:
        _need(h0, "h0", dtype=torch.float32, device=dev, shape=(q.shape[0], Hv, Dv, Dk))


def fwd_workspace_bytes(p: Problem) -> int:
    return int(lib().gdr_fwd_chunked_workspace(ctypes.byref(p)))


def bwd_workspace_bytes(p: Problem) -> int:
    return int(lib().gdr_bwd_chunked_workspace(ctypes.byref(p)))


def _workspace(query, p, device, workspace, missing=GDR_ERR_UNSUPPORTED):
    """(workspace, bytes) for the call whose size query is `query`: the caller's tensor after
    checking it, else a new uint8 buffer. A zero size means the call does not take this problem
    and raises as the status `missing` would."""
    nbytes = int(query(ctypes.byref(p)))
    if nbytes == 0:
        _check(missing)
    if workspace is not None:
        _need(workspace, "workspace", device=device)
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace too small: {workspace.numel() * workspace.element_size()} < {nbytes} bytes")
        return workspace, nbytes
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device), nbytes


def fwd_sequential(q, k, v, g, beta, h0=None, scale=None, use_qk_l2norm=True, output_final_state=True):
    """Token-by-token forward (gdr_fwd_sequential). Returns (o, ht or None)."""
    _check_inputs(q, k, v, g, beta, h0)
    p = _problem(q, v, g, scale, use_qk_l2norm)
    o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    ht = torch.empty((p.B, p.Hv, p.Dv, p.Dk), dtype=torch.float32, device=v.device) if output_final_state else None
    _check(lib().gdr_fwd_sequential(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(o), _ptr(ht), _stream(q.device)))
    return o, ht


def fwd_chunked(q, k, v, g, beta, h0=None, scale=None, use_qk_l2norm=True, output_final_state=True,
                workspace=None, save_states=False, save_all=False):
    """Chunked prefill forward (gdr_fwd_chunked: bf16 on the tensor cores, fp32 on the CUDA-core
    fp32 kernels). Returns (o, ht or None),
    or (o, ht, states) with save_states=True (gdr_fwd_chunked_states: the chunk-start states
    kept for bwd_chunked(..., states=states)), or (o, ht, saved) with save_all=True
    (gdr_fwd_chunked_saved: states and chunk operators kept for bwd_chunked(..., saved=saved))."""
    _check_inputs(q, k, v, g, beta, h0)
    p = _problem(q, v, g, scale, use_qk_l2norm)
    o = torch.empty(v.shape, dtype=v.dtype, device=v.device)
    ht = torch.empty((p.B, p.Hv, p.Dv, p.Dk), dtype=torch.float32, device=v.device) if output_final_state else None
    if save_all:
        L = lib()
        ws, nbytes = _workspace(L.gdr_fwd_chunked_saved_workspace, p, q.device, workspace)
        sb = int(L.gdr_chunk_saved_bytes(ctypes.byref(p)))
        saved = torch.empty(max(sb, 256), dtype=torch.uint8, device=q.device)
        _check(L.gdr_fwd_chunked_saved(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                       _ptr(o), _ptr(ht), _ptr(saved), ctypes.c_size_t(sb), _ptr(ws),
                                       ctypes.c_size_t(nbytes), _stream(q.device)))
        return o, ht, saved
    ws, nbytes = _workspace(lib().gdr_fwd_chunked_workspace, p, q.device, workspace)
    if not save_states:
        _check(lib().gdr_fwd_chunked(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                     _ptr(o), _ptr(ht), _ptr(ws), ctypes.c_size_t(nbytes), _stream(q.device)))
        return o, ht
    sb = int(lib().gdr_chunk_states_bytes(ctypes.byref(p)))
    states = torch.empty(max(sb, 256), dtype=torch.uint8, device=q.device)
    _check(lib().gdr_fwd_chunked_states(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                        _ptr(o), _ptr(ht), _ptr(states), ctypes.c_size_t(sb), _ptr(ws),
                                        ctypes.c_size_t(nbytes), _stream(q.device)))
    return o, ht, states


def bwd_chunked(q, k, v, g, beta, h0, do, dht=None, scale=None, use_qk_l2norm=True, workspace=None,
                states=None, saved=None):
    """Chunked backward (gdr_bwd_chunked) of <do,o> + <dht,ht>. Returns a dict of fp32
    gradients dq, dk, dv, dg, dbeta, dh0. With `states` from fwd_chunked(save_states=True)
    on the same inputs, gdr_bwd_chunked_states reads them instead of re-running the
    forward scan; with `saved` from fwd_chunked(save_all=True), gdr_bwd_chunked_saved runs
    neither prep nor the forward scan (h0 is unused in both cases)."""
    _check_inputs(q, k, v, g, beta, h0)
    _need(do, "do", dtype=v.dtype, device=v.device, shape=v.shape)
    p = _problem(q, v, g, scale, use_qk_l2norm)
    if dht is not None:
        _need(dht, "dht", dtype=torch.float32, device=v.device, shape=(p.B, p.Hv, p.Dv, p.Dk))
    f32 = dict(dtype=torch.float32, device=v.device)
    out = dict(dq=torch.empty(q.shape, **f32), dk=torch.empty(k.shape, **f32), dv=torch.empty(v.shape, **f32),
               dg=torch.empty(g.shape, **f32), dbeta=torch.empty(beta.shape, **f32),
               dh0=torch.empty((p.B, p.Hv, p.Dv, p.Dk), **f32))
    if saved is not None:
        _need(saved, "saved", dtype=torch.uint8, device=q.device)
        L = lib()
        ws, nbytes = _workspace(L.gdr_bwd_chunked_saved_workspace, p, q.device, workspace)
        _check(L.gdr_bwd_chunked_saved(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                       _ptr(saved), ctypes.c_size_t(saved.numel()), _ptr(do), _ptr(dht),
                                       _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                                       _ptr(out["dbeta"]), _ptr(out["dh0"]), _ptr(ws), ctypes.c_size_t(nbytes),
                                       _stream(q.device)))
        return out
    if states is None:
        ws, nbytes = _workspace(lib().gdr_bwd_chunked_workspace, p, q.device, workspace)
        _check(lib().gdr_bwd_chunked(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                     _ptr(do), _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                                     _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["dh0"]), _ptr(ws),
                                     ctypes.c_size_t(nbytes), _stream(q.device)))
        return out
    _need(states, "states", dtype=torch.uint8, device=q.device)
    ws, nbytes = _workspace(lib().gdr_bwd_chunked_states_workspace, p, q.device, workspace)
    _check(lib().gdr_bwd_chunked_states(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                        _ptr(states), ctypes.c_size_t(states.numel()), _ptr(do), _ptr(dht),
                                        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                                        _ptr(out["dbeta"]), _ptr(out["dh0"]), _ptr(ws), ctypes.c_size_t(nbytes),
                                        _stream(q.device)))
    return out


def bwd_sequential(q, k, v, g, beta, h0, do, dht=None, scale=None, use_qk_l2norm=True, workspace=None):
    """Sequential VJP (gdr_bwd_sequential) of <do,o> + <dht,ht>: every dtype, gate and head
    size. Returns a dict of fp32 gradients dq, dk, dv, dg, dbeta, dh0 (dg has g's shape)."""
    _check_inputs(q, k, v, g, beta, h0)
    _need(do, "do", dtype=v.dtype, device=v.device, shape=v.shape)
    p = _problem(q, v, g, scale, use_qk_l2norm)
    if dht is not None:
        _need(dht, "dht", dtype=torch.float32, device=v.device, shape=(p.B, p.Hv, p.Dv, p.Dk))
    f32 = dict(dtype=torch.float32, device=v.device)
    out = dict(dq=torch.empty(q.shape, **f32), dk=torch.empty(k.shape, **f32), dv=torch.empty(v.shape, **f32),
               dg=torch.empty(g.shape, **f32), dbeta=torch.empty(beta.shape, **f32),
               dh0=torch.empty((p.B, p.Hv, p.Dv, p.Dk), **f32))
    ws, nbytes = _workspace(lib().gdr_bwd_sequential_workspace, p, q.device, workspace, missing=GDR_ERR_INVALID_ARG)
    _check(lib().gdr_bwd_sequential(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                    _ptr(do), _ptr(dht), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                                    _ptr(out["dg"]), _ptr(out["dbeta"]), _ptr(out["dh0"]), _ptr(ws),
                                    ctypes.c_size_t(nbytes), _stream(q.device)))
    return out


def decode_step(q, k, v, g, beta, state, scale=None, use_qk_l2norm=True, out=None):
    """One decode step (gdr_decode_step): q,k [B,Hk,Dk]; v [B,Hv,Dv]; g [B,Hv] or [B,Hv,Dk];
    beta [B,Hv]; state [B,Hv,Dv,Dk] fp32 updated in place. Returns o [B,Hv,Dv]."""
    _check_inputs(q, k, v, g, beta)
    p = _problem(q, v, g, scale, use_qk_l2norm)
    _need(state, "state", dtype=torch.float32, device=q.device, shape=(p.B, p.Hv, p.Dv, p.Dk))
    o = out if out is not None else torch.empty(v.shape, dtype=v.dtype, device=v.device)
    _check(lib().gdr_decode_step(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                 _ptr(o), _stream(q.device)))
    return o


def workspace_status(ws) -> int:
    """Reads and clears the status word of a chunked workspace (0 = ok, 5 = a wait expired)."""
    return int(lib().gdr_workspace_status(_ptr(ws), ctypes.c_size_t(ws.numel()), _stream(ws.device)))


def selftest_wait_expiry(ws) -> None:
    """gdr_selftest_wait_expiry: one CTA's bounded wait on a phase that nothing completes gives up
    after about a second and records GDR_ERR_TIMEOUT in the status word of ``ws`` (uint8, >= 256
    bytes, on the GPU); read it back with workspace_status."""
    _check(lib().gdr_selftest_wait_expiry(_ptr(ws), ctypes.c_size_t(ws.numel()), _stream(ws.device)))


class trace:
    """Context manager recording (kernel name, ms) for every library launch inside it:
    ``with gdr.trace() as t: ...`` then ``t.records``."""

    def __enter__(self):
        lib().gdr_trace_collect(None, None, 0)
        lib().gdr_trace_enable(1)
        self.records = []
        return self

    def __exit__(self, *exc):
        L = lib()
        L.gdr_trace_enable(0)
        n = L.gdr_trace_collect(None, None, 0) if exc[0] is not None else None
        if n is None:
            cap = 1 << 16
            names = (ctypes.c_char_p * cap)()
            ms = (ctypes.c_float * cap)()
            n = L.gdr_trace_collect(names, ms, cap)
            self.records = [(names[i].decode(), float(ms[i])) for i in range(min(n, cap))]
        return False
