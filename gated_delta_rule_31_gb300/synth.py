"""Seeded synthetic inputs for the gated delta rule workloads.

This module only draws random numbers; it holds none of the method's arithmetic, so
both the CUDA path's tests and the oracle can consume the same inputs. Draws happen
on the CPU with ``torch.Generator().manual_seed(seed)`` in the order
q, k, v, g_raw, beta_raw, h0, do, dht, in fp32, and are then cast to the workload
dtype (the oracle consumes the cast values, so input rounding is not an error).

Distributions (the workloads of the gated delta rule pages' benchmark grid):
q, k, v ~ N(0, 1); g = -softplus(N(0, 1)) (log-decay, a = exp(g)); beta =
sigmoid(N(0, 1)); h0 ~ N(0, 0.02); do ~ N(0, 1); dht ~ N(0, 0.01). ``gate_scale``
multiplies g (e.g. 0.01 for a mild-decay case that keeps long-range state alive).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Shape:
    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int


def make_inputs(shape: Shape, dtype=torch.bfloat16, seed: int = 0, gate: str = "scalar",
                h0_std: float | None = 0.02, grads: bool = False, do_std: float = 1.0,
                dht_std: float | None = 0.01, gate_scale: float = 1.0, qk_std: float = 1.0):
    """Return a dict of CPU tensors: q,k [B,T,Hk,Dk] and v [B,T,Hv,Dv] in ``dtype``;
    g [B,T,Hv] (or [B,T,Hv,Dk] for gate='channel'), beta [B,T,Hv], h0 [B,Hv,Dv,Dk]
    in fp32 (None if h0_std is None); with grads=True also do (``dtype``) and dht
    (fp32, None if dht_std is None)."""
    s = shape
    gen = torch.Generator().manual_seed(seed)
    f32 = torch.float32

    def randn(*sz):
        return torch.randn(*sz, generator=gen, dtype=f32)

    q = (randn(s.B, s.T, s.Hk, s.Dk) * qk_std).to(dtype)
    k = (randn(s.B, s.T, s.Hk, s.Dk) * qk_std).to(dtype)
    v = randn(s.B, s.T, s.Hv, s.Dv).to(dtype)
    gshape = (s.B, s.T, s.Hv, s.Dk) if gate == "channel" else (s.B, s.T, s.Hv)
    g = (-torch.nn.functional.softplus(randn(*gshape))) * gate_scale
    beta = torch.sigmoid(randn(s.B, s.T, s.Hv))
    h0 = randn(s.B, s.Hv, s.Dv, s.Dk) * h0_std if h0_std is not None else None
    out = dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous(), h0=h0)
    if grads:
        out["do"] = (randn(s.B, s.T, s.Hv, s.Dv) * do_std).to(dtype)
        out["dht"] = randn(s.B, s.Hv, s.Dv, s.Dk) * dht_std if dht_std is not None else None
    return out


def make_decode_inputs(B: int, Hk: int, Hv: int, Dk: int, Dv: int, steps: int, seed: int = 0,
                       gate: str = "channel", dtype=torch.float32, state_std: float = 0.02):
    """Inputs for ``steps`` consecutive single-token decode steps, drawn up front:
    q,k [steps,B,Hk,Dk]; v [steps,B,Hv,Dv]; g [steps,B,Hv,Dk] (channel) or
    [steps,B,Hv]; beta [steps,B,Hv]; state0 [B,Hv,Dv,Dk] fp32."""
    gen = torch.Generator().manual_seed(seed)
    f32 = torch.float32

    def randn(*sz):
        return torch.randn(*sz, generator=gen, dtype=f32)

    q = randn(steps, B, Hk, Dk).to(dtype)
    k = randn(steps, B, Hk, Dk).to(dtype)
    v = randn(steps, B, Hv, Dv).to(dtype)
    gshape = (steps, B, Hv, Dk) if gate == "channel" else (steps, B, Hv)
    g = -torch.nn.functional.softplus(randn(*gshape))
    beta = torch.sigmoid(randn(steps, B, Hv))
    state0 = randn(B, Hv, Dv, Dk) * state_std
    return dict(q=q, k=k, v=v, g=g.contiguous(), beta=beta.contiguous(), state0=state0)


# The five workloads (seed = 1000 + index; the VJP sweep uses 1200 + point index).
TINY_SEQ = Shape(1, 64, 2, 2, 32, 32)            # fp32, h0 = 0, sequential forward
PREFILL = Shape(1, 4096, 16, 32, 128, 128)       # bf16 chunked forward, h0 ~ N(0, 0.02)
VJP_SWEEP = [Shape(b, t, 16, 32, 128, 128) for b in (1, 4, 8) for t in (8, 64, 512, 4096)]
DECODE = dict(B=32, Hk=16, Hv=32, Dk=128, Dv=128, steps=256)   # fp32, channel gate
LONG_TRAIN = Shape(1, 32768, 16, 32, 128, 128)   # bf16 forward + VJP, h0 = 0, dht = 0
