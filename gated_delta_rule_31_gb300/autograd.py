"""torch.autograd integration of the chunked gated delta rule.

``gated_delta_rule(q, k, v, g, beta, h0=None, scale=None, use_qk_l2norm=True)`` returns
``(o, ht)`` and is differentiable in q, k, v, g, beta and h0. Its forward runs
``gdr_fwd_chunked_states`` when any input needs a gradient (the chunk-start states are
kept for the backward, 32 KB per chunk and value head; ``gdr_fwd_chunked_saved`` with
``keep_operators=True``) and ``gdr_fwd_chunked`` otherwise; its backward runs the matching
``gdr_bwd_chunked_states`` / ``gdr_bwd_chunked_saved``. With ``use_qk_l2norm`` the kernels own the
q/k L2 normalisation (eps 1e-6), so no normalised copy of q or k is ever materialised or
kept for the backward — the point of "fold q/k L2-norm into the gated_delta_rule kernel"
(Megatron-LM PR #5396, "What" / "Why"). The VJP is the chunked backward of "Adding VJP for
gated delta net" (MLX PR #4565).

Every problem the C ABI accepts runs the chunked forward and the chunked VJP (scalar or
per-channel gate, Dk and Dv in {32, 64, 128}): bf16 q/k/v on the tensor cores, fp32 q/k/v on
the CUDA-core fp32 kernels of the same chunk algebra (fp32 chunk-start states, 64 KB per
chunk and value head at D = 128). The only torch operations here are argument marshalling: a
zero ``do`` when the output is unused, contiguity, and casting the fp32 gradients of q/k/v to
their dtype.
"""
from __future__ import annotations

import torch

from . import bwd_chunked, fwd_chunked

__all__ = ["gated_delta_rule", "GatedDeltaRuleFunction"]


class GatedDeltaRuleFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, g, beta, h0, scale, use_qk_l2norm, keep_operators):
        ctx.scale, ctx.norm, ctx.has_h0 = scale, bool(use_qk_l2norm), h0 is not None
        ctx.keep_operators = bool(keep_operators)
        kw = dict(scale=scale, use_qk_l2norm=use_qk_l2norm)
        if any(ctx.needs_input_grad[:6]):
            o, ht, kept = fwd_chunked(q, k, v, g, beta, h0, save_states=not ctx.keep_operators,
                                      save_all=ctx.keep_operators, **kw)
            ctx.save_for_backward(q, k, v, g, beta, kept)
        else:
            o, ht = fwd_chunked(q, k, v, g, beta, h0, **kw)
        return o, ht

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(ctx, do, dht):
        q, k, v, g, beta, kept = ctx.saved_tensors
        do = torch.zeros_like(v) if do is None else do.to(v.dtype).contiguous()
        dht = None if dht is None else dht.to(torch.float32).contiguous()
        kw = dict(scale=ctx.scale, use_qk_l2norm=ctx.norm)
        handoff = {"saved": kept} if ctx.keep_operators else {"states": kept}
        gr = bwd_chunked(q, k, v, g, beta, None, do, dht, **handoff, **kw)
        return (gr["dq"].to(q.dtype), gr["dk"].to(k.dtype), gr["dv"].to(v.dtype), gr["dg"], gr["dbeta"],
                gr["dh0"] if ctx.has_h0 else None, None, None, None)


def gated_delta_rule(q, k, v, g, beta, h0=None, scale=None, use_qk_l2norm=True, keep_operators=False):
    """Differentiable chunked gated delta rule: (o [B,T,Hv,Dv] in v's dtype, ht [B,Hv,Dv,Dk] fp32).

    q, k [B,T,Hk,Dk] and v [B,T,Hv,Dv] bf16 or fp32; g [B,T,Hv] (or [B,T,Hv,Dk] per key
    channel) fp32 log-decay; beta [B,T,Hv] fp32; h0 [B,Hv,Dv,Dk] fp32 or None (zero). scale
    defaults to Dk^-1/2. The forward keeps the chunk-start states (bf16: 32 KB per chunk and
    value head) for the backward; with keep_operators=True it keeps the chunk operators too
    (bf16: 144 KB per chunk and value head) and the backward then skips all recomputation.
    Both give bitwise the same results."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    return GatedDeltaRuleFunction.apply(q, k, v, g, beta, h0, float(scale), bool(use_qk_l2norm),
                                        bool(keep_operators))
