"""``torch.autograd`` over the library's kernels: the fixed-order softmax as a differentiable op.

``fixed_order_softmax(scores, ...)`` returns ``(P, LSE)``.  Its backward maps dP to dScores
with ``fos_softmax_bwd``: the VJP on the stored P, dScores_j = P_j * (dP_j - delta).  When the
per-head sink needs a gradient, ``fos_sink_grad`` gives it: d_sink[h] is minus the sum over the
head's rows of exp(sink_h - LSE_r) * delta_r, reduced in a fixed order ("[ROCm] Jax Add softmax
sink (learnable off-by-one) support", Description).  LSE is returned for callers that keep it
(e.g. to recompute P later); it is not differentiable here.

Argument marshalling only: every step runs in ``libfos_softmax.so``.  The masks (causal bound,
valid lengths, key mask) and the geometry mean what they mean for ``fos_softmax_fwd``.
"""

from __future__ import annotations

import torch
from torch.autograd.function import once_differentiable

from . import binding


class FixedOrderSoftmax(torch.autograd.Function):
    """P, LSE = softmax of each row of ``scores`` (see ``fixed_order_softmax``)."""

    @staticmethod
    def forward(ctx, scores, sink, batch, heads, q_len, causal, kv_valid_len, key_mask):
        p, lse = binding.fos_softmax_fwd(scores, batch=batch, heads=heads, q_len=q_len,
                                         causal=causal, kv_valid_len=kv_valid_len,
                                         key_mask=key_mask, sink=sink)
        ctx.save_for_backward(p, lse, sink, kv_valid_len, key_mask)
        ctx.geo = (batch, heads, q_len, causal)
        ctx.mark_non_differentiable(lse)
        return p, lse

    @staticmethod
    @once_differentiable
    def backward(ctx, dp, _dlse):
        p, lse, sink, kv_valid_len, key_mask = ctx.saved_tensors
        batch, heads, q_len, causal = ctx.geo
        if dp.dtype != p.dtype or dp.stride() != p.stride():
            # the kernels take P and dP in one row layout and dtype
            dp = torch.empty_strided(p.shape, p.stride(), dtype=p.dtype, device=p.device).copy_(dp)
        need_x, need_sink = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        ds, delta = binding.fos_softmax_bwd(p, dp, batch=batch, heads=heads, q_len=q_len,
                                            causal=causal, kv_valid_len=kv_valid_len,
                                            key_mask=key_mask, want_delta=True)
        d_sink = None
        if sink is not None and need_sink:
            d_sink = binding.fos_sink_grad(lse, delta, sink, batch=batch, heads=heads,
                                           q_len=q_len)
        return (ds if need_x else None), d_sink, None, None, None, None, None, None


def fixed_order_softmax(scores, *, batch=None, heads=None, q_len=None, causal=False,
                        kv_valid_len=None, key_mask=None, sink=None):
    """Differentiable fixed-order softmax over the last dimension of ``scores``.

    ``scores``: CUDA tensor (fp32, bf16 or fp16) whose rows, ordered [batch][heads][q_len],
    hold the keys with stride 1 (2-D ``[rows, keys]`` or 4-D ``[batch, heads, q_len, keys]``).
    ``sink``: optional fp32 ``[heads]`` logit per head (it may require grad).  Returns
    ``(P, LSE)``: P like ``scores``, LSE fp32 per row (not differentiable).
    """
    if not scores.is_cuda:
        raise ValueError("scores must be a CUDA tensor")
    _, _, _, batch, heads, q_len = binding._geometry(scores, batch, heads, q_len)
    return FixedOrderSoftmax.apply(scores, sink, batch, heads, q_len, bool(causal),
                                   kv_valid_len, key_mask)
