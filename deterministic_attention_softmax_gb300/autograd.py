"""``torch.autograd`` over the library's kernels: the fixed-order softmax, and attention built
on it, as differentiable ops.

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


class FixedOrderAttention(torch.autograd.Function):
    """out = softmax(scale Q K^T) V per (batch, query head) (see ``fixed_order_attention``)."""

    @staticmethod
    def forward(ctx, q, k, v, scale, causal, kv_valid_len):
        B, Hq, Sq, _ = q.shape
        masks = dict(batch=B, heads=Hq, q_len=Sq, causal=causal, kv_valid_len=kv_valid_len)
        s = binding.fos_qk_scores(q, k, scale, out_dtype=q.dtype)
        binding.fos_softmax_fwd(s, s, **masks)  # P in place of the scores; masked keys +0
        out = binding.fos_pv_out(s, v, out_dtype=q.dtype)
        ctx.save_for_backward(q, k, v, s, kv_valid_len)
        ctx.scale, ctx.causal = scale, causal
        return out

    @staticmethod
    @once_differentiable
    def backward(ctx, dout):
        q, k, v, p, kv_valid_len = ctx.saved_tensors
        B, Hq, Sq, _ = q.shape
        masks = dict(batch=B, heads=Hq, q_len=Sq, causal=ctx.causal, kv_valid_len=kv_valid_len)
        if dout.dtype != q.dtype or not dout.is_contiguous():
            dout = dout.to(q.dtype).contiguous()  # the kernels take one dense 16-bit layout
        dp = binding.fos_qk_scores(dout, v, 1.0, out_dtype=q.dtype)  # dP = dO V^T
        binding.fos_softmax_bwd(p, dp, dp, want_delta=False, **masks)  # dS in place of dP
        need_q, need_k, need_v = ctx.needs_input_grad[:3]
        dq = binding.fos_pv_out(dp, k, scale=ctx.scale, out_dtype=q.dtype) if need_q else None
        dk = binding.fos_grad_kv(dp, q, k.shape[1], ctx.scale, out_dtype=k.dtype) \
            if need_k else None
        dv = binding.fos_grad_kv(p, dout, k.shape[1], 1.0, out_dtype=v.dtype) if need_v else None
        return dq, dk, dv, None, None, None


def fixed_order_attention(q, k, v, scale=None, *, causal=False, kv_valid_len=None):
    """Differentiable attention on the library's kernels: scores = scale Q K^T (``fos_qk_scores``),
    P = the fixed-order softmax of each score row (``fos_softmax_fwd``, in place), out = P V
    (``fos_pv_out``); the backward is dP = dO V^T, dS = the softmax VJP, dQ = scale dS K,
    dK = scale dS^T Q and dV = P^T dO (``fos_grad_kv``), the group's query heads and positions
    in a fixed order ("Batch-invariant attention (standard softmax--cuda version)", Fixed
    Reduction Contract and GQA backward).

    ``q``: CUDA ``[batch, q_heads, q_len, D]``, ``k`` and ``v``: ``[batch, kv_heads, kv_len,
    D]``, all dense bf16 or all dense fp16, D = 64 or 128, q_heads a multiple of kv_heads.
    ``scale`` defaults to 1 / sqrt(D).  ``causal``: key j of query i is valid iff
    j <= kv_len - q_len + i ("Batch-invariant attention", Prefill / Decode / KV-cache Contract:
    one condition for full prefill, chunked prefill and decode); ``kv_valid_len``: optional
    int32 ``[batch]``, keys j >= kv_valid_len[b] masked.  The softmax applies the masks (masked
    P and dS are +0), so the contractions need none.  The output and the gradients have the
    inputs' dtype, each rounded once from float32.
    """
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k and v must be CUDA tensors")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4 or k.shape != v.shape:
        raise ValueError("q must be [B, Hq, Sq, D], k and v [B, Hkv, Skv, D]")
    scale = q.shape[-1] ** -0.5 if scale is None else float(scale)
    return FixedOrderAttention.apply(q.contiguous(), k.contiguous(), v.contiguous(), scale,
                                     bool(causal), kv_valid_len)
