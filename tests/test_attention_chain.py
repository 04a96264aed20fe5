"""Deterministic attention end to end on the library's kernels: the QK scores (fos_qk_scores),
the fixed-order softmax (fos_softmax_fwd, in place on the score rows) and the PV contraction
(fos_pv_out), chained in one 16-bit dtype, against the FP64 oracle's attention on the same Q, K
and V, within a bound derived from the chain's roundings; the gradients dQ, dK, dV through the
same kernels, the softmax backward and the key / value gradient contraction (fos_grad_kv)
against the oracle's; and the chain's bits for a batch entry embedded in a larger batch.  ("[WS1][kernels] Add fixed-order joint-attention softmax for
Qwen-Image", Summary: the QK GEMM -> softmax -> AV GEMM chain; "Batch-invariant attention
(standard softmax--cuda version)", Fixed Reduction Contract.)

The bound, per output (b, h, i, d), with u the unit roundoff of the 16-bit dtype (2^-8 bf16,
2^-11 fp16) and P, s the FP64 probabilities and scores of row (b, h, i):
  * the scores are rounded once to the dtype after a float32 dot product, so each is off by at
    most ds = u |s_j| + 2^-16 |scale| sum_d |q_d k_jd| (the QK check's float32 term);
  * a perturbation ds of the scores moves P_j by at most P_j (exp(2 max_j ds_j) - 1), about
    2 P_j max_j ds_j;
  * the softmax's float32 arithmetic and its one rounding to the dtype add u P_j (plus far less);
  * PV accumulates in float32 and writes float32: 2^-16 sum_j |P_j v_jd| (the PV check's term).
So |out - ref| <= (u + 2 max_j ds_j + 2^-16) sum_j P_j |v_jd|, taken here with a factor 1.25
for the second-order terms, plus, for fp16, half its subnormal spacing (2^-25) times sum_j
|v_jd| for probabilities that round into the subnormal range, where the error is absolute.
"""

import math

import numpy as np
import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
import oracle
from gpu_util import DTYPES, bits_equal, dev, np64
from oracle import gemm

pytestmark = pytest.mark.gpu

UNIT_ROUNDOFF = {"bfloat16": 2.0 ** -8, "float16": 2.0 ** -11}
SUBNORMAL_HALF_SPACING = {"bfloat16": 2.0 ** -134, "float16": 2.0 ** -25}


def inputs(B, Hq, Hkv, Sq, Skv, D, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(B, Hq, Sq, D, generator=g, device=dev()).to(dtype)
    k = torch.randn(B, Hkv, Skv, D, generator=g, device=dev()).to(dtype)
    v = torch.randn(B, Hkv, Skv, D, generator=g, device=dev()).to(dtype)
    return q, k, v


def chain(q, k, v, scale):
    """QK -> softmax (in place on the score rows) -> PV, every step in the library."""
    B, Hq, Sq, _ = q.shape
    s = fos.fos_qk_scores(q, k, scale, out_dtype=q.dtype)  # rows padded to 16 bytes
    fos.fos_softmax_fwd(s, s, batch=B, heads=Hq, q_len=Sq)
    return fos.fos_pv_out(s, v)


def reference(q, k, v, scale, **masks):
    qn, kn, vn = np64(q), np64(k), np64(v)
    B, Hq, Sq, _ = qn.shape
    Skv = kn.shape[2]
    s = gemm.qk_scores(qn, kn, scale)
    absqk = gemm.qk_scores(np.abs(qn), np.abs(kn), 1.0)
    p, _ = oracle.softmax_fwd(s.reshape(-1, Skv), batch=B, heads=Hq, q_len=Sq, **masks)
    p = p.reshape(s.shape)
    return s, absqk, p, gemm.pv(p, vn), gemm.pv(p, np.abs(vn))


def forward_bound(name, s, absqk, p, pv_abs, vn, scale):
    """The forward's bound (module docstring) per output."""
    u = UNIT_ROUNDOFF[name]
    ds = u * np.abs(s) + 2.0 ** -16 * abs(scale) * absqk
    coef = 1.25 * (u + 2.0 * ds.max(axis=-1, keepdims=True) + 2.0 ** -16)
    v_abs_sum = gemm.pv(np.ones_like(p), np.abs(vn))  # sum_j |v_jd| per output
    return coef * pv_abs + SUBNORMAL_HALF_SPACING[name] * v_abs_sum + 1e-30


def gradient_references(name, q, k, v, dout, scale, **masks):
    """The oracle's dQ, dK, dV and the bounds of the chain's roundings (see the gradient
    test): (reference, bound) per gradient."""
    B, Hq, Sq, _ = q.shape
    Skv = k.shape[2]
    qn, kn, vn, don = np64(q), np64(k), np64(v), np64(dout)
    s, absqk, p, _, _ = reference(q, k, v, scale, **masks)
    dp, dv_ref = gemm.pv_backward(don, p, vn)
    ds, delta = oracle.softmax_bwd(p.reshape(-1, Skv), dp.reshape(-1, Skv), batch=B, heads=Hq,
                                   q_len=Sq, **masks)
    ds, delta = ds.reshape(p.shape), delta.reshape(p.shape[:-1] + (1,))
    dq_ref, dk_ref = gemm.qk_backward(ds, qn, kn, scale)
    u = UNIT_ROUNDOFF[name]
    sub = SUBNORMAL_HALF_SPACING[name]
    eps = 1.25 * (u + 2.0 * (u * np.abs(s) + 2.0 ** -16 * scale * absqk).max(-1, keepdims=True))
    dp_abs = gemm.pv_backward(np.abs(don), p, np.abs(vn))[0]  # sum_d |dO_d v_jd|
    e_dp = u * np.abs(dp) + 2.0 ** -16 * dp_abs
    e_p = eps * p + sub
    e_delta = (e_p * np.abs(dp) + p * e_dp).sum(-1, keepdims=True) + \
        2.0 ** -20 * (p * np.abs(dp)).sum(-1, keepdims=True)
    e_ds = e_p * np.abs(dp - delta) + p * (e_dp + e_delta) + u * np.abs(ds) + sub
    # dQ = scale dS K, dK = scale sum_h dS^T Q: the error of dS carried through, plus the
    # float32 sums; dV = sum_h P^T dO: the error of P carried through, plus the float32 sum
    bq, bk = gemm.qk_backward(e_ds, np.abs(qn), np.abs(kn), scale)
    aq, ak = gemm.qk_backward(np.abs(ds), np.abs(qn), np.abs(kn), scale)
    _, bv = gemm.pv_backward(np.abs(don), e_p + 2.0 ** -16 * p, np.zeros_like(kn))
    return ((dq_ref, 1.5 * (bq + 2.0 ** -16 * aq) + 1e-30),
            (dk_ref, 1.5 * (bk + 2.0 ** -16 * ak) + 1e-30),
            (dv_ref, 1.5 * bv + 1e-30))


def assert_within(got, ref, bound, what):
    worst = float((np.abs(np64(got) - ref) / bound).max())
    assert worst <= 1.0, f"{what}: worst err/bound {worst:.3g}"


@pytest.mark.parametrize("name", ["bfloat16", "float16"])
@pytest.mark.parametrize("D", [64, 128])
def test_attention_matches_the_oracle(name, D):
    # grouped heads, two query tiles (the second ragged), 300 keys (ragged key tiles and blocks)
    B, Hq, Hkv, Sq, Skv = 2, 4, 2, 200, 300
    q, k, v = inputs(B, Hq, Hkv, Sq, Skv, D, DTYPES[name], seed=D + 41)
    scale = 1.0 / math.sqrt(D)
    out = chain(q, k, v, scale)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    s, absqk, p, ref, pv_abs = reference(q, k, v, scale)
    assert_within(out, ref, forward_bound(name, s, absqk, p, pv_abs, np64(v), scale), "out")


def test_attention_bits_do_not_depend_on_the_batch():
    # the same (q, k, v) of one batch entry, alone and as entry 1 of 3 with other data around it
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 150, 260, 128
    q, k, v = inputs(B, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=51)
    ref = chain(q, k, v, 0.09)
    q3, k3, v3 = inputs(3, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=52)
    q3[1], k3[1], v3[1] = q[0], k[0], v[0]
    out = chain(q3, k3, v3, 0.09)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    assert bits_equal(out[1:2].contiguous(), ref)


def chain_backward(q, k, v, dout, scale):
    """Forward as above, then dP = dO V^T (QK kernel), dS = P (dP - delta) in place of dP
    (softmax backward), dQ = scale dS K (PV kernel), dK = scale dS^T Q and dV = P^T dO
    (key / value gradient kernel): every step in the library."""
    B, Hq, Sq, _ = q.shape
    Hkv = k.shape[1]
    s = fos.fos_qk_scores(q, k, scale, out_dtype=q.dtype)
    fos.fos_softmax_fwd(s, s, batch=B, heads=Hq, q_len=Sq)  # P in place of the scores
    dp = fos.fos_qk_scores(dout, v, 1.0, out_dtype=q.dtype)
    fos.fos_softmax_bwd(s, dp, dp, batch=B, heads=Hq, q_len=Sq)  # dS in place of dP
    dq = fos.fos_pv_out(dp, k, scale=scale)
    dk = fos.fos_grad_kv(dp, q, Hkv, scale)
    dv = fos.fos_grad_kv(s, dout, Hkv)
    return dq, dk, dv


@pytest.mark.parametrize("name", ["bfloat16", "float16"])
@pytest.mark.parametrize("Hkv", [1, 2, 4])
def test_attention_gradients_match_the_oracle(name, Hkv):
    # The oracle's FP64 gradients of the same attention (its softmax VJP and the contractions'
    # gradients), against a bound carried through the chain's roundings (first order, with a
    # factor 1.5): P as in the forward bound (relative eps_i per row); dP rounded once after a
    # float32 dot product (u |dP| + 2^-16 sum |dO v|); delta summed in float32 from both; dS
    # rounded once; then the float32 contractions of dS (2^-16 of their absolute sums).
    B, Hq, Sq, Skv, D = 2, 4, 200, 300, 128
    dt = DTYPES[name]
    q, k, v = inputs(B, Hq, Hkv, Sq, Skv, D, dt, seed=Hkv + 71)
    g = torch.Generator(device="cuda").manual_seed(Hkv + 72)
    dout = torch.randn(B, Hq, Sq, D, generator=g, device=dev()).to(dt)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = chain_backward(q, k, v, dout, scale)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0

    for got, (ref, bound), what in zip((dq, dk, dv),
                                       gradient_references(name, q, k, v, dout, scale),
                                       ("dQ", "dK", "dV")):
        assert_within(got, ref, bound, what)


def test_attention_gradient_bits_do_not_depend_on_the_batch():
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 150, 260, 128
    q, k, v = inputs(B, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=81)
    g = torch.Generator(device="cuda").manual_seed(82)
    dout = torch.randn(B, Hq, Sq, D, generator=g, device=dev()).to(torch.bfloat16)
    ref = chain_backward(q, k, v, dout, 0.09)
    q3, k3, v3 = inputs(3, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=83)
    d3 = torch.randn(3, Hq, Sq, D, generator=g, device=dev()).to(torch.bfloat16)
    q3[1], k3[1], v3[1], d3[1] = q[0], k[0], v[0], dout[0]
    out = chain_backward(q3, k3, v3, d3, 0.09)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    for a, b in zip(out, ref):
        assert bits_equal(a[1:2].contiguous(), b)


@pytest.mark.parametrize("name", ["bfloat16", "float16"])
def test_masked_attention_and_its_gradients_match_the_oracle(name):
    # fixed_order_attention with the causal bound of a chunk (200 queries against 300 keys: key
    # j of query i valid iff j <= 100 + i) and valid lengths (300 and 230 keys per batch entry):
    # output and dQ, dK, dV against the oracle with the same masks, within the bounds above
    B, Hq, Hkv, Sq, Skv, D = 2, 4, 2, 200, 300, 64
    dt = DTYPES[name]
    q, k, v = inputs(B, Hq, Hkv, Sq, Skv, D, dt, seed=91)
    g = torch.Generator(device="cuda").manual_seed(92)
    dout = torch.randn(B, Hq, Sq, D, generator=g, device=dev()).to(dt)
    kv = torch.tensor([300, 230], dtype=torch.int32, device=dev())
    scale = D ** -0.5
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    out = fos.fixed_order_attention(qa, ka, va, scale, causal=True, kv_valid_len=kv)
    out.backward(dout)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    masks = dict(causal=True, kv_valid_len=kv.cpu().numpy())
    s, absqk, p, ref, pv_abs = reference(q, k, v, scale, **masks)
    # the output is in the input dtype: one more rounding, u |ref|
    bound = forward_bound(name, s, absqk, p, pv_abs, np64(v), scale) + \
        UNIT_ROUNDOFF[name] * np.abs(ref)
    assert_within(out.detach(), ref, bound, "out")
    for got, (ref_g, bound_g), what in zip((qa.grad, ka.grad, va.grad),
                                           gradient_references(name, q, k, v, dout, scale,
                                                               **masks),
                                           ("dQ", "dK", "dV")):
        assert_within(got, ref_g, bound_g + UNIT_ROUNDOFF[name] * np.abs(ref_g), what)


def test_chunked_prefill_and_decode_give_the_full_prefill_bits():
    # The pages' prefill / decode contract: one causal condition (key j of query i valid iff
    # j <= kv_len - q_len + i) for every mode.  Queries i0 .. i1 - 1 run against the first i1
    # keys (a prefill chunk; one query for decode) give the bits of the same rows of the full
    # causal prefill: a row's valid keys, tiles and key steps are the same, and the keys a
    # longer cache adds enter as exact zeros.
    B, Hq, Hkv, S, D = 1, 4, 2, 300, 128
    q, k, v = inputs(B, Hq, Hkv, S, S, D, torch.bfloat16, seed=95)
    full = fos.fixed_order_attention(q, k, v, causal=True)
    for i0, i1 in ((0, 100), (100, 237), (237, 300), (150, 151), (299, 300)):
        part = fos.fixed_order_attention(q[:, :, i0:i1], k[:, :, :i1], v[:, :, :i1],
                                         causal=True)
        assert bits_equal(part, full[:, :, i0:i1].contiguous()), (i0, i1)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
