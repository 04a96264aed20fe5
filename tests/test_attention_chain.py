"""Deterministic attention end to end on the library's kernels: the QK scores (fos_qk_scores),
the fixed-order softmax (fos_softmax_fwd, in place on the score rows) and the PV contraction
(fos_pv_out), chained in one 16-bit dtype, against the FP64 oracle's attention on the same Q, K
and V, within a bound derived from the chain's roundings; and the chain's bits for a batch entry
embedded in a larger batch.  ("[WS1][kernels] Add fixed-order joint-attention softmax for
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


def reference(q, k, v, scale):
    qn, kn, vn = np64(q), np64(k), np64(v)
    B, Hq, Sq, _ = qn.shape
    Skv = kn.shape[2]
    s = gemm.qk_scores(qn, kn, scale)
    absqk = gemm.qk_scores(np.abs(qn), np.abs(kn), 1.0)
    p, _ = oracle.softmax_fwd(s.reshape(-1, Skv), batch=B, heads=Hq, q_len=Sq)
    p = p.reshape(s.shape)
    return s, absqk, p, gemm.pv(p, vn), gemm.pv(p, np.abs(vn))


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
    u = UNIT_ROUNDOFF[name]
    ds = u * np.abs(s) + 2.0 ** -16 * abs(scale) * absqk
    coef = 1.25 * (u + 2.0 * ds.max(axis=-1, keepdims=True) + 2.0 ** -16)
    v_abs_sum = gemm.pv(np.ones_like(p), np.abs(np64(v)))  # sum_j |v_jd| per output
    bound = coef * pv_abs + SUBNORMAL_HALF_SPACING[name] * v_abs_sum + 1e-30
    err = np.abs(np64(out) - ref)
    worst = float((err / bound).max())
    assert worst <= 1.0, f"worst err/bound {worst:.3g}"


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
