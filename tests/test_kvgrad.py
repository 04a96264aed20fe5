"""The key / value gradient contraction (fos_grad_kv) against the FP64 oracle's attention
gradients (``oracle/gemm.py``: ``pv_backward`` gives dV = sum over the group's heads of P^T dO,
``qk_backward`` gives dK = scale * the same sum of dS^T Q), element by element, and its bitwise
invariance over the key's position and the batch entry; and the scale of the PV contraction
(dQ = scale * dS K).  ("Batch-invariant attention (standard softmax--cuda version)", GQA
backward: each dK / dV element accumulates the group's query heads and query positions in a
fixed order.)"""

import numpy as np
import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300 import _abi
from gpu_util import DTYPES, bits_equal, dev, np64, tol
from oracle import gemm

pytestmark = pytest.mark.gpu


def operands(B, Hq, Sq, Skv, D, dtype, seed, ld=None, prob_like=False):
    """`a` [B, Hq, Sq, Skv] in rows of `ld` elements (the padding is non-zero and must be
    ignored) and a dense `m` [B, Hq, Sq, D]."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    ld = ld or -(-Skv // 8) * 8
    buf = torch.full((B, Hq, Sq, ld), 5.0, dtype=dtype, device=dev())
    x = torch.rand(B, Hq, Sq, Skv, generator=g, device=dev())
    x = x.pow(4) * (5.0 / max(Skv, 1)) if prob_like else x * 2.0 - 1.0
    buf[..., :Skv] = x.to(dtype)
    m = torch.randn(B, Hq, Sq, D, generator=g, device=dev()).to(dtype)
    return buf[..., :Skv], m


def oracle_kv(a, m, hkv, scale):
    """scale * sum over each key head's query heads of a^T m, and the same of |a|^T |m|."""
    an, mn = np64(a), np64(m)
    vdummy = np.zeros((an.shape[0], hkv, an.shape[3], mn.shape[3]))
    _, ref = gemm.pv_backward(mn, an, vdummy)
    _, absd = gemm.pv_backward(np.abs(mn), np.abs(an), vdummy)
    return scale * ref, absd


def check(out, ref, absd, scale, out_name):
    ok, worst, idx = tol.check_scores(np64(out), ref, absd, scale, out_name)
    assert ok, f"worst err/bound {worst:.3g} at flat index {idx}"


@pytest.mark.parametrize("in_name", ["bfloat16", "float16"])
@pytest.mark.parametrize("out_name", ["float32", "bfloat16", "float16"])
@pytest.mark.parametrize("D", [64, 128])
def test_outputs_match_the_oracle(in_name, out_name, D):
    # two key heads of two query heads each; 200 query positions (four blocks of 64, the last
    # partial), 300 keys (three blocks of 128, the last partial), rows 304 elements apart
    B, Hq, Hkv, Sq, Skv = 2, 4, 2, 200, 300
    a, m = operands(B, Hq, Sq, Skv, D, DTYPES[in_name], seed=D + 5, ld=304)
    scale = 0.125
    out = fos.fos_grad_kv(a, m, Hkv, scale, out_dtype=DTYPES[out_name])
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    ref, absd = oracle_kv(a, m, Hkv, scale)
    check(out, ref, absd, scale, out_name)


@pytest.mark.parametrize("Hq,Hkv", [(3, 3), (4, 1), (8, 2)])
def test_head_groups_match_the_oracle(Hq, Hkv):
    # one query head per key head, all query heads on one key head, four per key head
    B, Sq, Skv, D = 1, 130, 260, 128
    a, m = operands(B, Hq, Sq, Skv, D, torch.bfloat16, seed=Hq * 10 + Hkv, prob_like=True)
    out = fos.fos_grad_kv(a, m, Hkv)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    ref, absd = oracle_kv(a, m, Hkv, 1.0)
    check(out, ref, absd, 1.0, "float32")


def test_qwen_image_shape_sampled():
    # 4 heads x 4,096 query positions, 4,352 keys, D = 128: dV from P and dO
    B, H, Sq, Skv, D = 1, 4, 4096, 4352, 128
    a, m = operands(B, H, Sq, Skv, D, torch.bfloat16, seed=9, prob_like=True)
    out = fos.fos_grad_kv(a, m, H)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    keys = np.unique(np.concatenate([[0, 127, 128, Skv - 1],
                                     np.random.default_rng(2).integers(0, Skv, 40)]))
    kt = torch.from_numpy(keys).to(dev())
    ref, absd = oracle_kv(a[..., kt], m, H, 1.0)
    check(out[:, :, kt], ref, absd, 1.0, "float32")


@pytest.mark.parametrize("out_name", ["float32", "bfloat16"])
def test_outputs_are_key_position_and_batch_invariant(out_name):
    # the same columns of a at other key positions (shifted by 37 keys) and the same group in
    # another batch entry of a bigger batch: the same bits
    odt = DTYPES[out_name]
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 150, 300, 128
    a, m = operands(B, Hq, Sq, Skv, D, torch.bfloat16, seed=31)
    ref = fos.fos_grad_kv(a, m, Hkv, 0.25, out_dtype=odt)
    a2, _ = operands(B, Hq, Sq, Skv + 37, D, torch.bfloat16, seed=32)
    a2[..., 37:] = a
    out = fos.fos_grad_kv(a2, m, Hkv, 0.25, out_dtype=odt)
    assert bits_equal(out[:, :, 37:].contiguous(), ref)
    a3, m3 = operands(3, Hq, Sq, Skv, D, torch.bfloat16, seed=33)
    a3[2], m3[2] = a[0], m[0]
    out = fos.fos_grad_kv(a3, m3, Hkv, 0.25, out_dtype=odt)
    assert bits_equal(out[2:3].contiguous(), ref)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0


def test_tiny_and_empty_problems():
    a, m = operands(1, 1, 1, 1, 64, torch.bfloat16, seed=3)
    ref, absd = oracle_kv(a, m, 1, 1.0)
    check(fos.fos_grad_kv(a, m, 1), ref, absd, 1.0, "float32")
    a, m = operands(1, 2, 17, 5, 128, torch.float16, seed=4)
    ref, absd = oracle_kv(a, m, 1, 0.5)
    check(fos.fos_grad_kv(a, m, 1, 0.5, out_dtype=torch.float16), ref, absd, 0.5, "float16")
    # no query position: a sum over nothing, +0 everywhere
    a, m = operands(1, 2, 0, 40, 64, torch.bfloat16, seed=5)
    out = fos.fos_grad_kv(a, m, 2, out=torch.full((1, 2, 40, 64), 3.0, device=dev()))
    torch.cuda.synchronize()
    assert torch.all(out == 0) and not torch.any(torch.signbit(out))
    # no key: nothing to write
    a, m = operands(1, 2, 8, 0, 64, torch.bfloat16, seed=6)
    assert fos.fos_grad_kv(a, m, 2).numel() == 0
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0


def test_refusals():
    a, m = operands(1, 2, 8, 16, 96, torch.bfloat16, seed=7)
    with pytest.raises(fos.FosError) as e:  # head dimension 96
        fos.fos_grad_kv(a, m, 1)
    assert e.value.status == _abi.FOS_ERR_UNSUPPORTED
    a, m = operands(1, 2, 8, 16, 64, torch.bfloat16, seed=8)
    with pytest.raises(fos.FosError) as e:  # a zero scale
        fos.fos_grad_kv(a, m, 1, 0.0)
    assert e.value.status == _abi.FOS_ERR_INVALID
    with pytest.raises(fos.FosError) as e:
        fos.fos_pv_out(a, torch.zeros(1, 1, 16, 64, dtype=torch.bfloat16, device=dev()),
                       scale=float("inf"))
    assert e.value.status == _abi.FOS_ERR_INVALID
    with pytest.raises(ValueError):  # 3 key heads do not divide 2 query heads
        fos.fos_grad_kv(a, m, 3)


@pytest.mark.parametrize("out_name", ["float32", "bfloat16"])
def test_pv_scale(out_name):
    # dQ = scale * dS K through fos_pv_out: the oracle's qk_backward; and the scale is one
    # float32 multiply of the sum (a scale of 2 is exact, so it doubles the float32 outputs)
    B, Hq, Hkv, Sq, Skv, D = 2, 4, 2, 140, 270, 128
    a, _ = operands(B, Hq, Sq, Skv, D, torch.bfloat16, seed=61, ld=280)
    g = torch.Generator(device="cuda").manual_seed(62)
    kk = torch.randn(B, Hkv, Skv, D, generator=g, device=dev()).to(torch.bfloat16)
    scale = 0.0884
    out = fos.fos_pv_out(a, kk, scale=scale, out_dtype=DTYPES[out_name])
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    an, kn = np64(a), np64(kk)
    qdummy = np.zeros((B, Hq, Sq, D))
    ref, _ = gemm.qk_backward(an, qdummy, kn, scale)
    absd, _ = gemm.qk_backward(np.abs(an), qdummy, np.abs(kn), 1.0)
    check(out, ref, absd, scale, out_name)
    assert bits_equal(fos.fos_pv_out(a, kk, scale=2.0), 2.0 * fos.fos_pv_out(a, kk))
