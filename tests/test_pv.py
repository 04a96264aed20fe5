"""The fixed-order PV contraction on the tensor cores (fos_pv_out) against the FP64 oracle
(``oracle/gemm.py:pv``), element by element, and its bitwise invariance: an output depends only
on its probability row and the value rows (and the key count), so it must have the same bits
wherever its row sits (query block position, batch entry, neighbouring heads).  ("Batch-invariant
attention (standard softmax--cuda version)", Fixed Reduction Contract; "[WS1][kernels] Add
fixed-order joint-attention softmax for Qwen-Image", Summary: the softmax's P feeds the AV
GEMM.)"""

import numpy as np
import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300 import _abi
from gpu_util import DTYPES, bits_equal, dev, np64, tol
from oracle import gemm

pytestmark = pytest.mark.gpu


def pv_inputs(B, Hq, Hkv, Sq, Skv, D, dtype, seed, ld=None):
    """Probability-shaped P (non-negative, rows summing to about 1) in rows of `ld` elements,
    and N(0, 1) values."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    ld = ld or -(-Skv // 8) * 8
    u = torch.rand(B, Hq, Sq, Skv, generator=g, device=dev())
    p = (u.pow(4) * (5.0 / Skv))
    buf = torch.full((B, Hq, Sq, ld), 3.0, dtype=dtype, device=dev())  # padding must be ignored
    buf[..., :Skv] = p.to(dtype)
    v = torch.randn(B, Hkv, Skv, D, generator=g, device=dev()).to(dtype)
    return buf[..., :Skv], v


def check_against_oracle(p, v, out, out_name):
    pn, vn = np64(p), np64(v)
    ref = gemm.pv(pn, vn)
    absd = gemm.pv(np.abs(pn), np.abs(vn))  # sum_j |p_j v_jd| per output
    ok, worst, idx = tol.check_pv(np64(out), ref, absd, out_name)
    assert ok, f"out: worst err/bound {worst:.3g} at flat index {idx}"


@pytest.mark.parametrize("in_name", ["bfloat16", "float16"])
@pytest.mark.parametrize("out_name", ["float32", "bfloat16", "float16"])
@pytest.mark.parametrize("D", [64, 128])
def test_outputs_match_the_oracle(in_name, out_name, D):
    # two query blocks (the second ragged), 300 keys = 5 blocks of 64 (the last partial), grouped
    # heads, P rows 304 elements apart with non-zero padding past the keys
    B, Hq, Hkv, Sq, Skv = 2, 4, 2, 200, 300
    p, v = pv_inputs(B, Hq, Hkv, Sq, Skv, D, DTYPES[in_name], seed=D + 3, ld=304)
    out = fos.fos_pv_out(p, v, out_dtype=DTYPES[out_name])
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    check_against_oracle(p, v, out, out_name)


def test_qwen_image_shape_sampled():
    # the benchmark's shape: 16,384 query rows (4 heads x 4,096) against 4,352 keys, D = 128
    B, H, Sq, Skv, D = 1, 4, 4096, 4352, 128
    p, v = pv_inputs(B, H, H, Sq, Skv, D, torch.bfloat16, seed=4)
    out = fos.fos_pv_out(p, v)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    rows = np.unique(np.concatenate([[0, 127, 128, Sq - 1],
                                     np.random.default_rng(1).integers(0, Sq, 40)]))
    r = torch.from_numpy(rows).to(dev())
    check_against_oracle(p[:, :, r], v, out[:, :, r], "float32")


@pytest.mark.parametrize("out_name", ["float32", "bfloat16"])
def test_outputs_are_position_and_batch_invariant(out_name):
    # the same probability rows at other query positions (shifted by 37 rows) and in another
    # batch entry of a bigger batch, with the same values and keys: the same bits
    odt = DTYPES[out_name]
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 300, 520, 128
    p, v = pv_inputs(B, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=21)
    ref = fos.fos_pv_out(p, v, out_dtype=odt)
    p2, _ = pv_inputs(B, Hq, Hkv, Sq + 37, Skv, D, torch.bfloat16, seed=22)
    p2[:, :, 37:] = p
    out = fos.fos_pv_out(p2, v, out_dtype=odt)
    assert bits_equal(out[:, :, 37:].contiguous(), ref)
    p3, v3 = pv_inputs(3, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=23)
    p3[1] = p[0]
    v3[1] = v[0]
    out = fos.fos_pv_out(p3, v3, out_dtype=odt)
    assert bits_equal(out[1:2].contiguous(), ref)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0


def test_tiny_problems():
    p, v = pv_inputs(1, 1, 1, 1, 1, 64, torch.bfloat16, seed=5)
    check_against_oracle(p, v, fos.fos_pv_out(p, v), "float32")
    p, v = pv_inputs(1, 3, 1, 5, 17, 128, torch.float16, seed=6)
    check_against_oracle(p, v, fos.fos_pv_out(p, v, out_dtype=torch.float16), "float16")
    p, v = pv_inputs(1, 1, 1, 0, 4, 64, torch.bfloat16, seed=7)
    assert fos.fos_pv_out(p, v).numel() == 0
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0


def test_refusals():
    p, v = pv_inputs(1, 2, 1, 8, 16, 96, torch.bfloat16, seed=8)
    with pytest.raises(fos.FosError) as e:  # head dimension 96
        fos.fos_pv_out(p, v)
    assert e.value.status == _abi.FOS_ERR_UNSUPPORTED
    p, v = pv_inputs(1, 3, 2, 8, 16, 64, torch.bfloat16, seed=9)
    with pytest.raises(fos.FosError) as e:  # 3 query heads over 2 value heads
        fos.fos_pv_out(p, v)
    assert e.value.status == _abi.FOS_ERR_INVALID
    p, v = pv_inputs(1, 1, 1, 8, 16, 64, torch.bfloat16, seed=10, ld=20)
    with pytest.raises(fos.FosError) as e:  # 40-byte probability rows
        fos.fos_pv_out(p, v)
    assert e.value.status == _abi.FOS_ERR_UNSUPPORTED
