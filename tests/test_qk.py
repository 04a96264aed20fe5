"""The fixed-order QK contraction on the tensor cores (fos_qk_scores) against the FP64 oracle
(``oracle/gemm.py:qk_scores``), element by element, and its bitwise invariance: a score depends
only on its query row and key row, so it must have the same bits wherever those rows sit (tile
position, batch entry, neighbouring heads, row stride of the output).  ("Batch-invariant
attention (standard softmax--cuda version)", Fixed Reduction Contract; "[WS1][kernels] Add
fixed-order joint-attention softmax for Qwen-Image", Summary: the QK GEMM in front of the
softmax.)"""

import math

import numpy as np
import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300 import _abi
from gpu_util import DTYPES, bits_equal, dev, np64, tol
from oracle import gemm

pytestmark = pytest.mark.gpu


def qk_inputs(B, Hq, Hkv, Sq, Skv, D, dtype, seed, sigma=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = (torch.randn(B, Hq, Sq, D, generator=g, device=dev()) * sigma).to(dtype)
    k = (torch.randn(B, Hkv, Skv, D, generator=g, device=dev()) * sigma).to(dtype)
    return q, k


def check_against_oracle(q, k, s, scale, out_name):
    qn, kn = np64(q), np64(k)
    ref = gemm.qk_scores(qn, kn, scale)
    absd = gemm.qk_scores(np.abs(qn), np.abs(kn), 1.0)  # sum_d |q_d k_d| per score
    ok, worst, idx = tol.check_scores(np64(s), ref, absd, scale, out_name)
    assert ok, f"scores: worst err/bound {worst:.3g} at flat index {idx}"
    return worst


@pytest.mark.parametrize("in_name", ["bfloat16", "float16"])
@pytest.mark.parametrize("out_name", ["float32", "bfloat16", "float16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("tile_n", [0, 128, 256])
def test_scores_match_the_oracle(in_name, out_name, D, tile_n):
    # two query tiles (the second ragged) x two or three key tiles (the last ragged), grouped
    # heads; 300 keys make 600-byte rows in a 16-bit output, so the binding pads the row stride.
    # tile_n 0: the persistent kernel (one CTA per SM over all tiles); 128 / 256: a CTA per tile
    B, Hq, Hkv, Sq, Skv = 2, 4, 2, 200, 300
    q, k = qk_inputs(B, Hq, Hkv, Sq, Skv, D, DTYPES[in_name], seed=D + 7)
    scale = 1.0 / math.sqrt(D)
    s = fos.fos_qk_scores(q, k, scale, out_dtype=DTYPES[out_name], tile_n=tile_n)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    check_against_oracle(q, k, s, scale, out_name)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("out_name", ["float32", "bfloat16"])
def test_runs_of_tiles_that_cross_query_tiles_and_heads(D, out_name):
    # 8 query tiles (the last ragged) x 16 key tiles (the last ragged) x 4 batch-heads = 512
    # tiles: the persistent kernel gives each CTA a contiguous run of three or four, so runs
    # cross key tiles, query tiles (a new Q block mid-run) and batch-head boundaries, with
    # grouped heads; every score against the oracle
    B, Hq, Hkv, Sq, Skv = 2, 2, 1, 1000, 2000
    q, k = qk_inputs(B, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=D + 31)
    scale = 1.0 / math.sqrt(D)
    s = fos.fos_qk_scores(q, k, scale, out_dtype=DTYPES[out_name])
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    check_against_oracle(q, k, s, scale, out_name)
    # and the bits of the CTA-per-tile kernel (same instructions on the same operands)
    s128 = fos.fos_qk_scores(q, k, scale, out_dtype=DTYPES[out_name], tile_n=128)
    assert bits_equal(s.contiguous(), s128.contiguous())


def test_qwen_image_shape_sampled():
    # the benchmark's shape: 16,384 query rows (4 heads x 4,096) against 4,352 keys, D = 128,
    # bf16 in, float32 scores; every score of a sample of query rows against the oracle
    B, H, Sq, Skv, D = 1, 4, 4096, 4352, 128
    q, k = qk_inputs(B, H, H, Sq, Skv, D, torch.bfloat16, seed=3)
    scale = 1.0 / math.sqrt(D)
    s = fos.fos_qk_scores(q, k, scale)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0
    rows = np.unique(np.concatenate([[0, 127, 128, Sq - 1],
                                     np.random.default_rng(0).integers(0, Sq, 40)]))
    r = torch.from_numpy(rows).to(dev())
    check_against_oracle(q[:, :, r], k, s[:, :, r], scale, "float32")


@pytest.mark.parametrize("out_name", ["float32", "bfloat16"])
def test_scores_are_position_and_batch_invariant(out_name):
    # The same query and key rows at other tile positions (shifted by 37 query rows and 29 keys),
    # in another batch entry of a bigger batch, between other heads, and into an output with a
    # wider row stride: every score has the same bits.
    odt = DTYPES[out_name]
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 300, 520, 128
    q, k = qk_inputs(B, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=11, sigma=2.0)
    ref = fos.fos_qk_scores(q, k, 0.125, out_dtype=odt)
    # shifted rows inside a longer head, and the other tile width
    q2, k2 = qk_inputs(B, Hq, Hkv, Sq + 37, Skv + 29, D, torch.bfloat16, seed=12, sigma=2.0)
    q2[:, :, 37:] = q
    k2[:, :, 29:] = k
    for tile_n in (128, 256):
        out = fos.fos_qk_scores(q2, k2, 0.125, out_dtype=odt, tile_n=tile_n)
        assert bits_equal(out[:, :, 37:, 29:].contiguous(), ref.contiguous()), tile_n
    # batch entry 2 of 3, with other noise around it
    q3, k3 = qk_inputs(3, Hq, Hkv, Sq, Skv, D, torch.bfloat16, seed=13, sigma=2.0)
    q3[2] = q[0]
    k3[2] = k[0]
    out = fos.fos_qk_scores(q3, k3, 0.125, out_dtype=odt)
    assert bits_equal(out[2:3].contiguous(), ref.contiguous())
    # a wider output row stride (a narrowed buffer), same bits, padding untouched
    ld = Skv + 24
    buf = torch.full((B, Hq, Sq, ld), 7.0, dtype=odt, device=dev())
    out = fos.fos_qk_scores(q, k, 0.125, scores=buf[..., :Skv])
    assert bits_equal(out.contiguous(), ref.contiguous())
    assert torch.all(buf[..., Skv:] == 7.0)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0


def test_tiny_and_empty_problems():
    q, k = qk_inputs(1, 1, 1, 1, 1, 64, torch.bfloat16, seed=5)
    s = fos.fos_qk_scores(q, k, 1.0)
    check_against_oracle(q, k, s, 1.0, "float32")
    q, k = qk_inputs(1, 3, 1, 5, 3, 128, torch.float16, seed=6)
    s = fos.fos_qk_scores(q, k, 0.3, out_dtype=torch.float16,
                          scores=torch.empty(1, 3, 5, 8, dtype=torch.float16,
                                             device=dev())[..., :3])
    check_against_oracle(q, k, s, 0.3, "float16")
    q, k = qk_inputs(1, 1, 1, 0, 4, 64, torch.bfloat16, seed=7)
    assert fos.fos_qk_scores(q, k).numel() == 0
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0


def test_refusals():
    q, k = qk_inputs(1, 2, 1, 8, 8, 96, torch.bfloat16, seed=8)
    with pytest.raises(fos.FosError) as e:  # head dimension 96
        fos.fos_qk_scores(q, k)
    assert e.value.status == _abi.FOS_ERR_UNSUPPORTED
    q, k = qk_inputs(1, 3, 2, 8, 8, 64, torch.bfloat16, seed=9)
    with pytest.raises(fos.FosError) as e:  # 3 query heads over 2 key heads
        fos.fos_qk_scores(q, k)
    assert e.value.status == _abi.FOS_ERR_INVALID
    q, k = qk_inputs(1, 1, 1, 8, 8, 64, torch.bfloat16, seed=10)
    out = torch.empty(1, 1, 8, 9, dtype=torch.float32, device=dev())[..., :8]
    with pytest.raises(fos.FosError) as e:  # 36-byte output rows
        fos.fos_qk_scores(q, k, scores=out)
    assert e.value.status == _abi.FOS_ERR_UNSUPPORTED
    with pytest.raises(fos.FosError) as e:  # keys per tile must be 128 or 256
        fos.fos_qk_scores(q, k, tile_n=64)
    assert e.value.status == _abi.FOS_ERR_INVALID
