"""The step from host buffers (fos_softmax_step_host): the bits of the device entry points
(fos_softmax_fwd, fos_softmax_bwd, fos_sink_grad) whatever the chunking, with masks, a sink and
padded rows; page-locked and pageable host memory; one workspace reused by consecutive calls;
the full Qwen-Image workload; and refusals with real tensors."""

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300 import workloads as W
from gpu_util import bits_equal, dev

pytestmark = pytest.mark.gpu


def device_step(x, dp, geo, sink=None):
    """Reference: the device entry points on device copies of the host inputs."""
    p, lse = fos.fos_softmax_fwd(x.to(dev()), sink=sink, **geo)
    ds, delta = fos.fos_softmax_bwd(p, dp.to(dev()), **geo)
    dsk = None
    if sink is not None:
        dsk = fos.fos_sink_grad(lse, delta, sink, batch=geo["batch"], heads=geo["heads"],
                                q_len=geo["q_len"]).cpu()
    return p.cpu(), lse.cpu(), ds.cpu(), delta.cpu(), dsk


def assert_same(out, ref):
    for h, r, name in zip(out, ref, ("P", "LSE", "dScores", "delta", "d_sink")):
        if r is None:
            assert h is None, name
        else:
            assert bits_equal(h.contiguous(), r.contiguous()), name


def inputs(rows, L, dtype=torch.bfloat16, seed=11, sigma=3.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(rows, L, generator=g) * sigma).to(dtype)
    dp = torch.randn(rows, L, generator=g).to(dtype)
    return x, dp


@pytest.mark.parametrize("chunk", [0, 1, 13, 64, 10_000])
def test_causal_valid_lengths_sink_any_chunking(chunk):
    B, H, Sq, L = 2, 3, 40, 300
    x, dp = inputs(B * H * Sq, L)
    kv = torch.tensor([260, 300], dtype=torch.int32, device=dev())
    sink = torch.randn(H, generator=torch.Generator().manual_seed(5)).to(dev())
    geo = dict(batch=B, heads=H, q_len=Sq, causal=True, kv_valid_len=kv)
    ref = device_step(x, dp, geo, sink)
    out = fos.fos_softmax_step_host(x.pin_memory(), dp.pin_memory(), sink=sink, chunk_rows=chunk,
                                    **geo)
    torch.cuda.synchronize()
    assert_same(out, ref)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_unmasked_rows_each_dtype(dtype):
    rows, L = 700, 4352
    x, dp = inputs(rows, L, dtype, seed=3, sigma=4.0)
    geo = dict(batch=1, heads=1, q_len=rows)
    ref = device_step(x, dp, geo)
    out = fos.fos_softmax_step_host(x.pin_memory(), dp.pin_memory(), chunk_rows=96, **geo)
    torch.cuda.synchronize()
    assert_same(out, ref)


def test_key_mask_and_padded_rows_leave_host_padding_alone():
    B, H, Sq, L, ld = 2, 2, 33, 300, 320
    rows = B * H * Sq
    x, dp = inputs(rows, L, seed=8)
    km = (torch.rand(B, L, generator=torch.Generator().manual_seed(2)) > 0.3).to(torch.uint8)
    geo = dict(batch=B, heads=H, q_len=Sq, key_mask=km.to(dev()))
    ref = device_step(x, dp, geo)

    def padded(t, fill):
        buf = torch.full((rows, ld), fill, dtype=t.dtype).pin_memory()
        buf[:, :L] = t
        return buf, buf[:, :L]

    _, hx = padded(x, -1.0)
    _, hdp = padded(dp, -1.0)
    pbuf, hp = padded(torch.zeros_like(x), 7.0)
    sbuf, hs = padded(torch.zeros_like(x), 7.0)
    out = fos.fos_softmax_step_host(hx, hdp, hp, None, hs, None, chunk_rows=20, **geo)
    torch.cuda.synchronize()
    assert_same(out, ref)
    assert bool((pbuf[:, L:] == 7.0).all()) and bool((sbuf[:, L:] == 7.0).all())


def test_pageable_host_memory_gives_the_same_bits():
    rows, L = 257, 1000
    x, dp = inputs(rows, L, seed=21)
    geo = dict(batch=1, heads=1, q_len=rows)
    ref = device_step(x, dp, geo)
    p, ds = torch.empty_like(x), torch.empty_like(x)
    lse, delta = torch.empty(rows), torch.empty(rows)
    out = fos.fos_softmax_step_host(x, dp, p, lse, ds, delta, chunk_rows=50, **geo)
    torch.cuda.synchronize()
    assert out[0] is p and out[2] is ds
    assert_same(out, ref)


def test_one_workspace_reused_by_consecutive_calls():
    rows, L = 400, 2048
    geo = dict(batch=1, heads=1, q_len=rows)
    sets = [inputs(rows, L, seed=40 + i) for i in range(3)]
    need = fos.fos_step_host_workspace_bytes(sets[0][0], chunk_rows=64, **geo)
    ws = torch.empty(need, dtype=torch.uint8, device=dev())
    outs = [fos.fos_softmax_step_host(x.pin_memory(), dp.pin_memory(), workspace=ws, chunk_rows=64,
                                      **geo) for x, dp in sets]
    torch.cuda.synchronize()
    for (x, dp), out in zip(sets, outs):
        assert_same(out, device_step(x, dp, geo))


def test_full_qwen_image_workload():
    w = W.WORKLOADS["qwen_image_bf16"]
    x = W.scores(w, "cpu")
    dp = W.dprobs(w, "cpu")
    geo = dict(batch=w.batch, heads=w.heads, q_len=w.q_len)
    ref = device_step(x, dp, geo)
    out = fos.fos_softmax_step_host(x.pin_memory(), dp.pin_memory(), **geo)
    torch.cuda.synchronize()
    assert_same(out, ref)
    assert fos.fos_device_error() == 0


def test_refusals_with_real_tensors():
    rows, L = 64, 512
    x, dp = inputs(rows, L)
    geo = dict(batch=1, heads=1, q_len=rows)
    need = fos.fos_step_host_workspace_bytes(x, chunk_rows=16, **geo)
    small = torch.empty(need - 256, dtype=torch.uint8, device=dev())
    with pytest.raises(fos.FosError) as e:
        fos.fos_softmax_step_host(x, dp, workspace=small, chunk_rows=16, **geo)
    assert e.value.status == 1
    with pytest.raises(ValueError):  # device tensors where host data are expected
        fos.fos_softmax_step_host(x.to(dev()), dp.to(dev()), **geo)
    empty = torch.empty(0, L, dtype=torch.bfloat16)
    out = fos.fos_softmax_step_host(empty, empty, batch=0, heads=1, q_len=0)
    assert out[0].numel() == 0
