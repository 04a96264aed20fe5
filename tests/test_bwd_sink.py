"""The backward with the sink gradient taken along (fos_softmax_bwd_sink).  Its results must be
the bits of fos_softmax_bwd followed by fos_sink_grad on every path and every strategy: rows of
at most 8 tiles (one warp per row: the two launches by default, octets of positions per warp
when the launch asks for them), longer staged rows (one CTA per row, octets per CTA when there
are enough of them, else the two launches), rows streamed in segments and rows copied with plain
loads.  Octets that straddle two batch entries (q_len not a multiple of
8), fully masked rows, -inf sinks and a given or absent delta are covered; the sink workload's
shape is also checked against the FP64 oracle end to end.  ("[ROCm] Jax Add softmax sink
(learnable off-by-one) support", Description and review thread: d_sink reduced per head in the
backward.)"""

import math

import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300 import workloads as W
from gpu_util import assert_check, bits_equal, check_bwd, dev, np64, oracle, tol

pytestmark = pytest.mark.gpu


def make(dt, B, H, Sq, L, seed, causal, kv=None, sink_vals=None):
    g = torch.Generator(device="cuda").manual_seed(seed)
    d = dev()
    x = (torch.randn(B * H * Sq, L, generator=g, device=d) * 3).to(dt)
    dp = torch.randn(B * H * Sq, L, generator=g, device=d).to(dt)
    sink = torch.randn(H, generator=g, device=d) if sink_vals is None else \
        torch.tensor(sink_vals, dtype=torch.float32, device=d)
    kvt = None if kv is None else torch.tensor(kv, dtype=torch.int32, device=d)
    kw = dict(batch=B, heads=H, q_len=Sq, causal=causal, kv_valid_len=kvt)
    p, lse = fos.fos_softmax_fwd(x, sink=sink, **kw)
    return p, dp, lse, sink, kw


def compare(p, dp, lse, sink, kw, launch=None):
    ds_ref, delta_ref = fos.fos_softmax_bwd(p, dp, launch=launch, **kw)
    d_ref = fos.fos_sink_grad(lse, delta_ref, sink, batch=kw["batch"], heads=kw["heads"],
                              q_len=kw["q_len"])
    # with delta given, and without (the workspace then holds what the sum needs)
    delta = torch.full_like(delta_ref, 5.0)
    ds, d_sink, delta = fos.fos_softmax_bwd_sink(p, dp, lse, sink, delta=delta, launch=launch,
                                                 **kw)
    assert bits_equal(ds, ds_ref) and bits_equal(d_sink, d_ref) and bits_equal(delta, delta_ref)
    ds2, d_sink2, _ = fos.fos_softmax_bwd_sink(p, dp, lse, sink, launch=launch, **kw)
    assert bits_equal(ds2, ds_ref) and bits_equal(d_sink2, d_ref)
    torch.cuda.synchronize()
    assert fos.fos_device_error() == 0


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32, torch.float16])
@pytest.mark.parametrize("L", [200, 600, 2048])
@pytest.mark.parametrize("causal", [False, True])
def test_short_rows_one_warp_per_row(dt, L, causal):
    # q_len 13: octets straddle batch entries; the second entry's valid length masks its tail
    p, dp, lse, sink, kw = make(dt, 3, 5, 13, L, seed=L + causal, causal=causal,
                                kv=[L, L // 3, L])
    compare(p, dp, lse, sink, kw)
    # the library's choice (two launches here), the octets forced, and never
    for opts in (dict(warps_per_cta=1), dict(warps_per_cta=7, stages=2), dict(ctas=3),
                 dict(sink_fusion=1), dict(sink_fusion=1, warps_per_cta=7, stages=2),
                 dict(sink_fusion=1, ctas=3), dict(sink_fusion=2)):
        compare(p, dp, lse, sink, kw, launch=fos.Launch(**opts))


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("opts", [dict(ctas=16), dict(ctas=16, generic=1),
                                  dict(ctas=12, warps_per_cta=3, stages=1), dict(), dict(generic=1),
                                  dict(ctas=16, sink_fusion=2)],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()) or "default")
def test_longer_rows_one_cta_per_row(dt, opts):
    # 17-tile rows, 75 octets: on a grid of at most 18 CTAs every CTA takes octets; the
    # default grid is too wide for them, so the two launches run (same bits)
    p, dp, lse, sink, kw = make(dt, 2, 3, 100, 4352, seed=5, causal=True, kv=[4352, 3000])
    compare(p, dp, lse, sink, kw, launch=fos.Launch(**opts))


@pytest.mark.parametrize("opts", [dict(load_path=3), dict(load_path=2, ctas=3)])
def test_streamed_and_plain_load_rows(opts):
    # streamed segments take no octets (two launches); plain loads on 3 CTAs take the 12 octets
    p, dp, lse, sink, kw = make(torch.bfloat16, 2, 2, 24, 3000, seed=7, causal=False,
                                kv=[3000, 1234])
    compare(p, dp, lse, sink, kw, launch=fos.Launch(**opts))


def test_fully_masked_rows_minus_inf_sinks_and_empty_batches():
    # batch entry 1 has no valid key; head 0's sink is -inf (its gradient is exactly 0)
    p, dp, lse, sink, kw = make(torch.bfloat16, 3, 3, 21, 700, seed=9, causal=False,
                                kv=[700, 0, 350], sink_vals=[-math.inf, 0.5, -1.0])
    compare(p, dp, lse, sink, kw)
    ds, d_sink, _ = fos.fos_softmax_bwd_sink(p, dp, lse, sink, **kw)
    assert d_sink[0].item() == 0.0
    # no rows at all: every head's gradient is 0
    e = torch.empty(0, 64, dtype=torch.bfloat16, device=dev())
    sk = torch.tensor([0.3, -0.2], device=dev())
    ds, d_sink, _ = fos.fos_softmax_bwd_sink(e, e, torch.empty(0, device=dev()), sk, batch=0,
                                             heads=2, q_len=4)
    torch.cuda.synchronize()
    assert torch.equal(d_sink, torch.zeros(2, device=dev()))


def test_sink_workload_shape_against_the_oracle():
    # the sink workload's shape with 4 of its 64 heads: forward on the GPU, backward with the
    # sink gradient taken along on the oracle's P rounded to bf16; the oracle chain on its own
    base = W.WORKLOADS["sink_causal_bf16"]
    w = W.Workload("sink_causal_bf16_4h", base.dtype, base.batch, 4, base.q_len, base.key_len,
                   base.score_sigma, seed=base.seed + 100, causal=True, sink=True)
    d = dev()
    geo = dict(batch=w.batch, heads=w.heads, q_len=w.q_len, causal=True)
    x = W.scores(w, d)
    dp = W.dprobs(w, d)
    sink = W.sink_logits(w)
    skn = sink.double().numpy()
    p, lse = fos.fos_softmax_fwd(x, sink=sink.to(d), **geo)
    p_ref, lse_ref = oracle.softmax_fwd(np64(x), sink=skn, **geo)
    p_in = torch.from_numpy(p_ref).to(torch.bfloat16).to(d)
    delta = torch.empty(w.rows, dtype=torch.float32, device=d)
    ds, d_sink, delta = fos.fos_softmax_bwd_sink(p_in, dp, lse, sink.to(d), delta=delta, **geo)
    pin, dpn = np64(p_in), np64(dp)
    ds_ref, delta_ref = oracle.softmax_bwd(pin, dpn, **geo)
    check_bwd(ds, delta, ds_ref, delta_ref, pin, dpn, "bfloat16", what="fused sink")
    ref = oracle.sink_grad(lse_ref, delta_ref, skn, batch=w.batch, heads=w.heads, q_len=w.q_len)
    assert_check(tol.check_dsink(np64(d_sink), ref, lse_ref, delta_ref, skn, w.batch, w.heads,
                                 w.q_len), "d_sink (fused)")


def test_refusals():
    p, dp, lse, sink, kw = make(torch.bfloat16, 1, 2, 8, 256, seed=3, causal=False)
    with pytest.raises(fos.FosError) as e:  # a workspace smaller than asked for
        small = torch.empty(16, dtype=torch.uint8, device=dev())
        fos.fos_softmax_bwd_sink(p, dp, lse, sink, workspace=small, **kw)
    assert e.value.status == 1
