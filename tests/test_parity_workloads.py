"""GPU vs FP64 oracle on the five workloads at full size, in the default launch configuration
(the one the benchmark times): every row for the two smaller workloads, sampled rows (first,
last and seeded random ones) for the larger ones, which the oracle computes one by one."""

import numpy as np
import pytest
import torch

import deterministic_attention_softmax_gb300 as fos
from deterministic_attention_softmax_gb300 import workloads as W
from gpu_util import assert_check, check_bwd, check_fwd, dev, np64, oracle, tol

pytestmark = pytest.mark.gpu


def dtype_name(w):
    return str(w.dtype).replace("torch.", "")


def sample_ids(rows, n=256, seed=0):
    rng = np.random.default_rng(seed)
    ids = np.concatenate([np.arange(4), rows - 4 + np.arange(4), rng.integers(0, rows, n)])
    return np.unique(ids)


def geometry(w):
    return dict(batch=w.batch, heads=w.heads, q_len=w.q_len, causal=w.causal)


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen_image_bf16"])
def test_workload_every_row(name):
    w = W.WORKLOADS[name]
    d = dev()
    x = W.scores(w, d)
    dp = W.dprobs(w, d)
    p, lse = fos.fos_softmax_fwd(x, **geometry(w))
    p_ref, lse_ref = oracle.softmax_fwd(np64(x), **geometry(w))
    check_fwd(p, lse, p_ref, lse_ref, dtype_name(w), name)
    del p
    p_in = torch.from_numpy(p_ref).to(w.dtype).to(d)
    del p_ref
    ds, delta = fos.fos_softmax_bwd(p_in, dp, **geometry(w))
    pin, dpn = np64(p_in), np64(dp)
    ds_ref, delta_ref = oracle.softmax_bwd(pin, dpn, **geometry(w))
    check_bwd(ds, delta, ds_ref, delta_ref, pin, dpn, dtype_name(w), what=name)
    assert fos.fos_device_error() == 0


@pytest.mark.parametrize("name", ["prompt_padding_bf16", "sink_causal_bf16", "large_bf16",
                                  "large_fp32", "long_rows_bf16"])
def test_workload_sampled_rows(name):
    w = W.WORKLOADS[name]
    d = dev()
    x = W.scores(w, d)  # the padding workload carries its -inf tail
    dp = W.dprobs(w, d)
    kv = W.valid_lengths(w)
    sink = W.sink_logits(w)
    sink_d = None if sink is None else sink.to(d)
    kv_d = None if kv is None else kv.to(d)
    kvn = None if kv is None else kv.numpy()
    skn = None if sink is None else sink.double().numpy()
    ids = sample_ids(w.rows, seed=w.seed)
    ids_d = torch.from_numpy(ids).to(d)

    # forward on the -inf padded scores, no explicit mask
    p, lse = fos.fos_softmax_fwd(x, sink=sink_d, **geometry(w))
    xs = np64(x.index_select(0, ids_d))
    p_ref, lse_ref = oracle.softmax_fwd(xs, sink=skn, row_ids=ids, **geometry(w))
    check_fwd(p.index_select(0, ids_d), lse.index_select(0, ids_d), p_ref, lse_ref,
              dtype_name(w), name)
    del p, x

    # backward on a probability-shaped input independent of the forward, with the mask
    p_in = W.probs_like(w, d)
    ds, delta = fos.fos_softmax_bwd(p_in, dp, kv_valid_len=kv_d, **geometry(w))
    pin = np64(p_in.index_select(0, ids_d))
    dpn = np64(dp.index_select(0, ids_d))
    ds_ref, delta_ref = oracle.softmax_bwd(pin, dpn, kv_valid_len=kvn, row_ids=ids,
                                           **geometry(w))
    from gpu_util import valid_matrix

    valid = valid_matrix(ids, w.key_len, w.batch, w.heads, w.q_len, w.causal, kvn, None)
    check_bwd(ds.index_select(0, ids_d), delta.index_select(0, ids_d), ds_ref, delta_ref, pin,
              dpn, dtype_name(w), valid=valid, what=name)
    del ds, p_in, dp

    if sink is not None:
        # d_sink over every row of every head, on LSE / delta inputs drawn independently
        g = torch.Generator(device="cpu").manual_seed(99)
        lse_in = (sink.repeat_interleave(w.q_len).repeat(w.batch) + 2.0 +
                  torch.randn(w.rows, generator=g).abs())
        delta_in = torch.randn(w.rows, generator=g) * 0.3
        d_sink = fos.fos_sink_grad(lse_in.to(d), delta_in.to(d), sink_d, batch=w.batch,
                                   heads=w.heads, q_len=w.q_len)
        ref = oracle.sink_grad(lse_in.double().numpy(), delta_in.double().numpy(), skn,
                               batch=w.batch, heads=w.heads, q_len=w.q_len)
        assert_check(tol.check_dsink(np64(d_sink), ref, lse_in.double().numpy(),
                                     delta_in.double().numpy(), skn, w.batch, w.heads, w.q_len),
                     "d_sink")
    assert fos.fos_device_error() == 0


def test_sink_workload_chain_small_heads():
    # forward -> backward -> d_sink end to end on the sink workload's shape restricted to 4
    # heads (the oracle then covers every row of those heads): GPU chain on its own outputs,
    # oracle chain on its own, the backward fed the oracle's P rounded to bf16 on both sides.
    base = W.WORKLOADS["sink_causal_bf16"]
    w = W.Workload("sink_causal_bf16_4h", base.dtype, base.batch, 4, base.q_len, base.key_len,
                   base.score_sigma, seed=base.seed, causal=True, sink=True)
    d = dev()
    x = W.scores(w, d)
    dp = W.dprobs(w, d)
    sink = W.sink_logits(w)
    skn = sink.double().numpy()
    p, lse = fos.fos_softmax_fwd(x, sink=sink.to(d), **geometry(w))
    p_ref, lse_ref = oracle.softmax_fwd(np64(x), sink=skn, **geometry(w))
    check_fwd(p, lse, p_ref, lse_ref, "bfloat16", "sink chain")
    p_in = torch.from_numpy(p_ref).to(torch.bfloat16).to(d)
    ds, delta = fos.fos_softmax_bwd(p_in, dp, **geometry(w))
    pin, dpn = np64(p_in), np64(dp)
    ds_ref, delta_ref = oracle.softmax_bwd(pin, dpn, **geometry(w))
    check_bwd(ds, delta, ds_ref, delta_ref, pin, dpn, "bfloat16", what="sink chain")
    d_sink = fos.fos_sink_grad(lse, delta, sink.to(d), batch=w.batch, heads=w.heads,
                               q_len=w.q_len)
    ref = oracle.sink_grad(lse_ref, delta_ref, skn, batch=w.batch, heads=w.heads, q_len=w.q_len)
    assert_check(tol.check_dsink(np64(d_sink), ref, lse_ref, delta_ref, skn, w.batch, w.heads,
                                 w.q_len), "d_sink chain")
