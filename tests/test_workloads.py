"""The workloads' algorithmic bytes, which every reported GB/s and roofline fraction divides by.
Per row the method must read the valid scores and write P and LSE (forward), read P and dP over
the valid keys and write dScores and delta (backward): esz*|V| + esz*L + 4 and
2*esz*|V| + esz*L + 4 bytes.  Pinned to worked values, and the mean number of valid keys under
a causal bound is checked by counting keys with the mask definition itself."""

import numpy as np
import pytest
import torch

from deterministic_attention_softmax_gb300 import workloads as W


def test_qwen_image_bytes():
    # 16,384 rows of 4,352 bf16 keys, nothing masked
    b = W.algorithmic_bytes(W.WORKLOADS["qwen_image_bf16"])
    assert b["fwd"] == 16384 * (2 * 4352 + 2 * 4352 + 4) == 285_278_208
    assert b["bwd"] == 16384 * (2 * 2 * 4352 + 2 * 4352 + 4) == 427_884_544
    assert b["sink"] == 0 and b["total"] == b["fwd"] + b["bwd"]


def test_tiny_fp32_bytes():
    b = W.algorithmic_bytes(W.WORKLOADS["tiny_fp32"])
    assert b["fwd"] == 2056 * (4 * 257 * 2 + 4) == 4_235_360
    assert b["bwd"] == 2056 * (4 * 257 * 3 + 4) == 6_348_928


@pytest.mark.parametrize("name,esz", [("large_bf16", 2), ("large_fp32", 4)])
def test_large_bytes(name, esz):
    b = W.algorithmic_bytes(W.WORKLOADS[name])
    rows, L = 24 * 8192, 8192
    assert b["fwd"] == rows * (2 * esz * L + 4)
    assert b["bwd"] == rows * (3 * esz * L + 4)


def brute_mean_valid(L, q_len, causal, lens=None):
    # count, per query row, the keys the mask definition makes valid (no -inf scores)
    j = np.arange(L)
    counts = []
    for b in range(1 if lens is None else len(lens)):
        for i in range(q_len):
            v = np.ones(L, dtype=bool)
            if causal:
                v &= j <= L - q_len + i
            if lens is not None:
                v &= j < lens[b]
            counts.append(v.sum())
    return float(np.mean(counts))


@pytest.mark.parametrize("L,q_len", [(2048, 2048), (4352, 1024), (300, 40), (9, 9)])
def test_causal_mean_valid_keys_matches_a_count(L, q_len):
    w = W.Workload("c", torch.bfloat16, 1, 1, q_len, L, 1.0, seed=0, causal=True)
    assert W.mean_valid_keys(w) == pytest.approx(brute_mean_valid(L, q_len, True), abs=1e-9)


def test_sink_causal_bytes():
    w = W.WORKLOADS["sink_causal_bf16"]
    v = W.mean_valid_keys(w)
    assert v == 1024.5  # query i of 2,048 sees i + 1 keys
    b = W.algorithmic_bytes(w, valid_keys=v)
    rows = 2 * 64 * 2048
    assert b["fwd"] == pytest.approx(rows * (2 * v + 2 * 2048 + 4))
    assert b["bwd"] == pytest.approx(rows * (2 * 2 * v + 2 * 2048 + 4))
    assert b["sink"] == rows * 8  # the sink gradient re-reads LSE and delta


def test_padding_mean_valid_keys_is_the_mean_valid_length():
    w = W.WORKLOADS["prompt_padding_bf16"]
    lens = W.valid_lengths(w).numpy()
    assert ((lens >= 4096 + 32) & (lens <= 4096 + 512)).all()
    assert W.mean_valid_keys(w) == pytest.approx(brute_mean_valid(w.key_len, 3, False, lens))


def small(**kw):
    base = dict(name="s", dtype=torch.bfloat16, batch=2, heads=3, q_len=4, key_len=300,
                score_sigma=4.0, seed=7)
    base.update(kw)
    return W.Workload(**base)


def test_inputs_are_reproducible_and_seeded():
    w = small()
    a, b = W.scores(w, "cpu"), W.scores(w, "cpu")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = W.scores(w, "cpu", seed_offset=1)
    assert not torch.equal(a, c)
    assert not torch.equal(W.dprobs(w, "cpu"), W.dprobs(w, "cpu", seed_offset=1))
    assert not torch.equal(W.scores(small(seed=8), "cpu"), a)
    assert a.shape == (24, 300) and a.dtype == torch.bfloat16


def test_inputs_are_rounded_once_from_float32():
    # sigma * N(0,1) in float32, then one round-to-nearest-even to the dtype
    w = small()
    x = W.scores(w, "cpu")
    ref = (torch.randn((24, 300), generator=torch.Generator().manual_seed(7 * 1000 + 1)) * 4.0)
    assert torch.equal(x, ref.to(torch.bfloat16))


def test_padding_tail_is_minus_infinity_past_each_valid_length():
    w = small(pad=(200, 10, 60))
    lens = W.valid_lengths(w)
    assert lens.dtype == torch.int32 and lens.shape == (2,)
    assert ((lens >= 210) & (lens <= 260)).all()
    x = W.scores(w, "cpu").view(2, 12, 300)
    for b in range(2):
        assert torch.isneginf(x[b, :, int(lens[b]):]).all()
        assert torch.isfinite(x[b, :, :int(lens[b])]).all()
    assert torch.isfinite(W.scores(w, "cpu", neg_inf_tail=False)).all()


def test_sink_logits_and_probability_inputs():
    assert W.sink_logits(small()) is None
    s = W.sink_logits(small(sink=True))
    assert s.shape == (3,) and s.dtype == torch.float32
    p = W.probs_like(small(), "cpu").float()
    assert (p >= 0).all() and float(p.max()) <= 5.0 / 300 + 1e-6
