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
