"""The oracle against the hand-derived worked examples in ``tests/golden/`` (CPU only).

Each fixture file states the passage it follows and, per case, the derivation of its exact
values (ratios of small integers and their logarithms), so a reader can check every number
without running anything.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def val(s):
    """'1/6' -> 1/6, 'log(6)' -> ln 6, '-inf' -> -inf, '5' -> 5."""
    s = s.strip()
    if s == "-inf":
        return -math.inf
    if s.startswith("log(") and s.endswith(")"):
        return math.log(float(Fraction(s[4:-1])))
    return float(Fraction(s))


def arr(rows):
    return np.array([[val(v) for v in row] for row in rows], dtype=np.float64)


def vec(items):
    return np.array([val(v) for v in items], dtype=np.float64)


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        data = json.load(f)
    assert data["citation"], "every fixture file cites the passage it follows"
    return data["cases"]


def masks(case):
    kv = case.get("kv_valid_len")
    km = case.get("key_mask")
    return (None if kv is None else np.array(kv, dtype=np.int32),
            None if km is None else np.array(km, dtype=np.uint8))


@pytest.mark.parametrize("case", load("fwd_rational.json"), ids=lambda c: c["name"])
def test_forward_worked_examples(case):
    kv, km = masks(case)
    sink = case.get("sink")
    p, lse = oracle.softmax_fwd(arr(case["scores"]), batch=case["batch"], heads=case["heads"],
                                q_len=case["q_len"], causal=bool(case.get("causal", 0)),
                                kv_valid_len=kv, key_mask=km,
                                sink=None if sink is None else vec(sink))
    np.testing.assert_allclose(p, arr(case["P"]), rtol=1e-14, atol=1e-300)
    exp_lse = vec(case["lse"])
    assert np.array_equal(np.isneginf(lse), np.isneginf(exp_lse))
    fin = np.isfinite(exp_lse)
    np.testing.assert_allclose(lse[fin], exp_lse[fin], rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("case", load("bwd_rational.json"), ids=lambda c: c["name"])
def test_backward_worked_examples(case):
    kv, km = masks(case)
    ds, delta = oracle.softmax_bwd(arr(case["P"]), arr(case["dP"]), batch=case["batch"],
                                   heads=case["heads"], q_len=case["q_len"],
                                   causal=bool(case.get("causal", 0)), kv_valid_len=kv,
                                   key_mask=km)
    np.testing.assert_allclose(delta, vec(case["delta"]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(ds, arr(case["dS"]), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("case", load("dsink_rational.json"), ids=lambda c: c["name"])
def test_sink_grad_worked_examples(case):
    d = oracle.sink_grad(vec(case["lse"]), vec(case["delta"]), vec(case["sink"]),
                         batch=case["batch"], heads=case["heads"], q_len=case["q_len"])
    np.testing.assert_allclose(d, vec(case["d_sink"]), rtol=1e-14, atol=1e-15)
