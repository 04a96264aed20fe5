"""Parity tolerances between the CUDA library and the FP64 oracle -- TEST INFRASTRUCTURE ONLY.

The bounds are the stated correctness bar of the kernels, read as follows:

* P, float32 I/O: max |gpu - ref| <= 1e-6.
* P, bf16/fp16 I/O: |gpu - ref| <= 1 ULP of the I/O dtype at the FP64 value.
* LSE (float32 output for every I/O dtype): |gpu - ref| <= 1e-5 * max(1, |ref|); -inf exactly.
* dScores: "1e-5 relative" is taken relative to the element's condition scale
  s_j = |ref_j| + P_j * (|dP_j| + sum_k P_k |dP_k|), because dP_j - delta cancels.
  float32 I/O: |err| <= 1e-5 * s_j.
  bf16/fp16 I/O: |err| <= max(1 ULP(ref_j), 2^-20 * P_j * (|dP_j| + sum_k P_k |dP_k|)): one
  ULP of the FP64 value, or, where dP_j - delta has cancelled below what a float32 delta can
  resolve, a float32 floor.  The floor scales with sum_k P_k |dP_k| rather than |delta|: the
  float32 sum's rounding errors are relative to its partial sums, whose size is set by the
  absolute terms, so no fixed-order float32 sum reaches 2^-20 * |delta| when delta cancels.
* delta (float32): |err| <= 1e-5 * sum_k P_k |dP_k|.
* QK scores: |err| <= 2^-16 * |scale| * sum_d |q_d k_d| (a float32 sum of the head dimension's
  products, whatever its order, stays within (D - 1) * 2^-24 of that absolute sum, 2^-17 at
  D = 128; 2^-16 leaves room for the final multiply by the scale), plus one ULP of the FP64 value
  for a 16-bit output dtype (its single rounding).
* PV outputs: the same form over the keys, |err| <= 2^-16 * sum_j |p_j v_jd| plus one ULP for a
  16-bit output (the scale is 1).  Over thousands of keys the worst-case float32 bound is looser
  than this, but the partial sums of terms of both signs stay far below the absolute sum, and the
  bound is the one an accurate float32 sum in any fixed order meets on such data.
* d_sink (float32): |err| <= 1e-5 * sum_r |c_r| with c_r = exp(sink_h - LSE_r) * delta_r.
"""

from __future__ import annotations

import numpy as np

_MANT = {"float32": 23, "bfloat16": 7, "float16": 10}
_EMIN = {"float32": -126, "bfloat16": -126, "float16": -14}


def ulp(ref, dtype: str):
    """Spacing of the I/O dtype's numbers at |ref| (ref in float64)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    m, emin = _MANT[dtype], _EMIN[dtype]
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    # zero and the subnormals share the smallest spacing, 2^(emin - m)
    e = np.where(a > 0, np.maximum(e, emin), emin)
    return np.ldexp(1.0, (e - m).astype(np.int64))


def _worst(err, bound):
    ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1), np.where(err > 0, np.inf, 0))
    i = int(np.argmax(ratio)) if ratio.size else 0
    return (float(ratio.ravel()[i]) if ratio.size else 0.0), i


def check_probs(gpu, ref, dtype: str):
    """Returns (ok, worst ratio err/bound, flat index of the worst element)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    bound = np.full_like(ref, 1e-6) if dtype == "float32" else ulp(ref, dtype)
    w, i = _worst(err, bound)
    return bool(np.all(err <= bound)), w, i


def check_lse(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    same_inf = np.array_equal(np.isneginf(gpu), np.isneginf(ref))
    fin = np.isfinite(ref)
    err = np.abs(gpu[fin] - ref[fin])
    bound = 1e-5 * np.maximum(1.0, np.abs(ref[fin]))
    w, i = _worst(err, bound)
    return bool(same_inf and np.all(np.isfinite(gpu[fin])) and np.all(err <= bound)), w, i


def dscores_scale(probs, dprobs, ref, valid=None):
    """s_j = |ref_j| + P_j (|dP_j| + sum_k P_k |dP_k|) over valid keys (all when valid=None)."""
    p = np.asarray(probs, dtype=np.float64)
    dp = np.asarray(dprobs, dtype=np.float64)
    pdp = np.abs(p * dp)
    if valid is not None:
        pdp = np.where(valid, pdp, 0.0)
    row = pdp.sum(axis=-1, keepdims=True)
    return np.abs(ref) + np.abs(p) * (np.abs(dp) + row), row[..., 0]


def check_dscores(gpu, ref, probs, dprobs, dtype: str, valid=None):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    s, row = dscores_scale(probs, dprobs, ref, valid)
    if dtype == "float32":
        bound = 1e-5 * s + 1e-30
    else:
        p = np.abs(np.asarray(probs, dtype=np.float64))
        dp = np.abs(np.asarray(dprobs, dtype=np.float64))
        floor = 2.0 ** -20 * p * (dp + row[..., None])
        bound = np.maximum(ulp(ref, dtype), floor)
    err = np.abs(gpu - ref)
    w, i = _worst(err, bound)
    return bool(np.all(err <= bound)), w, i


def check_delta(gpu, ref, probs, dprobs, valid=None):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    _, row = dscores_scale(probs, dprobs, np.zeros_like(np.asarray(probs, dtype=np.float64)), valid)
    bound = 1e-5 * row + 1e-30
    err = np.abs(gpu - ref)
    w, i = _worst(err, bound)
    return bool(np.all(err <= bound)), w, i


def check_dsink(gpu, ref, lse, delta, sink, batch, heads, q_len):
    """Bound 1e-5 * sum_r |exp(sink_h - LSE_r) * delta_r| per head (the oracle's LSE/delta)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64).reshape(batch, heads, q_len)
    delta = np.asarray(delta, dtype=np.float64).reshape(batch, heads, q_len)
    sk = np.asarray(sink, dtype=np.float64).reshape(1, heads, 1)
    with np.errstate(invalid="ignore", over="ignore"):
        c = np.where(np.isneginf(sk), 0.0, np.exp(sk - lse) * delta)
    bound = 1e-5 * np.abs(c).sum(axis=(0, 2)) + 1e-30
    err = np.abs(gpu - ref)
    w, i = _worst(err, bound)
    return bool(np.all(err <= bound)), w, i


def check_scores(gpu, ref, abs_dot, scale, dtype: str):
    """QK scores; abs_dot = sum_d |q_d k_d| per score (float64, same shape as ref)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = 2.0 ** -16 * abs(float(scale)) * np.asarray(abs_dot, dtype=np.float64) + 1e-30
    if dtype != "float32":
        bound = bound + ulp(ref, dtype)
    err = np.abs(gpu - ref)
    w, i = _worst(err, bound)
    return bool(np.all(err <= bound)), w, i


def check_pv(gpu, ref, abs_dot, dtype: str):
    """PV outputs; abs_dot = sum_j |p_j v_jd| per output (float64, same shape as ref)."""
    return check_scores(gpu, ref, abs_dot, 1.0, dtype)
