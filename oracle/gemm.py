"""FP64 oracle of the two contractions around the softmax -- TEST INFRASTRUCTURE ONLY.

scores = scale * Q K^T and out = P V, with grouped-query heads, and their backward products.
Only ``tests/`` import it; nothing on the product path does.  The library has no kernel for
these contractions yet: the oracle and its pins (``tests/test_oracle_gemm.py``) come first.

What the fixed-order QK and PV contractions compute ("Batch-invariant attention (standard
softmax--cuda version)", Fixed Reduction Contract): a score is the dot product of a query row
and a key row over the head dimension, an output element the probability-weighted sum of a
value column over the keys.  The fixed accumulation order there is the GPU's rounding order;
the exact result it approximates is written out here in float64, with numpy's matmul as the
one library step.  Grouped-query heads follow the same page (GQA backward): query head h reads
key / value head h // (Hq / Hkv), and dK, dV sum over the query heads of a group.

Layouts: q [B, Hq, Sq, D], k and v [B, Hkv, Skv, D], scores and P [B, Hq, Sq, Skv],
out [B, Hq, Sq, D].
"""

from __future__ import annotations

import numpy as np


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _group(hq: int, hkv: int) -> int:
    if hkv < 1 or hq % hkv != 0:
        raise ValueError("query heads must be a multiple of key/value heads")
    return hq // hkv


def _expand(t, g: int):
    """[B, Hkv, S, D] -> [B, Hkv * g, S, D]: key/value head j serves query heads j*g..j*g+g-1."""
    return np.repeat(t, g, axis=1)


def _fold(t, g: int):
    """[B, Hkv * g, S, D] -> [B, Hkv, S, D]: the sum over each group's query heads."""
    b, hq, s, d = t.shape
    return t.reshape(b, hq // g, g, s, d).sum(axis=2)


def qk_scores(q, k, scale: float = 1.0):
    """scores[b, h, i, j] = scale * sum_d q[b, h, i, d] * k[b, h // g, j, d]."""
    q, k = _f64(q), _f64(k)
    g = _group(q.shape[1], k.shape[1])
    return float(scale) * np.matmul(q, np.swapaxes(_expand(k, g), -1, -2))


def pv(p, v):
    """out[b, h, i, d] = sum_j p[b, h, i, j] * v[b, h // g, j, d]."""
    p, v = _f64(p), _f64(v)
    g = _group(p.shape[1], v.shape[1])
    return np.matmul(p, _expand(v, g))


def qk_backward(dscores, q, k, scale: float = 1.0):
    """(dq, dk) of scores = scale * Q K^T for the upstream gradient dscores."""
    ds, q, k = _f64(dscores), _f64(q), _f64(k)
    g = _group(q.shape[1], k.shape[1])
    dq = float(scale) * np.matmul(ds, _expand(k, g))
    dk = _fold(float(scale) * np.matmul(np.swapaxes(ds, -1, -2), q), g)
    return dq, dk


def pv_backward(dout, p, v):
    """(dp, dv) of out = P V for the upstream gradient dout."""
    do, p, v = _f64(dout), _f64(p), _f64(v)
    g = _group(p.shape[1], v.shape[1])
    dp = np.matmul(do, np.swapaxes(_expand(v, g), -1, -2))
    dv = _fold(np.matmul(np.swapaxes(p, -1, -2), do), g)
    return dp, dv
