"""Pins of the FP64 oracle of the QK and PV contractions (``oracle/gemm.py``), on the CPU.
Each check rests on something other than the oracle's own formula:
- exact closed forms (an identity query block, one-hot probabilities, a hand-computed example);
- brute-force loops over tiny shapes;
- the scale's linearity;
- central differences of scalar losses for every backward product (exact for these bilinear
  maps up to rounding), which pins the group sums of grouped-query heads."""

import numpy as np
import pytest

from oracle import gemm


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_hand_computed_example():
    q = np.array([[[[1.0, 2.0]]]])                      # B1 H1 Sq1 D2
    k = np.array([[[[3.0, 4.0], [5.0, 6.0]]]])          # Skv 2
    assert np.array_equal(gemm.qk_scores(q, k, 0.5), [[[[5.5, 8.5]]]])
    p = np.array([[[[0.25, 0.75]]]])
    v = np.array([[[[4.0, 8.0], [12.0, 16.0]]]])
    assert np.array_equal(gemm.pv(p, v), [[[[10.0, 14.0]]]])


def test_identity_queries_read_out_the_keys():
    # Sq = D and q = I: scores[b, h] is k[b, h // g] transposed, exactly
    B, Hq, Hkv, D, Skv = 2, 4, 2, 5, 7
    q = np.broadcast_to(np.eye(D), (B, Hq, D, D)).copy()
    k = rand((B, Hkv, Skv, D), 1)
    s = gemm.qk_scores(q, k)
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(s[b, h], k[b, h // (Hq // Hkv)].T)


def test_one_hot_probabilities_pick_value_rows():
    B, Hq, Hkv, Sq, Skv, D = 1, 6, 3, 4, 9, 3
    pick = np.random.default_rng(2).integers(0, Skv, size=(B, Hq, Sq))
    p = np.zeros((B, Hq, Sq, Skv))
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                p[b, h, i, pick[b, h, i]] = 1.0
    v = rand((B, Hkv, Skv, D), 3)
    out = gemm.pv(p, v)
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                assert np.array_equal(out[b, h, i], v[b, h // 2, pick[b, h, i]])


def test_brute_force_loops():
    B, Hq, Hkv, Sq, Skv, D = 2, 2, 1, 3, 4, 3
    q, k, v = rand((B, Hq, Sq, D), 4), rand((B, Hkv, Skv, D), 5), rand((B, Hkv, Skv, D), 6)
    p = rand((B, Hq, Sq, Skv), 7)
    s, o = gemm.qk_scores(q, k, 0.25), gemm.pv(p, v)
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                for j in range(Skv):
                    ref = 0.0
                    for d in range(D):
                        ref += q[b, h, i, d] * k[b, 0, j, d]
                    assert s[b, h, i, j] == pytest.approx(0.25 * ref, rel=1e-14, abs=1e-14)
                for d in range(D):
                    ref = 0.0
                    for j in range(Skv):
                        ref += p[b, h, i, j] * v[b, 0, j, d]
                    assert o[b, h, i, d] == pytest.approx(ref, rel=1e-14, abs=1e-14)


def test_scale_is_linear():
    q, k = rand((1, 2, 3, 8), 8), rand((1, 2, 5, 8), 9)
    assert np.allclose(gemm.qk_scores(q, k, 0.125), 0.125 * gemm.qk_scores(q, k, 1.0),
                       rtol=0, atol=1e-15)


def central_grad(f, x, h=1e-3):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        g[i] = (f(xp) - f(xm)) / (2 * h)
    return g


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (3, 1)])
def test_qk_backward_is_the_gradient(hq, hkv):
    B, Sq, Skv, D, scale = 1, 3, 4, 5, 0.3
    q, k = rand((B, hq, Sq, D), 10), rand((B, hkv, Skv, D), 11)
    g = rand((B, hq, Sq, Skv), 12)  # upstream gradient of the scores
    dq, dk = gemm.qk_backward(g, q, k, scale)
    fq = lambda x: float((g * gemm.qk_scores(x, k, scale)).sum())
    fk = lambda x: float((g * gemm.qk_scores(q, x, scale)).sum())
    assert np.allclose(dq, central_grad(fq, q), rtol=1e-8, atol=1e-9)
    assert np.allclose(dk, central_grad(fk, k), rtol=1e-8, atol=1e-9)


@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (3, 1)])
def test_pv_backward_is_the_gradient(hq, hkv):
    B, Sq, Skv, D = 1, 3, 4, 5
    p, v = rand((B, hq, Sq, Skv), 13), rand((B, hkv, Skv, D), 14)
    g = rand((B, hq, Sq, D), 15)  # upstream gradient of the output
    dp, dv = gemm.pv_backward(g, p, v)
    fp = lambda x: float((g * gemm.pv(x, v)).sum())
    fv = lambda x: float((g * gemm.pv(p, x)).sum())
    assert np.allclose(dp, central_grad(fp, p), rtol=1e-8, atol=1e-9)
    assert np.allclose(dv, central_grad(fv, v), rtol=1e-8, atol=1e-9)


def test_heads_must_group_evenly():
    with pytest.raises(ValueError):
        gemm.qk_scores(np.zeros((1, 3, 2, 4)), np.zeros((1, 2, 2, 4)))
    with pytest.raises(ValueError):
        gemm.pv(np.zeros((1, 4, 2, 3)), np.zeros((1, 3, 3, 4)))
