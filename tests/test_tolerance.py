"""Pins of the parity checker (``oracle/tolerance.py``), CPU only.

Every GPU parity test passes or fails through these functions, so a wrong mantissa width, a
wrong exponent floor or a bound that is too wide would loosen every check at once without a
single test failing.  The pins here come from outside the checker: the spacing of the I/O
dtypes read off their bit patterns (numpy's own float16/float32 types, and bf16 built from the
upper half of a float32), hand-computed worst-case values of each bound, and planted errors
just inside (0.99x) and just outside (1.01x) each bound.
"""

import math

import numpy as np
import pytest

from oracle import tolerance as tol


# ------------------------------------------------------------------ ulp()


@pytest.mark.parametrize("x,dtype,expect", [
    (1.0, "bfloat16", 2.0 ** -7),
    (1.99, "bfloat16", 2.0 ** -7),
    (2.0, "bfloat16", 2.0 ** -6),
    (3.0, "bfloat16", 2.0 ** -6),
    (-3.0, "bfloat16", 2.0 ** -6),
    (1e-40, "bfloat16", 2.0 ** -133),   # subnormal: spacing is fixed at 2^(-126-7)
    (0.0, "bfloat16", 2.0 ** -133),
    (1.0, "float16", 2.0 ** -10),
    (65504.0, "float16", 32.0),
    (1e-8, "float16", 2.0 ** -24),      # subnormal: 2^(-14-10)
    (1.0, "float32", 2.0 ** -23),
    (1e-45, "float32", 2.0 ** -149),
])
def test_ulp_hand_values(x, dtype, expect):
    assert tol.ulp(x, dtype) == expect


def _bf16_from_bits(u16):
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def test_ulp_matches_the_bit_patterns_of_every_dtype():
    # The spacing of a dtype at a finite positive value v is next(v) - v, read off the bit
    # pattern (the next representable value has the next integer bit pattern).
    rng = np.random.default_rng(0)
    # float32 and float16 through numpy's own types
    for npt, name, top in ((np.float32, "float32", 0x7f7fffff), (np.float16, "float16", 0x7bff)):
        it = np.uint32 if npt is np.float32 else np.uint16
        bits = rng.integers(1, top, 20000).astype(it)
        v = bits.view(npt).astype(np.float64)
        nxt = (bits + it(1)).view(npt).astype(np.float64)
        got = tol.ulp(v, name)
        # at a power of two the spacing below is half the spacing above; ulp() is the spacing
        # of the binade of |v|, i.e. the one above
        assert np.array_equal(got, nxt - v), name
    # bf16: the upper 16 bits of a float32
    bits = rng.integers(1, 0x7f7f, 20000).astype(np.uint32)
    v = _bf16_from_bits(bits)
    nxt = _bf16_from_bits(bits + 1)
    assert np.array_equal(tol.ulp(v, "bfloat16"), nxt - v)


# ------------------------------------------------------------------ P and LSE


@pytest.mark.parametrize("dtype,ref,bound", [
    ("float32", 0.3, 1e-6),
    ("bfloat16", 1.5, 2.0 ** -7),
    ("bfloat16", 0.01, 2.0 ** -14),   # 0.01 in [2^-7, 2^-6): spacing 2^-7 * 2^-7
    ("float16", 0.25, 2.0 ** -12),
])
def test_check_probs_at_its_bound(dtype, ref, bound):
    r = np.array([ref, 0.0])
    ok_in = tol.check_probs(np.array([ref + 0.99 * bound, 0.0]), r, dtype)
    ok_out = tol.check_probs(np.array([ref - 1.01 * bound, 0.0]), r, dtype)
    assert ok_in[0] and not ok_out[0]
    assert ok_out[2] == 0 and abs(ok_out[1] - 1.01) < 1e-6


def test_check_lse_bound_and_minus_inf():
    ref = np.array([100.0, 0.5, -math.inf])
    # bounds: 1e-5 * 100 = 1e-3, and 1e-5 * max(1, 0.5) = 1e-5
    assert tol.check_lse(np.array([100.00099, 0.5 - 0.99e-5, -math.inf]), ref)[0]
    assert not tol.check_lse(np.array([100.00101, 0.5, -math.inf]), ref)[0]
    assert not tol.check_lse(np.array([100.0, 0.5 + 1.01e-5, -math.inf]), ref)[0]
    # -inf must be matched exactly, in both directions
    assert not tol.check_lse(np.array([100.0, 0.5, -1e30]), ref)[0]
    assert not tol.check_lse(np.array([100.0, -math.inf, -math.inf]), ref)[0]


# ------------------------------------------------------------------ dScores and delta


def _two_key_row(dp1):
    # P = (1/2, 1/2), dP = (1, dp1): delta = (1 + dp1) / 2, dS = (1 - dp1) / 4 * (1, -1)
    p = np.array([[0.5, 0.5]])
    dp = np.array([[1.0, dp1]])
    delta = 0.5 * (1.0 + dp1)
    ds = np.array([[0.5 * (1.0 - delta), 0.5 * (dp1 - delta)]])
    return p, dp, ds, delta


def test_check_dscores_float32_bound():
    # dP = (1, 1 + 2^-10): dS = (-2^-12, 2^-12), sum_k P_k|dP_k| = 1 + 2^-11, so
    # s_0 = 2^-12 + 0.5 * (1 + 1 + 2^-11) = 1 + 2^-11 (by hand)
    p, dp, ds, _ = _two_key_row(1.0 + 2.0 ** -10)
    assert ds[0, 0] == -(2.0 ** -12)
    bound0 = 1e-5 * (1.0 + 2.0 ** -11)
    for f, ok in ((0.99, True), (1.01, False)):
        gpu = ds.copy()
        gpu[0, 0] += f * bound0
        assert tol.check_dscores(gpu, ds, p, dp, "float32")[0] is ok


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_check_dscores_half_bound_is_one_ulp_when_not_cancelled(dtype):
    # dP = (1, 3): delta = 2, dS = (-1/2, 1/2); one ULP at 1/2 is 2^-8 (bf16) or 2^-11 (fp16),
    # the float32 floor 2^-20 * 0.5 * (1 + 2) is far below either, so the bound is one ULP
    p, dp, ds, _ = _two_key_row(3.0)
    assert ds[0, 0] == -0.5
    one = 2.0 ** -8 if dtype == "bfloat16" else 2.0 ** -11
    for f, ok in ((0.99, True), (1.01, False)):
        gpu = ds.copy()
        gpu[0, 0] -= f * one
        assert tol.check_dscores(gpu, ds, p, dp, dtype)[0] is ok


@pytest.mark.parametrize("dtype", ["bfloat16", "float16"])
def test_check_dscores_half_floor_under_cancellation(dtype):
    # dP = (1, 1): delta = 1 and dS = (0, 0) exactly; the bound is the float32 floor
    # 2^-20 * P_j * (|dP_j| + sum_k P_k |dP_k|) = 2^-20 * 0.5 * 2 = 2^-20, not one ULP of 0
    p, dp, ds, delta = _two_key_row(1.0)
    assert delta == 1.0 and not ds.any()
    for f, ok in ((0.99, True), (1.01, False)):
        gpu = ds.copy()
        gpu[0, 1] = f * 2.0 ** -20
        assert tol.check_dscores(gpu, ds, p, dp, dtype)[0] is ok


def test_check_dscores_masked_keys_leave_the_row_sum():
    # a masked key (valid False) takes no part in sum_k P_k |dP_k|: with the second key masked
    # the floor of key 0 is 2^-20 * 0.5 * (1 + 0.5) instead of 2^-20 * 0.5 * (1 + 0.5 + 0.5 * 7)
    p = np.array([[0.5, 0.5]])
    dp = np.array([[1.0, 7.0]])
    ref = np.array([[0.0, 0.0]])
    valid = np.array([[True, False]])
    floor = 2.0 ** -20 * 0.5 * 1.5
    assert tol.check_dscores(np.array([[0.99 * floor, 0.0]]), ref, p, dp, "bfloat16", valid)[0]
    assert not tol.check_dscores(np.array([[1.01 * floor, 0.0]]), ref, p, dp, "bfloat16",
                                 valid)[0]


def test_check_delta_bound():
    p, dp, _, delta = _two_key_row(-3.0)
    # sum_k P_k |dP_k| = 0.5 * 1 + 0.5 * 3 = 2: bound 2e-5
    assert tol.check_delta(np.array([delta + 0.99 * 2e-5]), np.array([delta]), p, dp)[0]
    assert not tol.check_delta(np.array([delta - 1.01 * 2e-5]), np.array([delta]), p, dp)[0]


# ------------------------------------------------------------------ d_sink


def test_check_dsink_bound():
    # one head, two rows: sink 0, LSE (0, log 2) -> exp(sink - LSE) = (1, 1/2); delta (1, -2)
    # -> c = (1, -1), sum |c| = 2, bound 2e-5 around d_sink = -(1 - 1) = 0
    lse = np.array([0.0, math.log(2.0)])
    delta = np.array([1.0, -2.0])
    sink = np.array([0.0])
    ref = np.array([0.0])
    kw = dict(batch=1, heads=1, q_len=2)
    assert tol.check_dsink(np.array([0.99 * 2e-5]), ref, lse, delta, sink, **kw)[0]
    assert not tol.check_dsink(np.array([1.01 * 2e-5]), ref, lse, delta, sink, **kw)[0]
    # a -inf sink contributes nothing: the bound collapses to 1e-30 and only 0 passes
    assert tol.check_dsink(np.array([0.0]), ref, lse, delta, np.array([-math.inf]), **kw)[0]
    assert not tol.check_dsink(np.array([1e-20]), ref, lse, delta, np.array([-math.inf]), **kw)[0]


@pytest.mark.parametrize("dtype,spacing", [("bfloat16", 2.0 ** -133), ("float16", 2.0 ** -24)])
def test_a_zero_reference_allows_only_the_smallest_spacing(dtype, spacing):
    # masked keys have P = 0 and dS = 0 exactly in the oracle: a GPU value may differ from 0 by
    # at most the dtype's smallest (subnormal) spacing, not by the spacing at 1
    ref = np.zeros((1, 2))
    assert tol.check_probs(np.array([[spacing, 0.0]]), ref, dtype)[0]
    assert not tol.check_probs(np.array([[2 * spacing, 0.0]]), ref, dtype)[0]
    assert not tol.check_probs(np.array([[1e-3, 0.0]]), ref, dtype)[0]
    p = np.zeros((1, 2))  # P = 0 on the key: the float32 floor is 0 as well
    dp = np.ones((1, 2))
    assert not tol.check_dscores(np.array([[2 * spacing, 0.0]]), ref, p, dp, dtype)[0]



@pytest.mark.parametrize("dtype,one", [("float32", 0.0), ("bfloat16", 2.0 ** -7),
                                       ("float16", 2.0 ** -10)])
def test_check_scores_bound(dtype, one):
    # score 1.5 with scale 0.5 and sum_d |q_d k_d| = 8: floor 2^-16 * 0.5 * 8 = 2^-14, plus one
    # ULP at 1.5 for a 16-bit output (2^-7 bf16, 2^-10 fp16)
    ref = np.array([1.5])
    absd = np.array([8.0])
    bound = 2.0 ** -14 + one
    assert tol.check_scores(ref + 0.99 * bound, ref, absd, 0.5, dtype)[0]
    assert not tol.check_scores(ref - 1.01 * bound, ref, absd, 0.5, dtype)[0]
    # the scale's sign does not matter
    assert tol.check_scores(ref + 0.99 * bound, ref, absd, -0.5, dtype)[0]


def test_check_pv_bound():
    # output 2.0 with sum_j |p_j v_jd| = 4: floor 2^-16 * 4 = 2^-14, plus one bf16 ULP at 2 (2^-6)
    ref = np.array([2.0])
    absd = np.array([4.0])
    for dtype, one in (("float32", 0.0), ("bfloat16", 2.0 ** -6)):
        bound = 2.0 ** -14 + one
        assert tol.check_pv(ref + 0.99 * bound, ref, absd, dtype)[0]
        assert not tol.check_pv(ref + 1.01 * bound, ref, absd, dtype)[0]
