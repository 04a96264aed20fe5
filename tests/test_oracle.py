"""Pins for the FP64 oracle, against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a closed form, an invariant
of the definition, a finite difference, or a second, differently written formulation on tiny
inputs.  Between them they fail on the plausible mistakes: a dropped max-shift (overflow in
the shift test), a wrong sign or dropped term in the VJP or in d_sink (finite differences), a
wrong mask index or row decomposition (deletion, causal and three-way mask tests), a wrong
sink entry point (sigmoid and sink=-inf tests).

Definitions pinned: softmax along the key dimension ("[WS1][kernels] Add fixed-order
joint-attention softmax for Qwen-Image", Summary), its VJP (same page, "Fixed-order
backward"), LSE and fully masked rows ("Batch-invariant attention (standard softmax--cuda
version)", Implementation, Path Status), the causal condition (same page, Prefill / Decode /
KV-cache Contract), the per-head sink logit ("[ROCm] Jax Add softmax sink (learnable
off-by-one) support", Description and review thread).
"""

import math

import numpy as np
import pytest

import oracle

NEG_INF = -math.inf


def fwd1(x, sink=None, key_mask=None, causal=False, q_len=1):
    """Oracle forward on rows x [n, L] of a single (batch=1, heads=1) problem."""
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    n, L = x.shape
    sk = None if sink is None else np.array([sink], dtype=np.float64)
    km = None if key_mask is None else np.asarray(key_mask, dtype=np.uint8).reshape(1, L)
    return oracle.softmax_fwd(x, batch=1, heads=1, q_len=n, causal=causal, key_mask=km,
                              sink=sk)


def bwd1(p, dp, key_mask=None):
    p = np.atleast_2d(np.asarray(p, dtype=np.float64))
    dp = np.atleast_2d(np.asarray(dp, dtype=np.float64))
    n, L = p.shape
    km = None if key_mask is None else np.asarray(key_mask, dtype=np.uint8).reshape(1, L)
    return oracle.softmax_bwd(p, dp, batch=1, heads=1, q_len=n, key_mask=km)


# ----------------------------------------------------------------------------- forward


@pytest.mark.parametrize("L", [1, 2, 7, 256, 257, 1000])
@pytest.mark.parametrize("with_sink", [False, True])
def test_rows_sum_to_one(L, with_sink):
    rng = np.random.default_rng(L)
    x = rng.normal(0, 4, size=(5, L))
    sink = 0.7 if with_sink else None
    p, lse = fwd1(x, sink=sink)
    total = p.sum(axis=1)
    if with_sink:
        total = total + np.exp(sink - lse)
    np.testing.assert_allclose(total, 1.0, rtol=0, atol=1e-14)
    assert np.all(p >= 0)


@pytest.mark.parametrize("c", [0.0, -3.5, 17.0, 500.0, -800.0])
@pytest.mark.parametrize("L", [1, 3, 64, 4352])
def test_constant_row(c, L):
    p, lse = fwd1(np.full((1, L), c))
    np.testing.assert_allclose(p, 1.0 / L, rtol=1e-15, atol=0)
    np.testing.assert_allclose(lse, c + math.log(L), rtol=1e-15, atol=1e-13)


def test_constant_row_with_mask_counts_valid_keys_only():
    L = 10
    km = np.array([1, 0, 1, 1, 0, 0, 1, 1, 1, 0])
    p, lse = fwd1(np.full((1, L), 2.0), key_mask=km)
    nv = km.sum()
    np.testing.assert_allclose(p[0][km == 1], 1.0 / nv, rtol=1e-15)
    assert np.all(p[0][km == 0] == 0.0)
    np.testing.assert_allclose(lse, 2.0 + math.log(nv), rtol=1e-15)


@pytest.mark.parametrize("c", [1000.0, -1000.0, 88.5, 1e5])
def test_shift_invariance(c):
    # A missing max-shift overflows exp() at these offsets and fails here.
    rng = np.random.default_rng(1)
    x = rng.normal(0, 3, size=(4, 300))
    for sink in (None, 0.25):
        p0, l0 = fwd1(x, sink=sink)
        p1, l1 = fwd1(x + c, sink=None if sink is None else sink + c)
        np.testing.assert_allclose(p1, p0, rtol=1e-9, atol=1e-300)
        np.testing.assert_allclose(l1, l0 + c, rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("x0,x1", [(0.0, 0.0), (1.0, -2.0), (-3.0, 4.5), (30.0, -30.0),
                                   (700.0, 690.0), (-0.125, 0.125)])
def test_two_keys_logistic(x0, x1):
    p, lse = fwd1([[x0, x1]])
    p0 = 1.0 / (1.0 + math.exp(x1 - x0))
    np.testing.assert_allclose(p[0, 0], p0, rtol=1e-14)
    np.testing.assert_allclose(p[0, 1], 1.0 / (1.0 + math.exp(x0 - x1)), rtol=1e-14)
    ref_lse = max(x0, x1) + math.log1p(math.exp(-abs(x0 - x1)))
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-15, atol=1e-15)


# ----------------------------------------------------------------------------- sink


def test_sink_minus_inf_is_vanilla_exactly():
    rng = np.random.default_rng(2)
    x = rng.normal(0, 3, size=(6, 129))
    x[2, :] = NEG_INF  # a fully masked row too
    p0, l0 = fwd1(x)
    p1, l1 = fwd1(x, sink=NEG_INF)
    assert np.array_equal(p0, p1) and np.array_equal(l0, l1)


@pytest.mark.parametrize("x0,s", [(0.0, 0.0), (2.0, -1.0), (-4.0, 3.0), (50.0, 49.0)])
def test_one_key_with_sink_is_sigmoid(x0, s):
    p, lse = fwd1([[x0]], sink=s)
    np.testing.assert_allclose(p[0, 0], 1.0 / (1.0 + math.exp(s - x0)), rtol=1e-14)
    ref_lse = max(x0, s) + math.log1p(math.exp(-abs(x0 - s)))
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-15)


def test_fully_masked_rows():
    x = np.full((1, 8), NEG_INF)
    p, lse = fwd1(x)
    assert np.all(p == 0) and lse[0] == NEG_INF
    p, lse = fwd1(x, sink=1.5)
    assert np.all(p == 0) and lse[0] == 1.5
    p, lse = fwd1(np.ones((1, 8)), key_mask=np.zeros(8))
    assert np.all(p == 0) and lse[0] == NEG_INF
    ds, delta = bwd1(np.zeros((1, 8)), np.arange(8.0), key_mask=np.zeros(8))
    assert np.all(ds == 0) and delta[0] == 0


# ----------------------------------------------------------------------------- masks


def test_masked_keys_equal_deleting_them():
    rng = np.random.default_rng(3)
    L = 97
    x = rng.normal(0, 4, size=(1, L))
    km = (rng.random(L) < 0.6).astype(np.uint8)
    for sink in (None, -0.3):
        p, lse = fwd1(x, key_mask=km, sink=sink)
        pc, lc = fwd1(x[:, km == 1], sink=sink)
        np.testing.assert_allclose(p[0, km == 1], pc[0], rtol=1e-14)
        assert np.all(p[0, km == 0] == 0)
        np.testing.assert_allclose(lse, lc, rtol=1e-15)


def test_causal_square_is_lower_triangular():
    rng = np.random.default_rng(4)
    L = 33
    x = rng.normal(0, 3, size=(L, L))
    p, lse = fwd1(x, causal=True)
    for i in range(L):
        assert np.all(p[i, i + 1:] == 0)
        pc, lc = fwd1(x[i:i + 1, :i + 1])
        np.testing.assert_allclose(p[i, :i + 1], pc[0], rtol=1e-14)
        np.testing.assert_allclose(lse[i], lc[0], rtol=1e-15)


def test_causal_rectangular_key_sets():
    # q_len = 3 queries at the end of L = 5 keys: query i sees keys 0 .. 2 + i.
    expected_valid = [[1, 1, 1, 0, 0], [1, 1, 1, 1, 0], [1, 1, 1, 1, 1]]
    x = np.zeros((3, 5))
    p, _ = fwd1(x, causal=True)
    for i in range(3):
        v = np.array(expected_valid[i], dtype=bool)
        np.testing.assert_allclose(p[i, v], 1.0 / v.sum(), rtol=1e-15)
        assert np.all(p[i, ~v] == 0)


def test_valid_len_equals_key_mask_equals_neg_inf_fill():
    rng = np.random.default_rng(5)
    B, H, Sq, L = 3, 2, 4, 40
    lens = np.array([40, 17, 1], dtype=np.int32)
    x = rng.normal(0, 4, size=(B * H * Sq, L))
    sink = rng.normal(0, 1, size=H)
    km = np.zeros((B, L), dtype=np.uint8)
    fill = x.copy()
    for b in range(B):
        km[b, :lens[b]] = 1
    for r in range(B * H * Sq):
        b = r // (H * Sq)  # rows are ordered [batch][heads][q_len]
        fill[r, lens[b]:] = NEG_INF
    kw = dict(batch=B, heads=H, q_len=Sq, sink=sink)
    a = oracle.softmax_fwd(x, kv_valid_len=lens, **kw)
    b_ = oracle.softmax_fwd(x, key_mask=km, **kw)
    c = oracle.softmax_fwd(fill, **kw)
    for u, v in ((a, b_), (a, c)):
        assert np.array_equal(u[0], v[0]) and np.array_equal(u[1], v[1])
    # and the sink is per head: rows of head 1 use sink[1]
    r = 1 * H * Sq + 1 * Sq + 2  # b=1, h=1, i=2
    pc, lc = fwd1(x[r:r + 1, :lens[1]], sink=sink[1])
    np.testing.assert_allclose(a[0][r, :lens[1]], pc[0], rtol=1e-14)
    np.testing.assert_allclose(a[1][r], lc[0], rtol=1e-15)


def test_row_ids_select_the_same_rows():
    rng = np.random.default_rng(6)
    B, H, Sq, L = 2, 3, 5, 11
    x = rng.normal(0, 2, size=(B * H * Sq, L))
    kv = np.array([11, 6], dtype=np.int32)
    sink = np.array([0.1, -0.2, 0.3])
    full_p, full_l = oracle.softmax_fwd(x, batch=B, heads=H, q_len=Sq, causal=True,
                                        kv_valid_len=kv, sink=sink)
    ids = np.array([29, 0, 17, 5])
    p, lse = oracle.softmax_fwd(x[ids], batch=B, heads=H, q_len=Sq, causal=True,
                                kv_valid_len=kv, sink=sink, row_ids=ids)
    assert np.array_equal(p, full_p[ids]) and np.array_equal(lse, full_l[ids])


def test_row_ids_past_2_31_find_their_batch_entry_and_position():
    # A problem of 65536 x 4097 x 8 rows (more than 2^31): a row's batch entry and query
    # position decide its mask, so each given row must equal the same query position of a
    # one-entry, one-head problem with that entry's valid length, forward and backward.
    B, H, Sq, L = 65536, 4097, 8, 8
    rng = np.random.default_rng(8)
    kv = rng.integers(0, L + 1, size=B).astype(np.int32)
    base = (1 << 31) // Sq * Sq
    ids = np.array([base - 1, base, base + 5, base + 8 * Sq + 7, B * H * Sq - 1], dtype=np.int64)
    x = rng.normal(0, 2, size=(len(ids), L))
    dp = rng.normal(0, 1, size=(len(ids), L))
    geo = dict(batch=B, heads=H, q_len=Sq, causal=True, kv_valid_len=kv)
    p, lse = oracle.softmax_fwd(x, row_ids=ids, **geo)
    ds, delta = oracle.softmax_bwd(p, dp, row_ids=ids, **geo)
    for k, r in enumerate(ids):
        b, i = int(r) // (H * Sq), int(r) % Sq
        one = dict(batch=1, heads=1, q_len=Sq, causal=True, kv_valid_len=kv[b:b + 1])
        p1, l1 = oracle.softmax_fwd(x[k:k + 1], row_ids=[i], **one)
        ds1, d1 = oracle.softmax_bwd(p1, dp[k:k + 1], row_ids=[i], **one)
        assert np.array_equal(p[k], p1[0]) and np.array_equal(lse[k], l1[0], equal_nan=True)
        assert np.array_equal(ds[k], ds1[0]) and np.array_equal(delta[k], d1[0])
        # and the mask it applied is the definition's: causal bound and valid length
        allowed = (np.arange(L) <= L - Sq + i) & (np.arange(L) < kv[b])
        assert np.all(p[k][~allowed] == 0) and (not allowed.any() or np.all(p[k][allowed] > 0))


# ----------------------------------------------------------------------------- brute force


def brute_softmax(x, sink=None):
    """P_j = 1 / sum_k exp(x_k - x_j): the definition rearranged, with exactly rounded sums."""
    terms = list(x) + ([sink] if sink is not None else [])
    p = [1.0 / math.fsum(math.exp(xk - xj) for xk in terms) for xj in x]
    lse = x[0] - math.log(p[0])
    return p, lse


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 6])
def test_brute_force_tiny(L):
    rng = np.random.default_rng(10 + L)
    for _ in range(20):
        x = list(rng.normal(0, 3, size=L))
        for sink in (None, float(rng.normal())):
            p, lse = fwd1([x], sink=sink)
            bp, bl = brute_softmax(x, sink)
            np.testing.assert_allclose(p[0], bp, rtol=1e-13)
            np.testing.assert_allclose(lse[0], bl, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("L", [1, 2, 4, 6])
def test_backward_equals_jacobian_transpose(L):
    # dS = J^T dP with J_jk = dP_j/dx_k = P_j (delta_jk - P_k): a matrix-vector product,
    # not the oracle's P*(dP - delta) form.
    rng = np.random.default_rng(20 + L)
    for sink in (None, 0.4):
        x = rng.normal(0, 2, size=(1, L))
        dp = rng.normal(0, 1, size=(1, L))
        p, _ = fwd1(x, sink=sink)
        ds, delta = bwd1(p, dp)
        P = p[0]
        J = np.diag(P) - np.outer(P, P)
        np.testing.assert_allclose(ds[0], J.T @ dp[0], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(delta[0], math.fsum(P * dp[0]), rtol=1e-14, atol=1e-16)


# ----------------------------------------------------------------------------- gradients


def loss(x, dp, sink=None, key_mask=None):
    """f(x) = sum_j dP_j P_j(x): its gradient in x is dScores."""
    p, _ = fwd1(x, sink=sink, key_mask=key_mask)
    return math.fsum((p * dp).ravel())


@pytest.mark.parametrize("L", [1, 2, 5, 8])
@pytest.mark.parametrize("sink", [None, 0.8])
@pytest.mark.parametrize("masked", [False, True])
def test_dscores_central_difference(L, sink, masked):
    rng = np.random.default_rng(30 + L)
    x = rng.normal(0, 2, size=(1, L))
    dp = rng.normal(0, 1, size=(1, L))
    km = None
    if masked:
        km = np.ones(L, dtype=np.uint8)
        km[::3] = 0
        if km.sum() == 0:
            km[-1] = 1
    p, _ = fwd1(x, sink=sink, key_mask=km)
    ds, delta = bwd1(p, dp, key_mask=km)
    h = 1e-6
    fd = np.zeros(L)
    for j in range(L):
        xp = x.copy()
        xm = x.copy()
        xp[0, j] += h
        xm[0, j] -= h
        fd[j] = (loss(xp, dp, sink, km) - loss(xm, dp, sink, km)) / (2 * h)
    np.testing.assert_allclose(ds[0], fd, rtol=1e-7, atol=1e-9)
    # sum_j dS_j = delta * P_sink (zero without a sink)
    _, lse = fwd1(x, sink=sink, key_mask=km)
    p_sink = 0.0 if sink is None else math.exp(sink - lse[0])
    np.testing.assert_allclose(ds[0].sum(), delta[0] * p_sink, rtol=0, atol=1e-14)


def test_dsink_central_difference():
    rng = np.random.default_rng(40)
    B, H, Sq, L = 2, 3, 4, 6
    x = rng.normal(0, 2, size=(B * H * Sq, L))
    dp = rng.normal(0, 1, size=x.shape)
    sink = rng.normal(0, 1, size=H)
    kv = np.array([6, 3], dtype=np.int32)
    kw = dict(batch=B, heads=H, q_len=Sq, causal=True, kv_valid_len=kv)

    def total_loss(s):
        p, _ = oracle.softmax_fwd(x, sink=s, **kw)
        return math.fsum((p * dp).ravel())

    p, lse = oracle.softmax_fwd(x, sink=sink, **kw)
    _, delta = oracle.softmax_bwd(p, dp, **kw)
    dsink = oracle.sink_grad(lse, delta, sink, batch=B, heads=H, q_len=Sq)
    h = 1e-6
    for hh in range(H):
        sp = sink.copy()
        sm = sink.copy()
        sp[hh] += h
        sm[hh] -= h
        fd = (total_loss(sp) - total_loss(sm)) / (2 * h)
        np.testing.assert_allclose(dsink[hh], fd, rtol=1e-7, atol=1e-9)


def test_dsink_minus_inf_head_is_zero():
    lse = np.array([1.0, 2.0, -math.inf, 0.5])
    delta = np.array([0.5, -1.0, 0.0, 2.0])
    d = oracle.sink_grad(lse, delta, np.array([NEG_INF, NEG_INF]), batch=1, heads=2, q_len=2)
    assert np.all(d == 0)


def test_oracle_rejects_bad_sizes():
    with pytest.raises(ValueError):
        oracle.softmax_fwd(np.zeros((3, 4)), batch=1, heads=1, q_len=2)
    with pytest.raises(ValueError):  # causal needs q_len <= key length
        oracle.softmax_fwd(np.zeros((5, 2)), batch=1, heads=1, q_len=5, causal=True)
