"""Pins for the fp64 oracle: each test checks it against something other than
itself (a hand derivation, a closed form, a library routine, brute force or a
derived identity), chosen so that a dropped term, a wrong sign, index or
constant, or a transposed operand fails at least one of them.

Source of what is computed: the "Nyströmformer" review page, section
"Proposed method", bullets 1-6.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.signal
import scipy.special

from oracle import nystrom_ref as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_n4_m2.json")
GOLDEN_RAGGED = os.path.join(os.path.dirname(__file__), "golden", "closed_form_n8_m3.json")


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- golden ----

@pytest.mark.parametrize("path", [GOLDEN, GOLDEN_RAGGED], ids=["n4_m2", "n8_m3"])
def test_closed_form_worked_example(path):
    """Hand-derived (n, m) = (4, 2) and (8, 3), d=64 examples (tests/golden):
    pin the 1/sqrt(d) scale, segment means (n=8: segments of 2, 3, 3 rows), which
    axis each softmax runs over, Z_0, the update's constants, the F (Z (B V))
    association and the conv orientation."""
    f = json.load(open(path))
    q, k, v = (np.array(f[x]) for x in ("q", "k", "v"))
    for case in f["cases"]:
        r = R.nystrom_head(q, k, v, np.array(f["conv_w"]), f["m"], case["iters"])
        np.testing.assert_allclose(r["a_s"], f["a_s"], atol=1e-14)
        np.testing.assert_allclose(r["g"], f["g"], atol=1e-14)
        np.testing.assert_allclose(r["conv"], f["conv"], atol=1e-14)
        np.testing.assert_allclose(r["z"], case["z"], atol=1e-13)
        np.testing.assert_allclose(r["w"], case["w"], atol=1e-13)
        np.testing.assert_allclose(r["out"], case["out"], atol=1e-13)


# ---------------------------------------------------------- segment means ----

def brute_segment_means(x, m):
    """Row t belongs to segment i iff floor(i n/m) <= t < floor((i+1) n/m),
    i.e. i = ceil((t+1) m / n) - 1: each row is sent to its segment by that
    formula and the rows of a segment are averaged one by one."""
    n, d = len(x), len(x[0])
    sums = [[0.0] * d for _ in range(m)]
    counts = [0] * m
    for t in range(n):
        i = ((t + 1) * m + n - 1) // n - 1
        counts[i] += 1
        for c in range(d):
            sums[i][c] += x[t][c]
    return np.array([[sums[i][c] / counts[i] for c in range(d)] for i in range(m)])


@pytest.mark.parametrize("n,m,d", [(12, 3, 2), (8, 8, 3), (9, 1, 4), (64, 16, 5),
                                   (10, 3, 2), (1000, 48, 3), (300, 256, 2), (5, 2, 3)])
def test_segment_means_brute_force(n, m, d):
    x = rng(n * 31 + m).standard_normal((n, d))
    np.testing.assert_allclose(R.segment_means(x, m), brute_segment_means(x.tolist(), m),
                               rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("n,m", [(10, 3), (1000, 48), (300, 256), (7, 7), (64, 16), (9, 1)])
def test_segment_bounds_cover_the_rows_evenly(n, m):
    b = R.segment_bounds(n, m)
    assert b[0][0] == 0 and b[-1][1] == n
    assert all(b[i][1] == b[i + 1][0] for i in range(m - 1))
    assert {hi - lo for lo, hi in b} <= {n // m, -(-n // m)}
    if n % m == 0:
        assert all(hi - lo == n // m for lo, hi in b)


def test_segment_means_of_piecewise_constant_rows_are_the_constants():
    n, m = 1000, 48
    vals = rng(5).standard_normal((m, 3))
    x = np.empty((n, 3))
    for i, (lo, hi) in enumerate(R.segment_bounds(n, m)):
        x[lo:hi] = vals[i]
    np.testing.assert_allclose(R.segment_means(x, m), vals, rtol=1e-15, atol=1e-15)


def test_segment_means_reject_more_landmarks_than_rows():
    with pytest.raises(ValueError):
        R.segment_means(np.zeros((10, 2)), 11)


# ---------------------------------------------------------------- softmax ----

def test_softmax_rows_library_and_invariants():
    s = rng(1).standard_normal((7, 11)) * 5
    p = R.softmax_rows(s)
    np.testing.assert_allclose(p, scipy.special.softmax(s, axis=1), rtol=1e-14)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert (p > 0).all()
    # invariant to adding a constant per row; equal scores give 1/n
    np.testing.assert_allclose(R.softmax_rows(s + 100.0 * np.arange(7)[:, None]), p, rtol=1e-12)
    np.testing.assert_allclose(R.softmax_rows(np.full((2, 4), 3.0)), 0.25, atol=1e-16)
    # huge scores do not overflow
    assert np.isfinite(R.softmax_rows(np.array([[1e4, 0.0, -1e4]]))).all()


def test_landmark_kernel_scale_by_hand():
    """Scores q.k/sqrt(d) with d=4: q=(2,0,0,0), keys (1,0,0,0), (0,0,0,0) ->
    scores (1, 0) -> row (e/(e+1), 1/(e+1)), on the key axis."""
    qt = np.array([[2.0, 0, 0, 0], [0, 0, 0, 0]])
    kt = np.array([[1.0, 0, 0, 0], [0, 0, 0, 0]])
    a = R.landmark_kernel(qt, kt)
    e = math.e
    np.testing.assert_allclose(a[0], [e / (e + 1), 1 / (e + 1)], rtol=1e-15)
    np.testing.assert_allclose(a[1], [0.5, 0.5], rtol=1e-15)


# ------------------------------------------------------------------ pinv ----

def test_pinv_initial_norms_library():
    a = rng(2).standard_normal((5, 5))
    z0 = R.pinv_initial(a)
    expect = a.T / (np.linalg.norm(a, 1) * np.linalg.norm(a, np.inf))
    np.testing.assert_allclose(z0, expect, rtol=1e-15)


@pytest.mark.parametrize("seed", range(5))
def test_pinv_step_residual_recurrence(seed):
    """For ANY A, Z: with E = I - A Z, one update gives
    I - A Z' = 3/4 E^3 + 1/4 E^4 (derived by expanding the update's
    polynomial at X = I - E). Pins the constants 13, 15, 7, 1/4, the nesting,
    and that Z multiplies from the left."""
    g = rng(10 + seed)
    m = 6
    a = g.standard_normal((m, m))
    z = g.standard_normal((m, m)) * 0.1
    e = np.eye(m) - a @ z
    e_next = np.eye(m) - a @ R.pinv_step(a, z)
    np.testing.assert_allclose(e_next, 0.75 * np.linalg.matrix_power(e, 3)
                               + 0.25 * np.linalg.matrix_power(e, 4), atol=1e-10)


def test_pinv_diagonal_scalar_recurrence():
    """Diagonal A = diag(s): Z_0 = diag(s)/max(s)^2 and each diagonal entry's
    residual e = 1 - s z follows e' = 3/4 e^3 + 1/4 e^4 exactly ``iters``
    times (pins Z_0's normalisation and the update count)."""
    s = np.array([1.5, 0.7, 0.2, 0.05])
    a = np.diag(s)
    for iters in range(0, 9):
        z = R.pinv_iterative(a, iters)
        for i, si in enumerate(s):
            e = 1.0 - si * si / (s.max() ** 2)
            for _ in range(iters):
                e = 0.75 * e ** 3 + 0.25 * e ** 4
            assert abs(z[i, i] - (1.0 - e) / si) <= 1e-12 * max(1.0, abs(z[i, i]))
        assert np.abs(z - np.diag(np.diag(z))).max() == 0.0


@pytest.mark.parametrize("m,seed", [(4, 0), (8, 1), (16, 2)])
def test_pinv_matches_svd_when_converged(m, seed):
    """Well-conditioned softmax A_S (landmarks scaled up so A_S is near
    diagonal): 40 updates reach the SVD Moore-Penrose inverse."""
    g = rng(100 + seed)
    qt = g.standard_normal((m, 8)) * 3
    a = R.landmark_kernel(qt, qt)
    assert np.linalg.cond(a) < 50
    z = R.pinv_iterative(a, 40)
    np.testing.assert_allclose(z, R.svd_pinv(a), atol=1e-12)
    # Penrose conditions
    np.testing.assert_allclose(a @ z @ a, a, atol=1e-12)
    np.testing.assert_allclose(z @ a @ z, z, atol=1e-12)
    np.testing.assert_allclose((a @ z).T, a @ z, atol=1e-12)
    np.testing.assert_allclose((z @ a).T, z @ a, atol=1e-12)


def test_pinv_rank_deficient_projector():
    """Constant keys give A_S = J/m (all entries 1/m), a rank-1 projector:
    Z_0 = A_S and every update leaves it there (closed form)."""
    m = 8
    qt = rng(3).standard_normal((m, 4))
    kt = np.tile(rng(4).standard_normal((1, 4)), (m, 1))
    a = R.landmark_kernel(qt, kt)
    np.testing.assert_allclose(a, 1.0 / m, atol=1e-15)
    for iters in (0, 1, 6, 10):
        np.testing.assert_allclose(R.pinv_iterative(a, iters), 1.0 / m, atol=1e-14)
    np.testing.assert_allclose(R.svd_pinv(a), 1.0 / m, atol=1e-14)


# ------------------------------------------------------------------ conv ----

def brute_conv(v, w):
    n, d = len(v), len(v[0])
    ks = len(w)
    r = (ks - 1) // 2
    out = [[0.0] * d for _ in range(n)]
    for t in range(n):
        for c in range(d):
            tot = 0.0
            for j in range(ks):
                u = t + j - r
                if 0 <= u < n:
                    tot += w[j] * v[u][c]
            out[t][c] = tot
    return np.array(out)


@pytest.mark.parametrize("n,ks", [(10, 3), (7, 5), (5, 9), (40, 33), (3, 1)])
def test_conv_brute_force_and_library(n, ks):
    g = rng(n + ks)
    v = g.standard_normal((n, 3))
    w = g.standard_normal(ks)  # asymmetric: a flipped filter would fail
    got = R.depthwise_conv_seq(v, w)
    np.testing.assert_allclose(got, brute_conv(v.tolist(), w.tolist()), atol=1e-13)
    for c in range(3):
        lib = scipy.signal.correlate(v[:, c], w, mode="same", method="direct")
        np.testing.assert_allclose(got[:, c], lib, atol=1e-13)


def test_conv_closed_forms():
    n, ks = 12, 5
    w = np.array([0.5, -1.0, 2.0, 0.25, 3.0])
    delta = np.zeros(ks)
    delta[ks // 2] = 1.0
    v = rng(5).standard_normal((n, 4))
    np.testing.assert_allclose(R.depthwise_conv_seq(v, delta), v, atol=0)
    ones = R.depthwise_conv_seq(np.ones((n, 2)), w)
    # interior rows see every tap, edge rows a partial sum of taps
    np.testing.assert_allclose(ones[2:-2], w.sum(), atol=1e-15)
    np.testing.assert_allclose(ones[0], w[2:].sum(), atol=1e-15)
    np.testing.assert_allclose(ones[1], w[1:].sum(), atol=1e-15)
    np.testing.assert_allclose(ones[-1], w[:3].sum(), atol=1e-15)
    np.testing.assert_allclose(ones[-2], w[:4].sum(), atol=1e-15)
    np.testing.assert_allclose(R.depthwise_conv_seq(v, np.zeros(0)), 0.0)


# -------------------------------------------------- whole-head special cases ----

def test_constant_keys_give_mean_of_values():
    """K constant: every key scores alike, so exact attention and the
    Nyström output both equal mean(V) in every row, for any iters."""
    n, d, m = 64, 8, 8
    g = rng(6)
    q = g.standard_normal((n, d))
    k = np.tile(g.standard_normal((1, d)), (n, 1))
    v = g.standard_normal((n, d))
    exact = R.softmax_attention(q, k, v)
    np.testing.assert_allclose(exact, np.tile(v.mean(axis=0), (n, 1)), atol=1e-14)
    for iters in (0, 6):
        att = R.nystrom_head(q, k, v, np.zeros(0), m, iters)["att"]
        np.testing.assert_allclose(att, exact, atol=1e-13)


def test_single_landmark():
    """m = 1: A_S = [[1]], Z = [[1]] for every iters; each output row is the
    softmax over all keys of the mean query, applied to V."""
    n, d = 32, 8
    g = rng(7)
    q, k, v = (g.standard_normal((n, d)) for _ in range(3))
    r = R.nystrom_head(q, k, v, np.zeros(0), 1, 6)
    assert r["a_s"].shape == (1, 1) and abs(r["a_s"][0, 0] - 1) < 1e-15
    assert abs(r["z"][0, 0] - 1) < 1e-15
    qbar = q.mean(axis=0)
    p = scipy.special.softmax(k @ qbar / math.sqrt(d))
    np.testing.assert_allclose(r["att"], np.tile(p @ v, (n, 1)), atol=1e-14)


def test_m_equals_n_svd_pinv_is_exact_attention():
    """m = n (segments of one row): Q~ = Q, K~ = K, so all three softmax
    factors equal S and S S^+ S = S (a Penrose identity): with the SVD
    inverse the Nyström product is exact softmax attention."""
    n, d = 16, 8
    g = rng(8)
    q, k, v = (g.standard_normal((n, d)) for _ in range(3))
    r = R.nystrom_head(q, k, v, np.zeros(0), n, 0)
    s = R.landmark_kernel(q, k)
    att_svd = R.token_rows(q, k, R.svd_pinv(r["a_s"]) @ r["g"])
    np.testing.assert_allclose(att_svd, R.softmax_attention(q, k, v), atol=1e-10)
    np.testing.assert_allclose(r["a_s"], s, atol=1e-15)


def test_m_equals_n_iteration_converged_is_exact_attention():
    """m = n with a well-conditioned S and enough updates: the iterative
    inverse reaches the SVD one, so the output is exact attention."""
    n, d = 16, 16
    g = rng(9)
    basis = np.linalg.qr(g.standard_normal((d, d)))[0]
    q = basis[:n] * 6.0
    k = basis[:n] * 6.0
    v = g.standard_normal((n, d))
    r = R.nystrom_head(q, k, v, np.zeros(0), n, 40)
    assert np.linalg.cond(r["a_s"]) < 10
    np.testing.assert_allclose(r["att"], R.softmax_attention(q, k, v), atol=1e-10)


def test_softmax_factors_are_stochastic():
    n, d, m = 48, 8, 6
    g = rng(11)
    q, k, v = (g.standard_normal((n, d)) for _ in range(3))
    r = R.nystrom_head(q, k, v, np.zeros(0), m, 6)
    np.testing.assert_allclose(r["a_s"].sum(axis=1), 1.0, atol=1e-14)
    # G rows are convex combinations of V rows
    assert (r["g"] <= v.max(axis=0) + 1e-12).all() and (r["g"] >= v.min(axis=0) - 1e-12).all()


def test_approximation_error_vs_exact_attention_is_reported():
    """Nothing on the page bounds the approximation error for random inputs;
    this records it (relative max error of the attention term) and checks
    only that more landmarks with a converged inverse close the gap."""
    n, d = 64, 16
    g = rng(12)
    q, k, v = (g.standard_normal((n, d)) * 0.5 for _ in range(3))
    exact = R.softmax_attention(q, k, v)
    errs = {}
    for m in (8, 16, 64):
        att = R.nystrom_head(q, k, v, np.zeros(0), m, 60)["att"]
        errs[m] = np.abs(att - exact).max() / np.abs(exact).max()
    assert all(np.isfinite(list(errs.values())))
    assert errs[64] < 1e-8 < errs[8]


# ---------------------------------------------------------------- variants ----

def test_per_channel_conv_matches_scipy_column_by_column():
    g = rng(41)
    n, d, ks = 50, 6, 9
    v = g.standard_normal((n, d))
    w = g.standard_normal((d, ks))
    got = R.depthwise_conv_seq_channels(v, w)
    for c in range(d):
        np.testing.assert_allclose(got[:, c], scipy.signal.correlate(v[:, c], w[c], mode="same"),
                                   atol=1e-13)


def test_per_channel_conv_with_equal_filters_is_the_shared_conv():
    g = rng(42)
    v = g.standard_normal((40, 5))
    w = g.standard_normal(7)
    np.testing.assert_allclose(R.depthwise_conv_seq_channels(v, np.tile(w, (5, 1))),
                               R.depthwise_conv_seq(v, w), atol=1e-14)


def test_per_channel_delta_filters_shift_each_channel():
    """Channel c's filter is a delta at tap c: out[t, c] = V[t + c - 2, c]."""
    n, d, ks = 12, 5, 5
    v = rng(43).standard_normal((n, d))
    w = np.eye(d, ks)
    out = R.depthwise_conv_seq_channels(v, w)
    for c in range(d):
        shift = c - 2
        for t in range(n):
            want = v[t + shift, c] if 0 <= t + shift < n else 0.0
            assert out[t, c] == want


@pytest.mark.parametrize("n,length,m,ks", [(64, 64, 8, 5), (64, 40, 8, 5), (100, 77, 16, 9),
                                           (33, 1, 1, 3), (48, 48, 48, 0)])
def test_padded_head_is_its_unpadded_prefix(n, length, m, ks):
    """Masked formulation (key mask, zeroed V rows, zeroed output rows) against
    the plain forward pass on the first ``length`` rows alone."""
    g = rng(n + length)
    q, k, v = (g.standard_normal((n, 16)) for _ in range(3))
    w = g.standard_normal(ks)
    pad = R.nystrom_head_padded(q, k, v, w, m, 6, length)
    ref = R.nystrom_head(q[:length], k[:length], v[:length], w, m, 6)
    np.testing.assert_allclose(pad["out"][:length], ref["out"], atol=1e-12)
    assert (pad["out"][length:] == 0).all()
    np.testing.assert_allclose(pad["g"], ref["g"], atol=1e-13)


def test_padded_head_with_per_channel_filters():
    g = rng(44)
    n, length, d = 70, 50, 8
    q, k, v = (g.standard_normal((n, d)) for _ in range(3))
    w = g.standard_normal((d, 7))
    pad = R.nystrom_head_padded(q, k, v, w, 10, 6, length)
    ref = R.nystrom_head(q[:length], k[:length], v[:length], w, 10, 6)
    np.testing.assert_allclose(pad["out"][:length], ref["out"], atol=1e-12)


def test_batched_lengths_and_channel_filters():
    g = rng(45)
    B, H, n, d = 2, 2, 40, 8
    q, k, v = (g.standard_normal((B, H, n, d)) for _ in range(3))
    w = g.standard_normal((H, d, 5))
    out = R.nystrom_attention(q, k, v, w, 4, 6, lengths=[40, 25])
    for b, length in ((0, 40), (1, 25)):
        for h in range(H):
            ref = R.nystrom_head(q[b, h, :length], k[b, h, :length], v[b, h, :length], w[h], 4, 6)
            np.testing.assert_allclose(out[b, h, :length], ref["out"], atol=1e-12)
            assert (out[b, h, length:] == 0).all()
