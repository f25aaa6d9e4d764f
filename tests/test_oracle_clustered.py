"""Pins of the clustered-attention oracle (centroid path), each against
something other than itself: brute-force K-means on tiny inputs, exact
recovery of well-separated clusters, C = n (every query its own cluster:
exact softmax attention), and planted mistakes."""
import numpy as np

from oracle import clustered_ref as CR
from oracle import nystrom_ref as R


def brute_kmeans(q, C, iters):
    """Pure-Python loops, the textbook algorithm."""
    n, d = len(q), len(q[0])
    mu = []
    for i in range(C):
        lo, hi = i * n // C, (i + 1) * n // C
        mu.append([sum(q[t][j] for t in range(lo, hi)) / (hi - lo) for j in range(d)])
    for _ in range(iters):
        prev = [row[:] for row in mu]
        assign = []
        for t in range(n):
            best, best_c = None, -1
            for c in range(C):
                dist = sum((q[t][j] - mu[c][j]) ** 2 for j in range(d))
                if best is None or dist < best:
                    best, best_c = dist, c
            assign.append(best_c)
        for c in range(C):
            members = [t for t in range(n) if assign[t] == c]
            if members:
                mu[c] = [sum(q[t][j] for t in members) / len(members) for j in range(d)]
    return assign, prev, mu


def test_kmeans_matches_brute_force():
    rng = np.random.default_rng(1)
    for n, C, d, iters in [(12, 3, 2, 1), (20, 4, 3, 3), (17, 5, 4, 6)]:
        q = rng.standard_normal((n, d))
        a, prev, mu = CR.kmeans_queries(q, C, iters)
        ba, bprev, bmu = brute_kmeans(q.tolist(), C, iters)
        assert a.tolist() == ba
        np.testing.assert_allclose(prev, bprev, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(mu, bmu, rtol=1e-12, atol=1e-12)


def test_well_separated_clusters_are_recovered():
    """Queries around C far-apart centres, in contiguous runs: the segment
    means start inside the right clusters, so one round assigns every query
    to its own centre's cluster and the centroids are the run means."""
    rng = np.random.default_rng(2)
    C, per, d = 4, 10, 8
    centres = rng.standard_normal((C, d)) * 50.0
    q = np.repeat(centres, per, axis=0) + rng.standard_normal((C * per, d))
    a, _, mu = CR.kmeans_queries(q, C, 3)
    assert a.tolist() == np.repeat(np.arange(C), per).tolist()
    np.testing.assert_allclose(mu, q.reshape(C, per, d).mean(axis=1), rtol=1e-12, atol=1e-12)


def test_one_cluster_per_query_is_exact_attention():
    """C = n: the segment means are the queries themselves, every query is
    its own nearest centroid, and the centroid attention is exact softmax
    attention."""
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((24, 8)) for _ in range(3))
    out = CR.clustered_head(q, k, v, 24, 2)["out"]
    np.testing.assert_allclose(out, R.softmax_attention(q, k, v), rtol=1e-12, atol=1e-12)


def test_empty_cluster_keeps_its_centroid():
    q = np.array([[0.0], [0.1], [10.0], [10.1], [10.2], [9.9]])
    mu = np.array([[0.05], [10.0], [100.0]])
    a = CR.kmeans_assign(q, mu)
    assert a.tolist() == [0, 0, 1, 1, 1, 1]
    new = CR.kmeans_update(q, a, mu)
    np.testing.assert_allclose(new[:, 0], [0.05, 10.05, 100.0])


def test_ties_go_to_the_lowest_index():
    q = np.array([[1.0, 0.0]])
    mu = np.array([[0.0, 0.0], [2.0, 0.0]])  # both at distance 1
    assert CR.kmeans_assign(q, mu).tolist() == [0]


def test_pins_reject_planted_mistakes(monkeypatch):
    """Three plausible bugs each fail a pin above: a distance without the
    square (L1-like sum of differences), centroids not updated, and the
    attention scaled by 1/d instead of 1/sqrt(d)."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((20, 3))
    ba, _, bmu = brute_kmeans(q.tolist(), 4, 3)

    def assign_no_square(q_, mu_):
        return np.argmin(np.abs(np.asarray(q_)[:, None, :] - np.asarray(mu_)[None]).sum(axis=2), axis=1)

    with monkeypatch.context() as mp:
        mp.setattr(CR, "kmeans_assign", assign_no_square)
        a, _, mu = CR.kmeans_queries(q, 4, 3)
        assert a.tolist() != ba or not np.allclose(mu, bmu)
    with monkeypatch.context() as mp:
        mp.setattr(CR, "kmeans_update", lambda q_, a_, mu_: np.asarray(mu_, np.float64))
        _, _, mu = CR.kmeans_queries(q, 4, 3)
        assert not np.allclose(mu, bmu)
    k, v = rng.standard_normal((20, 3)), rng.standard_normal((20, 3))
    with monkeypatch.context() as mp:
        mp.setattr(R, "landmark_rows",
                   lambda qt, k_, v_: R.softmax_rows(np.asarray(qt) @ np.asarray(k_).T / 3.0) @ v_)
        out = CR.clustered_head(q, k, v, 20, 1)["out"]
        assert not np.allclose(out, R.softmax_attention(q, k, v))
