"""fp64 CPU oracle for clustered attention (centroid path).

TEST INFRASTRUCTURE. Only the tests and the benchmark's CPU leg may import
or run this module; the CUDA library never calls it and shares no code with
it.

Source: the review page "Fast Transformers with Clustered Attention"
(nubint.ai), section "Proposed method" (提出的方法): queries are grouped into
clusters by K-means (bullet 1), attention is computed once per cluster
centroid (bullet 2) and used for every query of the cluster; the cost is
linear in the sequence length for a fixed number of clusters (bullet 4).
The refinement that recomputes each query's top keys exactly (bullet 3,
"i-clustered") is not part of this path.

Readings where the page is silent:
* K-means is Lloyd's algorithm on each head's queries Q [n, d], squared
  Euclidean distance, run for a fixed number of iterations (no early exit);
  each iteration assigns every query to its nearest centroid (ties go to the
  lowest cluster index) and then moves every centroid to the mean of its
  queries (a cluster with no query keeps its centroid);
* the initial centroids are the segment means of the queries over C
  contiguous segments (the landmarks of the Nyström method);
* the centroid attention uses the scale 1/sqrt(d): G_c = softmax(mu_c K^T /
  sqrt(d)) V, and query i receives row G_{a(i)} of its cluster a(i);
* the output is that broadcast alone (no convolution term).
"""
from __future__ import annotations

import numpy as np

from oracle import nystrom_ref as R

__all__ = ["kmeans_assign", "kmeans_update", "kmeans_queries", "clustered_head",
           "clustered_attention"]


def kmeans_assign(q, mu):
    """Index of the nearest centroid for every row of q (squared Euclidean
    distance; ties go to the lowest index)."""
    q, mu = np.asarray(q, np.float64), np.asarray(mu, np.float64)
    dist = ((q[:, None, :] - mu[None, :, :]) ** 2).sum(axis=2)  # [n, C]
    return np.argmin(dist, axis=1)  # first minimum: the lowest index


def kmeans_update(q, assign, mu):
    """Every centroid moves to the mean of its queries; a centroid with no
    query stays where it is."""
    q = np.asarray(q, np.float64)
    new = np.array(mu, dtype=np.float64, copy=True)
    for c in range(new.shape[0]):
        members = q[assign == c]
        if len(members):
            new[c] = members.mean(axis=0)
    return new


def kmeans_queries(q, C, iters):
    """Lloyd's K-means on the queries of one head: `iters` >= 1 rounds of
    (assign, update) from the segment means. Returns (assignment after the
    last round, centroids before the last update, centroids after it)."""
    if iters < 1:
        raise ValueError("at least one K-means iteration")
    mu = R.segment_means(q, C)
    for _ in range(iters):
        prev = mu
        assign = kmeans_assign(q, mu)
        mu = kmeans_update(q, assign, mu)
    return assign, prev, mu


def clustered_head(q, k, v, C, iters):
    """One head of clustered attention; returns every intermediate."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    assign, prev, mu = kmeans_queries(q, C, iters)
    g = R.landmark_rows(mu, k, v)  # softmax(mu K^T / sqrt(d)) V, [C, d]
    return {"assign": assign, "mu_prev": prev, "mu": mu, "g": g, "out": g[assign]}


def clustered_attention(q, k, v, C, iters):
    """[B, H, n, d] -> [B, H, n, d] (float64)."""
    B, H, n, d = q.shape
    out = np.empty((B, H, n, d))
    for b in range(B):
        for h in range(H):
            out[b, h] = clustered_head(q[b, h], k[b, h], v[b, h], C, iters)["out"]
    return out
