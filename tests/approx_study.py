"""Approximation study on the fp64 oracle: how far Nyström attention lies from
exact softmax attention as the number of landmarks m and of pseudo-inverse
updates grows.

The Nyströmformer review page ("Proposed method", bullets 3-5) replaces the
n x n softmax matrix by a product through m segment-mean landmarks and an
iterative Moore-Penrose inverse that is said to settle after about six
updates. Nothing on the page bounds the resulting error for a given input, so
this study only reports it: the relative Frobenius error of the attention
term (conv off) against the O(n^2) result, per (m, updates), with the SVD inverse
beside it to separate the landmark error from the iteration error.

Two input families, both drawn by ``workloads.make_inputs``:
* ``normal``: Q, K, V standard normal (the 512-token BERT-base-like workload);
* ``clustered``: the same plus a rank-4 drift shared by each of 128 segments
  (the 8192-token clustered workload's recipe, at this length).

Test infrastructure: it runs only the oracle. ``python tests/approx_study.py``
prints the table; ``tests/test_approx_study.py`` runs a small grid of it.
"""
from __future__ import annotations

import argparse
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402
from oracle import nystrom_ref as R  # noqa: E402

FAMILIES = {"normal": 0.0, "clustered": 0.5}


def draw(family: str, n: int, d: int, heads: int, seed: int):
    """[heads, n, d] float64 Q, K, V of one input family."""
    wl = workloads.custom(1, heads, n, d, 128 if n % 128 == 0 else n, 0, 0, "f32",
                          drift=FAMILIES[family])
    inp = workloads.make_inputs(wl, seed=seed, ks=0)
    return (inp.q[0].astype(np.float64), inp.k[0].astype(np.float64),
            inp.v[0].astype(np.float64))


def rel_err(att, exact):
    """Relative Frobenius error ||att - exact||_F / ||exact||_F."""
    return float(np.linalg.norm(att - exact) / np.linalg.norm(exact))


def approx_errors(family: str, n: int, d: int, ms, iters_list, heads: int = 2, seed: int = 7):
    """Relative Frobenius error of the attention term against exact attention,
    the worst over ``heads`` heads, for every m in ``ms`` and every update count
    in ``iters_list``; key ``(m, "svd")`` holds the error with the SVD inverse
    of A_S in place of the iteration."""
    q, k, v = draw(family, n, d, heads, seed)
    out = {}
    for h in range(heads):
        exact = R.softmax_attention(q[h], k[h], v[h])
        for m in ms:
            q_t, k_t = R.segment_means(q[h], m), R.segment_means(k[h], m)
            a_s = R.landmark_kernel(q_t, k_t)
            g = R.landmark_rows(q_t, k[h], v[h])
            cols = [(it, R.pinv_iterative(a_s, it)) for it in iters_list]
            cols.append(("svd", R.svd_pinv(a_s)))
            for key, z in cols:
                e = rel_err(R.token_rows(q[h], k_t, z @ g), exact)
                out[(m, key)] = max(out.get((m, key), 0.0), e)
    return out


def table(family, n, d, ms, iters_list, heads):
    errs = approx_errors(family, n, d, ms, iters_list, heads)
    head = "| m | " + " | ".join(f"{it} upd." for it in iters_list) + " | SVD |"
    rows = [head, "|" + "---|" * (len(iters_list) + 2)]
    for m in ms:
        vals = [errs[(m, it)] for it in iters_list] + [errs[(m, "svd")]]
        rows.append(f"| {m} | " + " | ".join(f"{x:.3f}" for x in vals) + " |")
    return "\n".join(rows)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--n", type=int, nargs="+", default=[512, 2048])
    p.add_argument("--d", type=int, default=64)
    p.add_argument("--heads", type=int, default=2)
    args = p.parse_args()
    iters_list = [0, 2, 4, 6, 8, 12]
    for n in args.n:
        ms = [m for m in (16, 32, 64, 128, 256) if m <= n and n % m == 0]
        for family in FAMILIES:
            t0 = time.perf_counter()
            print(f"\n{family}, n={n}, d={args.d}, worst of {args.heads} heads "
                  f"(relative Frobenius error of the attention term vs exact attention)\n")
            print(table(family, n, args.d, ms, iters_list, args.heads))
            print(f"\n({time.perf_counter() - t0:.1f} s)")


if __name__ == "__main__":
    main()
