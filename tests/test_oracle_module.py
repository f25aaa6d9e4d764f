"""Pins of the oracle's attention module (split / merge of heads and the
projections around the op), each against something other than itself."""
import numpy as np

import workloads
from oracle import nystrom_ref as R


def test_split_heads_by_brute_force_indexing():
    x = np.random.default_rng(1).standard_normal((2, 5, 12))
    s = R.split_heads(x, 3)
    for b in range(2):
        for t in range(5):
            for c in range(12):
                assert s[b, c // 4, t, c % 4] == x[b, t, c]
    assert np.array_equal(R.merge_heads(s), x)


def test_biases_alone_give_the_closed_form():
    """w_qkv = 0: every query, key and value row of head h is the bias, so
    the keys are constant, each attention row is the mean of V (= b_v of the
    head) and, with no conv, y = b_v w_o + b_o in every row."""
    wl = workloads.custom(2, 3, 24, 8, 4, 6, 0, "f32")
    inp = workloads.module_inputs(wl, seed=3)
    D = wl.H * wl.d
    y = R.mha_forward(inp.x, np.zeros((D, 3 * D)), inp.b_qkv, inp.w_o, inp.b_o,
                      np.zeros((wl.H, 0)), wl.H, wl.m, wl.iters)
    expect = inp.b_qkv[2 * D:].astype(np.float64) @ inp.w_o.astype(np.float64) + inp.b_o
    np.testing.assert_allclose(y, np.broadcast_to(expect, y.shape), rtol=1e-12, atol=1e-12)


def test_identity_projections_reduce_to_the_op():
    """w_qkv = [I | I | I], w_o = I, no biases: y is the op on the split x."""
    wl = workloads.custom(1, 2, 32, 8, 4, 6, 3, "f32")
    inp = workloads.module_inputs(wl, seed=4)
    D = wl.H * wl.d
    eye = np.eye(D)
    y = R.mha_forward(inp.x, np.hstack([eye, eye, eye]), None, eye, None, inp.conv_w, wl.H, wl.m,
                      wl.iters)
    xs = R.split_heads(inp.x, wl.H)
    op = R.nystrom_attention(xs, xs, xs, inp.conv_w, wl.m, wl.iters)
    np.testing.assert_allclose(y, R.merge_heads(op), rtol=1e-12, atol=1e-12)


def test_head_permutation_equivariance():
    """Relabelling the heads (columns of each of the Q, K, V blocks, rows of
    w_o and rows of conv_w, blockwise) leaves y unchanged."""
    wl = workloads.custom(1, 3, 40, 8, 5, 6, 5, "f32")
    inp = workloads.module_inputs(wl, seed=5)
    H, d, D = wl.H, wl.d, wl.H * wl.d
    perm = [2, 0, 1]
    cols = np.concatenate([np.arange(p * d, (p + 1) * d) for p in perm])
    w2 = np.hstack([inp.w_qkv[:, blk * D:(blk + 1) * D][:, cols] for blk in range(3)])
    b2 = np.concatenate([inp.b_qkv[blk * D:(blk + 1) * D][cols] for blk in range(3)])
    y1 = R.mha_forward(inp.x, inp.w_qkv, inp.b_qkv, inp.w_o, inp.b_o, inp.conv_w, H, wl.m, wl.iters)
    y2 = R.mha_forward(inp.x, w2, b2, inp.w_o[cols], inp.b_o, inp.conv_w[perm], H, wl.m, wl.iters)
    np.testing.assert_allclose(y1, y2, rtol=1e-10, atol=1e-10)


def test_pins_reject_planted_mistakes():
    """A transposed w_o, the K and V blocks swapped, or a dropped output
    bias each fail the closed form above."""
    wl = workloads.custom(2, 3, 24, 8, 4, 6, 0, "f32")
    inp = workloads.module_inputs(wl, seed=3)
    D = wl.H * wl.d
    zero = np.zeros((D, 3 * D))
    expect = inp.b_qkv[2 * D:].astype(np.float64) @ inp.w_o.astype(np.float64) + inp.b_o

    def bad(b_qkv, w_o, b_o):
        y = R.mha_forward(inp.x, zero, b_qkv, w_o, b_o, np.zeros((wl.H, 0)), wl.H, wl.m, wl.iters)
        return not np.allclose(y, np.broadcast_to(expect, y.shape), rtol=1e-9, atol=1e-9)

    swapped = np.concatenate([inp.b_qkv[:D], inp.b_qkv[2 * D:], inp.b_qkv[D:2 * D]])
    assert bad(inp.b_qkv, inp.w_o.T, inp.b_o)
    assert bad(swapped, inp.w_o, inp.b_o)
    assert bad(inp.b_qkv, inp.w_o, None)
