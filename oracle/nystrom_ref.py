"""fp64 CPU oracle for Nyström self-attention (forward pass).

TEST INFRASTRUCTURE. Only the tests, the package's ``smoke()`` check and the
benchmark's CPU-baseline leg may import or run this module. The CUDA library
never calls it, shares no code with it, and has no path through it.

Source: the review page "Nyströmformer: A Nyström-Based Algorithm for
Approximating Self-Attention" (nubint.ai), section "Proposed method"
(提出的方法), bullets 1-6, cited below as "Proposed method, bullet k". The
page gives the method at formula level:

* bullet 1: exact attention S = softmax(Q K^T / sqrt(d_q));
* bullet 2: landmarks of Q and K give a small m x m matrix A_S by a softmax,
  whose Moore-Penrose inverse is used;
* bullet 3: S ~ S_hat = softmax(Q K~^T / sqrt(d_q)) A_S^+ softmax(Q~ K^T / sqrt(d_q));
* bullet 4: the landmarks Q~, K~ are segment means;
* bullet 5: A_S^+ is computed by an iterative method (no SVD) that settles
  after about 6 iterations;
* bullet 6: the output is S_hat V plus a depthwise convolution of V (a skip
  connection).

The page does not print the iteration. This oracle uses the third-order
iteration of the Nyströmformer paper (Xiong et al., 2021), which takes it
from Razavi et al. (2014):
    Z_0 = A^T / (||A||_1 ||A||_inf),
    Z <- 1/4 Z (13 I - A Z (15 I - A Z (7 I - A Z))),
run a fixed number of times with no early exit.

Readings where the page is silent (each listed in the design notes):
* all three softmaxes use the scale 1/sqrt(d) (d = head dimension);
* segment i is rows [floor(i*n/m), floor((i+1)*n/m)), which is n/m rows each
  when m divides n and otherwise lengths floor(n/m) and ceil(n/m); m <= n;
* ||.||_1 is the largest column abs-sum and ||.||_inf the largest row
  abs-sum, of each head's own A_S;
* the depthwise convolution runs along the sequence with one filter of odd
  width ks per head, shared by all d channels, as a cross-correlation with
  (ks-1)/2 zero rows padded on each side, no bias, and is added to S_hat V;
* ks = 0 means no convolution term;
* variants (not on the page): per-channel filters [d, ks] apply channel c's
  own taps to channel c; a padded sequence (``nystrom_head_padded``) behaves
  as its unpadded prefix, with zero output rows for the padding.

Every function works in float64 on numpy arrays and is written for a reader
to check against the page by eye, not for speed.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "segment_bounds", "segment_means", "softmax_rows", "landmark_kernel", "pinv_initial",
    "pinv_step", "pinv_iterative", "landmark_rows", "token_rows",
    "depthwise_conv_seq", "nystrom_head", "nystrom_attention",
    "softmax_attention", "svd_pinv", "depthwise_conv_seq_channels", "conv_of",
    "masked_softmax_rows", "nystrom_head_padded", "split_heads", "merge_heads", "mha_forward",
]


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def segment_bounds(n, m):
    """Row ranges of the m contiguous segments of n rows: segment i is rows
    [floor(i n / m), floor((i + 1) n / m)). When m divides n every segment
    has n/m rows; otherwise the lengths are floor(n/m) and ceil(n/m), spread
    evenly (the reading used where n is not a multiple of m). Needs
    1 <= m <= n so that no segment is empty."""
    if m < 1 or m > n:
        raise ValueError(f"segment means need 1 <= m <= n (n={n}, m={m})")
    return [(i * n // m, (i + 1) * n // m) for i in range(m)]


def segment_means(x, m):
    """Segment-means landmarks (Proposed method, bullet 4).

    x: [n, d]. Returns [m, d] whose row i is the plain average of the rows of
    segment i (see ``segment_bounds``).
    """
    x = _f64(x)
    n, d = x.shape
    out = np.empty((m, d))
    for i, (lo, hi) in enumerate(segment_bounds(n, m)):
        out[i] = x[lo:hi].mean(axis=0)
    return out


def softmax_rows(s):
    """Row-wise softmax (Proposed method, bullets 1-3): each row of s becomes
    exp(s_ij - max_j s_ij) / sum_j exp(s_ij - max_j s_ij)."""
    s = _f64(s)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def landmark_kernel(q_tilde, k_tilde):
    """A_S = softmax(Q~ K~^T / sqrt(d)), the m x m landmark matrix
    (Proposed method, bullet 2)."""
    q_tilde, k_tilde = _f64(q_tilde), _f64(k_tilde)
    d = q_tilde.shape[1]
    return softmax_rows(q_tilde @ k_tilde.T / np.sqrt(d))


def pinv_initial(a):
    """Z_0 = A^T / (||A||_1 ||A||_inf): ||A||_1 is the largest column
    abs-sum, ||A||_inf the largest row abs-sum (Proposed method, bullet 5;
    initialisation of the Nyströmformer paper's iteration)."""
    a = _f64(a)
    norm1 = np.abs(a).sum(axis=0).max()
    norminf = np.abs(a).sum(axis=1).max()
    return a.T / (norm1 * norminf)


def pinv_step(a, z):
    """One update Z <- 1/4 Z (13 I - A Z (15 I - A Z (7 I - A Z)))
    (Proposed method, bullet 5), evaluated inside-out as written."""
    a, z = _f64(a), _f64(z)
    eye = np.eye(a.shape[0])
    az = a @ z
    inner = 7.0 * eye - az
    middle = 15.0 * eye - az @ inner
    outer = 13.0 * eye - az @ middle
    return 0.25 * (z @ outer)


def pinv_iterative(a, iters):
    """Z ~ A^+ after exactly ``iters`` updates from Z_0, no early exit
    (Proposed method, bullet 5: iterative, avoids the SVD, about 6 updates)."""
    z = pinv_initial(a)
    for _ in range(iters):
        z = pinv_step(a, z)
    return z


def landmark_rows(q_tilde, k, v):
    """G = softmax(Q~ K^T / sqrt(d)) V, the [m, d] product of the right
    Nyström factor with V (Proposed method, bullets 3 and 6)."""
    q_tilde, k, v = _f64(q_tilde), _f64(k), _f64(v)
    d = k.shape[1]
    return softmax_rows(q_tilde @ k.T / np.sqrt(d)) @ v


def token_rows(q, k_tilde, w):
    """softmax(Q K~^T / sqrt(d)) W, the left Nyström factor applied to the
    [m, d] matrix W = Z G (Proposed method, bullets 3 and 6)."""
    q, k_tilde, w = _f64(q), _f64(k_tilde), _f64(w)
    d = q.shape[1]
    return softmax_rows(q @ k_tilde.T / np.sqrt(d)) @ w


def depthwise_conv_seq(v, w):
    """Depthwise convolution of V along the sequence (Proposed method,
    bullet 6): out[t] = sum_j w[j] * V[t + j - (ks-1)/2], rows of V outside
    [0, n) read as zero. One filter w [ks] (odd ks) for all channels."""
    v, w = _f64(v), _f64(w)
    n, _ = v.shape
    ks = w.shape[0]
    out = np.zeros_like(v)
    if ks == 0:
        return out
    if ks % 2 != 1:
        raise ValueError("conv width must be odd")
    r = (ks - 1) // 2
    for j in range(ks):
        shift = j - r  # out[t] takes V[t + shift]
        lo, hi = max(0, -shift), min(n, n - shift)
        if lo < hi:
            out[lo:hi] += w[j] * v[lo + shift:hi + shift]
    return out


def nystrom_head(q, k, v, w, m, iters):
    """One head of Nyström self-attention, returning every intermediate.

    q, k, v: [n, d]; w: [ks] conv filter shared by the channels (ks may be
    0), or [d, ks] filters, one per channel; m landmarks;
    ``iters`` pseudo-inverse updates. The output uses the association
    F (Z (B V)), which never forms an n x n or n x m product with V
    (Proposed method, bullet 6: linear time).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    q_tilde = segment_means(q, m)
    k_tilde = segment_means(k, m)
    a_s = landmark_kernel(q_tilde, k_tilde)
    z = pinv_iterative(a_s, iters)
    g = landmark_rows(q_tilde, k, v)
    w_mat = z @ g
    att = token_rows(q, k_tilde, w_mat)
    conv = conv_of(v, w)
    return {
        "q_tilde": q_tilde, "k_tilde": k_tilde, "a_s": a_s, "z": z,
        "g": g, "w": w_mat, "att": att, "conv": conv, "out": att + conv,
    }


def nystrom_attention(q, k, v, conv_w, m, iters, heads=None, lengths=None):
    """Forward pass over [B, H, n, d] inputs with conv weights [H, ks] (one
    filter per head) or [H, d, ks] (one per channel).

    Returns out [B, H, n, d] in float64. ``heads`` optionally restricts the
    work to a list of (b, h) pairs; the other heads are left as NaN.
    ``lengths`` optionally gives each batch entry's number of tokens; the
    rows past it are padding (see ``nystrom_head_padded``).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    conv_w = _f64(conv_w)
    B, H, n, d = q.shape
    out = np.full((B, H, n, d), np.nan)
    todo = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in todo:
        if lengths is None:
            out[b, h] = nystrom_head(q[b, h], k[b, h], v[b, h], conv_w[h], m, iters)["out"]
        else:
            out[b, h] = nystrom_head_padded(q[b, h], k[b, h], v[b, h], conv_w[h], m, iters,
                                            int(lengths[b]))["out"]
    return out


# ------------------------------------------------------------------ variants
# Two points the page leaves open, each with the reading used here: a
# depthwise filter per channel instead of per head, and padded sequences.

def depthwise_conv_seq_channels(v, w):
    """Depthwise convolution along the sequence with one filter per channel
    (bullet 6 says only "depthwise convolution"; this reading gives channel
    c its own taps): out[t, c] = sum_j w[c, j] * V[t + j - (ks-1)/2, c],
    rows of V outside [0, n) read as zero. w: [d, ks], odd ks."""
    v, w = _f64(v), _f64(w)
    n, d = v.shape
    if w.ndim != 2 or w.shape[0] != d:
        raise ValueError("per-channel filters need shape [d, ks]")
    ks = w.shape[1]
    out = np.zeros_like(v)
    if ks == 0:
        return out
    if ks % 2 != 1:
        raise ValueError("conv width must be odd")
    r = (ks - 1) // 2
    for t in range(n):
        for j in range(ks):
            u = t + j - r
            if 0 <= u < n:
                out[t] += w[:, j] * v[u]
    return out


def conv_of(v, w):
    """The conv term for a shared filter [ks] or per-channel filters [d, ks]."""
    w = _f64(w)
    return depthwise_conv_seq_channels(v, w) if w.ndim == 2 else depthwise_conv_seq(v, w)


def masked_softmax_rows(s, valid):
    """Row-wise softmax over the columns where ``valid`` is true; the other
    columns get weight 0."""
    return softmax_rows(np.where(np.asarray(valid)[None, :], _f64(s), -np.inf))


def nystrom_head_padded(q, k, v, w, m, iters, length):
    """One head whose n rows hold ``length`` tokens followed by padding (the
    page mentions no masking; this is the reading that padding takes part in
    nothing):

    * the landmarks are the segment means of the ``length`` tokens
      (``segment_bounds(length, m)``; needs m <= length);
    * padded keys are masked out of softmax(Q~ K^T / sqrt(d)); A_S and
      softmax(Q K~^T / sqrt(d)) see only landmarks;
    * padded rows of V read as zero in the convolution;
    * the output rows of padding are zero.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, d = q.shape
    if not 1 <= length <= n:
        raise ValueError(f"length must be in [1, n] (n={n}, length={length})")
    valid = np.arange(n) < length
    q_tilde = segment_means(q[:length], m)
    k_tilde = segment_means(k[:length], m)
    a_s = landmark_kernel(q_tilde, k_tilde)
    z = pinv_iterative(a_s, iters)
    g = masked_softmax_rows(q_tilde @ k.T / np.sqrt(d), valid) @ v
    w_mat = z @ g
    att = token_rows(q, k_tilde, w_mat)
    conv = conv_of(np.where(valid[:, None], v, 0.0), w)
    return {
        "q_tilde": q_tilde, "k_tilde": k_tilde, "a_s": a_s, "z": z, "g": g, "w": w_mat,
        "att": np.where(valid[:, None], att, 0.0), "conv": np.where(valid[:, None], conv, 0.0),
        "out": np.where(valid[:, None], att + conv, 0.0),
    }


def softmax_attention(q, k, v):
    """Exact O(n^2) softmax attention S V with S = softmax(Q K^T / sqrt(d))
    for one head (Proposed method, bullet 1): what the method approximates."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    d = q.shape[1]
    return softmax_rows(q @ k.T / np.sqrt(d)) @ v


def svd_pinv(a):
    """Moore-Penrose inverse by the SVD (what bullet 5's iteration avoids)."""
    return np.linalg.pinv(_f64(a))


# -------------------------------------------------------------- the module
# The multi-head attention module the page's model wraps around the op
# (abstract; Proposed method, bullet 6: Nyström self-attention replaces
# softmax attention in the Transformer): projections in, heads, projection
# out. Random weights only; no residual, normalisation or dropout (those
# belong to the layer).

def split_heads(x, H):
    """[B, n, H*d] -> [B, H, n, d]: head h takes columns [h*d, (h+1)*d)."""
    x = _f64(x)
    B, n, D = x.shape
    d = D // H
    out = np.empty((B, H, n, d))
    for h in range(H):
        out[:, h] = x[:, :, h * d:(h + 1) * d]
    return out


def merge_heads(o):
    """[B, H, n, d] -> [B, n, H*d]: the inverse of ``split_heads``."""
    o = _f64(o)
    B, H, n, d = o.shape
    out = np.empty((B, n, H * d))
    for h in range(H):
        out[:, :, h * d:(h + 1) * d] = o[:, h]
    return out


def mha_forward(x, w_qkv, b_qkv, w_o, b_o, conv_w, H, m, iters):
    """y = merge(Nystrom(Q, K, V)) w_o + b_o with [Q | K | V] = x w_qkv +
    b_qkv split into H heads. x [B, n, D], w_qkv [D, 3D] (the Q block, then K,
    then V), b_qkv [3D] or None, w_o [D, D], b_o [D] or None, conv_w [H, ks]."""
    x = _f64(x)
    D = x.shape[2]
    qkv = x @ _f64(w_qkv)
    if b_qkv is not None:
        qkv = qkv + _f64(b_qkv)
    q = split_heads(qkv[..., :D], H)
    k = split_heads(qkv[..., D:2 * D], H)
    v = split_heads(qkv[..., 2 * D:], H)
    y = merge_heads(nystrom_attention(q, k, v, conv_w, m, iters)) @ _f64(w_o)
    if b_o is not None:
        y = y + _f64(b_o)
    return y
