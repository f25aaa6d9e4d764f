"""Seeded synthetic workloads for Nyström self-attention (forward).

This module only draws inputs. It holds none of the method's arithmetic, so
the fp64 oracle, the tests and the benchmark can all use it without sharing
any computation with the CUDA path.

The five shapes below stand in for the workloads of the Nyströmformer review
page ("Experiments": GLUE and IMDB at BERT-base length, Long Range Arena at
several thousand tokens). No dataset is read: every tensor is drawn from a
seeded normal distribution with the shape, scale and (for ``c4``) clustered
structure stated per workload.

Draw order per workload, from ``numpy.random.default_rng(20260 + index)``:
Q, K, V (each ``[B, H, n, d]``, standard normal, times ``scale``), then the
depthwise-conv weights ``[H, ks]`` (normal with variance ``1/ks``), then, only
for ``drift > 0``, the per-(b, h) rank-4 factors ``U [B, H, m, 4]`` and
``P [B, H, 4, d]``. The drift ``drift * U @ P / 2`` of segment ``i`` is added
to every row of segment ``i`` of Q, K and V alike.

For bf16 workloads the fp32 draws are rounded to bfloat16 with
round-to-nearest-even before anyone sees them; both sides receive the same
rounded values (as fp32 arrays that hold bf16-representable numbers, and as
raw uint16 bit patterns for upload).
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    d: int
    m: int
    iters: int
    ks: int
    dtype: str  # "f32" or "bf16": the element type of q, k, v and out
    scale: float = 1.0
    drift: float = 0.0
    label: str = ""

    @property
    def heads(self) -> int:
        return self.B * self.H

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.n

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} H={self.H} n={self.n} d={self.d} m={self.m} "
                f"iters={self.iters} ks={self.ks} {self.dtype}")


WORKLOADS = {
    "c1": Workload("c1", 1, 1, 512, 64, 64, 6, 33, "f32",
                   label="fp32 single head, n=512"),
    "c2": Workload("c2", 32, 12, 512, 64, 64, 6, 33, "bf16",
                   label="BERT-base-like, n=512"),
    "c3": Workload("c3", 32, 2, 4096, 32, 64, 6, 35, "bf16", scale=0.5,
                   label="long-sequence classifier, n=4096"),
    "c4": Workload("c4", 8, 8, 8192, 64, 128, 6, 33, "bf16", drift=0.5,
                   label="clustered (rank-4 segment drift), n=8192"),
    "c5": Workload("c5", 2, 16, 32768, 128, 256, 8, 65, "bf16",
                   label="long context, n=32768"),
}
ORDER = ["c1", "c2", "c3", "c4", "c5"]


def seed_of(name: str) -> int:
    return 20260 + ORDER.index(name)


def round_to_bf16(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round fp32 values to bfloat16 (nearest, ties to even).

    Returns (values as fp32, raw uint16 bit patterns). Inputs are finite.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    hi = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    back = (hi.astype(np.uint32) << 16).view(np.float32)
    return back, hi


@dataclasses.dataclass
class Inputs:
    """One drawn workload. ``q, k, v`` are fp32 arrays ``[B, H, n, d]`` holding
    exactly the values both sides use; ``*_bits`` are the bf16 patterns (bf16
    workloads only); ``conv_w`` is fp32 ``[H, ks]``."""
    wl: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    conv_w: np.ndarray
    q_bits: np.ndarray | None = None
    k_bits: np.ndarray | None = None
    v_bits: np.ndarray | None = None


def make_inputs(wl: Workload, seed: int | None = None, ks: int | None = None) -> Inputs:
    """Draw ``wl``'s tensors. ``seed`` defaults to the workload's own seed;
    ``ks`` overrides the conv width (0 draws no weights)."""
    rng = np.random.default_rng(seed_of(wl.name) if seed is None else seed)
    ks = wl.ks if ks is None else ks
    shape = (wl.B, wl.H, wl.n, wl.d)
    q = rng.standard_normal(shape, dtype=np.float32)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    if wl.scale != 1.0:
        for t in (q, k, v):
            t *= np.float32(wl.scale)
    if ks > 0:
        w = (rng.standard_normal((wl.H, ks), dtype=np.float32)
             * np.float32(1.0 / np.sqrt(ks))).astype(np.float32)
    else:
        w = np.zeros((wl.H, 0), dtype=np.float32)
    if wl.drift > 0:
        if wl.n % wl.m != 0:
            raise ValueError("the segment drift needs n to be a multiple of m")
        u = rng.standard_normal((wl.B, wl.H, wl.m, 4), dtype=np.float32)
        p = rng.standard_normal((wl.B, wl.H, 4, wl.d), dtype=np.float32)
        seg_off = (np.float32(wl.drift) * np.matmul(u, p) / np.float32(2.0)).astype(np.float32)
        per_row = np.repeat(seg_off, wl.n // wl.m, axis=2)
        for t in (q, k, v):
            t += per_row
    out = Inputs(wl, q, k, v, w)
    if wl.dtype == "bf16":
        out.q, out.q_bits = round_to_bf16(q)
        out.k, out.k_bits = round_to_bf16(k)
        out.v, out.v_bits = round_to_bf16(v)
    return out


def custom(B, H, n, d, m, iters, ks, dtype, scale=1.0, drift=0.0, name="custom") -> Workload:
    """A workload of any shape (tests use it for tiny, ragged and edge cases).
    Its seed must be passed to :func:`make_inputs` explicitly."""
    return Workload(name, B, H, n, d, m, iters, ks, dtype, scale, drift)


def conv_channels(H: int, d: int, ks: int, seed: int) -> np.ndarray:
    """Per-channel depthwise-conv weights ``[H, d, ks]`` (float32), normal
    with variance ``1/ks`` like the per-head filters, from their own seeded
    generator (the per-channel variant of the convolution)."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((H, d, ks), dtype=np.float32)
            * np.float32(1.0 / np.sqrt(ks))).astype(np.float32)


def lengths_for(B: int, n: int, m: int, seed: int) -> np.ndarray:
    """Tokens per batch entry for the padded-sequence variant: int32 ``[B]``
    uniform in ``[m, n]``, with the first entry at ``n`` (no padding) and,
    for ``B > 1``, the second at ``m`` (the shortest allowed)."""
    rng = np.random.default_rng(seed)
    out = rng.integers(m, n + 1, size=B).astype(np.int32)
    out[0] = n
    if B > 1:
        out[1] = m
    return out


@dataclasses.dataclass
class ModuleInputs:
    """Inputs of the attention module around the op: x ``[B, n, H*d]``,
    w_qkv ``[D, 3D]``, b_qkv ``[3D]``, w_o ``[D, D]``, b_o ``[D]`` (fp32
    arrays holding the values both sides use; ``*_bits`` the bf16 patterns
    of x, w_qkv, w_o for bf16 workloads) and the per-head conv weights."""
    wl: Workload
    x: np.ndarray
    w_qkv: np.ndarray
    b_qkv: np.ndarray
    w_o: np.ndarray
    b_o: np.ndarray
    conv_w: np.ndarray
    bits: dict | None = None


def module_inputs(wl: Workload, seed: int) -> ModuleInputs:
    """Random weights for the module (no trained model exists here): x
    standard normal, weights normal with variance 1/D (so Q, K, V have about
    unit variance), biases normal with standard deviation 0.1, conv weights as
    in ``make_inputs``. Draw order: x, w_qkv, b_qkv, w_o, b_o, conv_w."""
    rng = np.random.default_rng(seed)
    D = wl.H * wl.d
    x = rng.standard_normal((wl.B, wl.n, D), dtype=np.float32)
    w_qkv = (rng.standard_normal((D, 3 * D), dtype=np.float32) / np.float32(np.sqrt(D))).astype(np.float32)
    b_qkv = (rng.standard_normal(3 * D, dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    w_o = (rng.standard_normal((D, D), dtype=np.float32) / np.float32(np.sqrt(D))).astype(np.float32)
    b_o = (rng.standard_normal(D, dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    ks = wl.ks
    conv_w = ((rng.standard_normal((wl.H, ks), dtype=np.float32) * np.float32(1.0 / np.sqrt(ks))).astype(np.float32)
              if ks > 0 else np.zeros((wl.H, 0), dtype=np.float32))
    out = ModuleInputs(wl, x, w_qkv, b_qkv, w_o, b_o, conv_w)
    if wl.dtype == "bf16":
        out.bits = {}
        for name in ("x", "w_qkv", "w_o"):
            vals, bits = round_to_bf16(getattr(out, name))
            setattr(out, name, vals)
            out.bits[name] = bits
    return out
