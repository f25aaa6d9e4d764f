"""GPU parity of the two variants the page leaves open, through
nystrom_attn_fwd_ex, against the oracle's readings of them (Proposed method,
bullets 4 and 6): per-channel depthwise filters [H][d][ks], and padded
sequences (a batch entry's rows past its length take part in nothing and
come out zero). Same bars as the plain path: max|out - ref| / max|ref| <=
2e-2 for bf16 inputs, <= 1e-4 for float32, on the full output and on the
attention term alone."""
import numpy as np
import pytest

import workloads
from oracle import nystrom_ref as R
from tests.gpu_helpers import TOL, dtype_code, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    import torch
    from nystr_self_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    torch.cuda.set_device(0)


def run_ex(inp, conv_w, ks, layout, lengths):
    import torch
    import nystr_self_attention_gb300 as N
    wl = inp.wl
    q, k, v, _ = to_device(inp)
    w = torch.from_numpy(np.ascontiguousarray(conv_w)).cuda() if ks > 0 else None
    out = torch.full_like(q, float("nan"))  # every element must be written
    N.nystrom_attn_fwd_ex(q, k, v, w, out, wl.B, wl.H, wl.n, wl.d, wl.m, wl.iters, ks,
                          dtype_code(wl.dtype), layout, lengths)
    torch.cuda.synchronize()
    assert N.nystrom_get_status() == N.NYS_OK
    return out.float().cpu().numpy()


def check(inp, conv_w, layout, lengths, heads=None):
    """Full output and attention term alone, every head (or `heads`), and
    exact zeros in the padding rows."""
    import nystr_self_attention_gb300 as N
    wl = inp.wl
    ks = conv_w.shape[-1]
    got = run_ex(inp, conv_w, ks, layout, lengths)
    got_att = run_ex(inp, conv_w, 0, layout, lengths)
    assert np.isfinite(got).all() and np.isfinite(got_att).all()
    todo = heads or [(b, h) for b in range(wl.B) for h in range(wl.H)]
    worst = 0.0
    for b, h in todo:
        L = int(lengths[b]) if lengths is not None else wl.n
        w = conv_w[h]
        if lengths is None:
            ref = R.nystrom_head(inp.q[b, h], inp.k[b, h], inp.v[b, h], w, wl.m, wl.iters)
        else:
            ref = R.nystrom_head_padded(inp.q[b, h], inp.k[b, h], inp.v[b, h], w, wl.m, wl.iters, L)
        e_out = rel_err(got[b, h], ref["out"])
        e_att = rel_err(got_att[b, h], ref["att"])
        worst = max(worst, e_out, e_att)
        assert e_out <= TOL[wl.dtype] and e_att <= TOL[wl.dtype], ((b, h), L, e_out, e_att)
        assert (got[b, h, L:] == 0).all() and (got_att[b, h, L:] == 0).all()
    return worst


SHAPES = [
    # B, H, n, d, m, iters, ks
    (3, 2, 512, 64, 32, 6, 9),
    (2, 2, 1000, 32, 64, 6, 35),      # n not a multiple of the tile
    (2, 1, 640, 128, 160, 6, 33),     # m > 128
    (4, 3, 256, 64, 128, 4, 5),       # pseudo-inverse after the landmark rows
    (2, 2, 384, 128, 64, 6, 65),      # d = 128
]
IDS = [f"B{s[0]}H{s[1]}n{s[2]}d{s[3]}m{s[4]}i{s[5]}k{s[6]}" for s in SHAPES]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_per_channel_filters(shape, dtype):
    import nystr_self_attention_gb300 as N
    B, H, n, d, m, iters, ks = shape
    wl = workloads.custom(B, H, n, d, m, iters, ks, dtype)
    inp = workloads.make_inputs(wl, seed=31)
    w = workloads.conv_channels(H, d, ks, seed=32)
    check(inp, w, N.NYS_CONV_PER_CHANNEL, None)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_padded_sequences(shape, dtype):
    import nystr_self_attention_gb300 as N
    B, H, n, d, m, iters, ks = shape
    wl = workloads.custom(B, H, n, d, m, iters, ks, dtype)
    inp = workloads.make_inputs(wl, seed=41)
    lengths = workloads.lengths_for(B, n, m, seed=42)
    check(inp, inp.conv_w, N.NYS_CONV_PER_HEAD, lengths)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES[:3], ids=IDS[:3])
def test_padded_sequences_with_per_channel_filters(shape, dtype):
    import nystr_self_attention_gb300 as N
    B, H, n, d, m, iters, ks = shape
    wl = workloads.custom(B, H, n, d, m, iters, ks, dtype)
    inp = workloads.make_inputs(wl, seed=51)
    w = workloads.conv_channels(H, d, ks, seed=52)
    lengths = workloads.lengths_for(B, n, m, seed=53)
    check(inp, w, N.NYS_CONV_PER_CHANNEL, lengths)


def test_plain_layout_without_lengths_equals_the_fused_path():
    """NYS_CONV_PER_HEAD and no lengths: the fused path, bit for bit."""
    import torch
    import nystr_self_attention_gb300 as N
    from tests.gpu_helpers import run_gpu
    wl = workloads.custom(2, 3, 512, 64, 64, 6, 33, "bf16")
    inp = workloads.make_inputs(wl, seed=61)
    a, _ = run_gpu(inp)
    b = run_ex(inp, inp.conv_w, wl.ks, N.NYS_CONV_PER_HEAD, None)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("name", ["c2", "c3", "c4", "c5"])
def test_full_workload_variants(name):
    """Each workload at full size with padded sequences and per-channel
    filters together, every head against the oracle."""
    import nystr_self_attention_gb300 as N
    wl = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(wl)
    w = workloads.conv_channels(wl.H, wl.d, wl.ks, seed=70 + workloads.ORDER.index(name))
    lengths = workloads.lengths_for(wl.B, wl.n, wl.m, seed=80 + workloads.ORDER.index(name))
    worst = check(inp, w, N.NYS_CONV_PER_CHANNEL, lengths)
    print(f"{name} variants: lengths {lengths.tolist()[:6]}..., worst {worst:.2e}")
