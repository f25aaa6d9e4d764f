"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs. Bar: max|out - ref| / max|ref| <= 2e-2 for bf16 inputs,
<= 1e-4 for float32, on the full output AND on the attention term alone
(conv_ks = 0), since the convolution term would otherwise dominate max|ref|.
"""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import nystrom_ref as R
from tests.gpu_helpers import TOL, dtype_code, rel_err, run_gpu, stage, to_device

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_n4_m2.json")


@pytest.fixture(scope="module", autouse=True)
def library():
    import torch
    from nystr_self_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    torch.cuda.set_device(0)


def oracle_heads(inp, heads, ks=None):
    """Oracle intermediates for the listed (b, h) heads."""
    wl = inp.wl
    res = {}
    for b, h in heads:
        w = inp.conv_w[h] if (ks is None or ks > 0) else np.zeros(0)
        res[(b, h)] = R.nystrom_head(inp.q[b, h], inp.k[b, h], inp.v[b, h], w, wl.m, wl.iters)
    return res


# ------------------------------------------------------------------ golden ----

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_golden_closed_form(dtype):
    f = json.load(open(GOLDEN))
    n, d, m = f["n"], f["d"], f["m"]
    for case in f["cases"]:
        wl = workloads.custom(1, 1, n, d, m, case["iters"], 3, dtype)
        q = np.array(f["q"], np.float32)[None, None]
        v = np.array(f["v"], np.float32)[None, None]
        inp = workloads.Inputs(wl, q, q.copy(), v, np.array([f["conv_w"]], np.float32))
        if dtype == "bf16":
            for name in ("q", "k", "v"):
                vals, bits = workloads.round_to_bf16(getattr(inp, name))
                assert (vals == getattr(inp, name)).all()  # exactly representable
                setattr(inp, name + "_bits", bits)
        got, _ = run_gpu(inp)
        err = rel_err(got[0, 0], np.array(case["out"]))
        assert err <= TOL[dtype], (case["iters"], err)


# ------------------------------------------------------------- small shapes ----

SMALL = [
    # B, H, n, d, m, iters, ks
    (1, 2, 256, 64, 32, 6, 9),
    (2, 1, 200, 32, 8, 6, 5),      # n not a multiple of any tile
    (1, 1, 64, 64, 64, 6, 3),      # m = n (segments of one row)
    (1, 2, 96, 128, 1, 6, 7),      # one landmark
    (1, 1, 512, 128, 256, 8, 65),  # largest m
    (1, 3, 1000, 64, 40, 4, 0),    # m not a power of two, no conv
    (1, 1, 8, 32, 2, 0, 1),        # no pinv update, 1-tap conv
    (1, 1, 1, 32, 1, 6, 3),        # a single token
    (1, 1, 384, 64, 128, 6, 127),  # widest conv
    (1, 2, 960, 128, 192, 6, 33),  # d = 128 with m > 128, ragged last tile
    (2, 1, 640, 128, 160, 6, 0),   # d = 128, m = 160, no conv
    (1, 2, 528, 64, 132, 6, 5),    # m > 128 not a multiple of 8: the fp16 operands' rows padded to 136
    (2, 10, 1152, 128, 192, 6, 33),  # several heads per CTA range
    (20, 1, 1152, 128, 192, 4, 9),   # consecutive heads sharing conv taps
    (4, 32, 256, 64, 128, 6, 9),     # pseudo-inverse after the landmark rows (128 CTAs)
    (8, 48, 128, 64, 64, 6, 5),      # pseudo-inverse two CTAs per SM beside the rows
    (1, 152, 128, 64, 64, 4, 3),     # 76 pseudo-inverse CTAs: one per SM, the last such shape
    (1, 154, 128, 64, 64, 4, 3),     # 77 CTAs: two per SM
    (2, 210, 128, 32, 64, 2, 3),     # 210 CTAs: too many beside the rows, two head groups
    (2, 1, 777, 32, 64, 6, 5),       # n not a multiple of m: segments of 12 and 13 rows
    (1, 2, 5000, 64, 64, 6, 9),      # segments of 78 and 79 rows (long-segment landmark kernel)
    (1, 1, 300, 128, 256, 8, 33),    # segments of 1 and 2 rows, m > 128
    (1, 2, 640, 64, 192, 6, 9),      # m > 128 with d = 64: W in 32-column halves
    (2, 1, 384, 32, 160, 0, 5),      # m > 128, d = 32, no update: W = Z_0 G
    (1, 1, 512, 128, 256, 1, 3),     # m > 128, a single (odd) update
]

# float32 only: head sizes outside {32, 64, 128} (the CUDA-core landmark
# kernel), with and without ragged segments
SMALL_F32 = [
    (1, 2, 333, 96, 16, 6, 5),
    (2, 1, 250, 8, 32, 4, 3),
    (1, 1, 1000, 40, 48, 6, 0),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL, ids=[f"B{s[0]}H{s[1]}n{s[2]}d{s[3]}m{s[4]}i{s[5]}k{s[6]}" for s in SMALL])
def test_small_shapes(shape, dtype):
    B, H, n, d, m, iters, ks = shape
    wl = workloads.custom(B, H, n, d, m, iters, ks, dtype)
    inp = workloads.make_inputs(wl, seed=hash(shape) % 1000)
    ref = R.nystrom_attention(inp.q, inp.k, inp.v, inp.conv_w, m, iters)
    got, _ = run_gpu(inp)
    assert rel_err(got, ref) <= TOL[dtype]
    if ks > 0:  # the attention term on its own
        att_ref = R.nystrom_attention(inp.q, inp.k, inp.v, np.zeros((H, 0)), m, iters)
        got_att, _ = run_gpu(inp, ks=0)
        assert rel_err(got_att, att_ref) <= TOL[dtype]


@pytest.mark.parametrize("shape", SMALL_F32, ids=[f"B{s[0]}H{s[1]}n{s[2]}d{s[3]}m{s[4]}i{s[5]}k{s[6]}" for s in SMALL_F32])
def test_small_shapes_f32_head_sizes(shape):
    test_small_shapes(shape, "f32")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("d,m", [(128, 256), (64, 128), (64, 64)])
def test_scores_rising_along_the_landmarks(d, m, dtype):
    """Keys whose segments grow steadily in norm (the last ~16x the first),
    so that a token's scores rise from one block of landmarks to the next by
    far more than the softmax's exponent range: the row maximum must come
    from the last blocks, not the first (most rows here have a block maximum
    2^8 above every earlier block's, several times over)."""
    n = 8 * m
    wl = workloads.custom(1, 2, n, d, m, 6, 0, dtype)
    inp = workloads.make_inputs(wl, seed=77 + m)
    seg = np.arange(n) // (n // m)
    k = inp.k * (1.0 + 15.0 * seg / (m - 1)).astype(np.float32)[None, None, :, None]
    if dtype == "bf16":
        inp.k, inp.k_bits = workloads.round_to_bf16(k)
    else:
        inp.k = k.astype(np.float32)
    ref = R.nystrom_attention(inp.q, inp.k, inp.v, inp.conv_w, m, wl.iters)
    got, _ = run_gpu(inp)
    assert rel_err(got, ref) <= TOL[dtype]


@pytest.mark.parametrize("rising", [False, True])
def test_f32_landmark_rows_over_several_key_tiles(rising):
    """160 heads (more than there are SMs): the fp32 landmark-row pass then
    runs each head's key tiles in one CTA, one tile after another (the next
    tile's loads during P V, the online softmax rescaling O), with a ragged
    last tile; with keys rising along the sequence the running maximum grows
    from tile to tile."""
    import nystr_self_attention_gb300 as N
    B, H, n, d, m = 1, 160, 1000, 64, 40
    plan = N.nystrom_plan_describe(B, H, n, d, m, 6, 9, N.NYS_FP32)
    assert "rows=rows_x3[splits=1,tiles_per_split=8]" in plan, plan
    wl = workloads.custom(B, H, n, d, m, 6, 9, "f32")
    inp = workloads.make_inputs(wl, seed=31 + rising)
    if rising:
        inp.k = (inp.k * (1.0 + 3.0 * np.arange(n) / n).astype(np.float32)[None, None, :, None]).astype(np.float32)
    got, _ = run_gpu(inp)
    ref = R.nystrom_attention(inp.q, inp.k, inp.v, inp.conv_w, m, wl.iters)
    for h in range(H):
        assert rel_err(got[0, h], ref[0, h]) <= TOL["f32"], h


@pytest.mark.parametrize("shape", [
    (2, 4, 384, 64, 32),   # four heads stacked per CTA (m_pad 32)
    (2, 4, 384, 32, 32),   # four heads, d = 32
    (1, 6, 256, 32, 64),   # two heads per CTA, d = 32, three CTAs
    (1, 3, 200, 64, 24),   # three heads in one CTA (N = 96 products)
    (1, 5, 200, 64, 24),   # four heads, then one in the last CTA
], ids=lambda s: "B%dH%dn%dd%dm%d" % s)
def test_f32_pseudo_inverse_with_stacked_heads(shape):
    """The fp32 pseudo-inverse on the tensor cores (three tf32 products per
    product) with several heads stacked along the TMEM lanes of one CTA."""
    import nystr_self_attention_gb300 as N
    B, H, n, d, m = shape
    assert "pinv=pinv_tc[" in N.nystrom_plan_describe(B, H, n, d, m, 6, 5, N.NYS_FP32)
    wl = workloads.custom(B, H, n, d, m, 6, 5, "f32")
    inp = workloads.make_inputs(wl, seed=41 + m)
    got, ws = run_gpu(inp, workspace=True)
    ref = R.nystrom_attention(inp.q, inp.k, inp.v, inp.conv_w, m, wl.iters)
    assert rel_err(got, ref) <= TOL["f32"]
    heads = [(b, h) for b in range(B) for h in range(H)]
    st = stage(ws, wl, N.NYS_STAGE_Z, m, m)
    for (b, h), r in oracle_heads(inp, heads).items():
        assert rel_err(st[b * H + h], r["z"]) <= 1e-4, (b, h)


# ------------------------------------------------------------------ stages ----

# few heads: the pseudo-inverse runs beside the landmark-row pass and W = Z G
# is formed afterwards; 128 heads of m = 128 (one CTA each, more than half of
# the SMs): the pseudo-inverse runs after the landmark rows, merges G and
# forms W itself
STAGE_SHAPES = [(2, 2, 512, 64, 64), (16, 8, 512, 64, 128), (1, 2, 1024, 128, 256),
                (2, 1, 640, 128, 160)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", STAGE_SHAPES, ids=[f"B{s[0]}H{s[1]}" for s in STAGE_SHAPES])
def test_stage_intermediates(shape, dtype):
    import nystr_self_attention_gb300 as N
    B, H, n, d, m = shape
    wl = workloads.custom(B, H, n, d, m, 6, 33, dtype)
    inp = workloads.make_inputs(wl, seed=3)
    _, ws = run_gpu(inp, workspace=True)
    heads = [(0, 0), (B - 1, H - 1)]
    ref = oracle_heads(inp, heads)
    st = {name: stage(ws, wl, code, rows, cols) for name, code, rows, cols in (
        ("q_tilde", N.NYS_STAGE_Q_TILDE, wl.m, wl.d), ("k_tilde", N.NYS_STAGE_K_TILDE, wl.m, wl.d),
        ("g", N.NYS_STAGE_G, wl.m, wl.d), ("a_s", N.NYS_STAGE_A_S, wl.m, wl.m),
        ("z", N.NYS_STAGE_Z, wl.m, wl.m), ("w", N.NYS_STAGE_W, wl.m, wl.d))}
    # Z: the iterate after 6 updates, fp32 (CUDA cores) or tf32 products
    # with fp32 storage (tensor cores), relative to its largest entry
    tol = {"q_tilde": 1e-6, "k_tilde": 1e-6, "a_s": 1e-5, "z": 1e-4 if dtype == "f32" else 1e-2,
           "g": 1e-5 if dtype == "f32" else 1e-2, "w": 1e-4 if dtype == "f32" else 2e-2}
    for (b, h) in heads:
        i = b * wl.H + h
        for name in st:
            assert rel_err(st[name][i], ref[(b, h)][name]) <= tol[name], name
        np.testing.assert_allclose(st["a_s"][i].sum(axis=1), 1.0, atol=1e-5)


# ----------------------------------------------------------- full workloads ----

FULL = ["c1", "c2", "c3", "c4", "c5"]
_cache = {}


def full_inputs(name):
    if name not in _cache:
        _cache.clear()
        _cache[name] = workloads.make_inputs(workloads.WORKLOADS[name])
    return _cache[name]


@pytest.mark.parametrize("name", FULL)
def test_full_workload(name):
    """Every configuration at its full size, in the launch configuration the
    benchmark times, compared with the oracle on EVERY head (heads are
    independent, so the oracle runs head by head): the full output and the
    attention term alone, each head against the bar."""
    inp = full_inputs(name)
    wl = inp.wl
    got, _ = run_gpu(inp)
    got_att, _ = run_gpu(inp, ks=0)
    assert np.isfinite(got).all() and np.isfinite(got_att).all()
    worst = (0.0, 0.0)
    failed = []
    for b in range(wl.B):
        for h in range(wl.H):
            ref = R.nystrom_head(inp.q[b, h], inp.k[b, h], inp.v[b, h], inp.conv_w[h], wl.m,
                                 wl.iters)
            e_out = rel_err(got[b, h], ref["out"])
            e_att = rel_err(got_att[b, h], ref["att"])
            worst = (max(worst[0], e_out), max(worst[1], e_att))
            if e_out > TOL[wl.dtype] or e_att > TOL[wl.dtype]:
                failed.append(((b, h), e_out, e_att))
    print(f"{name}: {wl.heads} heads, worst out {worst[0]:.2e}, worst attention {worst[1]:.2e}")
    assert not failed, failed[:8]


# ------------------------------------------------------------ entry points ----

def test_host_entry_matches_device_entry():
    import torch
    import nystr_self_attention_gb300 as N
    wl = workloads.custom(2, 3, 512, 64, 64, 6, 33, "bf16")
    inp = workloads.make_inputs(wl, seed=11)
    dev_out, _ = run_gpu(inp)
    out_bits = np.zeros(inp.q_bits.shape, np.uint16)
    N.nystrom_attn_fwd_host(inp.q_bits, inp.k_bits, inp.v_bits, inp.conv_w, out_bits, wl.B, wl.H,
                            wl.n, wl.d, wl.m, wl.iters, wl.ks, N.NYS_BF16)
    host_out = (out_bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(host_out, dev_out)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_host_entry_in_head_range_chunks(dtype):
    """One batch entry of 16 heads: the host-buffer entry pipelines it in
    eight chunks of two heads (each with its own rows of the conv filters)."""
    import nystr_self_attention_gb300 as N
    wl = workloads.custom(1, 16, 640, 64, 64, 6, 9, dtype)
    inp = workloads.make_inputs(wl, seed=23)
    ref = R.nystrom_attention(inp.q, inp.k, inp.v, inp.conv_w, wl.m, wl.iters)
    if dtype == "bf16":
        out_bits = np.zeros(inp.q_bits.shape, np.uint16)
        N.nystrom_attn_fwd_host(inp.q_bits, inp.k_bits, inp.v_bits, inp.conv_w, out_bits, wl.B, wl.H,
                                wl.n, wl.d, wl.m, wl.iters, wl.ks, N.NYS_BF16)
        got = (out_bits.astype(np.uint32) << 16).view(np.float32)
    else:
        got = np.zeros(inp.q.shape, np.float32)
        N.nystrom_attn_fwd_host(inp.q, inp.k, inp.v, inp.conv_w, got, wl.B, wl.H, wl.n, wl.d, wl.m,
                                wl.iters, wl.ks, N.NYS_FP32)
    for h in range(wl.H):
        assert rel_err(got[0, h], ref[0, h]) <= TOL[dtype], h


def test_repeatable_and_workspace_entry_agrees():
    wl = workloads.custom(1, 4, 1024, 64, 64, 6, 33, "bf16")
    inp = workloads.make_inputs(wl, seed=12)
    a, _ = run_gpu(inp)
    b, _ = run_gpu(inp)
    c, _ = run_gpu(inp, workspace=True)
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_output_not_written_outside_bounds():
    import torch
    import nystr_self_attention_gb300 as N
    wl = workloads.custom(1, 2, 200, 64, 8, 6, 5, "bf16")
    inp = workloads.make_inputs(wl, seed=13)
    q, k, v, w = to_device(inp)
    total = q.numel()
    canary = torch.full((total + 4096,), 12345, dtype=torch.int16, device="cuda")
    out = canary[2048:2048 + total].view(torch.bfloat16).view(q.shape)
    N.nystrom_attn_fwd(q, k, v, w, out, wl.B, wl.H, wl.n, wl.d, wl.m, wl.iters, wl.ks, N.NYS_BF16)
    torch.cuda.synchronize()
    c = canary.cpu().numpy()
    assert (c[:2048] == 12345).all() and (c[2048 + total:] == 12345).all()
