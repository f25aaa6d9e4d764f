"""Host-side plan of the forward pass (no GPU): which kernels a shape
launches and the sizes the plan gives them, through nystrom_plan_describe."""
import ctypes

import pytest

import workloads


@pytest.fixture(scope="module")
def N():
    from nystr_self_attention_gb300 import build
    build.build()
    import nystr_self_attention_gb300 as N
    return N


def plan(N, B, H, n, d, m, dtype, iters=6, ks=5):
    text = N.nystrom_plan_describe(B, H, n, d, m, iters, ks, dtype)
    return dict(item.split("=", 1) for item in text.split())


def workload_plan(N, name):
    w = workloads.WORKLOADS[name]
    return plan(N, w.B, w.H, w.n, w.d, w.m, N.NYS_BF16 if w.dtype == "bf16" else N.NYS_FP32,
                w.iters, w.ks)


def test_fp32_runs_three_tf32_products_on_the_tensor_cores(N):
    # c1: one head, n 512 -> four 128-key tiles, one landmark-row CTA each
    p = workload_plan(N, "c1")
    assert p["plan"] == "serial"
    assert p["rows"] == "rows_x3[splits=4,tiles_per_split=1]"
    assert p["pinv"].startswith("pinv_tc[") and p["tokens"] == "tokens_x3"
    assert "conv" not in p  # the convolution inside the token pass


@pytest.mark.parametrize("d,m,iters,rows,pinv,tokens", [
    (64, 128, 6, "rows_x3", "pinv_simt", "tokens_x3"),     # pseudo-inverse: m <= 64 only
    (64, 64, 13, "rows_x3", "pinv_simt", "tokens_x3"),     # past the three-product update limit
    (128, 64, 6, "rows_simt", "pinv_simt", "tokens_simt"),  # d > 64
    (40, 64, 6, "rows_x3", "pinv_simt", "tokens_x3"),      # d not a multiple of 32
    (8, 16, 6, "rows_x3", "pinv_simt", "tokens_x3"),
])
def test_fp32_kernel_choice(N, d, m, iters, rows, pinv, tokens):
    p = plan(N, 1, 2, 512, d, m, N.NYS_FP32, iters=iters)
    assert (p["rows"].split("[")[0], p["pinv"].split("[")[0], p["tokens"]) == (rows, pinv, tokens)


@pytest.mark.parametrize("name,pinv,rows_ctas", [
    ("c2", "pinv_tc[z-only,ctas=192,sms=96]", 152 - 96),  # two pseudo-inverse CTAs per SM
    ("c3", "pinv_tc[z-only,ctas=32,sms=32]", 152 - 32),
    ("c4", "pinv_tc[z-only,ctas=64,sms=64]", 152 - 64),
])
def test_z_beside_rows_for_the_bf16_workloads_up_to_m128(N, name, pinv, rows_ctas):
    p = workload_plan(N, name)
    assert p["plan"] == "z-beside-rows" and p["groups"] == "1"
    assert p["pinv"] == pinv
    assert p["merge"] == "merge_g" and p["w"] == "w_tc" and p["tokens"] == "tokens_tc"
    # the landmark-row pass spreads its tiles over at most the SMs left to it
    ctas = int(p["rows"].split("ctas=")[1].split(",")[0])
    assert p["rows"].startswith("rows_tc[") and ctas <= rows_ctas


def test_long_context_m256_is_serial_on_the_clustered_kernels(N):
    p = workload_plan(N, "c5")
    assert p["plan"] == "serial"
    assert p["pinv"] == "pinv_big[clusters=32]" and p["tokens"] == "tokens_big"
    assert p["rows"].startswith("rows_tc[ctas=152,")


@pytest.mark.parametrize("H,pinv", [
    (152, "pinv_tc[z-only,ctas=76,sms=76]"),   # fits one CTA per SM in half the GPU
    (154, "pinv_tc[z-only,ctas=77,sms=39]"),   # two CTAs per SM from here on
])
def test_pinv_packing_threshold(N, H, pinv):
    assert plan(N, 1, H, 128, 64, 64, N.NYS_BF16)["pinv"] == pinv


def test_too_many_heads_beside_the_rows_split_into_head_groups(N):
    p = plan(N, 2, 210, 128, 32, 64, N.NYS_BF16)
    assert p["plan"] == "head-groups" and p["groups"] == "2"
    assert p["pinv"] == "pinv_tc[ctas=105]"  # one group's 210 heads, two per CTA


def test_m128_with_many_heads_runs_the_pseudo_inverse_after_the_rows(N):
    p = plan(N, 4, 32, 256, 64, 128, N.NYS_BF16)
    assert p["plan"] == "serial" and p["pinv"] == "pinv_tc[ctas=128]"


@pytest.mark.parametrize("n,d,dtype,kernel", [
    (512, 64, 1, "landmarks_small"),   # 8-row segments
    (777, 32, 1, "landmarks_small"),   # segments of 12 and 13 rows
    (4096, 32, 1, "landmarks_vec"),    # 64-row segments
    (5000, 64, 0, "landmarks_vec"),
    (333, 96, 0, "landmarks_simt"),    # 24 vectors per row: does not divide 32
])
def test_landmark_kernel_choice(N, n, d, dtype, kernel):
    assert plan(N, 1, 2, n, d, 64 if n >= 64 else 16, dtype)["landmarks"] == kernel


def test_errors_and_truncation(N):
    lib = N.load_library()
    assert lib.nystrom_plan_describe(1, 1, 32, 64, 64, 6, 5, 1, None, 0) == N.NYS_ERR_SHAPE
    assert lib.nystrom_plan_describe(1, 1, 512, 64, 64, 6, 5, 1, None, 8) == N.NYS_ERR_ARG
    assert lib.nystrom_plan_describe(1, 1, 512, 64, 64, 6, 5, 1, None, -1) == N.NYS_ERR_ARG
    full = lib.nystrom_plan_describe(1, 1, 512, 64, 64, 6, 5, 1, None, 0)
    buf = ctypes.create_string_buffer(b"#" * 16)
    assert lib.nystrom_plan_describe(1, 1, 512, 64, 64, 6, 5, 1, buf, 10) == full > 9
    assert buf.raw[:10] == N.nystrom_plan_describe(1, 1, 512, 64, 64, 6, 5, 1)[:9].encode() + b"\0"
    assert buf.raw[10:16] == b"#" * 6  # nothing written past len


def test_many_updates_leave_the_tensor_core_pseudo_inverse(N):
    """Past 8 updates the bf16 path's pseudo-inverse runs in fp32 (CUDA cores)."""
    assert plan(N, 1, 2, 512, 64, 64, N.NYS_BF16, iters=8)["pinv"].startswith("pinv_tc")
    assert plan(N, 1, 2, 512, 64, 64, N.NYS_BF16, iters=9)["pinv"] == "pinv_simt"
    assert plan(N, 1, 2, 512, 128, 256, N.NYS_BF16, iters=8)["pinv"].startswith("pinv_big")
    assert plan(N, 1, 2, 512, 128, 256, N.NYS_BF16, iters=12)["pinv"] == "pinv_simt"
