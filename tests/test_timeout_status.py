"""The device-side timeout path, without a fault: nystrom_debug_stall_pinv
makes the tensor-core pseudo-inverse kernel wait on a barrier phase that
nothing completes; the bounded wait runs out after 1 ms, the kernel records
NYS_ERR_TIMEOUT and winds down, and nystrom_get_status reports it with the
CUDA context intact. With the switch off again, the next call is correct."""
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


@pytest.mark.parametrize("shape,dtype", [((1, 2, 256, 64, 32), "bf16"), ((16, 8, 512, 64, 128), "bf16"),
                                         ((1, 2, 256, 64, 32), "f32")],
                         ids=["z-beside-rows", "serial", "fp32-three-products"])
def test_timeout_is_reported_and_the_next_call_is_correct(shape, dtype):
    import torch
    import nystr_self_attention_gb300 as N
    B, H, n, d, m = shape
    wl = workloads.custom(B, H, n, d, m, 6, 9, dtype)
    assert "pinv_tc" in N.nystrom_plan_describe(B, H, n, d, m, 6, 9, dtype_code(dtype))
    inp = workloads.make_inputs(wl, seed=77)
    q, k, v, w = to_device(inp)
    out = torch.empty_like(q)
    args = (B, H, n, d, m, wl.iters, wl.ks, dtype_code(dtype))
    try:
        N.nystrom_debug_stall_pinv(True)
        N.nystrom_attn_fwd(q, k, v, w, out, *args)
        torch.cuda.synchronize()  # no CUDA error: the kernels returned
        assert N.nystrom_get_status() == N.NYS_ERR_TIMEOUT
    finally:
        N.nystrom_debug_stall_pinv(False)
    assert N.nystrom_get_status() == N.NYS_OK  # read once, then cleared
    N.nystrom_attn_fwd(q, k, v, w, out, *args)
    torch.cuda.synchronize()
    assert N.nystrom_get_status() == N.NYS_OK
    ref = R.nystrom_attention(inp.q, inp.k, inp.v, inp.conv_w, m, wl.iters, heads=[(0, 0), (B - 1, H - 1)])
    got = out.float().cpu().numpy()
    for b, h in [(0, 0), (B - 1, H - 1)]:
        assert rel_err(got[b, h], ref[b, h]) <= TOL[dtype]


def test_switch_rejects_other_values():
    import nystr_self_attention_gb300 as N
    assert N.load_library().nystrom_debug_stall_pinv(2) == N.NYS_ERR_ARG
