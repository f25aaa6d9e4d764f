"""GPU parity of the attention module around the op (nystrom_mha_fwd:
projections in, heads, Nyström attention, heads merged, projection out)
against the oracle's mha_forward on the same seeded random weights. Bars as
for the op: max|y - ref| / max|ref| <= 2e-2 for bf16, <= 1e-4 for float32."""
import numpy as np
import pytest

import workloads
from oracle import nystrom_ref as R
from tests.gpu_helpers import TOL, dtype_code, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    import torch
    from nystr_self_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    torch.cuda.set_device(0)


def run_module(inp, workspace=False):
    import torch
    import nystr_self_attention_gb300 as N
    wl = inp.wl

    def dev(name):
        if wl.dtype == "bf16":
            return torch.from_numpy(inp.bits[name].view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(getattr(inp, name)).cuda()

    x, w_qkv, w_o = dev("x"), dev("w_qkv"), dev("w_o")
    b_qkv, b_o = torch.from_numpy(inp.b_qkv).cuda(), torch.from_numpy(inp.b_o).cuda()
    conv = torch.from_numpy(np.ascontiguousarray(inp.conv_w)).cuda() if wl.ks > 0 else None
    y = torch.full_like(x, float("nan"))
    ws, nbytes = None, 0
    if workspace:
        nbytes = N.nystrom_mha_workspace_bytes(wl.B, wl.n, wl.H, wl.d, wl.m, dtype_code(wl.dtype))
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    N.nystrom_mha_fwd(x, w_qkv, b_qkv, w_o, b_o, conv, y, wl.B, wl.n, wl.H, wl.d, wl.m, wl.iters,
                      wl.ks, dtype_code(wl.dtype), ws, nbytes)
    torch.cuda.synchronize()
    assert N.nystrom_get_status() == N.NYS_OK
    return y.float().cpu().numpy()


SHAPES = [
    # B, n, H, d, m, iters, ks
    (2, 512, 4, 64, 64, 6, 33),
    (1, 1000, 2, 128, 160, 6, 9),
    (3, 384, 3, 32, 48, 4, 0),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{s[0]}n{s[1]}H{s[2]}d{s[3]}m{s[4]}" for s in SHAPES])
def test_module(shape, dtype):
    B, n, H, d, m, iters, ks = shape
    wl = workloads.custom(B, H, n, d, m, iters, ks, dtype)
    inp = workloads.module_inputs(wl, seed=90 + n)
    got = run_module(inp)
    assert np.isfinite(got).all()
    ref = R.mha_forward(inp.x, inp.w_qkv, inp.b_qkv, inp.w_o, inp.b_o, inp.conv_w, H, m, iters)
    assert rel_err(got, ref) <= TOL[dtype]


def test_module_bert_base_size():
    """The BERT-base-sized module (B=32, n=512, H=12, d=64: D=768) in bf16,
    the page's GLUE / IMDB setting, with its own workspace."""
    wl = workloads.custom(32, 12, 512, 64, 64, 6, 33, "bf16")
    inp = workloads.module_inputs(wl, seed=95)
    got = run_module(inp, workspace=True)
    ref = R.mha_forward(inp.x, inp.w_qkv, inp.b_qkv, inp.w_o, inp.b_o, inp.conv_w, wl.H, wl.m,
                        wl.iters)
    err = rel_err(got, ref)
    print(f"module B32 n512 H12 d64 bf16: {err:.2e}")
    assert err <= TOL["bf16"]
