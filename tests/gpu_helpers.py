"""Shared helpers of the GPU tests: upload seeded inputs, run the library
through the C ABI, compare with the oracle."""
import numpy as np

import workloads

TOL = {"bf16": 2e-2, "f32": 1e-4}


def dtype_code(dtype):
    import nystr_self_attention_gb300 as N
    return N.NYS_BF16 if dtype == "bf16" else N.NYS_FP32


def to_device(inp):
    import torch
    if inp.wl.dtype == "bf16":
        conv = lambda bits: torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
        q, k, v = conv(inp.q_bits), conv(inp.k_bits), conv(inp.v_bits)
    else:
        q, k, v = (torch.from_numpy(x).cuda() for x in (inp.q, inp.k, inp.v))
    w = torch.from_numpy(np.ascontiguousarray(inp.conv_w)).cuda()
    return q, k, v, w


def run_gpu(inp, ks=None, workspace=False):
    """Forward pass through the C ABI; returns (out as fp32 numpy, ws tensor or None)."""
    import torch
    import nystr_self_attention_gb300 as N
    wl = inp.wl
    ks = wl.ks if ks is None else ks
    q, k, v, w = to_device(inp)
    out = torch.empty_like(q)
    dt = dtype_code(wl.dtype)
    ws = None
    if workspace:
        nbytes = N.nystrom_attn_workspace_bytes(wl.B, wl.H, wl.n, wl.d, wl.m, dt)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        N.nystrom_attn_fwd_ws(q, k, v, w if ks > 0 else None, out, wl.B, wl.H, wl.n, wl.d, wl.m,
                              wl.iters, ks, dt, ws, nbytes)
    else:
        N.nystrom_attn_fwd(q, k, v, w if ks > 0 else None, out, wl.B, wl.H, wl.n, wl.d, wl.m,
                           wl.iters, ks, dt)
    torch.cuda.synchronize()
    assert N.nystrom_get_status() == N.NYS_OK
    return out.float().cpu().numpy(), ws


def stage(ws, wl, which, rows, cols):
    """Read one stage array [B*H, rows, cols] (float32) from a workspace."""
    import torch
    import nystr_self_attention_gb300 as N
    off = N.nystrom_attn_stage_offset(wl.B, wl.H, wl.n, wl.d, wl.m, dtype_code(wl.dtype), which)
    assert off >= 0
    nbytes = wl.B * wl.H * rows * cols * 4
    return ws[off:off + nbytes].view(torch.float32).cpu().numpy().reshape(wl.B * wl.H, rows, cols)


def rel_err(got, ref):
    return float(np.abs(got - ref).max() / np.abs(ref).max())
