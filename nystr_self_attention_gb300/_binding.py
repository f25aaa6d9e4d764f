"""ctypes binding of libnystrom.so: same names as the C ABI
(include/nystrom.h), argument marshalling only. Every step of the forward
pass runs in the library's CUDA kernels; there is no Python or CPU path, and
calling without the built library raises."""
from __future__ import annotations

import ctypes
import os

NYS_FP32, NYS_BF16 = 0, 1
NYS_OK, NYS_ERR_ARG, NYS_ERR_SHAPE, NYS_ERR_ALIGN = 0, -1, -2, -3
NYS_ERR_UNSUPPORTED, NYS_ERR_NOMEM, NYS_ERR_CUDA, NYS_ERR_TIMEOUT = -4, -5, -6, -7
NYS_STAGE_Q_TILDE, NYS_STAGE_K_TILDE, NYS_STAGE_G, NYS_STAGE_A_S, NYS_STAGE_W, NYS_STAGE_Z = range(6)
NYS_CONV_PER_HEAD, NYS_CONV_PER_CHANNEL = 0, 1
NYS_CSTAGE_ASSIGN, NYS_CSTAGE_CENTROIDS_PREV, NYS_CSTAGE_CENTROIDS, NYS_CSTAGE_G = range(4)

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnystrom.so")
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIG = {
    "nystrom_attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "nystrom_attn_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "nystrom_attn_fwd_ws": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P,
                                 ctypes.c_size_t, _P]),
    "nystrom_attn_fwd_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "nystrom_attn_fwd_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "nystrom_attn_fwd_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P,
                                 ctypes.c_size_t, _P]),
    "nystrom_attn_stage_offset": (ctypes.c_longlong, [_I, _I, _I, _I, _I, _I, _I]),
    "nystrom_plan_describe": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.c_char_p, _I]),
    "nystrom_get_status": (_I, [_P]),
    "nystrom_strerror": (ctypes.c_char_p, [_I]),
    "nystrom_last_error_string": (ctypes.c_char_p, []),
    "nystrom_launch_count": (ctypes.c_ulonglong, []),
    "nystrom_profile_enable": (_I, [_I]),
    "nystrom_debug_stall_pinv": (_I, [_I]),
    "nystrom_mha_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "nystrom_clustered_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I]),
    "nystrom_clustered_stage_offset": (ctypes.c_longlong, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "nystrom_clustered_attn_fwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                                        ctypes.c_size_t, _P]),
    "nystrom_mha_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P,
                             ctypes.c_size_t, _P]),
    "nystrom_profile_read": (_I, [_I, ctypes.c_char_p, _I, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_longlong)]),
}


class NystromError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if code == NYS_ERR_CUDA:
            detail = ": " + load_library().nystrom_last_error_string().decode()
        super().__init__(f"{where} returned {code} ({nystrom_strerror(code)}){detail}")


def load_library(path: str | None = None):
    """Load libnystrom.so (built by __graft_entry__.build()). Raises if it
    is missing: there is no fallback."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIG.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):  # numpy array (host buffers)
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc < 0:
        raise NystromError(rc, where)
    return rc


def nystrom_attn_fwd(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype, stream=None):
    lib = load_library()
    return _check(lib.nystrom_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(conv_w), _ptr(out),
                                       B, H, n, d, m, iters, conv_ks, dtype, _stream(stream)),
                  "nystrom_attn_fwd")


def nystrom_attn_workspace_bytes(B, H, n, d, m, dtype) -> int:
    return load_library().nystrom_attn_workspace_bytes(B, H, n, d, m, dtype)


def nystrom_attn_fwd_ws(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype,
                        workspace, ws_bytes, stream=None):
    lib = load_library()
    return _check(lib.nystrom_attn_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(conv_w), _ptr(out),
                                          B, H, n, d, m, iters, conv_ks, dtype, _ptr(workspace),
                                          ws_bytes, _stream(stream)),
                  "nystrom_attn_fwd_ws")


def nystrom_attn_fwd_noalloc(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype,
                             stream=None):
    """The forward pass with no device allocation: scratch is a fixed 32 MiB
    array inside the library (see include/nystrom.h)."""
    lib = load_library()
    return _check(lib.nystrom_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(conv_w), _ptr(out),
                                               B, H, n, d, m, iters, conv_ks, dtype,
                                               _stream(stream)),
                  "nystrom_attn_fwd_noalloc")


def nystrom_attn_fwd_ex(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype,
                        conv_layout=NYS_CONV_PER_HEAD, lengths=None, workspace=None, ws_bytes=0,
                        stream=None):
    """The forward pass with per-channel conv filters and/or padded sequences
    (see include/nystrom.h). `lengths`: a host sequence of B ints, or None."""
    lib = load_library()
    lens = None
    if lengths is not None:
        lens = (ctypes.c_int * B)(*[int(x) for x in lengths])
    return _check(lib.nystrom_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(conv_w), _ptr(out),
                                          B, H, n, d, m, iters, conv_ks, dtype, conv_layout,
                                          ctypes.cast(lens, ctypes.c_void_p) if lens is not None
                                          else None, _ptr(workspace), ws_bytes, _stream(stream)),
                  "nystrom_attn_fwd_ex")


def nystrom_attn_fwd_host(q, k, v, conv_w, out, B, H, n, d, m, iters, conv_ks, dtype, stream=None):
    lib = load_library()
    return _check(lib.nystrom_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(conv_w), _ptr(out),
                                            B, H, n, d, m, iters, conv_ks, dtype, _stream(stream)),
                  "nystrom_attn_fwd_host")


def nystrom_attn_stage_offset(B, H, n, d, m, dtype, stage) -> int:
    return load_library().nystrom_attn_stage_offset(B, H, n, d, m, dtype, stage)


def nystrom_plan_describe(B, H, n, d, m, iters, conv_ks, dtype) -> str:
    """The kernels a forward call of this shape launches (host only)."""
    lib = load_library()
    need = _check(lib.nystrom_plan_describe(B, H, n, d, m, iters, conv_ks, dtype, None, 0),
                  "nystrom_plan_describe")
    buf = ctypes.create_string_buffer(need + 1)
    lib.nystrom_plan_describe(B, H, n, d, m, iters, conv_ks, dtype, buf, need + 1)
    return buf.value.decode()


def nystrom_get_status(stream=None) -> int:
    return load_library().nystrom_get_status(_stream(stream))


def nystrom_strerror(code: int) -> str:
    return load_library().nystrom_strerror(code).decode()


def nystrom_last_error_string() -> str:
    return load_library().nystrom_last_error_string().decode()


def nystrom_attention(q, k, v, conv_w, m: int, iters: int, out=None, stream=None):
    """Convenience call on CUDA torch tensors q, k, v [B, H, n, d] (float32
    or bfloat16, contiguous) and conv_w [H, ks] float32 (or None): allocates
    `out` if not given and calls nystrom_attn_fwd on the current stream."""
    import torch
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dim() == 4 and t.dtype == q.dtype):
            raise ValueError("q, k, v must be contiguous CUDA tensors [B, H, n, d] of one dtype")
    if q.dtype == torch.float32:
        dtype = NYS_FP32
    elif q.dtype == torch.bfloat16:
        dtype = NYS_BF16
    else:
        raise ValueError("dtype must be float32 or bfloat16")
    B, H, n, d = q.shape
    ks = 0
    if conv_w is not None:
        if not (conv_w.is_cuda and conv_w.dtype == torch.float32 and conv_w.is_contiguous()
                and conv_w.dim() == 2 and conv_w.shape[0] == H):
            raise ValueError("conv_w must be a contiguous float32 CUDA tensor [H, ks]")
        ks = conv_w.shape[1]
    if out is None:
        out = torch.empty_like(q)
    nystrom_attn_fwd(q, k, v, conv_w if ks > 0 else None, out, B, H, n, d, m, iters, ks, dtype,
                     stream)
    return out


def nystrom_mha_workspace_bytes(B, n, H, d, m, dtype) -> int:
    return load_library().nystrom_mha_workspace_bytes(B, n, H, d, m, dtype)


def nystrom_mha_fwd(x, w_qkv, b_qkv, w_o, b_o, conv_w, y, B, n, H, d, m, iters, conv_ks, dtype,
                    workspace=None, ws_bytes=0, stream=None):
    """The attention module around the op (see include/nystrom.h)."""
    lib = load_library()
    return _check(lib.nystrom_mha_fwd(_ptr(x), _ptr(w_qkv), _ptr(b_qkv), _ptr(w_o), _ptr(b_o),
                                      _ptr(conv_w), _ptr(y), B, n, H, d, m, iters, conv_ks, dtype,
                                      _ptr(workspace), ws_bytes, _stream(stream)),
                  "nystrom_mha_fwd")


def nystrom_clustered_workspace_bytes(B, H, n, d, C, dtype) -> int:
    return load_library().nystrom_clustered_workspace_bytes(B, H, n, d, C, dtype)


def nystrom_clustered_stage_offset(B, H, n, d, C, iters, dtype, stage) -> int:
    return load_library().nystrom_clustered_stage_offset(B, H, n, d, C, iters, dtype, stage)


def nystrom_clustered_attn_fwd(q, k, v, out, B, H, n, d, C, iters, dtype, workspace=None,
                               ws_bytes=0, stream=None):
    """Clustered attention, centroid path (see include/nystrom.h)."""
    lib = load_library()
    return _check(lib.nystrom_clustered_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, n, d,
                                                 C, iters, dtype, _ptr(workspace), ws_bytes,
                                                 _stream(stream)),
                  "nystrom_clustered_attn_fwd")


def nystrom_debug_stall_pinv(on: bool) -> int:
    """Timeout-path test switch (see include/nystrom.h)."""
    return _check(load_library().nystrom_debug_stall_pinv(1 if on else 0),
                  "nystrom_debug_stall_pinv")


def nystrom_launch_count() -> int:
    return load_library().nystrom_launch_count()


def nystrom_profile_enable(on: bool) -> int:
    return load_library().nystrom_profile_enable(1 if on else 0)


def nystrom_profile_read(max_kernels: int = 16) -> dict:
    """{kernel name: (total ms, launches)} recorded since the last read."""
    lib = load_library()
    name_len = 64
    names = ctypes.create_string_buffer(max_kernels * name_len)
    ms = (ctypes.c_double * max_kernels)()
    cnt = (ctypes.c_longlong * max_kernels)()
    n = _check(lib.nystrom_profile_read(max_kernels, names, name_len, ms, cnt), "nystrom_profile_read")
    out = {}
    for i in range(min(n, max_kernels)):
        nm = names.raw[i * name_len:(i + 1) * name_len].split(b"\0", 1)[0].decode()
        out[nm] = (ms[i], cnt[i])
    return out
