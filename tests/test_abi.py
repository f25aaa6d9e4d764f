"""The C ABI without a GPU: the library builds and loads, exports every
function include/nystrom.h declares, and rejects bad arguments with the
documented codes before touching CUDA. No compute call runs here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nystrom.h")


@pytest.fixture(scope="module")
def N():
    from nystr_self_attention_gb300 import build
    build.build()
    import nystr_self_attention_gb300 as pkg
    pkg.load_library()
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nystrom_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("nystrom_attn_fwd", "nystrom_attn_fwd_ws", "nystrom_attn_workspace_bytes",
                     "nystrom_attn_fwd_host", "nystrom_get_status", "nystrom_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(N):
    lib = ctypes.CDLL(N.LIB_PATH)
    missing = [name for name in declared_functions() if not hasattr(lib, name)]
    assert not missing, f"not exported: {missing}"


def test_binding_wraps_every_declared_symbol(N):
    for name in declared_functions():
        assert hasattr(N, name), f"binding lacks {name}"


def test_strerror_covers_codes(N):
    for code in range(0, -8, -1):
        assert N.nystrom_strerror(code) not in ("", "unknown status code")
    assert N.nystrom_strerror(5) == "unknown status code"


GOOD = dict(B=2, H=3, n=64, d=64, m=8, iters=6, ks=5, dtype=1)


def call(N, q=16, k=16, v=16, w=16, out=16, **kw):
    a = dict(GOOD, **kw)
    lib = N.load_library()
    return lib.nystrom_attn_fwd(q, k, v, w, out, a["B"], a["H"], a["n"], a["d"], a["m"], a["iters"],
                                a["ks"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(out=None), -1), (dict(w=None), -1), (dict(dtype=2), -1),
    (dict(B=0), -2), (dict(n=4), -2), (dict(m=512, n=512), -2), (dict(d=48), -2),
    (dict(d=12, dtype=0), -2), (dict(d=256), -2), (dict(iters=-1), -2), (dict(iters=65), -2),
    (dict(ks=4), -2), (dict(ks=129), -2), (dict(ks=-1), -2),
    (dict(q=24), -3), (dict(out=8), -3), (dict(w=18), -3),
])
def test_argument_errors_before_any_launch(N, kw, code):
    assert call(N, **kw) == code


def test_conv_weights_may_be_null_without_conv(N):
    # with ks = 0 a NULL conv_w is accepted by the checks; the call then
    # needs a GPU, which this machine may lack (NYS_ERR_UNSUPPORTED)
    assert call(N, w=None, ks=0, q=24) == -3


def test_workspace_sizes(N):
    assert N.nystrom_attn_workspace_bytes(32, 12, 512, 64, 64, 1) > 0
    assert N.nystrom_attn_workspace_bytes(1, 1, 100, 64, 64, 1) > 0  # ragged segments
    assert N.nystrom_attn_workspace_bytes(1, 1, 48, 64, 64, 1) == 0  # m > n
    assert N.nystrom_attn_workspace_bytes(1, 1, 512, 64, 64, 1) % 256 == 0
    a = N.nystrom_attn_workspace_bytes(2, 16, 32768, 128, 256, 1)
    b = N.nystrom_attn_workspace_bytes(4, 16, 32768, 128, 256, 1)
    assert b > a
    for stage in range(5):
        off = N.nystrom_attn_stage_offset(2, 3, 64, 64, 8, 1, stage)
        assert 0 <= off < N.nystrom_attn_workspace_bytes(2, 3, 64, 64, 8, 1) and off % 256 == 0
    assert N.nystrom_attn_stage_offset(2, 3, 64, 64, 8, 1, 9) == -1


def test_workspace_entry_checks(N):
    lib = N.load_library()
    ws_need = N.nystrom_attn_workspace_bytes(2, 3, 64, 64, 8, 1)
    args = (16, 16, 16, 16, 16, 2, 3, 64, 64, 8, 6, 5, 1)
    assert lib.nystrom_attn_fwd_ws(*args, None, ws_need, None) == -1
    assert lib.nystrom_attn_fwd_ws(*args, 128, ws_need, None) == -3
    assert lib.nystrom_attn_fwd_ws(*args, 256, ws_need - 1, None) == -5


def test_host_entry_checks(N):
    lib = N.load_library()
    assert lib.nystrom_attn_fwd_host(None, 16, 16, 16, 16, 2, 3, 64, 64, 8, 6, 5, 1, None) == -1
    assert lib.nystrom_attn_fwd_host(16, 16, 16, 16, 16, 2, 3, 4, 64, 8, 6, 5, 1, None) == -2


def test_binding_raises_on_error(N):
    with pytest.raises(N.NystromError) as e:
        N.nystrom_attn_fwd(16, 16, 16, 16, 16, 2, 3, 4, 64, 8, 6, 5, 1, stream=0)
    assert e.value.code == -2


def test_no_cpu_path(N):
    """There is no CPU implementation behind the ABI: CPU tensors are refused
    and, on a machine without a GB300, a well-formed call fails instead of
    computing anything."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("checks the behaviour without a GPU")
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        N.nystrom_attention(q, q, q, None, 8, 6)
    with pytest.raises(N.NystromError) as e:
        N.nystrom_attn_fwd(16, 16, 16, 16, 16, 1, 1, 64, 64, 8, 6, 5, N.NYS_BF16, stream=0)
    assert e.value.code == N.NYS_ERR_UNSUPPORTED


def test_fwd_ex_rejects_bad_variant_arguments(N):
    lib = N.load_library()
    a = GOOD

    def ex(layout=0, lengths=None, ws=None, ws_bytes=0):
        arr = None
        if lengths is not None:
            arr = (ctypes.c_int * len(lengths))(*lengths)
        return lib.nystrom_attn_fwd_ex(16, 16, 16, 16, 16, a["B"], a["H"], a["n"], a["d"], a["m"],
                                       a["iters"], a["ks"], a["dtype"], layout,
                                       ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None,
                                       ws, ws_bytes, None)
    assert ex(layout=2) == N.NYS_ERR_ARG
    assert ex(lengths=[a["m"] - 1, a["n"]]) == N.NYS_ERR_SHAPE   # shorter than m
    assert ex(lengths=[a["n"] + 1, a["n"]]) == N.NYS_ERR_SHAPE   # longer than n
    assert ex(ws=256 + 16) == N.NYS_ERR_ALIGN                    # workspace not 256-aligned
    assert ex(ws=256, ws_bytes=8) == N.NYS_ERR_NOMEM              # workspace too small


def test_stall_switch_rejects_other_values(N):
    lib = N.load_library()
    assert lib.nystrom_debug_stall_pinv(2) == N.NYS_ERR_ARG
    assert lib.nystrom_debug_stall_pinv(0) == N.NYS_OK


def test_module_rejects_bad_arguments(N):
    lib = N.load_library()

    def mha(x=256, w=256, wo=256, y=256, b=None, ws=None, nbytes=0, **kw):
        a = dict(dict(B=2, n=64, H=2, d=64, m=8, iters=6, ks=0, dtype=1), **kw)
        return lib.nystrom_mha_fwd(x, w, b, wo, b, None, y, a["B"], a["n"], a["H"], a["d"], a["m"],
                                   a["iters"], a["ks"], a["dtype"], ws, nbytes, None)
    assert mha(x=None) == N.NYS_ERR_ARG
    assert mha(ks=5) == N.NYS_ERR_ARG            # a conv width without weights
    assert mha(d=48) == N.NYS_ERR_SHAPE          # bf16 head width outside {32, 64, 128}
    assert mha(x=264) == N.NYS_ERR_ALIGN
    assert mha(ws=256 + 64) == N.NYS_ERR_ALIGN
    assert mha(ws=256, nbytes=16) == N.NYS_ERR_NOMEM
    assert N.nystrom_mha_workspace_bytes(2, 64, 2, 64, 8, 1) > 0
    assert N.nystrom_mha_workspace_bytes(2, 64, 2, 48, 8, 1) == 0


def test_clustered_rejects_bad_arguments(N):
    lib = N.load_library()

    def cl(q=256, iters=3, C=8, d=64, ws=None, nbytes=0):
        return lib.nystrom_clustered_attn_fwd(q, 256, 256, 256, 2, 2, 64, d, C, iters, 1, ws, nbytes,
                                              None)
    assert cl(q=None) == N.NYS_ERR_ARG
    assert cl(iters=0) == N.NYS_ERR_SHAPE
    assert cl(iters=65) == N.NYS_ERR_SHAPE
    assert cl(C=65) == N.NYS_ERR_SHAPE     # more clusters than queries
    assert cl(q=264) == N.NYS_ERR_ALIGN
    assert cl(ws=256, nbytes=8) == N.NYS_ERR_NOMEM
    for it in (1, 2, 3):
        last = N.nystrom_clustered_stage_offset(2, 2, 64, 64, 8, it, 1, N.NYS_CSTAGE_CENTROIDS)
        prev = N.nystrom_clustered_stage_offset(2, 2, 64, 64, 8, it, 1, N.NYS_CSTAGE_CENTROIDS_PREV)
        assert last >= 0 and prev >= 0 and last != prev
    assert N.nystrom_clustered_stage_offset(2, 2, 64, 64, 8, 1, 1, 9) == -1
