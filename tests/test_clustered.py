"""GPU parity of clustered attention (centroid path, nystrom_clustered_attn_fwd)
against the oracle (oracle/clustered_ref.py).

K-means decides integers (each query's cluster) from fp32 distances on the
GPU and fp64 ones in the oracle, so queries that sit almost exactly between
two centroids may legitimately go either way. Where the clusters are well
separated the assignment is unique and is compared exactly; on random inputs
what is unique is checked instead, and the rest for validity: every query
sits at a centroid that is nearest within fp32 rounding (of the centroids
the last assignment used), every centroid is the mean of its queries (or
unchanged if it has none), and every output row is its centroid's attention
row. Output bars as for the Nyström path: 2e-2 bf16, 1e-4 float32."""
import numpy as np
import pytest

import workloads
from oracle import clustered_ref as CR
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


def upload(x, dtype):
    import torch
    if dtype == "bf16":
        vals, bits = workloads.round_to_bf16(x)
        return vals, torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    x = np.ascontiguousarray(x, dtype=np.float32)
    return x, torch.from_numpy(x).cuda()


def run_clustered(q, k, v, C, iters, dtype):
    """Returns (out, assign, mu_prev, mu, q, k, v) with q, k, v the values the
    GPU saw (bf16-rounded where bf16)."""
    import torch
    import nystr_self_attention_gb300 as N
    B, H, n, d = q.shape
    qv, qd = upload(q, dtype)
    kv, kd = upload(k, dtype)
    vv, vd = upload(v, dtype)
    out = torch.full_like(qd, float("nan"))
    dt = dtype_code(dtype)
    nbytes = N.nystrom_clustered_workspace_bytes(B, H, n, d, C, dt)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    N.nystrom_clustered_attn_fwd(qd, kd, vd, out, B, H, n, d, C, iters, dt, ws, nbytes)
    torch.cuda.synchronize()
    assert N.nystrom_get_status() == N.NYS_OK

    def stage(code, dtype_, shape):
        off = N.nystrom_clustered_stage_offset(B, H, n, d, C, iters, dt, code)
        nb = int(np.prod(shape)) * 4
        return ws[off:off + nb].view(dtype_).cpu().numpy().reshape(shape)
    a = stage(N.NYS_CSTAGE_ASSIGN, torch.int32, (B, H, n))
    mp = stage(N.NYS_CSTAGE_CENTROIDS_PREV, torch.float32, (B, H, C, d))
    mu = stage(N.NYS_CSTAGE_CENTROIDS, torch.float32, (B, H, C, d))
    return out.float().cpu().numpy(), a, mp, mu, qv, kv, vv


def check_valid(out, a, mp, mu, q, k, v, dtype):
    """The properties of a K-means round and of the centroid path, per head."""
    B, H, n, d = q.shape
    C = mu.shape[2]
    for b in range(B):
        for h in range(H):
            qh = q[b, h].astype(np.float64)
            prev = mp[b, h].astype(np.float64)
            # fp64 squared distances (the expansion is exact enough in fp64)
            dist = (qh * qh).sum(1)[:, None] - 2.0 * qh @ prev.T + (prev * prev).sum(1)[None, :]
            mine = dist[np.arange(n), a[b, h]]
            best = dist.min(axis=1)
            assert np.all(mine <= best + 1e-5 * (best + 1.0)), "a query is not at a nearest centroid"
            for c in range(C):
                members = qh[a[b, h] == c]
                want = members.mean(axis=0) if len(members) else prev[c]
                np.testing.assert_allclose(mu[b, h, c], want, rtol=1e-5, atol=1e-5)
            g = R.landmark_rows(mu[b, h].astype(np.float64), k[b, h], v[b, h])
            assert rel_err(out[b, h], g[a[b, h]]) <= TOL[dtype]


def separated(B, H, n, d, C, seed):
    """Queries in C contiguous runs around far-apart centres (so that the
    segment means start inside the right clusters); keys and values normal."""
    rng = np.random.default_rng(seed)
    centres = rng.standard_normal((B, H, C, d)).astype(np.float32) * 8.0
    runs = [(i * n // C, (i + 1) * n // C) for i in range(C)]
    q = np.empty((B, H, n, d), np.float32)
    for c, (lo, hi) in enumerate(runs):
        q[:, :, lo:hi] = centres[:, :, c:c + 1]
    q += rng.standard_normal(q.shape, dtype=np.float32) * 0.5
    k = rng.standard_normal(q.shape, dtype=np.float32)
    v = rng.standard_normal(q.shape, dtype=np.float32)
    return q, k, v, runs


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(2, 2, 512, 64, 16, 3), (1, 3, 1000, 32, 40, 5),
                                   (1, 2, 640, 128, 160, 2)],
                         ids=["n512d64C16", "n1000d32C40", "n640d128C160"])
def test_well_separated_clusters_match_exactly(shape, dtype):
    B, H, n, d, C, iters = shape
    q, k, v, runs = separated(B, H, n, d, C, seed=n + C)
    out, a, mp, mu, qv, kv, vv = run_clustered(q, k, v, C, iters, dtype)
    for b in range(B):
        for h in range(H):
            ref = CR.clustered_head(qv[b, h], kv[b, h], vv[b, h], C, iters)
            assert np.array_equal(a[b, h], ref["assign"])
            np.testing.assert_allclose(mu[b, h], ref["mu"], rtol=1e-5, atol=1e-5)
            assert rel_err(out[b, h], ref["out"]) <= TOL[dtype]
    check_valid(out, a, mp, mu, qv, kv, vv, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_one_cluster_per_query_is_exact_attention(dtype):
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((1, 2, 256, 64), dtype=np.float32) for _ in range(3))
    out, a, _, _, qv, kv, vv = run_clustered(q, k, v, 256, 2, dtype)
    for h in range(2):
        assert np.array_equal(a[0, h], np.arange(256))
        assert rel_err(out[0, h], R.softmax_attention(qv[0, h], kv[0, h], vv[0, h])) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(2, 3, 512, 64, 64, 10), (1, 2, 777, 32, 48, 4),
                                   (1, 1, 1024, 128, 256, 6), (1, 2, 1000, 128, 100, 4),
                                   (2, 2, 300, 64, 128, 5)],
                         ids=["n512d64C64", "n777d32C48", "n1024d128C256", "n1000d128C100",
                              "n300d64C128"])
def test_random_inputs_give_a_valid_result(shape, dtype):
    B, H, n, d, C, iters = shape
    wl = workloads.custom(B, H, n, d, C, iters, 0, dtype)
    inp = workloads.make_inputs(wl, seed=500 + C)
    out, a, mp, mu, qv, kv, vv = run_clustered(inp.q, inp.k, inp.v, C, iters, dtype)
    check_valid(out, a, mp, mu, qv, kv, vv, dtype)
    agree = np.mean([np.mean(a[b, h] == CR.clustered_head(qv[b, h], kv[b, h], vv[b, h], C, iters)["assign"])
                     for b in range(B) for h in range(H)])
    print(f"clustered {shape} {dtype}: assignments equal to the fp64 oracle's: {agree:.4f}")


def test_full_size_clustered_workload():
    """The clustered-input workload (B=8 H=8 n=8192 d=64, rank-4 segment
    drift) with C = 128 clusters and 10 K-means rounds, every head checked
    for validity."""
    wl = workloads.WORKLOADS["c4"]
    inp = workloads.make_inputs(wl)
    out, a, mp, mu, qv, kv, vv = run_clustered(inp.q, inp.k, inp.v, 128, 10, "bf16")
    check_valid(out, a, mp, mu, qv, kv, vv, "bf16")


@pytest.mark.parametrize("shape", [(2, 2, 1000, 64, 96, 6), (1, 2, 640, 128, 128, 3)],
                         ids=["n1000d64C96", "n640d128C128"])
def test_rounds_are_deterministic(shape):
    """The members' sums are added across CTAs in a fixed order: two calls
    give the same assignments, centroids and output, bit for bit."""
    B, H, n, d, C, iters = shape
    wl = workloads.custom(B, H, n, d, C, iters, 0, "bf16")
    inp = workloads.make_inputs(wl, seed=900 + C)
    first = run_clustered(inp.q, inp.k, inp.v, C, iters, "bf16")
    second = run_clustered(inp.q, inp.k, inp.v, C, iters, "bf16")
    for x, y in zip(first[:4], second[:4]):
        assert np.array_equal(x, y)
