"""GPU parity of the low-M projections (kda_skinny_proj) against the fp64 oracle.

The shapes are those of the skinny-GEMM test in the vLLM PR report "[Bugfix] Fix Kimi-K3
KDA projection overlap compile on Hopper": hidden 7168 -> 144, the first 128 columns ->
1536, m = 2, 8, 14 (and 1 and 16 here).  Tolerances follow from the arithmetic: y is the
fp32 sum of k products rounded to bf16 (half a bf16 ulp: at most 2^-8 of the value, for a
value just above a power of two; plus a bound on the fp32 summation); z multiplies y's
bf16 values, which may sit one bf16 ulp (at most 2^-7 of the value) from the oracle's
rounding of its fp64 y where the two sums straddle a rounding boundary.
"""
import numpy as np
import pytest
import torch

import kda_gated_delta_chunk_gb300 as kda
from oracle.proj import bf16_round, skinny_proj as proj_oracle

pytestmark = pytest.mark.gpu

K, NAB, R, NB = 7168, 144, 128, 1536


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kda_gated_delta_chunk_gb300 import build as kbuild
    kbuild.build()
    assert kda.device_check(torch.cuda.current_device()) == kda.OK


def inputs(m, k=K, n_ab=NAB, r=R, n_b=NB, seed=0):
    g = torch.Generator().manual_seed(43 + m + seed)
    x = torch.randn(m, k, generator=g).to(torch.bfloat16)
    w_ab = torch.randn(n_ab, k, generator=g).to(torch.bfloat16)
    w_b = torch.randn(n_b, r, generator=g).to(torch.bfloat16)
    return x, w_ab, w_b


def check(x, w_ab, w_b, r, y, z):
    f = lambda t: t.double().numpy()
    y64, z64 = proj_oracle(f(x), f(w_ab), f(w_b), r)
    k = x.shape[1]
    absdot = np.abs(f(x)) @ np.abs(f(w_ab)).T
    tol_y = 2.0 ** -8 * np.abs(y64) + k * 2.0 ** -23 * absdot
    dy = np.abs(f(y.cpu()) - y64)
    assert np.all(dy <= tol_y), float((dy / np.maximum(tol_y, 1e-30)).max())
    yb = bf16_round(y64)[:, :r]
    tol_z = 2.0 ** -8 * np.abs(z64) + 2.0 ** -7 * (np.abs(yb) @ np.abs(f(w_b)).T) \
        + r * 2.0 ** -23 * (np.abs(yb) @ np.abs(f(w_b)).T)
    dz = np.abs(f(z.cpu()) - z64)
    assert np.all(dz <= tol_z), float((dz / np.maximum(tol_z, 1e-30)).max())
    return dy.max(), dz.max()


@pytest.mark.parametrize("m", [1, 2, 8, 14, 16])
def test_pages_shapes(m):
    x, w_ab, w_b = inputs(m)
    y, z = kda.skinny_proj(x.cuda(), w_ab.cuda(), w_b.cuda(), R)
    torch.cuda.synchronize()
    dy, dz = check(x, w_ab, w_b, R, y, z)
    print(f"m={m}: max |dy| {dy:.3e}  max |dz| {dz:.3e}")


def test_deterministic_and_reusable_workspace():
    """The split-K partial sums are added in a fixed order: two calls give the same bits,
    and the workspace's arrival counters are left ready for the next call."""
    x, w_ab, w_b = (t.cuda() for t in inputs(8))
    ws = torch.zeros(kda.skinny_proj_workspace_size(K, NAB), dtype=torch.uint8, device="cuda")
    a = kda.skinny_proj(x, w_ab, w_b, R, workspace=ws)
    b = kda.skinny_proj(x, w_ab, w_b, R, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_small_shapes_and_strided_outputs():
    """The smallest shapes the call accepts, and y / z written as views of wider buffers
    (rows of the buffers the next kernels read), strided x rows."""
    m, k, n_ab, r, n_b = 5, 512, 32, 16, 48
    x, w_ab, w_b = inputs(m, k, n_ab, r, n_b, seed=9)
    xw = torch.zeros(m, k + 64, dtype=torch.bfloat16, device="cuda")
    xw[:, 8:8 + k] = x.cuda()
    yb = torch.full((m, n_ab + 24), 7.0, dtype=torch.bfloat16, device="cuda")
    zb = torch.full((m, n_b + 10), 7.0, dtype=torch.bfloat16, device="cuda")
    y, z = kda.skinny_proj(xw[:, 8:8 + k], w_ab.cuda(), w_b.cuda(), r, y=yb[:, 8:8 + n_ab],
                           z=zb[:, 2:2 + n_b])
    torch.cuda.synchronize()
    check(x, w_ab, w_b, r, y, z)
    assert torch.all(yb[:, :8].float() == 7.0) and torch.all(yb[:, 8 + n_ab:].float() == 7.0)
    assert torch.all(zb[:, :2].float() == 7.0) and torch.all(zb[:, 2 + n_b:].float() == 7.0)


def test_cuda_graph_replay():
    x, w_ab, w_b = (t.cuda() for t in inputs(14, seed=3))
    ws = torch.zeros(kda.skinny_proj_workspace_size(K, NAB), dtype=torch.uint8, device="cuda")
    y = torch.empty(14, NAB, dtype=torch.bfloat16, device="cuda")
    z = torch.empty(14, NB, dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        kda.skinny_proj(x, w_ab, w_b, R, y=y, z=z, workspace=ws, stream=side)
    side.synchronize()
    ref = (y.clone(), z.clone())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        kda.skinny_proj(x, w_ab, w_b, R, y=y, z=z, workspace=ws, stream=side)
    for _ in range(3):
        y.zero_()
        z.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref[0]) and torch.equal(z, ref[1])


@pytest.mark.parametrize("over", [dict(m=17), dict(m=0), dict(k=7424), dict(r=24), dict(r=160),
                                  dict(n_b=40)])
def test_refused_shapes(over):
    a = dict(m=4, k=K, n_ab=NAB, r=R, n_b=NB)
    a.update(over)
    x = torch.zeros(max(a["m"], 1), a["k"], dtype=torch.bfloat16, device="cuda")
    w_ab = torch.zeros(a["n_ab"], a["k"], dtype=torch.bfloat16, device="cuda")
    w_b = torch.zeros(a["n_b"], a["r"], dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kda.KDAError) as e:
        kda.skinny_proj(x[:a["m"]] if a["m"] > 0 else x[:0], w_ab, w_b, a["r"])
    assert e.value.code == kda.ERR_INVALID_ARG
