"""GPU parity of the Gaussian-RBF grid (hg_rbf_fwd / hg_rbf_bwd: DInf-Grid's
normalised Gaussian interpolation over a ring neighbourhood) against the
oracle, element by element.

Cases: d = 2 and 3; rings 1 to 4; kernel widths 0.5 to 2; dense (the page's
grids) and hashed levels; fp32 and fp16 tables; F = 1, 2, 4; both layouts;
masks; points at the grid's border (clipped neighbourhoods) and the edge
coordinates; stratified (coherent) points in 2D and 3D (runs of same-cell
points, tiles over several rows of strata) and the same points shuffled (runs
of one point, tap boxes too large for a CTA's tile); coarse levels with many
points per vertex.  Tolerance 1e-5 of the oracle's
condition magnitude (every term of the quotient rule in absolute value)."""
import zlib

import numpy as np
import pytest

from _harness import check_close, dev, host
from test_parity_gpu import _coords

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


# (id, d, L, F, n_min, n_max, log2T, dtype, layout, n, mask, eps, rings)
CASES = [
    ("2d_F2_ring3_dense", 2, 3, 2, 16, 64, 13, "f32", 1, 3000, None, 1.0, 3),
    ("2d_F1_ring1_hashed_point_major", 2, 3, 1, 8, 200, 10, "f32", 0, 1500, None, 0.5, 1),
    ("2d_F2_f16_ring2", 2, 4, 2, 4, 40, 12, "f16", 1, 2000, None, 2.0, 2),
    ("2d_F4_ring4", 2, 2, 4, 8, 30, 11, "f32", 1, 700, None, 0.7, 4),
    ("3d_F2_ring3_dense", 3, 3, 2, 4, 16, 13, "f32", 1, 1500, None, 1.0, 3),
    ("3d_F2_ring2_hashed_point_major", 3, 3, 2, 4, 40, 11, "f32", 0, 900, None, 1.5, 2),
    ("3d_F1_f16_ring1_mask", 3, 3, 1, 4, 30, 12, "f16", 1, 800, 0b101, 1.0, 1),
    ("3d_F2_ring4", 3, 2, 2, 3, 9, 12, "f32", 1, 300, None, 0.8, 4),
    ("2d_F2_stratified", 2, 3, 2, 16, 64, 13, "f32", 1, 16384, None, 1.0, 3),
    ("2d_F2_coarse_many_points", 2, 2, 2, 4, 8, 10, "f32", 1, 20000, None, 1.0, 3),
    ("3d_F2_coarse_many_points", 3, 2, 2, 2, 5, 10, "f32", 0, 30000, None, 1.0, 2),
    ("3d_one_point", 3, 2, 2, 4, 8, 10, "f32", 1, 1, None, 1.0, 3),
    # 3D stratified points: runs of same-cell points, tiles of two or more rows of strata
    ("3d_F2_stratified", 3, 3, 2, 7, 28, 15, "f32", 1, 13824, None, 1.0, 3),
    ("3d_F1_stratified_hashed_point_major", 3, 2, 1, 5, 20, 12, "f32", 0, 8000, None, 0.8, 2),
    ("3d_F4_stratified_ring4", 3, 2, 4, 4, 12, 12, "f32", 1, 4096, None, 1.2, 4),
    ("3d_F2_stratified_shuffled", 3, 3, 2, 7, 28, 15, "f32", 1, 13824, None, 1.0, 3),
    ("2d_F2_stratified_shuffled", 2, 3, 2, 16, 64, 13, "f32", 1, 16384, None, 1.0, 3),
]


def _build(case, seed=0):
    import multiresolution_hash_grid_02_b300 as m
    import oracle
    cid, d, L, F, nmin, nmax, log2T, dt, layout, n, mask, eps, rings = case
    rng = np.random.default_rng(zlib.crc32(cid.encode()) + seed)
    res = oracle.level_resolutions(L, nmin, nmax)
    x = _coords(rng, n, d, res, stratified="stratified" in cid)
    if "shuffled" in cid:  # the same strata in a random order: runs of one point, boxes past the tile
        x = np.ascontiguousarray(x[rng.permutation(n)])
    npdt = np.float16 if dt == "f16" else np.float32
    table = (rng.random((L, 1 << log2T, F), dtype=np.float32) * 2 - 1).astype(npdt)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=nmin, n_max=nmax, log2_T=(log2T,), level_mask=mask,
                      dtype=m.HG_F16 if dt == "f16" else m.HG_F32, layout=layout)
    return m, oracle, desc, res, x, table, rng


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rbf_forward_parity(case):
    from multiresolution_hash_grid_02_b300 import workloads as W
    m, oracle, desc, res, x, table, rng = _build(case)
    n, d, L, F = x.shape[0], desc.d, desc.L, desc.F
    eps, rings = case[11], case[12]
    fm = desc.layout == m.HG_FEATURE_MAJOR
    g = torch.full((L, F, n) if fm else (n, L, F), float("nan"), device="cuda")
    dg = torch.full((d, L, F, n) if fm else (n, d, L, F), float("nan"), device="cuda")
    lp = torch.full((L, F, n) if fm else (n, L, F), float("nan"), device="cuda")
    m.hg.hg_rbf_fwd(desc, n, dev(x), eps, rings, m.linear_view(dev(table)), g, dg, lp)
    torch.cuda.synchronize()
    got = [host(g), host(dg), host(lp)]
    if fm:
        got = [W.from_feature_major(got[0], False), W.from_feature_major(got[1], True),
               W.from_feature_major(got[2], False)]
    ref = oracle.rbf_fwd(d, F, res, case[6], table, x, eps, rings, level_mask=case[10])
    for k, a in zip(("gamma", "dgamma", "lap"), got):
        check_close(k, a, ref[k], ref["m" + k])


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_rbf_backward_parity(case):
    from multiresolution_hash_grid_02_b300 import workloads as W
    m, oracle, desc, res, x, table, rng = _build(case, seed=1)
    n, d, L, F = x.shape[0], desc.d, desc.L, desc.F
    eps, rings = case[11], case[12]
    up = {"g_gamma": rng.standard_normal((n, L, F), dtype=np.float32),
          "g_dgamma": rng.standard_normal((n, d, L, F), dtype=np.float32),
          "g_lap": rng.standard_normal((n, L, F), dtype=np.float32)}
    fm = desc.layout == m.HG_FEATURE_MAJOR
    conv = lambda k, a: dev(W.to_feature_major(a, k == "g_dgamma") if fm else a)
    for use in ("all", "g_gamma", "g_lap"):
        sel = up if use == "all" else {use: up[use]}
        grad = torch.zeros((L, 1 << case[6], F), device="cuda")
        m.hg.hg_rbf_bwd(desc, n, dev(x), eps, rings,
                        *[conv(k, sel[k]) if k in sel else None for k in ("g_gamma", "g_dgamma", "g_lap")],
                        m.linear_view(grad))
        torch.cuda.synchronize()
        want, mag = oracle.rbf_bwd(d, F, res, case[6], x, eps, rings, level_mask=case[10], **sel)
        check_close(f"grad ({use})", host(grad), want, mag)
