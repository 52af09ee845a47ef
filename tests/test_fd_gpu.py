"""GPU parity of the INGP-FD entry points (hg_linear_fd_fwd / hg_linear_fd_bwd:
the d-linear encoding with central finite differences, the Hermite-NGP
page's baseline) against the oracle, element by element.

Cases span several tiles and a ragged tail, both layouts, fp32 and fp16
tables, F = 1, 2, 4, d = 2, 3, 4, masks, steps that stay inside cells and
steps that cross one or several cells, the edge coordinates (0, 1, cell
faces, out of range, NaN, infinities: the shifted coordinate is clamped),
and coarse one-to-one levels with many points per vertex (the privatised
backward).  Tolerance 1e-5 of the oracle's condition magnitude, which for
the differences carries the 1/eps and 1/eps^2 factors of their terms."""
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


# (id, d, L, F, n_min, n_max, log2T, dtype, layout, n, mask, eps)
CASES = [
    ("3d_F2_eps_half_finest_cell", 3, 6, 2, 4, 128, 12, "f32", 1, 3000, None, 2.0 ** -8),
    ("3d_F2_point_major", 3, 5, 2, 4, 64, 11, "f32", 0, 1001, None, 1e-3),
    ("2d_F2_f16", 2, 6, 2, 4, 300, 10, "f16", 1, 2500, None, 2.0 ** -10),
    ("2d_F1_large_eps_multi_cell", 2, 4, 1, 8, 200, 12, "f32", 1, 1500, None, 0.05),
    ("3d_F4_mask", 3, 4, 4, 4, 60, 10, "f32", 0, 700, 0b1010, 2.0 ** -9),
    ("4d_F2", 4, 3, 2, 2, 12, 12, "f32", 1, 900, None, 2.0 ** -7),
    ("3d_F2_coarse_many_points", 3, 3, 2, 2, 8, 12, "f32", 1, 30000, None, 2.0 ** -6),
    ("2d_F1_f16_coarse_many_points", 2, 3, 1, 4, 16, 10, "f16", 0, 20000, None, 2.0 ** -8),
    ("3d_one_point", 3, 4, 2, 4, 60, 10, "f32", 1, 1, None, 1e-3),
]


def _build(case, seed=0):
    import multiresolution_hash_grid_02_b300 as m
    import oracle
    cid, d, L, F, nmin, nmax, log2T, dt, layout, n, mask, eps = case
    rng = np.random.default_rng(zlib.crc32(cid.encode()) + seed)
    res = oracle.level_resolutions(L, nmin, nmax)
    x = _coords(rng, n, d, res)
    npdt = np.float16 if dt == "f16" else np.float32
    table = (rng.random((L, 1 << log2T, F), dtype=np.float32) * 2 - 1).astype(npdt)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=nmin, n_max=nmax, log2_T=(log2T,), level_mask=mask,
                      dtype=m.HG_F16 if dt == "f16" else m.HG_F32, layout=layout)
    return m, oracle, desc, res, x, table, eps, rng


def _fwd(m, desc, x, table, eps, want=("dgamma", "lap", "stencil")):
    from multiresolution_hash_grid_02_b300 import workloads as W
    n, d, L, F = x.shape[0], desc.d, desc.L, desc.F
    fm = desc.layout == m.HG_FEATURE_MAJOR
    shp = lambda k: ((k, L, F, n) if fm else (n, k, L, F)) if k else ((L, F, n) if fm else (n, L, F))
    out = {"gamma": torch.full(shp(0), float("nan"), device="cuda")}
    if "dgamma" in want:
        out["dgamma"] = torch.full(shp(d), float("nan"), device="cuda")
    if "lap" in want:
        out["lap"] = torch.full(shp(0), float("nan"), device="cuda")
    if "stencil" in want:
        out["stencil"] = torch.full(shp(2 * d), float("nan"), device="cuda")
    t = dev(table)
    m.hg.hg_linear_fd_fwd(desc, n, dev(x), eps, m.linear_view(t), out["gamma"], out.get("dgamma"), out.get("lap"),
                          out.get("stencil"))
    torch.cuda.synchronize()
    res = {}
    for k, v in out.items():
        a = host(v)
        res[k] = W.from_feature_major(a, k in ("dgamma", "stencil")) if fm else a
    return res


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fd_forward_parity(case):
    m, oracle, desc, res, x, table, eps, rng = _build(case)
    ref = oracle.linear_fd_fwd(desc.d, desc.F, res, case[6], table, x, eps, level_mask=case[10])
    got = _fwd(m, desc, x, table, eps)
    for k in ("gamma", "dgamma", "lap", "stencil"):
        check_close(k, got[k], ref[k], ref["m" + k])
    # outputs not requested leave the others unchanged
    g2 = _fwd(m, desc, x, table, eps, want=())
    assert np.array_equal(g2["gamma"], got["gamma"], equal_nan=True)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fd_backward_parity(case):
    from multiresolution_hash_grid_02_b300 import workloads as W
    m, oracle, desc, res, x, table, eps, rng = _build(case, seed=1)
    n, d, L, F = x.shape[0], desc.d, desc.L, desc.F
    up = {"g_gamma": rng.standard_normal((n, L, F), dtype=np.float32),
          "g_dgamma": rng.standard_normal((n, d, L, F), dtype=np.float32),
          "g_lap": rng.standard_normal((n, L, F), dtype=np.float32),
          "g_stencil": rng.standard_normal((n, 2 * d, L, F), dtype=np.float32)}
    fm = desc.layout == m.HG_FEATURE_MAJOR
    conv = lambda k, a: dev(W.to_feature_major(a, k in ("g_dgamma", "g_stencil")) if fm else a)
    for use in ("all", "g_gamma", "g_lap", "g_stencil"):
        sel = up if use == "all" else {use: up[use]}
        grad = torch.zeros((L, 1 << case[6], F), device="cuda")
        m.hg.hg_linear_fd_bwd(desc, n, dev(x), eps, *[conv(k, sel[k]) if k in sel else None
                                                      for k in ("g_gamma", "g_dgamma", "g_lap", "g_stencil")],
                              m.linear_view(grad))
        torch.cuda.synchronize()
        want, mag = oracle.linear_fd_bwd(d, F, res, case[6], x, eps, level_mask=case[10], **sel)
        check_close(f"grad ({use})", host(grad), want, mag)


def test_fd_with_stencil_inside_cells_matches_the_linear_encoding():
    """gamma(x) of the FD forward is the d-linear encoding itself."""
    m, oracle, desc, res, x, table, eps, rng = _build(CASES[0])
    got = _fwd(m, desc, x, table, eps, want=())
    lin = torch.full((desc.L, desc.F, x.shape[0]), float("nan"), device="cuda")
    m.hg.hg_linear_fwd(desc, x.shape[0], dev(x), m.linear_view(dev(table)), lin)
    torch.cuda.synchronize()
    from multiresolution_hash_grid_02_b300 import workloads as W
    assert np.array_equal(W.from_feature_major(host(lin), False), got["gamma"], equal_nan=True)
