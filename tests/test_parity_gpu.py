"""GPU parity: the CUDA library (called through its C ABI) against the oracle,
element by element, on seeded inputs.

Indices are compared bit for bit; floats within 1e-5 of the oracle's
condition magnitude (see tests/_harness.py).  Small cases span several
256-thread tiles plus a ragged tail, both output layouts, packed and
separate order tables, fp32 and fp16 coefficients, F = 1, 2, 4, 8, mixed
per-order table sizes, active-level masks and the edge coordinates (0, 1,
cell faces, out of range, NaN, infinities).
"""
import zlib
from math import comb

import numpy as np
import pytest

from _harness import RTOL, check_close, dev, gpu_hermite_bwd, gpu_hermite_fwd, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _mods():
    import multiresolution_hash_grid_02_b300 as m
    from multiresolution_hash_grid_02_b300 import workloads as W
    import oracle
    return m, W, oracle


EDGE = [0.0, 1.0, 0.5, 0.25, 1.0 - 2 ** -24, 2 ** -24, -0.5, 1.5, float("nan"), float("inf"), float("-inf"), -0.0]


def _coords(rng, n, d, res, stratified=False):
    if stratified:
        # one point per stratum, strata in row-major order: consecutive points
        # are neighbours (coherent scatter, as the PINN collocation workload)
        side = round(n ** (1.0 / d))
        assert side ** d == n
        cells = np.stack([(np.arange(n) // side ** i) % side for i in range(d)], axis=1)
        return ((cells + rng.random((n, d))) / side).astype(np.float32)
    x = rng.random((n, d), dtype=np.float32)
    m = min(n, 64)
    if n >= 8:
        # edge values and exact cell faces of a few levels
        for i in range(m // 2):
            x[i] = [EDGE[(i * (j + 3)) % len(EDGE)] for j in range(d)]
        for i in range(m // 2, m):
            N = res[i % len(res)]
            x[i] = (rng.integers(0, N + 1, size=d) / N).astype(np.float32)
    return x


# (id, d, L, F, n_min, n_max, log2T per order, dtype, layout, packed, n, level_mask)
CASES = [
    ("cfg1_feature_major", 2, 4, 2, 4, 32, (12, 12, 12), "f32", 1, True, 4096, None),
    ("cfg1_point_major", 2, 4, 2, 4, 32, (12, 12, 12), "f32", 0, True, 4096, None),
    ("cfg1_f16", 2, 4, 2, 4, 32, (12, 12, 12), "f16", 1, True, 4096, None),
    ("2d_F1_hashed", 2, 6, 1, 8, 300, (10, 10, 10), "f32", 1, True, 3001, None),
    ("2d_orders_11_11_7", 2, 6, 2, 8, 300, (11, 11, 7), "f32", 1, False, 2500, None),
    ("2d_F4_point_major", 2, 5, 4, 4, 100, (9, 9, 9), "f32", 0, True, 1000, None),
    ("2d_F8_f16", 2, 3, 8, 4, 50, (8, 8, 8), "f16", 1, True, 700, None),
    ("3d_F2", 3, 6, 2, 4, 64, (12, 12, 12, 12), "f32", 1, True, 3000, None),
    ("3d_F2_point_major", 3, 6, 2, 4, 64, (12, 12, 12, 12), "f32", 0, True, 777, None),
    ("3d_F1_f16", 3, 5, 1, 4, 40, (10, 10, 10, 10), "f16", 1, True, 2049, None),
    ("3d_F2_f16", 3, 5, 2, 4, 40, (10, 10, 10, 10), "f16", 1, True, 1025, None),
    ("3d_orders_11_10_9_8", 3, 5, 2, 4, 40, (11, 10, 9, 8), "f32", 1, False, 1500, None),
    ("3d_F4_separate", 3, 4, 4, 4, 30, (9, 9, 9, 9), "f32", 0, False, 500, None),
    ("3d_F8_f16", 3, 3, 8, 4, 20, (9, 9, 9, 9), "f16", 1, True, 300, None),
    ("3d_mask_1010", 3, 4, 2, 4, 60, (10, 10, 10, 10), "f32", 1, True, 600, 0b1010),
    ("3d_one_point", 3, 4, 2, 4, 60, (10, 10, 10, 10), "f32", 1, True, 1, None),
    ("2d_32_levels_max_res", 2, 32, 2, 2, 1 << 22, (12, 12, 12), "f32", 1, True, 1500, None),
    # many points per vertex on small one-to-one levels: the backward takes the
    # shared-memory (privatised) path for these levels
    ("2d_F1_coarse_many_points", 2, 3, 1, 4, 16, (10, 10, 10), "f32", 1, True, 20000, None),
    ("2d_F2_coarse_many_points", 2, 3, 2, 4, 16, (10, 10, 10), "f32", 0, True, 20000, None),
    ("3d_F1_coarse_many_points", 3, 3, 1, 2, 8, (10, 10, 10, 10), "f32", 0, True, 20000, None),
    ("3d_F2_f16_coarse_many_points", 3, 3, 2, 2, 6, (9, 9, 9, 9), "f16", 1, True, 30000, 0b011),
    # stratified (coherent) points: runs of points in one cell are summed in
    # the warp before the scatter
    ("2d_F2_stratified", 2, 5, 2, 4, 160, (11, 11, 11), "f32", 1, True, 16384, None),
    ("2d_F1_stratified", 2, 4, 1, 4, 64, (10, 10, 10), "f32", 0, True, 10000, None),
    ("3d_F2_stratified", 3, 4, 2, 2, 40, (12, 12, 12, 12), "f32", 1, True, 13824, None),
    ("3d_F1_f16_stratified", 3, 3, 1, 2, 20, (10, 10, 10, 10), "f16", 1, True, 8000, None),
    # 4D (space-time): 16 corners x 16 multi-indices, five order tables
    ("4d_F2", 4, 3, 2, 2, 8, (12, 12, 12, 12, 12), "f32", 1, True, 1500, None),
    ("4d_F2_point_major_hashed", 4, 3, 2, 4, 30, (10, 10, 10, 10, 10), "f32", 0, True, 900, None),
    ("4d_F1_f16", 4, 3, 1, 2, 10, (10, 10, 10, 10, 10), "f16", 1, True, 700, None),
    ("4d_F2_f16", 4, 2, 2, 3, 12, (11, 11, 11, 11, 11), "f16", 1, True, 600, None),
    ("4d_orders_12_11_10_9_8", 4, 3, 2, 2, 9, (12, 11, 10, 9, 8), "f32", 1, False, 500, None),
    ("4d_F4_mask_101", 4, 3, 4, 2, 12, (9, 9, 9, 9, 9), "f32", 0, True, 300, 0b101),
    ("4d_one_point", 4, 2, 2, 2, 5, (10, 10, 10, 10, 10), "f32", 1, True, 1, None),
    ("4d_F2_stratified", 4, 2, 2, 2, 6, (12, 12, 12, 12, 12), "f32", 1, True, 4096, None),
]


def _build_case(case, seed=0):
    m, W, oracle = _mods()
    cid, d, L, F, nmin, nmax, log2T, dt, layout, packed, n, mask = case
    rng = np.random.default_rng(zlib.crc32(cid.encode()) + seed)
    res = oracle.level_resolutions(L, nmin, nmax)
    coords = _coords(rng, n, d, res, stratified="stratified" in cid)
    npdt = np.float16 if dt == "f16" else np.float32
    if packed:
        assert len(set(log2T)) == 1
        table = (rng.random((L, 1 << log2T[0], 1 << d, F), dtype=np.float32) * 2 - 1).astype(npdt)
        orders = W.split_orders(table, d)
        t_dev = dev(table)
        views = m.packed_views(t_dev, d)
        keep = [t_dev]
    else:
        orders = [(rng.random((L, 1 << log2T[k], comb(d, k), F), dtype=np.float32) * 2 - 1).astype(npdt)
                  for k in range(d + 1)]
        keep = [dev(o) for o in orders]
        views = m.order_views(keep)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=nmin, n_max=nmax, log2_T=log2T, level_mask=mask,
                      dtype=m.HG_F16 if dt == "f16" else m.HG_F32, layout=layout)
    gg = rng.standard_normal((n, L, F), dtype=np.float32)
    gd = rng.standard_normal((n, d, L, F), dtype=np.float32)
    gl = rng.standard_normal((n, L, F), dtype=np.float32)
    return dict(desc=desc, res=res, coords=coords, orders=orders, views=views, keep=keep, packed=packed,
                gg=gg, gd=gd, gl=gl, log2T=log2T, mask=mask)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_hermite_forward_parity(case):
    m, W, oracle = _mods()
    c = _build_case(case)
    desc = c["desc"]
    ref = oracle.encode_fwd(desc.d, desc.F, c["res"], c["log2T"], c["orders"], c["coords"], level_mask=c["mask"])
    g, dg, lp = gpu_hermite_fwd(desc, c["coords"], c["views"])
    check_close("gamma", g, ref["gamma"], ref["mgamma"])
    check_close("dgamma", dg, ref["dgamma"], ref["mdgamma"])
    check_close("lap", lp, ref["lap"], ref["mlap"])
    # gamma alone (derivative outputs not requested) is the same gamma
    g2, _, _ = gpu_hermite_fwd(desc, c["coords"], c["views"], want_d=False, want_l=False)
    assert np.array_equal(g2, g, equal_nan=True)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_hermite_backward_parity(case):
    m, W, oracle = _mods()
    c = _build_case(case, seed=1)
    desc = c["desc"]
    d, L, F = desc.d, desc.L, desc.F
    n = c["coords"].shape[0]
    if c["packed"]:
        gt = torch.zeros((L, 1 << c["log2T"][0], 1 << d, F), device="cuda")
        got = gpu_hermite_bwd(desc, c["coords"], c["gg"], c["gd"], c["gl"], [gt], m.packed_views(gt, d))[0]
        got = W.split_orders(got, d)
    else:
        gts = [torch.zeros((L, 1 << c["log2T"][k], comb(d, k), F), device="cuda") for k in range(d + 1)]
        got = gpu_hermite_bwd(desc, c["coords"], c["gg"], c["gd"], c["gl"], gts, m.order_views(gts))
    grads, mags = oracle.encode_bwd(d, F, c["res"], c["log2T"], c["coords"], c["gg"], c["gd"], c["gl"],
                                    level_mask=c["mask"])
    for k in range(d + 1):
        check_close(f"grad order {k}", got[k], grads[k], mags[k])
    assert n >= 1


def test_hermite_backward_partial_upstream():
    """Upstream gradients given for gamma only / for the Laplacian only."""
    m, W, oracle = _mods()
    c = _build_case(CASES[7], seed=2)
    desc = c["desc"]
    d, L, F = desc.d, desc.L, desc.F
    for use in ("gamma", "lap", "dgamma"):
        gg = c["gg"] if use == "gamma" else None
        gd = c["gd"] if use == "dgamma" else None
        gl = c["gl"] if use == "lap" else None
        gt = torch.zeros((L, 1 << c["log2T"][0], 1 << d, F), device="cuda")
        got = W.split_orders(gpu_hermite_bwd(desc, c["coords"], gg, gd, gl, [gt], m.packed_views(gt, d))[0], d)
        grads, mags = oracle.encode_bwd(d, F, c["res"], c["log2T"], c["coords"], gg, gd, gl)
        for k in range(d + 1):
            check_close(f"{use}: grad order {k}", got[k], grads[k], mags[k])


def test_backward_accumulates():
    """The backward adds into the gradient tables (+=), it does not overwrite."""
    m, W, oracle = _mods()
    c = _build_case(CASES[0], seed=3)
    desc = c["desc"]
    d, L, F = desc.d, desc.L, desc.F
    gt = torch.zeros((L, 1 << 12, 1 << d, F), device="cuda")
    once = gpu_hermite_bwd(desc, c["coords"], c["gg"], c["gd"], c["gl"], [gt], m.packed_views(gt, d))[0].copy()
    twice = gpu_hermite_bwd(desc, c["coords"], c["gg"], c["gd"], c["gl"], [gt], m.packed_views(gt, d))[0]
    assert np.allclose(twice, 2 * once, rtol=1e-6, atol=1e-6 * np.abs(once).max())


LIN_CASES = [
    ("cfg2_shape_small", 2, 16, 2, 16, 2048, 12, "f32", 1, 5000, None),
    ("2d_point_major", 2, 8, 2, 4, 500, 10, "f32", 0, 3333, None),
    ("2d_F1_f16", 2, 6, 1, 4, 200, 9, "f16", 1, 1000, None),
    ("3d_F2", 3, 8, 2, 4, 128, 12, "f32", 1, 2500, None),
    ("3d_F4_f16_mask", 3, 5, 4, 4, 64, 10, "f16", 0, 700, 0b10110),
    ("3d_F8", 3, 3, 8, 2, 16, 8, "f32", 1, 257, None),
    ("2d_F1_coarse_many_points", 2, 3, 1, 4, 16, 10, "f32", 1, 30000, None),
    ("3d_F4_f16_coarse_many_points", 3, 3, 4, 2, 8, 9, "f16", 0, 30000, 0b101),
    ("2d_F2_stratified", 2, 6, 2, 4, 300, 12, "f32", 1, 16384, None),
    ("4d_F2", 4, 4, 2, 2, 16, 12, "f32", 1, 2000, None),
    ("4d_F1_f16_point_major", 4, 3, 1, 2, 9, 10, "f16", 0, 700, None),
    ("4d_F2_coarse_many_points", 4, 2, 2, 2, 3, 12, "f32", 1, 20000, None),
]


@pytest.mark.parametrize("case", LIN_CASES, ids=[c[0] for c in LIN_CASES])
def test_linear_parity(case):
    m, W, oracle = _mods()
    from multiresolution_hash_grid_02_b300 import hg
    cid, d, L, F, nmin, nmax, log2T, dt, layout, n, mask = case
    rng = np.random.default_rng(zlib.crc32(cid.encode()))
    res = oracle.level_resolutions(L, nmin, nmax)
    coords = _coords(rng, n, d, res, stratified="stratified" in cid)
    npdt = np.float16 if dt == "f16" else np.float32
    table = (rng.random((L, 1 << log2T, F), dtype=np.float32) * 2 - 1).astype(npdt)
    gg = rng.standard_normal((n, L, F), dtype=np.float32)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=nmin, n_max=nmax, log2_T=(log2T,), level_mask=mask,
                      dtype=m.HG_F16 if dt == "f16" else m.HG_F32, layout=layout)
    t_dev = dev(table)
    fm = layout == m.HG_FEATURE_MAJOR
    out = torch.full((L, F, n) if fm else (n, L, F), float("nan"), device="cuda")
    hg.hg_linear_fwd(desc, n, dev(coords), m.linear_view(t_dev), out)
    torch.cuda.synchronize()
    got = host(out)
    if fm:
        got = W.from_feature_major(got, False)
    want, mag = oracle.linear_fwd(d, F, res, log2T, table, coords, level_mask=mask)
    check_close("linear gamma", got, want, mag)
    grad = torch.zeros((L, 1 << log2T, F), device="cuda")
    hg.hg_linear_bwd(desc, n, dev(coords), dev(W.to_feature_major(gg, False) if fm else gg), m.linear_view(grad))
    torch.cuda.synchronize()
    gw, gm = oracle.linear_bwd(d, F, res, log2T, coords, gg, level_mask=mask)
    check_close("linear grad", host(grad), gw, gm)


INDEX_GEOMS = [
    ("cfg1", 2, 4, 4, 32, (12, 12, 12)),
    ("cfg2", 2, 16, 16, 2048, (19, 19, 19)),
    ("cfg3", 2, 16, 16, 1024, (19, 19, 19)),
    ("cfg4", 3, 16, 16, 512, (19, 19, 19, 19)),
    ("cfg5", 3, 16, 16, 2048, (22, 22, 22, 22)),
    ("2d_orders_14_14_10", 2, 16, 16, 1024, (14, 14, 10)),
    ("3d_orders_14_10_14_12", 3, 12, 4, 300, (14, 10, 14, 12)),
    ("2d_max_res", 2, 32, 2, 1 << 22, (30, 30, 30)),
    ("4d_dense_and_hashed", 4, 8, 2, 200, (16, 15, 14, 13, 12)),
    ("4d_max_res", 4, 16, 2, 1 << 22, (20, 20, 20, 20, 20)),
]


@pytest.mark.parametrize("geom", INDEX_GEOMS, ids=[g[0] for g in INDEX_GEOMS])
def test_vertex_indices_bit_exact(geom):
    m, W, oracle = _mods()
    from multiresolution_hash_grid_02_b300 import hg
    gid, d, L, nmin, nmax, log2T = geom
    rng = np.random.default_rng(zlib.crc32(gid.encode()))
    res = oracle.level_resolutions(L, nmin, nmax)
    coords = _coords(rng, 5000, d, res)
    desc = m.GridDesc(d=d, L=L, F=2, n_min=nmin, n_max=nmax, log2_T=log2T)
    out = torch.zeros((coords.shape[0], L, d + 1, 1 << d), dtype=torch.int32, device="cuda")
    hg.hg_hash_indices(desc, coords.shape[0], dev(coords), out)
    torch.cuda.synchronize()
    got = host(out).view(np.uint32)
    want = oracle.hash_indices(d, res, log2T, coords)
    assert np.array_equal(got, want)
    assert hg.hg_level_resolutions(desc) == res


def test_zero_points_is_a_no_op():
    m, W, oracle = _mods()
    from multiresolution_hash_grid_02_b300 import hg
    desc = m.GridDesc(d=3, L=4, F=2, n_min=4, n_max=32, log2_T=(8, 8, 8, 8))
    t = torch.zeros((4, 256, 8, 2), device="cuda")
    lin = torch.zeros((4, 256, 2), device="cuda")
    hg.hg_encode_fwd(desc, 0, None, m.packed_views(t, 3), None)
    hg.hg_encode_bwd(desc, 0, None, None, None, None, m.packed_views(t, 3))
    hg.hg_linear_fwd(desc, 0, None, m.linear_view(lin), None)
    hg.hg_linear_bwd(desc, 0, None, None, m.linear_view(lin))
    torch.cuda.synchronize()
    assert float(t.abs().sum()) == 0.0 and float(lin.abs().sum()) == 0.0


@pytest.mark.parametrize("mask", [None, 0b1011], ids=["all_levels", "mask_1011"])
def test_fp16_pipelined_forward_steady_state(mask):
    """The fp16 3D F = 2 packed forward is a persistent kernel: a CTA of 128
    threads walks 64-point batches, copying batch b + gridDim.x into the
    other shared-memory stage while it blends batch b.  Its grid holds at
    most (SMs x CTAs per SM) CTAs, and CTAs per SM are at most the SM's
    thread limit / 128.  With 2^19 points every CTA walks at least three
    batches, so the prefetch and the stage toggle run; every output
    (Laplacian and full-Hessian forwards) is compared with the oracle."""
    m, W, oracle = _mods()
    from multiresolution_hash_grid_02_b300 import hg
    from test_hessian_gpu import gpu_hessian_fwd
    n, d, L, F, nmin, nmax, log2T = 1 << 19, 3, 4, 2, 4, 64, 12
    props = torch.cuda.get_device_properties(0)
    max_ctas = props.multi_processor_count * (props.max_threads_per_multi_processor // 128)
    assert (n + 63) // 64 >= 3 * max_ctas
    rng = np.random.default_rng(1902)
    res = oracle.level_resolutions(L, nmin, nmax)
    coords = _coords(rng, n, d, res)
    table = (rng.random((L, 1 << log2T, 1 << d, F), dtype=np.float32) * 2 - 1).astype(np.float16)
    orders = W.split_orders(table, d)
    t_dev = dev(table)
    views = m.packed_views(t_dev, d)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=nmin, n_max=nmax, log2_T=(log2T,) * 4, level_mask=mask,
                      dtype=m.HG_F16, layout=m.HG_FEATURE_MAJOR)
    ref = oracle.encode_fwd(d, F, res, (log2T,) * 4, orders, coords, level_mask=mask)
    g, dg, lp = gpu_hermite_fwd(desc, coords, views)
    check_close("gamma", g, ref["gamma"], ref["mgamma"])
    check_close("dgamma", dg, ref["dgamma"], ref["mdgamma"])
    check_close("lap", lp, ref["lap"], ref["mlap"])
    ref = oracle.encode_fwd_hessian(d, F, res, (log2T,) * 4, orders, coords, level_mask=mask)
    g, dg, h = gpu_hessian_fwd(desc, coords, views)
    check_close("hessian gamma", g, ref["gamma"], ref["mgamma"])
    check_close("hessian dgamma", dg, ref["dgamma"], ref["mdgamma"])
    check_close("hess", h, ref["hess"], ref["mhess"])
