"""GPU parity of the full-Hessian entry points (hg_encode_fwd_hessian,
hg_encode_bwd_hessian) against the oracle, element by element.

The cases are the small cases of the Laplacian parity tests, so every kernel
variant is covered: lane-pair and generic forwards, lane-split, privatised
and generic backwards, both output layouts, packed and separate order
tables, fp32 and fp16 coefficients, F = 1..8, masks, coherent points and
the edge coordinates.  Tolerance as there: 1e-5 of the oracle's condition
magnitude.  Beyond the oracle, gamma and grad gamma of the Hessian forward
must be bit-identical to the Laplacian forward's (the same sums in the same
order), and a backward whose Hessian upstream is the Laplacian's on the
diagonal must reproduce the Laplacian backward.
"""
from math import comb

import numpy as np
import pytest

from _harness import check_close, dev, gpu_hermite_fwd, host
from test_parity_gpu import CASES, _build_case

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


def gpu_hessian_fwd(desc, coords, views, want_d=True):
    """hg_encode_fwd_hessian -> point-major numpy (gamma, dgamma, hess)."""
    m, W, _ = _mods()
    n, d, L, F = coords.shape[0], desc.d, desc.L, desc.F
    P = d * (d + 1) // 2
    fm = desc.layout == m.HG_FEATURE_MAJOR
    g = torch.full((L, F, n) if fm else (n, L, F), float("nan"), device="cuda")
    dg = torch.full((d, L, F, n) if fm else (n, d, L, F), float("nan"), device="cuda") if want_d else None
    h = torch.full((P, L, F, n) if fm else (n, P, L, F), float("nan"), device="cuda")
    m.hg.hg_encode_fwd_hessian(desc, n, dev(coords), views, g, dg, h)
    torch.cuda.synchronize()
    g, h = host(g), host(h)
    dg = host(dg) if want_d else None
    if fm:
        g, h = W.from_feature_major(g, False), W.from_feature_major(h, True)
        dg = W.from_feature_major(dg, True) if want_d else None
    return g, dg, h


def gpu_hessian_bwd(desc, coords, gg, gd, gh, grad_tensors, grad_views):
    """hg_encode_bwd_hessian on point-major numpy upstream gradients."""
    m, W, _ = _mods()
    fm = desc.layout == m.HG_FEATURE_MAJOR
    conv = (lambda a, ax: W.to_feature_major(a, ax)) if fm else (lambda a, ax: a)
    up = [None if a is None else dev(conv(a, ax)) for a, ax in ((gg, False), (gd, True), (gh, True))]
    m.hg.hg_encode_bwd_hessian(desc, coords.shape[0], dev(coords), up[0], up[1], up[2], grad_views)
    torch.cuda.synchronize()
    return [host(t) for t in grad_tensors]


def _grad_tables(c):
    m, W, _ = _mods()
    desc = c["desc"]
    d, L, F = desc.d, desc.L, desc.F
    if c["packed"]:
        gt = torch.zeros((L, 1 << c["log2T"][0], 1 << d, F), device="cuda")
        return [gt], m.packed_views(gt, d), lambda got: W.split_orders(got[0], d)
    gts = [torch.zeros((L, 1 << c["log2T"][k], comb(d, k), F), device="cuda") for k in range(d + 1)]
    return gts, m.order_views(gts), lambda got: got


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_hessian_forward_parity(case):
    m, W, oracle = _mods()
    c = _build_case(case)
    desc = c["desc"]
    ref = oracle.encode_fwd_hessian(desc.d, desc.F, c["res"], c["log2T"], c["orders"], c["coords"],
                                    level_mask=c["mask"])
    g, dg, h = gpu_hessian_fwd(desc, c["coords"], c["views"])
    check_close("gamma", g, ref["gamma"], ref["mgamma"])
    check_close("dgamma", dg, ref["dgamma"], ref["mdgamma"])
    check_close("hess", h, ref["hess"], ref["mhess"])
    # gamma and grad gamma are the Laplacian forward's, bit for bit
    g0, dg0, _ = gpu_hermite_fwd(desc, c["coords"], c["views"])
    assert np.array_equal(g, g0, equal_nan=True)
    assert np.array_equal(dg, dg0, equal_nan=True)
    # without grad gamma requested the other outputs are unchanged
    g2, _, h2 = gpu_hessian_fwd(desc, c["coords"], c["views"], want_d=False)
    assert np.array_equal(g2, g, equal_nan=True) and np.array_equal(h2, h, equal_nan=True)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_hessian_backward_parity(case):
    m, W, oracle = _mods()
    c = _build_case(case, seed=1)
    desc = c["desc"]
    d, L, F = desc.d, desc.L, desc.F
    n = c["coords"].shape[0]
    rng = np.random.default_rng(n + 17 * d + F)
    gh = rng.standard_normal((n, d * (d + 1) // 2, L, F), dtype=np.float32)
    tensors, views, to_orders = _grad_tables(c)
    got = to_orders(gpu_hessian_bwd(desc, c["coords"], c["gg"], c["gd"], gh, tensors, views))
    grads, mags = oracle.encode_bwd_hessian(d, F, c["res"], c["log2T"], c["coords"], c["gg"], c["gd"], gh,
                                            level_mask=c["mask"])
    for k in range(d + 1):
        check_close(f"grad order {k}", got[k], grads[k], mags[k])


@pytest.mark.parametrize("which", ["3d_F2", "2d_F1_coarse_many_points", "3d_F1_f16_stratified"])
def test_hessian_backward_partial_upstream(which):
    """Upstream gradients for one output only (the others NULL)."""
    m, W, oracle = _mods()
    case = next(cs for cs in CASES if cs[0] == which)
    c = _build_case(case, seed=2)
    desc = c["desc"]
    d, L, F = desc.d, desc.L, desc.F
    n = c["coords"].shape[0]
    gh_full = np.random.default_rng(5).standard_normal((n, d * (d + 1) // 2, L, F), dtype=np.float32)
    for use in ("gamma", "dgamma", "hess"):
        gg = c["gg"] if use == "gamma" else None
        gd = c["gd"] if use == "dgamma" else None
        gh = gh_full if use == "hess" else None
        tensors, views, to_orders = _grad_tables(c)
        got = to_orders(gpu_hessian_bwd(desc, c["coords"], gg, gd, gh, tensors, views))
        grads, mags = oracle.encode_bwd_hessian(d, F, c["res"], c["log2T"], c["coords"], gg, gd, gh,
                                                level_mask=c["mask"])
        for k in range(d + 1):
            check_close(f"{use}: grad order {k}", got[k], grads[k], mags[k])


@pytest.mark.parametrize("which", ["cfg1_feature_major", "3d_F2", "3d_F1_f16", "3d_F2_f16_coarse_many_points"])
def test_hessian_backward_with_diagonal_upstream_is_laplacian_backward(which):
    """g_hess = g_lap on every diagonal entry and 0 off it: the Laplacian
    backward's result (the Laplacian is the Hessian's trace)."""
    m, W, oracle = _mods()
    case = next(cs for cs in CASES if cs[0] == which)
    c = _build_case(case, seed=3)
    desc = c["desc"]
    d, L, F = desc.d, desc.L, desc.F
    n = c["coords"].shape[0]
    pairs = oracle.hess_pairs(d)
    gh = np.zeros((n, len(pairs), L, F), np.float32)
    for q, (i, j) in enumerate(pairs):
        if i == j:
            gh[:, q] = c["gl"]
    tensors, views, to_orders = _grad_tables(c)
    got = to_orders(gpu_hessian_bwd(desc, c["coords"], c["gg"], c["gd"], gh, tensors, views))
    grads, mags = oracle.encode_bwd(d, F, c["res"], c["log2T"], c["coords"], c["gg"], c["gd"], c["gl"],
                                    level_mask=c["mask"])
    for k in range(d + 1):
        check_close(f"grad order {k}", got[k], grads[k], mags[k])


def test_hessian_inactive_levels_are_zero():
    m, W, oracle = _mods()
    case = next(cs for cs in CASES if cs[0] == "3d_mask_1010")
    c = _build_case(case)
    g, dg, h = gpu_hessian_fwd(c["desc"], c["coords"], c["views"])
    for l in (0, 2):
        assert not np.any(g[:, l]) and not np.any(dg[:, :, l]) and not np.any(h[:, :, l])
