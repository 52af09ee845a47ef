"""Pins for the oracle's full-Hessian output (the widening of the Laplacian
of "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
关键设计 2, to every second derivative d2 gamma / dx_i dx_j): hand-derived
single-coefficient values, exact reproduction of a tensor cubic's Hessian,
finite differences of the gradient, trace = Laplacian, and the adjoint
identity / brute-force Jacobian of the backward."""
import json
import os
from math import comb

import numpy as np
import pytest

from test_oracle_pins import _fill_from_polys, _poly_eval, _vertex_index_map

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hessian_single_coefficient_closed_forms(oracle_mod):
    with open(os.path.join(GOLDEN, "single_coefficient.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        d, N = case["d"], case["N"]
        log2T = [12] * (d + 1)
        tabs = [np.zeros((1, 1 << 12, comb(d, k), 1)) for k in range(d + 1)]
        alpha = sum(a << i for i, a in enumerate(case["alpha"]))
        k = sum(case["alpha"])
        vert = tuple(c + v for c, v in zip(case["cell"], case["corner"]))
        vmap = _vertex_index_map(oracle_mod, d, [N], log2T)
        tabs[k][0, vmap[(0, k, vert)], oracle_mod.slot_in_bucket(d, alpha), 0] = 1.0
        x = np.array([[(c + t) / N for c, t in zip(case["cell"], case["t"])]], np.float32)
        out = oracle_mod.encode_fwd_hessian(d, 1, [N], log2T, tabs, x)
        assert np.allclose(out["hess"][0, :, 0, 0], case["hess"], rtol=0, atol=1e-13)
        assert abs(out["gamma"][0, 0, 0] - case["gamma"]) < 1e-15


@pytest.mark.parametrize("d,res,log2T", [(2, [4, 8, 20], [12, 12, 12]), (3, [4, 6, 10], [11, 11, 11, 11]),
                                          (4, [2, 3], [9, 9, 9, 9, 9])])
def test_exact_tensor_cubic_hessian(oracle_mod, d, res, log2T):
    rng = np.random.default_rng(21)
    F = 2
    polys = [[rng.uniform(-1, 1, size=(4,) * d) for _ in range(F)] for _ in res]
    tabs = _fill_from_polys(oracle_mod, d, F, res, log2T, polys, 3)
    xs = (rng.integers(0, 1 << 16, size=(48, d)) / float(1 << 16)).astype(np.float32)
    out = oracle_mod.encode_fwd_hessian(d, F, res, log2T, tabs, xs)
    lap = oracle_mod.encode_fwd(d, F, res, log2T, tabs, xs)["lap"]
    pairs = oracle_mod.hess_pairs(d)
    for n in range(len(xs)):
        x = xs[n].astype(np.float64)
        for l in range(len(res)):
            for f in range(F):
                for q, (i, j) in enumerate(pairs):
                    der = [0] * d
                    der[i] += 1
                    der[j] += 1
                    want = _poly_eval(polys[l][f], x, der)
                    assert abs(out["hess"][n, q, l, f] - want) < 1e-9 * max(1, res[l] ** 2)
    # the trace is the Laplacian
    tr = sum(out["hess"][:, q] for q, (i, j) in enumerate(pairs) if i == j)
    assert np.allclose(tr, lap, rtol=1e-12, atol=1e-12 * max(res) ** 2)


@pytest.mark.parametrize("d", [2, 3, 4])
def test_hessian_by_finite_differences_of_the_gradient(oracle_mod, d):
    rng = np.random.default_rng(22)
    F, N, log2T = 2, 29, [7] * (d + 1)
    tabs = [rng.uniform(-1, 1, size=(1 << log2T[k], comb(d, k), F)) for k in range(d + 1)]
    pairs = oracle_mod.hess_pairs(d)
    for _ in range(8):
        c = rng.integers(0, N, size=d)
        t = rng.uniform(0.2, 0.8, size=d)
        _, _, hess = oracle_mod.eval_cell_hessian(d, F, N, log2T, tabs, c, t)
        h = 1e-4
        for q, (i, j) in enumerate(pairs):
            tp, tm = t.copy(), t.copy()
            tp[j] += h
            tm[j] -= h
            dgp = oracle_mod.eval_cell_hessian(d, F, N, log2T, tabs, c, tp)[1]
            dgm = oracle_mod.eval_cell_hessian(d, F, N, log2T, tabs, c, tm)[1]
            fd = (dgp[i] - dgm[i]) / (2 * h) * N          # d/dx_j of d gamma/dx_i
            assert np.allclose(fd, hess[q], rtol=1e-6, atol=1e-6 * N * N)


@pytest.mark.parametrize("d,res,log2T", [(2, [4, 9, 30], [4, 5, 4]), (3, [3, 7, 11], [5, 6, 5, 4]),
                                          (4, [2, 5, 9], [6, 5, 7, 6, 4])])
def test_hessian_backward_adjoint_identity(oracle_mod, d, res, log2T):
    rng = np.random.default_rng(23)
    F, n = 2, 200
    L = len(res)
    P = oracle_mod.hess_entries(d)
    tabs = [rng.uniform(-1, 1, size=(L, 1 << log2T[k], comb(d, k), F)) for k in range(d + 1)]
    xs = rng.random((n, d), dtype=np.float32)
    gg = rng.standard_normal((n, L, F), dtype=np.float32)
    gd = rng.standard_normal((n, d, L, F), dtype=np.float32)
    gh = rng.standard_normal((n, P, L, F), dtype=np.float32)
    out = oracle_mod.encode_fwd_hessian(d, F, res, log2T, tabs, xs)
    grads, mags = oracle_mod.encode_bwd_hessian(d, F, res, log2T, xs, gg, gd, gh)
    lhs = sum(float((g * t).sum()) for g, t in zip(grads, tabs))
    rhs = float((gg * out["gamma"]).sum() + (gd * out["dgamma"]).sum() + (gh * out["hess"]).sum())
    scale = sum(float((m * np.abs(t)).sum()) for m, t in zip(mags, tabs))
    assert abs(lhs - rhs) <= 1e-12 * scale


def test_hessian_backward_equals_bruteforce_jacobian(oracle_mod):
    rng = np.random.default_rng(24)
    d, F, res, log2T = 2, 1, [3, 6], [4, 4, 3]
    L, P = len(res), oracle_mod.hess_entries(2)
    shapes = [(L, 1 << log2T[k], comb(d, k), F) for k in range(d + 1)]
    xs = rng.random((20, d), dtype=np.float32)
    gh = rng.standard_normal((20, P, L, F), dtype=np.float32)
    grads, _ = oracle_mod.encode_bwd_hessian(d, F, res, log2T, xs, None, None, gh)
    for k, shp in enumerate(shapes):
        for e in np.ndindex(*shp):
            tabs = [np.zeros(s) for s in shapes]
            tabs[k][e] = 1.0
            out = oracle_mod.encode_fwd_hessian(d, F, res, log2T, tabs, xs, with_mags=False)
            col = float((gh * out["hess"]).sum())
            assert abs(grads[k][e] - col) < 1e-12 * (1 + abs(col)), (k, e)
