"""Pins of the oracle's INGP-FD functions (the d-linear encoding with central
finite differences, the Hermite-NGP page's baseline: "研究背景与动机",
"关键设计 2"), tied to closed forms rather than to the oracle itself:

- a linear field stored at the vertices is reproduced by the d-linear
  encoding, so every stencil value is the field at the shifted point, the
  central gradient is the field's gradient and the Laplacian is zero;
- at a vertex of a field quadratic along one axis the FD Laplacian is
  exactly 2 / (N eps) and the FD gradient the exact derivative 2x, while
  inside a cell it is 0 (the encoding is linear along each axis there);
- at x = 1 the shifted coordinate clamps, giving half the slope;
- the backward is the transpose of the forward (adjoint identity, and the
  brute-force Jacobian of a tiny table).
Coordinates are dyadic and eps = 2^-10, so the fp32 shifts are exact."""
from math import comb

import numpy as np
import pytest

EPS = 2.0 ** -10


def _linear_tables(oracle_mod, d, res, log2T, coef):
    """[L][T][F] d-linear table holding p(x_g) = coef[l][f] . (1, x_g) at every vertex."""
    L, F = len(res), coef.shape[1]
    tab = np.zeros((L, 1 << log2T, F))
    for l, N in enumerate(res):
        assert (N + 1) ** d <= (1 << log2T)
        for g in np.ndindex(*([N + 1] * d)):
            idx = sum(g[i] * (N + 1) ** i for i in range(d))      # the one-to-one index (pinned elsewhere)
            x = np.array(g, float) / N
            tab[l, idx] = coef[l, :, 0] + coef[l, :, 1:] @ x
    return tab


def _dyadic_points(rng, n, d, lo=EPS, hi=1 - EPS):
    x = rng.integers(0, 1 << 16, size=(n, d)) / float(1 << 16)
    return np.clip(x, lo, hi).astype(np.float32)


@pytest.mark.parametrize("d,res,log2T", [(2, [4, 16, 32], 11), (3, [4, 8], 10), (4, [2, 4], 10)])
def test_fd_of_a_linear_field_is_exact(oracle_mod, d, res, log2T):
    rng = np.random.default_rng(21)
    F = 2
    coef = rng.uniform(-1, 1, size=(len(res), F, d + 1))
    tab = _linear_tables(oracle_mod, d, res, log2T, coef)
    x = _dyadic_points(rng, 40, d)
    out = oracle_mod.linear_fd_fwd(d, F, res, log2T, tab, x, EPS)
    for l in range(len(res)):
        for f in range(F):
            b = coef[l, f]
            p = lambda y: b[0] + b[1:] @ y
            for n in range(len(x)):
                xn = x[n].astype(np.float64)
                assert abs(out["gamma"][n, l, f] - p(xn)) < 1e-13
                for i in range(d):
                    e = np.zeros(d)
                    e[i] = EPS
                    assert abs(out["stencil"][n, 2 * i, l, f] - p(xn + e)) < 1e-13        # x + eps e_i
                    assert abs(out["stencil"][n, 2 * i + 1, l, f] - p(xn - e)) < 1e-13    # x - eps e_i
                    assert abs(out["dgamma"][n, i, l, f] - b[1 + i]) < 1e-9
                assert abs(out["lap"][n, l, f]) < 1e-6


def test_fd_laplacian_closed_forms_for_a_quadratic(oracle_mod):
    """p(g) = (g_0 / N)^2 at the vertices: at the interior vertex x_0 = g / N
    the FD Laplacian is N (p_{g+1} - 2 p_g + p_{g-1}) / eps = 2 / (N eps) and
    the FD gradient N (p_{g+1} - p_{g-1}) / 2 = 2 x_0; inside a cell the
    stencil stays in the cell and the FD Laplacian is 0."""
    d, N, log2T, F = 2, 16, 9, 1
    tab = np.zeros((1, 1 << log2T, F))
    for g in np.ndindex(N + 1, N + 1):
        tab[0, g[0] + (N + 1) * g[1], 0] = (g[0] / N) ** 2
    x = np.array([[5 / 16, 0.5], [11 / 16, 3 / 16], [0.5 + 1 / 64, 0.25 + 1 / 64]], np.float32)
    out = oracle_mod.linear_fd_fwd(d, F, [N], log2T, tab, x, EPS)
    for n in range(2):
        assert abs(out["lap"][n, 0, 0] - 2.0 / (N * EPS)) < 1e-9
        assert abs(out["dgamma"][n, 0, 0, 0] - 2.0 * float(x[n, 0])) < 1e-12
        assert abs(out["dgamma"][n, 1, 0, 0]) < 1e-12
    assert abs(out["lap"][2, 0, 0]) < 1e-9                       # cell interior: the stencil stays in the cell


def test_fd_clamps_the_shifted_coordinate(oracle_mod):
    """At x_0 = 1, x_0 + eps clamps back to 1: the central difference of a
    linear field gives half its slope along that axis, and at x_0 = 0 too."""
    d, res, log2T, F = 2, [8], 8, 1
    coef = np.array([[[0.25, -3.0, 0.5]]])
    tab = _linear_tables(None, d, res, log2T, coef)
    x = np.array([[1.0, 0.5], [0.0, 0.5]], np.float32)
    out = oracle_mod.linear_fd_fwd(d, F, res, log2T, tab, x, EPS)
    assert abs(out["dgamma"][0, 0, 0, 0] - (-1.5)) < 1e-9
    assert abs(out["dgamma"][1, 0, 0, 0] - (-1.5)) < 1e-9
    assert abs(out["dgamma"][0, 1, 0, 0] - 0.5) < 1e-9


@pytest.mark.parametrize("d,res,log2T", [(2, [4, 9, 30], 6), (3, [3, 7, 20], 7), (4, [2, 5], 8)])
def test_fd_backward_adjoint_identity(oracle_mod, d, res, log2T):
    """<bwd(g), theta> = <g, fwd(theta)> over all four outputs (hashed levels
    with collisions included)."""
    rng = np.random.default_rng(23)
    F, n, L = 2, 60, len(res)
    theta = rng.standard_normal((L, 1 << log2T, F))
    x = rng.random((n, d), dtype=np.float32)
    x[:4] = [[0.0] * d, [1.0] * d, [0.5] * d, [1.0 - 2 ** -20] * d]
    up = {"g_gamma": rng.standard_normal((n, L, F)).astype(np.float32),
          "g_dgamma": rng.standard_normal((n, d, L, F)).astype(np.float32),
          "g_lap": rng.standard_normal((n, L, F)).astype(np.float32),
          "g_stencil": rng.standard_normal((n, 2 * d, L, F)).astype(np.float32)}
    fwd = oracle_mod.linear_fd_fwd(d, F, res, log2T, theta, x, EPS, with_mags=False)
    grad = oracle_mod.linear_fd_bwd(d, F, res, log2T, x, EPS, with_mags=False, **up)
    lhs = float((grad * theta).sum())
    rhs = sum(float((up["g_" + k].astype(np.float64) * fwd[k]).sum()) for k in ("gamma", "dgamma", "lap", "stencil"))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs))


def test_fd_backward_equals_bruteforce_jacobian(oracle_mod):
    d, res, log2T, F = 2, [3, 6], 3, 1
    rng = np.random.default_rng(24)
    n, L, T = 7, 2, 1 << 3
    x = rng.random((n, d), dtype=np.float32)
    cols = []
    for l in range(L):
        for i in range(T):
            e = np.zeros((L, T, F))
            e[l, i, 0] = 1.0
            o = oracle_mod.linear_fd_fwd(d, F, res, log2T, e, x, EPS, with_mags=False)
            cols.append(np.concatenate([o[k].ravel() for k in ("gamma", "dgamma", "lap", "stencil")]))
    J = np.stack(cols, axis=1)
    up = {"g_gamma": rng.standard_normal((n, L, F)).astype(np.float32),
          "g_dgamma": rng.standard_normal((n, d, L, F)).astype(np.float32),
          "g_lap": rng.standard_normal((n, L, F)).astype(np.float32),
          "g_stencil": rng.standard_normal((n, 2 * d, L, F)).astype(np.float32)}
    g = np.concatenate([up[k].astype(np.float64).ravel() for k in ("g_gamma", "g_dgamma", "g_lap", "g_stencil")])
    want = (J.T @ g).reshape(L, T, F)
    got = oracle_mod.linear_fd_bwd(d, F, res, log2T, x, EPS, with_mags=False, **up)
    assert np.allclose(got, want, rtol=1e-10, atol=1e-9)
