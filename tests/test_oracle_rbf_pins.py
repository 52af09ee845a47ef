"""Pins of the oracle's Gaussian-RBF grid ("DInf-Grid：一种基于可微特征网格的神经微分方程求解器",
可微的径向基函数插值 and 多分辨率特征网格), tied to mathematics rather than to
the oracle's own formulas:

- partition of unity: a constant field is reproduced with zero gradient
  and Laplacian, also where the ring neighbourhood is clipped at the border;
- separability: exp(-eps^2 |y - g|^2) factorises over the axes and the ring
  neighbourhood is a box, so the normalised weight is a product of 1D
  normalised Gaussian weights -- the test rebuilds gamma, its gradient and
  its Laplacian from 1D weights and their 1D quotient-rule derivatives and
  tensor contractions, an independent route to the oracle's d-dimensional
  quotient rule;
- the nearest-vertex limit of a narrow kernel;
- finite differences of gamma and of its gradient inside a cell;
- the backward is the transpose (adjoint identity, brute-force Jacobian)."""
import itertools

import numpy as np
import pytest


def _dense_table(rng, d, res, log2T, F):
    for N in res:
        assert (N + 1) ** d <= (1 << log2T)
    return rng.uniform(-1, 1, size=(len(res), 1 << log2T, F))


def _dense_index(g, N):
    return sum(int(g[i]) * (N + 1) ** i for i in range(len(g)))


@pytest.mark.parametrize("d,rings", [(2, 1), (2, 3), (3, 2), (4, 1)])
def test_partition_of_unity(oracle_mod, d, rings):
    res, log2T, F = [3, 7], 12, 2
    x = np.random.default_rng(31).random((30, d), dtype=np.float32)
    x[:3] = [[0.0] * d, [1.0] * d, [0.5] * d]
    table = np.empty((len(res), 1 << log2T, F))
    table[..., 0], table[..., 1] = 0.75, -2.5
    out = oracle_mod.rbf_fwd(d, F, res, log2T, table, x, 1.0, rings)
    assert np.allclose(out["gamma"][..., 0], 0.75, rtol=0, atol=1e-14)
    assert np.allclose(out["gamma"][..., 1], -2.5, rtol=0, atol=1e-14)
    assert np.all(np.abs(out["dgamma"]) <= 1e-12 * np.maximum(out["mdgamma"], 1))
    assert np.all(np.abs(out["lap"]) <= 1e-12 * np.maximum(out["mlap"], 1))


def _weights_1d(y, c, N, eps, rings):
    """Normalised 1D Gaussian weights over g = c-rings+1 .. c+rings clipped to
    [0, N], and their first and second y-derivatives (1D quotient rule)."""
    g = np.arange(c - rings + 1, c + rings + 1)
    g = g[(g >= 0) & (g <= N)]
    r = y - g
    e = np.exp(-eps * eps * r * r)
    e1 = -2 * eps * eps * r * e
    e2 = (4 * eps ** 4 * r * r - 2 * eps * eps) * e
    s, s1, s2 = e.sum(), e1.sum(), e2.sum()
    w = e / s
    w1 = (e1 - w * s1) / s
    w2 = (e2 - 2 * w1 * s1 - w * s2) / s
    return g, w, w1, w2


@pytest.mark.parametrize("d,rings,eps", [(2, 1, 1.0), (2, 3, 1.0), (2, 2, 0.5), (3, 3, 1.0), (3, 2, 2.0)])
def test_separable_tensor_form(oracle_mod, d, rings, eps):
    rng = np.random.default_rng(32 + rings)
    res, log2T, F = [4, 9], 12, 1
    table = _dense_table(rng, d, res, log2T, F)
    x = rng.random((25, d), dtype=np.float32)
    x[:2] = [[0.0] * d, [1.0 - 2 ** -20] * d]
    out = oracle_mod.rbf_fwd(d, F, res, log2T, table, x, eps, rings)
    for l, N in enumerate(res):
        for n in range(len(x)):
            pos = (np.clip(x[n], 0, 1) * np.float32(N)).astype(np.float32).astype(np.float64)
            c = np.minimum(np.floor(pos).astype(int), N - 1)
            ax = [_weights_1d(pos[i], c[i], N, eps, rings) for i in range(d)]
            gam, grad, lap = 0.0, np.zeros(d), 0.0
            for combo in itertools.product(*[range(len(a[0])) for a in ax]):
                g = [ax[i][0][combo[i]] for i in range(d)]
                th = table[l, _dense_index(g, N), 0]
                w = [ax[i][1][combo[i]] for i in range(d)]
                gam += np.prod(w) * th
                for i in range(d):
                    others = np.prod([w[k] for k in range(d) if k != i])
                    grad[i] += N * ax[i][2][combo[i]] * others * th
                    lap += N * N * ax[i][3][combo[i]] * others * th
            assert abs(out["gamma"][n, l, 0] - gam) < 1e-12
            assert np.allclose(out["dgamma"][n, :, l, 0], grad, rtol=0, atol=1e-11 * N)
            assert abs(out["lap"][n, l, 0] - lap) < 1e-10 * N * N


def test_narrow_kernel_tends_to_the_nearest_vertex(oracle_mod):
    """eps = 8 in grid units: at a vertex every other weight is below
    e^-64, so gamma is that vertex's value."""
    rng = np.random.default_rng(33)
    d, res, log2T, F = 2, [8], 8, 2
    table = _dense_table(rng, d, res, log2T, F)
    g = np.array([[3, 5], [0, 8], [8, 0], [4, 4]])
    x = (g / 8.0).astype(np.float32)
    out = oracle_mod.rbf_fwd(d, F, res, log2T, table, x, 8.0, 2)
    for n in range(len(g)):
        assert np.allclose(out["gamma"][n, 0], table[0, _dense_index(g[n], 8)], rtol=0, atol=1e-20)


@pytest.mark.parametrize("d", [2, 3])
def test_derivatives_by_finite_differences(oracle_mod, d):
    """Central differences of gamma (gradient) and of the gradient (Laplacian)
    inside one cell, where the neighbourhood does not change."""
    rng = np.random.default_rng(34)
    res, log2T, F, N = [6], 12, 1, 6
    table = _dense_table(rng, d, res, log2T, F)
    h = 2.0 ** -12
    base = (np.array([2.5, 3.25, 1.75][:d]) / N)
    xs = [base]
    for i in range(d):
        for sgn in (1, -1):
            e = np.zeros(d)
            e[i] = sgn * h
            xs.append(base + e)
    x = np.array(xs, np.float32)
    out = oracle_mod.rbf_fwd(d, F, res, log2T, table, x, 1.0, 3)
    lap_fd = 0.0
    for i in range(d):
        hp = float(x[1 + 2 * i, i]) - float(x[0, i])
        hm = float(x[0, i]) - float(x[2 + 2 * i, i])
        g_fd = (out["gamma"][1 + 2 * i, 0, 0] - out["gamma"][2 + 2 * i, 0, 0]) / (hp + hm)
        assert abs(g_fd - out["dgamma"][0, i, 0, 0]) < 1e-4 * max(1.0, out["mdgamma"][0, i, 0, 0])
        lap_fd += (out["dgamma"][1 + 2 * i, i, 0, 0] - out["dgamma"][2 + 2 * i, i, 0, 0]) / (hp + hm)
    assert abs(lap_fd - out["lap"][0, 0, 0]) < 1e-3 * max(1.0, out["mlap"][0, 0, 0])


@pytest.mark.parametrize("d,res,log2T,rings", [(2, [3, 9, 40], 7, 2), (3, [2, 5, 12], 8, 3)])
def test_rbf_backward_adjoint_identity(oracle_mod, d, res, log2T, rings):
    rng = np.random.default_rng(35)
    F, n, L = 2, 40, len(res)
    theta = rng.standard_normal((L, 1 << log2T, F))
    x = rng.random((n, d), dtype=np.float32)
    x[:3] = [[0.0] * d, [1.0] * d, [0.5] * d]
    up = {"g_gamma": rng.standard_normal((n, L, F)).astype(np.float32),
          "g_dgamma": rng.standard_normal((n, d, L, F)).astype(np.float32),
          "g_lap": rng.standard_normal((n, L, F)).astype(np.float32)}
    fwd = oracle_mod.rbf_fwd(d, F, res, log2T, theta, x, 1.0, rings, with_mags=False)
    grad = oracle_mod.rbf_bwd(d, F, res, log2T, x, 1.0, rings, with_mags=False, **up)
    lhs = float((grad * theta).sum())
    rhs = sum(float((up["g_" + k].astype(np.float64) * fwd[k]).sum()) for k in ("gamma", "dgamma", "lap"))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs))


def test_rbf_backward_equals_bruteforce_jacobian(oracle_mod):
    d, res, log2T, F, rings = 2, [2, 4], 5, 1, 2
    rng = np.random.default_rng(36)
    n, L, T = 6, 2, 1 << 5
    x = rng.random((n, d), dtype=np.float32)
    cols = []
    for l in range(L):
        for i in range(T):
            e = np.zeros((L, T, F))
            e[l, i, 0] = 1.0
            o = oracle_mod.rbf_fwd(d, F, res, log2T, e, x, 1.0, rings, with_mags=False)
            cols.append(np.concatenate([o[k].ravel() for k in ("gamma", "dgamma", "lap")]))
    J = np.stack(cols, axis=1)
    up = {"g_gamma": rng.standard_normal((n, L, F)).astype(np.float32),
          "g_dgamma": rng.standard_normal((n, d, L, F)).astype(np.float32),
          "g_lap": rng.standard_normal((n, L, F)).astype(np.float32)}
    g = np.concatenate([up[k].astype(np.float64).ravel() for k in ("g_gamma", "g_dgamma", "g_lap")])
    want = (J.T @ g).reshape(L, T, F)
    got = oracle_mod.rbf_bwd(d, F, res, log2T, x, 1.0, rings, with_mags=False, **up)
    assert np.allclose(got, want, rtol=1e-10, atol=1e-9)
