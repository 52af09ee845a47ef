"""Pins for the oracle: each check ties it to something other than itself --
the formulas the pages print, hand-derived closed forms, exact polynomial
reproduction, finite differences, brute force and the adjoint identity.

Sources (page title, section):
  "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs":
      关键设计 1 (encoding equation, bases, order-bucketed tables),
      关键设计 2 (derivative bases, factorised derivative), 关键设计 3 (the
      coarse-to-fine active-level mask).
  "SIGGRAPH 2022｜InstantNGP 与多分辨率哈希编码": 流程与原理 (d-linear
      interpolation, one-to-one vs hashed levels).
  "英偉達將訓練 NeRF 模型從 5 小時縮至 5 秒": the geometric progression of
      level resolutions (formula lost in extraction).
"""
import json
import os
from decimal import Decimal, getcontext
from math import comb

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PRIMES = (1, 2654435761, 805459861, 3674653429)   # the spatial-hash primes (one per axis; the 4th for 4D)


def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# bases
# ---------------------------------------------------------------------------

def test_bases_match_printed_polynomials(oracle_mod):
    g = _load_golden("hermite_bases.json")
    for name, p in g["polynomials"].items():
        for t in np.linspace(0.0, 1.0, 17):
            want = sum(c * t ** i for i, c in enumerate(p["coeffs"]))
            got = oracle_mod.basis_1d(p["vertex_side"], p["order"], t)[p["derivative"]]
            assert abs(got - want) < 1e-14, (name, t, got, want)


def test_bases_hermite_interpolation_conditions(oracle_mod):
    # value bases: 1 at their own vertex, 0 at the other, zero slope at both;
    # slope bases: 0 at both vertices, unit slope (d/dt) at their own vertex.
    for v in (0, 1):
        for at in (0, 1):
            b0 = oracle_mod.basis_1d(v, 0, float(at))
            b1 = oracle_mod.basis_1d(v, 1, float(at))
            assert b0[0] == (1.0 if at == v else 0.0)
            assert b0[1] == 0.0
            assert b1[0] == 0.0
            assert b1[1] == (1.0 if at == v else 0.0)


def test_bases_partition_of_unity_and_mirror(oracle_mod):
    for t in np.linspace(0.0, 1.0, 33):
        assert abs(oracle_mod.basis_1d(0, 0, t)[0] + oracle_mod.basis_1d(1, 0, t)[0] - 1.0) < 1e-15
        # mirror image: the low-side bases are the high-side ones reflected
        lo0, hi0 = oracle_mod.basis_1d(0, 0, t), oracle_mod.basis_1d(1, 0, 1.0 - t)
        lo1, hi1 = oracle_mod.basis_1d(0, 1, t), oracle_mod.basis_1d(1, 1, 1.0 - t)
        assert abs(lo0[0] - hi0[0]) < 1e-15 and abs(lo0[1] + hi0[1]) < 1e-14 and abs(lo0[2] - hi0[2]) < 1e-13
        assert abs(lo1[0] + hi1[0]) < 1e-15 and abs(lo1[1] - hi1[1]) < 1e-14 and abs(lo1[2] + hi1[2]) < 1e-13


def test_bases_derivatives_by_finite_differences(oracle_mod):
    h = 1e-5
    for v in (0, 1):
        for order in (0, 1):
            for t in np.linspace(0.1, 0.9, 9):
                f = lambda s: oracle_mod.basis_1d(v, order, s)
                d1 = (f(t + h)[0] - f(t - h)[0]) / (2 * h)
                d2 = (f(t + h)[1] - f(t - h)[1]) / (2 * h)
                assert abs(d1 - f(t)[1]) < 1e-8
                assert abs(d2 - f(t)[2]) < 1e-8


# ---------------------------------------------------------------------------
# level schedule
# ---------------------------------------------------------------------------

def _decimal_schedule(L, n_min, n_max):
    """floor(N_min * (N_max/N_min)^(l/(L-1))) at 80 significant digits; a value
    within 1e-50 of an integer is that integer (for these small arguments an
    irrational value cannot come that close to one)."""
    getcontext().prec = 80
    out = []
    for l in range(L):
        v = Decimal(n_min) * (((Decimal(n_max) / Decimal(n_min)).ln() * Decimal(l) / Decimal(L - 1)).exp())
        r = v.to_integral_value()
        out.append(int(r) if abs(v - r) < Decimal("1e-50") else int(v))
    return out


@pytest.mark.parametrize("L,n_min,n_max", [
    (4, 4, 32), (16, 16, 2048), (16, 16, 1024), (16, 16, 512), (8, 3, 1000), (5, 7, 7), (32, 2, 65536),
    (12, 10, 999), (2, 5, 9)])
def test_level_schedule_matches_high_precision(oracle_mod, L, n_min, n_max):
    res = oracle_mod.level_resolutions(L, n_min, n_max)
    assert res == _decimal_schedule(L, n_min, n_max)
    assert res[0] == n_min and res[-1] == n_max
    assert all(a <= b for a, b in zip(res, res[1:]))


def test_level_schedule_exact_powers(oracle_mod):
    # 16 -> 1024 over 16 levels is 16 * 2^(0.4 l): every fifth level is an
    # exact power of two, where a plain floating-point floor can land one low.
    res = oracle_mod.level_resolutions(16, 16, 1024)
    assert res[5] == 64 and res[10] == 256 and res[15] == 1024
    assert oracle_mod.level_resolutions(1, 9, 9) == [9]


# ---------------------------------------------------------------------------
# vertex indexing
# ---------------------------------------------------------------------------

def _vertex_probe_points(d, N):
    """One query point per grid vertex g (0..N per axis) and the corner of its
    cell that is g.  Points are cell centres, written dyadically."""
    pts, corners, verts = [], [], []
    for g in np.ndindex(*([N + 1] * d)):
        cell = [min(gi, N - 1) for gi in g]
        corner = sum(((g[i] - cell[i]) << i) for i in range(d))
        pts.append([(cell[i] + 0.5) / N for i in range(d)])
        corners.append(corner)
        verts.append(g)
    return np.array(pts, np.float32), np.array(corners), verts


@pytest.mark.parametrize("d,N,log2T", [(2, 3, 4), (2, 15, 8), (2, 31, 10), (3, 3, 6), (3, 7, 9), (3, 4, 7),
                                        (4, 3, 8), (4, 5, 11)])
def test_dense_levels_are_a_bijection(oracle_mod, d, N, log2T):
    assert (N + 1) ** d <= (1 << log2T)
    pts, corners, verts = _vertex_probe_points(d, N)
    idx = oracle_mod.hash_indices(d, [N], [log2T] * (d + 1), pts)
    got = idx[np.arange(len(pts)), 0, 0, corners]
    assert sorted(got.tolist()) == list(range((N + 1) ** d))
    # axis 0 runs fastest (the reading for the unstated dense order)
    by_vertex = dict(zip(verts, got.tolist()))
    assert by_vertex[tuple([1] + [0] * (d - 1))] == 1
    assert by_vertex[tuple([0, 1] + [0] * (d - 2))] == N + 1


@pytest.mark.parametrize("d,N,log2T", [(2, 40, 8), (3, 12, 9), (3, 40, 12), (2, 4, 4), (4, 6, 9), (4, 9, 12)])
def test_hashed_levels_xor_structure(oracle_mod, d, N, log2T):
    T = 1 << log2T
    assert (N + 1) ** d > T
    pts, corners, verts = _vertex_probe_points(d, N)
    idx = oracle_mod.hash_indices(d, [N], [log2T] * (d + 1), pts)
    got = dict(zip(verts, idx[np.arange(len(pts)), 0, 0, corners].tolist()))
    assert all(0 <= v < T for v in got.values())
    # the first axis' prime is 1, so the axis-0 line is the identity mod T
    for g0 in range(N + 1):
        assert got[tuple([g0] + [0] * (d - 1))] == g0 % T
    # unit steps along the other axes land on the primes mod T
    for i in range(1, d):
        e = [0] * d
        e[i] = 1
        assert got[tuple(e)] == PRIMES[i] % T
    # XOR of per-axis terms: idx(g) = idx(g0 e0) ^ idx(g1 e1) [^ idx(g2 e2)]
    for g, v in got.items():
        acc = 0
        for i in range(d):
            e = [0] * d
            e[i] = g[i]
            acc ^= got[tuple(e)]
        assert v == acc


def test_hash_is_roughly_uniform(oracle_mod):
    d, N, log2T = 3, 63, 10
    pts, corners, verts = _vertex_probe_points(d, N)
    idx = oracle_mod.hash_indices(d, [N], [log2T] * (d + 1), pts)
    got = idx[np.arange(len(pts)), 0, 0, corners]
    counts = np.bincount(got, minlength=1 << log2T)
    expect = len(got) / (1 << log2T)
    chi2 = ((counts - expect) ** 2 / expect).sum()
    dof = (1 << log2T) - 1
    assert chi2 < dof + 6 * np.sqrt(2 * dof)


def test_dense_hashed_switch_per_order(oracle_mod):
    # (N+1)^d <= T_k decides per order table: T = (16, 8 bits) at N = 15 gives
    # a one-to-one order-0 table and a hashed order-1 table.
    pts = np.array([[0.5, 0.5]], np.float32)
    idx = oracle_mod.hash_indices(2, [15], [8, 7, 8], pts)
    c = 7  # cell (7, 7), corner 0 is vertex (7, 7)
    assert idx[0, 0, 0, 0] == 7 + 16 * 7
    assert idx[0, 0, 1, 0] == (7 ^ ((7 * PRIMES[1]) & 0xffffffff)) % 128
    assert idx[0, 0, 2, 0] == 7 + 16 * 7
    assert c == 7


def test_corner_numbering_and_clamping(oracle_mod):
    N = 8
    pts = np.array([[0.0, 0.0], [1.0, 1.0], [-3.0, 2.0], [np.nan, 0.5], [np.inf, -np.inf]], np.float32)
    idx = oracle_mod.hash_indices(2, [N], [12, 12, 12], pts)
    side = N + 1
    # x = 0 -> cell 0, t = 0; x = 1 -> last cell with t = 1; out of range clamps; NaN -> 0
    assert idx[0, 0, 0].tolist() == [0, 1, side, side + 1]
    c = N - 1
    assert idx[1, 0, 0].tolist() == [c + side * c, c + 1 + side * c, c + side * (c + 1), c + 1 + side * (c + 1)]
    assert idx[2, 0, 0].tolist() == [side * c, 1 + side * c, side * (c + 1), 1 + side * (c + 1)]
    assert idx[3, 0, 0, 0] == 0 + side * 4
    assert idx[4, 0, 0, 0] == c


# ---------------------------------------------------------------------------
# blend: exact reproduction, vertex values, single coefficients
# ---------------------------------------------------------------------------

def _vertex_index_map(oracle_mod, d, res, log2T):
    """{(level, order, vertex tuple): table index}, asked from the oracle."""
    out = {}
    for l, N in enumerate(res):
        pts, corners, verts = _vertex_probe_points(d, N)
        idx = oracle_mod.hash_indices(d, [N], log2T, pts)
        for k in range(d + 1):
            for g, v in zip(verts, idx[np.arange(len(pts)), 0, k, corners].tolist()):
                out[(l, k, g)] = v
    return out


def _alpha_list(d):
    """(alpha mask, order k, slot within bucket k) for all 2^d multi-indices."""
    return [(a, bin(a).count("1")) for a in range(1 << d)]


def _poly_eval(coef, x, deriv):
    """Tensor polynomial sum_c coef[c] prod_i x_i^c_i and its partial derivative
    of per-axis orders ``deriv``."""
    d = coef.ndim
    tot = 0.0
    for c in np.ndindex(*coef.shape):
        term = coef[c]
        for i in range(d):
            m = deriv[i]
            if c[i] < m:
                term = 0.0
                break
            fac = 1.0
            for j in range(m):
                fac *= c[i] - j
            term *= fac * x[i] ** (c[i] - m)
        tot += term
    return tot


def _fill_from_polys(oracle_mod, d, F, res, log2T, polys, degree_limit):
    """Order tables [L][T_k][C(d,k)][F] holding theta^(alpha)(g) = d^alpha p(x_g)."""
    L = len(res)
    tabs = [np.zeros((L, 1 << log2T[k], comb(d, k), F)) for k in range(d + 1)]
    vmap = _vertex_index_map(oracle_mod, d, res, log2T)
    for l, N in enumerate(res):
        for g in np.ndindex(*([N + 1] * d)):
            xg = [g[i] / N for i in range(d)]
            for a, k in _alpha_list(d):
                deriv = [(a >> i) & 1 for i in range(d)]
                s = oracle_mod.slot_in_bucket(d, a)
                for f in range(F):
                    tabs[k][l, vmap[(l, k, g)], s, f] = _poly_eval(polys[l][f], xg, deriv)
    return tabs


@pytest.mark.parametrize("d,res,log2T", [(2, [4, 8, 16, 32], [12, 12, 12]), (2, [5, 20, 25], [10, 11, 12]),
                                          (3, [4, 6, 10], [11, 11, 11, 11]), (4, [2, 3], [9, 9, 9, 9, 9])])
def test_exact_tensor_cubic_reproduction(oracle_mod, d, res, log2T):
    """On one-to-one levels, coefficients sampled from a polynomial of degree
    <= 3 per axis reproduce it, its gradient and its Laplacian exactly."""
    rng = np.random.default_rng(11)
    F = 2
    for N in res:
        assert all((N + 1) ** d <= (1 << t) for t in log2T)
    polys = [[rng.uniform(-1, 1, size=(4,) * d) for _ in range(F)] for _ in res]
    tabs = _fill_from_polys(oracle_mod, d, F, res, log2T, polys, 3)
    # dyadic query points: x * N is exact in fp32 for these N, so the cell
    # polynomial is evaluated at x itself
    xs = (rng.integers(0, 1 << 16, size=(64, d)) / float(1 << 16)).astype(np.float32)
    xs[0] = 0.0
    xs[1] = 1.0
    out = oracle_mod.encode_fwd(d, F, res, log2T, tabs, xs)
    for n in range(len(xs)):
        x = xs[n].astype(np.float64)
        for l in range(len(res)):
            for f in range(F):
                p = polys[l][f]
                assert abs(out["gamma"][n, l, f] - _poly_eval(p, x, [0] * d)) < 1e-12
                lap = 0.0
                for j in range(d):
                    e1 = [0] * d
                    e1[j] = 1
                    e2 = [0] * d
                    e2[j] = 2
                    assert abs(out["dgamma"][n, j, l, f] - _poly_eval(p, x, e1)) < 1e-10 * max(1, res[l])
                    lap += _poly_eval(p, x, e2)
                assert abs(out["lap"][n, l, f] - lap) < 1e-9 * max(1, res[l] ** 2)


def test_vertex_interpolation_with_collisions(oracle_mod):
    """At x = x_g the encoding is the stored value and its gradient the stored
    first-order slopes -- also on hashed levels with collisions."""
    rng = np.random.default_rng(5)
    d, F, res, log2T = 3, 2, [4, 16, 64], [5, 6, 7, 8]
    tabs = [rng.uniform(-1, 1, size=(len(res), 1 << log2T[k], comb(d, k), F)) for k in range(d + 1)]
    g = rng.integers(0, 5, size=(40, d))
    for l, N in enumerate(res):
        gl = g * (N // 4)
        xs = (gl / N).astype(np.float32)
        idx = oracle_mod.hash_indices(d, res, log2T, xs)
        out = oracle_mod.encode_fwd(d, F, res, log2T, tabs, xs)
        cells = np.minimum(gl, N - 1)
        corner = ((gl - cells) << np.arange(d)).sum(1)
        for n in range(len(xs)):
            i0 = idx[n, l, 0, corner[n]]
            assert np.allclose(out["gamma"][n, l], tabs[0][l, i0, 0], rtol=0, atol=1e-15)
            i1 = idx[n, l, 1, corner[n]]
            for j in range(d):
                assert np.allclose(out["dgamma"][n, j, l], tabs[1][l, i1, j], rtol=0, atol=1e-13)


def test_single_coefficient_closed_forms(oracle_mod):
    g = _load_golden("single_coefficient.json")
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
        out = oracle_mod.encode_fwd(d, 1, [N], log2T, tabs, x)
        assert abs(out["gamma"][0, 0, 0] - case["gamma"]) < 1e-15
        for j in range(d):
            assert abs(out["dgamma"][0, j, 0, 0] - case["dgamma"][j]) < 1e-14
        assert abs(out["lap"][0, 0, 0] - case["lap"]) < 1e-13


def test_slot_order_within_buckets(oracle_mod):
    # k=1: x, y, z; k=2: xy, xz, yz; k=3: xyz (the reading of the bucket order)
    assert [oracle_mod.slot_in_bucket(3, a) for a in (1, 2, 4)] == [0, 1, 2]
    assert [oracle_mod.slot_in_bucket(3, a) for a in (3, 5, 6)] == [0, 1, 2]
    assert oracle_mod.slot_in_bucket(3, 7) == 0
    assert [oracle_mod.slot_in_bucket(2, a) for a in (0, 1, 2, 3)] == [0, 0, 1, 0]
    # 4D: k=1 x, y, z, w; k=2 xy, xz, xw, yz, yw, zw; k=3 xyz, xyw, xzw, yzw; k=4 xyzw
    assert [oracle_mod.slot_in_bucket(4, a) for a in (1, 2, 4, 8)] == [0, 1, 2, 3]
    assert [oracle_mod.slot_in_bucket(4, a) for a in (3, 5, 9, 6, 10, 12)] == [0, 1, 2, 3, 4, 5]
    assert [oracle_mod.slot_in_bucket(4, a) for a in (7, 11, 13, 14)] == [0, 1, 2, 3]
    assert oracle_mod.slot_in_bucket(4, 15) == 0


# ---------------------------------------------------------------------------
# continuity and finite differences (one cell, fp64 local coordinates)
# ---------------------------------------------------------------------------

def _level_tables(rng, d, F, log2T):
    return [rng.uniform(-1, 1, size=(1 << log2T[k], comb(d, k), F)) for k in range(d + 1)]


@pytest.mark.parametrize("d", [2, 3, 4])
def test_c1_continuity_across_faces(oracle_mod, d):
    rng = np.random.default_rng(7)
    F, N, log2T = 2, 37, [6] * (d + 1)    # hashed, with collisions
    tabs = _level_tables(rng, d, F, log2T)
    for _ in range(20):
        c = rng.integers(0, N - 1, size=d)
        t = rng.uniform(0, 1, size=d)
        for j in range(d):
            tl, tr = t.copy(), t.copy()
            tl[j], tr[j] = 1.0, 0.0
            cr = c.copy()
            cr[j] += 1
            gl, dl, _ = oracle_mod.eval_cell(d, F, N, log2T, tabs, c, tl)
            gr, dr, _ = oracle_mod.eval_cell(d, F, N, log2T, tabs, cr, tr)
            assert np.allclose(gl, gr, rtol=0, atol=1e-13)
            assert np.allclose(dl, dr, rtol=0, atol=1e-11)


@pytest.mark.parametrize("d", [2, 3, 4])
def test_gradient_and_laplacian_by_finite_differences(oracle_mod, d):
    rng = np.random.default_rng(8)
    F, N, log2T = 2, 23, [7] * (d + 1)
    tabs = _level_tables(rng, d, F, log2T)
    for _ in range(10):
        c = rng.integers(0, N, size=d)
        t = rng.uniform(0.2, 0.8, size=d)
        g0, dg, lp = oracle_mod.eval_cell(d, F, N, log2T, tabs, c, t)
        lap_fd = np.zeros(F)
        for j in range(d):
            h = 1e-4
            tp, tm = t.copy(), t.copy()
            tp[j] += h
            tm[j] -= h
            gp = oracle_mod.eval_cell(d, F, N, log2T, tabs, c, tp)[0]
            gm = oracle_mod.eval_cell(d, F, N, log2T, tabs, c, tm)[0]
            # d/dx = N d/dt; central difference error O(h^2)
            assert np.allclose((gp - gm) / (2 * h) * N, dg[j], rtol=1e-6, atol=1e-6 * N)
            # second difference is exact for a cubic along the axis
            h2 = 1e-2
            tp[j], tm[j] = t[j] + h2, t[j] - h2
            gp = oracle_mod.eval_cell(d, F, N, log2T, tabs, c, tp)[0]
            gm = oracle_mod.eval_cell(d, F, N, log2T, tabs, c, tm)[0]
            lap_fd += (gp - 2 * g0 + gm) / h2 ** 2 * N * N
        assert np.allclose(lap_fd, lp, rtol=1e-8, atol=1e-8 * N * N)


# ---------------------------------------------------------------------------
# reduction to d-linear
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", [2, 3, 4])
def test_multilinear_reproduction_and_reduction(oracle_mod, d):
    """A multilinear p is reproduced by both the d-linear and the Hermite
    encodings (the latter with p's values and mixed partials stored)."""
    rng = np.random.default_rng(9)
    F, res = 2, [4, 8]
    lt = 13 if d == 4 else 12             # one-to-one levels: (N+1)^d <= T
    assert all((N + 1) ** d <= (1 << lt) for N in res)
    log2T = [lt] * (d + 1)
    polys = [[rng.uniform(-1, 1, size=(2,) * d) for _ in range(F)] for _ in res]
    tabs = _fill_from_polys(oracle_mod, d, F, res, log2T, polys, 1)
    lin_table = tabs[0][:, :, 0, :]
    xs = (rng.integers(0, 1 << 16, size=(50, d)) / float(1 << 16)).astype(np.float32)
    her = oracle_mod.encode_fwd(d, F, res, log2T, tabs, xs)
    lin, _ = oracle_mod.linear_fwd(d, F, res, lt, lin_table, xs)
    for n in range(len(xs)):
        for l in range(len(res)):
            for f in range(F):
                want = _poly_eval(polys[l][f], xs[n].astype(np.float64), [0] * d)
                assert abs(lin[n, l, f] - want) < 1e-13
                assert abs(her["gamma"][n, l, f] - want) < 1e-13


def test_linear_vertex_values_and_weights(oracle_mod):
    rng = np.random.default_rng(10)
    d, F, res, log2T = 2, 2, [8, 32], 6     # second level hashed
    table = rng.uniform(-1, 1, size=(2, 1 << log2T, F))
    xs = np.array([[0.25, 0.5], [1.0, 0.0]], np.float32)
    idx = oracle_mod.hash_indices(d, res, [log2T] * 3, xs)
    out, _ = oracle_mod.linear_fwd(d, F, res, log2T, table, xs)
    assert np.allclose(out[0, 0], table[0, idx[0, 0, 0, 0]], atol=1e-15)
    assert np.allclose(out[1, 1], table[1, idx[1, 1, 0, 1]], atol=1e-15)   # x = 1: corner (1, 0)
    # at the cell centre every corner weighs 1/4
    xc = np.array([[2.5 / 8, 5.5 / 8]], np.float32)
    idx = oracle_mod.hash_indices(d, res, [log2T] * 3, xc)
    out, _ = oracle_mod.linear_fwd(d, F, res, log2T, table, xc)
    assert np.allclose(out[0, 0], 0.25 * table[0, idx[0, 0, 0]].sum(0), atol=1e-15)


# ---------------------------------------------------------------------------
# backward: adjoint identity and the brute-force Jacobian
# ---------------------------------------------------------------------------

def _inner_tables(a, b):
    return sum(float((x * y).sum()) for x, y in zip(a, b))


@pytest.mark.parametrize("d,res,log2T", [(2, [4, 9, 30], [4, 5, 4]), (3, [3, 7, 11], [5, 6, 5, 4]),
                                          (4, [2, 5, 9], [6, 5, 7, 6, 4])])
def test_backward_adjoint_identity(oracle_mod, d, res, log2T):
    rng = np.random.default_rng(12)
    F, n = 2, 300
    L = len(res)
    tabs = [rng.uniform(-1, 1, size=(L, 1 << log2T[k], comb(d, k), F)) for k in range(d + 1)]
    xs = rng.random((n, d), dtype=np.float32)
    gg = rng.standard_normal((n, L, F), dtype=np.float32)
    gd = rng.standard_normal((n, d, L, F), dtype=np.float32)
    gl = rng.standard_normal((n, L, F), dtype=np.float32)
    out = oracle_mod.encode_fwd(d, F, res, log2T, tabs, xs)
    grads, mags = oracle_mod.encode_bwd(d, F, res, log2T, xs, gg, gd, gl)
    lhs = _inner_tables(grads, tabs)
    rhs = float((gg * out["gamma"]).sum() + (gd * out["dgamma"]).sum() + (gl * out["lap"]).sum())  # fp64 products
    scale = _inner_tables(mags, [np.abs(t) for t in tabs])
    assert abs(lhs - rhs) <= 1e-12 * scale


def test_backward_equals_bruteforce_jacobian(oracle_mod):
    """Tiny hashed grid (T = 16, many collisions): the backward equals J^T g
    for the Jacobian built column by column from forwards of unit tables."""
    rng = np.random.default_rng(13)
    d, F, res, log2T = 2, 1, [3, 6], [4, 4, 3]
    L = len(res)
    shapes = [(L, 1 << log2T[k], comb(d, k), F) for k in range(d + 1)]
    xs = rng.random((25, d), dtype=np.float32)
    gg = rng.standard_normal((25, L, F), dtype=np.float32)
    gd = rng.standard_normal((25, d, L, F), dtype=np.float32)
    gl = rng.standard_normal((25, L, F), dtype=np.float32)
    grads, _ = oracle_mod.encode_bwd(d, F, res, log2T, xs, gg, gd, gl)
    for k, shp in enumerate(shapes):
        for e in np.ndindex(*shp):
            tabs = [np.zeros(s) for s in shapes]
            tabs[k][e] = 1.0
            out = oracle_mod.encode_fwd(d, F, res, log2T, tabs, xs, with_mags=False)
            col = float((gg * out["gamma"]).sum() + (gd * out["dgamma"]).sum() + (gl * out["lap"]).sum())
            assert abs(grads[k][e] - col) < 1e-12 * (1 + abs(col)), (k, e)


def test_linear_backward_adjoint_and_jacobian(oracle_mod):
    rng = np.random.default_rng(14)
    d, F, res, log2T = 3, 2, [2, 5], 4
    L = len(res)
    xs = rng.random((40, d), dtype=np.float32)
    gg = rng.standard_normal((40, L, F), dtype=np.float32)
    grad, _ = oracle_mod.linear_bwd(d, F, res, log2T, xs, gg)
    for e in np.ndindex(L, 1 << log2T, F):
        table = np.zeros((L, 1 << log2T, F))
        table[e] = 1.0
        out, _ = oracle_mod.linear_fwd(d, F, res, log2T, table, xs)
        assert abs(grad[e] - float((gg * out).sum())) < 1e-12


# ---------------------------------------------------------------------------
# coarse-to-fine active-level mask
# ---------------------------------------------------------------------------

def test_level_mask(oracle_mod):
    rng = np.random.default_rng(15)
    d, F, res, log2T = 3, 2, [4, 8, 16, 32], [9, 9, 9, 9]
    L = len(res)
    tabs = [rng.uniform(-1, 1, size=(L, 1 << 9, comb(d, k), F)) for k in range(d + 1)]
    xs = rng.random((100, d), dtype=np.float32)
    full = oracle_mod.encode_fwd(d, F, res, log2T, tabs, xs)
    mask = 0b0101
    part = oracle_mod.encode_fwd(d, F, res, log2T, tabs, xs, level_mask=mask)
    gg = rng.standard_normal((100, L, F), dtype=np.float32)
    gfull, _ = oracle_mod.encode_bwd(d, F, res, log2T, xs, gg)
    gpart, _ = oracle_mod.encode_bwd(d, F, res, log2T, xs, gg, level_mask=mask)
    for l in range(L):
        on = (mask >> l) & 1
        for key in ("gamma", "lap"):
            assert np.array_equal(part[key][:, l], full[key][:, l] if on else np.zeros_like(full[key][:, l]))
        assert np.array_equal(part["dgamma"][:, :, l], full["dgamma"][:, :, l] if on else 0 * full["dgamma"][:, :, l])
        for k in range(d + 1):
            assert np.array_equal(gpart[k][l], gfull[k][l] if on else np.zeros_like(gfull[k][l]))
