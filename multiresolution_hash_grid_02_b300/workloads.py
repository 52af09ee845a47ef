"""Seeded synthetic workloads for the hash-grid encoding.

This module only draws random inputs and describes their shapes; it holds none
of the encoding's arithmetic and imports neither the CUDA library nor the
oracle, so both sides can be fed from it.

The five workloads follow the shapes the pages work with: a tiny 2D Hermite
grid, the Instant-NGP 2D d-linear grid (L=16, F=2, T=2^19, the parameters the
InstantNGP article fixes in its experiments section), a PINN-sized 2D Hermite
grid with stratified collocation points (the stratified sampling of the
DInf-Grid article, "可微的径向基函数插值"), 3D Hermite grids, the largest
with fp16 coefficients and a coarse-to-fine active-level mask ("关键设计 3" of
the Hermite-NGP notes), and a 4D space-time Hermite grid (the extension the
Hermite-NGP notes name as the method's main storage cost; they give no 4D
configuration, so it takes the 3D grid's parameters).  No public dataset is
involved.

Draw order for one workload (``numpy.random.default_rng(seed)``): coordinates,
then the coefficient table(s), then the upstream gradients g_gamma, g_dgamma,
g_lap.  All draws are float32 (``dtype=np.float32`` in numpy's generator); fp16
tables are the float32 draw rounded to fp16.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from math import comb

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "hermite", "linear", "linear_fd" (d-linear with central differences) or "rbf"
    d: int
    n_points: int
    L: int
    F: int
    n_min: int
    n_max: int
    log2_T: tuple             # per order table k = 0..d (hermite) or (T,) (linear)
    dtype: str                # "f32" or "f16" table storage
    coef_range: float         # tables ~ U[-r, r)
    coords: str = "uniform"   # "uniform", "stratified" or "stratified_shuffled"
    level_masks: tuple = field(default=())  # extra active-level masks to exercise
    seed: int = 0
    eps: float = 0.0          # finite-difference step (linear_fd); Gaussian width in grid units (rbf)
    rings: int = 0            # rbf: ring neighbourhood

    @property
    def V(self) -> int:
        return 1 << self.d

    def scaled(self, n_points: int) -> "Workload":
        return replace(self, n_points=n_points)


WORKLOADS = {
    1: Workload("2d_hermite_tiny", "hermite", 2, 4096, 4, 2, 4, 32, (12, 12, 12), "f32", 1.0, seed=1),
    2: Workload("2d_linear_ingp", "linear", 2, 1 << 20, 16, 2, 16, 2048, (19,), "f32", 1e-4, seed=2),
    3: Workload("2d_hermite_pinn", "hermite", 2, 1 << 20, 16, 2, 16, 1024, (19, 19, 19), "f32", 1e-2,
                coords="stratified", seed=3),
    4: Workload("3d_hermite", "hermite", 3, 1 << 21, 16, 2, 16, 512, (19, 19, 19, 19), "f32", 1e-2, seed=4),
    5: Workload("3d_hermite_large_fp16", "hermite", 3, 1 << 23, 16, 2, 16, 2048, (22, 22, 22, 22), "f16", 1e-2,
                level_masks=((1 << 4) - 1, (1 << 10) - 1, (1 << 16) - 1), seed=5),
    # space-time (x, y, z, t): workload 4's grid with a fourth axis, half the points
    6: Workload("4d_hermite_spacetime", "hermite", 4, 1 << 20, 16, 2, 16, 512, (19, 19, 19, 19, 19), "f32", 1e-2,
                seed=6),
    # the pages' finite-difference baseline (INGP-FD) on workload 4's grid: 2d+1 = 7 d-linear encodes per point;
    # eps = 2^-10, half the finest cell (the pages leave the step to hand tuning)
    7: Workload("3d_linear_fd", "linear_fd", 3, 1 << 21, 16, 2, 16, 512, (19,), "f32", 1e-4, seed=7, eps=2.0 ** -10),
    # DInf-Grid's Gaussian-RBF grids with the page's settings: eps = 1 with 3 rings, 4 dense levels, the
    # finest 512 in 2D and 56 in 3D; stratified collocation points (its structured sampling)
    8: Workload("2d_dinf_rbf", "rbf", 2, 1 << 20, 4, 2, 64, 512, (19,), "f32", 1e-2, coords="stratified", seed=8,
                eps=1.0, rings=3),
    9: Workload("3d_dinf_rbf", "rbf", 3, 1 << 21, 4, 2, 7, 56, (18,), "f32", 1e-2, coords="stratified", seed=9,
                eps=1.0, rings=3),
    # workload 3 with its collocation points in a seeded random order, as a training loop that shuffles its
    # mini-batches would present them (the DInf-Grid page fixes the strata, not their order); the tables and
    # upstream gradients are workload 3's draws
    10: Workload("2d_hermite_pinn_shuffled", "hermite", 2, 1 << 20, 16, 2, 16, 1024, (19, 19, 19), "f32", 1e-2,
                 coords="stratified_shuffled", seed=3),
}

SHUFFLE_SEED_OFFSET = 3000   # the permutation of the shuffled order comes from default_rng(seed + 3000)


def draw_coords(rng: np.random.Generator, w: Workload) -> np.ndarray:
    """float32 [N][d] in [0,1]^d.  "stratified_shuffled": the stratified
    points (the same draws from ``rng``) permuted by a second generator,
    ``default_rng(seed + SHUFFLE_SEED_OFFSET)``, so every other draw of the
    workload is unchanged."""
    if w.coords == "stratified_shuffled":
        x = draw_coords(rng, replace(w, coords="stratified"))
        perm = np.random.default_rng(w.seed + SHUFFLE_SEED_OFFSET).permutation(w.n_points)
        return np.ascontiguousarray(x[perm])
    if w.coords == "stratified":
        side = int(round(w.n_points ** (1.0 / w.d)))
        if side ** w.d != w.n_points:
            raise ValueError("stratified sampling needs N = side^d")
        u = rng.random((w.n_points, w.d), dtype=np.float32).astype(np.float64)
        # stratum number n = sum_i s_i side^i: axis 0 fastest (row-major in y)
        n = np.arange(w.n_points, dtype=np.int64)
        cells = np.stack([(n // side ** i) % side for i in range(w.d)], axis=1)
        x = (cells + u) / side
        return np.minimum(x, 1.0).astype(np.float32)
    return rng.random((w.n_points, w.d), dtype=np.float32)


def draw_packed_table(rng: np.random.Generator, w: Workload) -> np.ndarray:
    """The coefficient tables of all orders, drawn as one interleaved array.

    Hermite: [L][T][2^d][F], the 2^d slots of a vertex ordered by derivative
    order, then lexicographically (f, fx, fy, [fz], fxy, [fxz, fyz, fxyz]).
    Linear, linear_fd and rbf: [L][T][F].  float32 or float16 (the float32 draw rounded).
    """
    T = 1 << w.log2_T[0]
    if w.kind == "hermite":
        if len(set(w.log2_T)) != 1:
            raise ValueError("the interleaved table needs one T for all orders")
        shape = (w.L, T, w.V, w.F)
    else:
        shape = (w.L, T, w.F)
    a = rng.random(shape, dtype=np.float32)
    a *= np.float32(2.0 * w.coef_range)
    a -= np.float32(w.coef_range)
    return a.astype(np.float16) if w.dtype == "f16" else a


def slot_offsets(d: int) -> list[int]:
    """Offset of order bucket k inside an interleaved vertex row (in slots)."""
    offs, o = [], 0
    for k in range(d + 1):
        offs.append(o)
        o += comb(d, k)
    return offs


def split_orders(packed: np.ndarray, d: int) -> list[np.ndarray]:
    """Views of the order-k tables [L][T][C(d,k)][F] inside an interleaved table."""
    offs = slot_offsets(d)
    return [packed[:, :, offs[k]:offs[k] + comb(d, k), :] for k in range(d + 1)]


def draw_order_tables(rng: np.random.Generator, w: Workload) -> list[np.ndarray]:
    """Separate, contiguous order tables [L][T_k][C(d,k)][F] (T_k may differ)."""
    out = []
    for k in range(w.d + 1):
        a = rng.random((w.L, 1 << w.log2_T[k], comb(w.d, k), w.F), dtype=np.float32)
        a *= np.float32(2.0 * w.coef_range)
        a -= np.float32(w.coef_range)
        out.append(a.astype(np.float16) if w.dtype == "f16" else a)
    return out


def draw_upstream(rng: np.random.Generator, w: Workload, with_derivs: bool = True):
    """N(0,1) upstream gradients in the point-major logical layout:
    g_gamma [N][L][F], g_dgamma [N][d][L][F], g_lap [N][L][F] (Hermite);
    for linear_fd the third is g_stencil [N][2d][L][F], the upstream of the
    stencil encodings."""
    n, L, F, d = w.n_points, w.L, w.F, w.d
    gg = rng.standard_normal((n, L, F), dtype=np.float32)
    if not with_derivs or w.kind == "linear":
        return gg, None, None
    # hermite and rbf: gradient and Laplacian upstream
    if w.kind == "linear_fd":
        return gg, None, rng.standard_normal((n, 2 * d, L, F), dtype=np.float32)
    gd = rng.standard_normal((n, d, L, F), dtype=np.float32)
    gl = rng.standard_normal((n, L, F), dtype=np.float32)
    return gg, gd, gl


def draw_upstream_hessian(rng: np.random.Generator, w: Workload) -> np.ndarray:
    """N(0,1) upstream gradient of the full Hessian, point-major
    [N][P][L][F] with P = d(d+1)/2 upper-triangle entries."""
    P = w.d * (w.d + 1) // 2
    return rng.standard_normal((w.n_points, P, w.L, w.F), dtype=np.float32)


def make(w: Workload, seed: int | None = None, separate_orders: bool = False):
    """Draw a complete workload: dict with coords, table (interleaved) or
    order_tables (separate), and upstream gradients."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    out = {"coords": draw_coords(rng, w)}
    if separate_orders and w.kind == "hermite":
        out["order_tables"] = draw_order_tables(rng, w)
    else:
        out["table"] = draw_packed_table(rng, w)
    gg, gd, third = draw_upstream(rng, w)
    out["g_gamma"], out["g_dgamma"] = gg, gd
    out["g_stencil" if w.kind == "linear_fd" else "g_lap"] = third
    return out


def to_feature_major(a: np.ndarray, has_axis: bool) -> np.ndarray:
    """Point-major [N]([d])[L][F] -> feature-major ([d])[L][F][N] (a copy)."""
    if has_axis:
        return np.ascontiguousarray(np.transpose(a, (1, 2, 3, 0)))
    return np.ascontiguousarray(np.transpose(a, (1, 2, 0)))


def from_feature_major(a: np.ndarray, has_axis: bool) -> np.ndarray:
    """Inverse of :func:`to_feature_major`."""
    if has_axis:
        return np.ascontiguousarray(np.transpose(a, (3, 0, 1, 2)))
    return np.ascontiguousarray(np.transpose(a, (2, 0, 1)))


# ---------------------------------------------------------------------------
# the SIREN consumer of the encoding (Hermite-NGP, 关键设计 2)
# ---------------------------------------------------------------------------

SIREN_H = 64        # hidden width: the page does not fix it
SIREN_O = 1         # a scalar field u
SIREN_OMEGA = 30.0  # omega_0 of the page's training setup ("损失函数 / 训练策略")


def siren_weights(rng: np.random.Generator, K: int, H: int = SIREN_H, O: int = SIREN_O,
                  omega: float = SIREN_OMEGA) -> dict:
    """SIREN initialisation (first layer U(-1/K, 1/K); bias U(-1/sqrt K, 1/sqrt K);
    output layer U(-sqrt(6/H)/omega, sqrt(6/H)/omega); zero output bias), float32."""
    f32 = np.float32
    return {"W1": rng.uniform(-1 / K, 1 / K, (H, K)).astype(f32),
            "b1": (rng.uniform(-1, 1, H) / np.sqrt(K)).astype(f32),
            "W2": (rng.uniform(-1, 1, (O, H)) * np.sqrt(6 / H) / omega).astype(f32),
            "b2": np.zeros(O, f32)}


def siren_upstream(rng: np.random.Generator, n: int, d: int, O: int = SIREN_O) -> dict:
    """N(0,1) gradients of a loss with respect to u [n][O], grad u [n][d][O]
    and lap u [n][O] (point-major), float32."""
    return {"g_u": rng.standard_normal((n, O), dtype=np.float32),
            "g_du": rng.standard_normal((n, d, O), dtype=np.float32),
            "g_lapu": rng.standard_normal((n, O), dtype=np.float32)}
