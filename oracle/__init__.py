"""Oracle for the multiresolution hash-grid encoding -- TEST INFRASTRUCTURE.

A plain, slow, fp64 CPU restatement of what the encoding computes, used only by
``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference arm.  The product library never imports, links or calls anything
here, and nothing here imports the product library.

The arithmetic lives in ``hg_oracle.c`` (built with gcc into
``_build/libhg_oracle.so`` by :func:`build`); this module marshals numpy arrays
and adds the one piece that needs arbitrary-precision integers, the level
schedule.

Sources (page title, section):

* "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
  sections "整体框架", "关键设计 1", "关键设计 2" -- the Hermite encoding,
  order-bucketed tables, bases and derivatives.
* "SIGGRAPH 2022｜InstantNGP 与多分辨率哈希编码", section
  "InstantNGP 与多分辨率哈希编码流程与原理" -- d-linear interpolation, the
  one-to-one vs hashed levels.
* "英偉達將訓練 NeRF 模型從 5 小時縮至 5 秒" -- the geometric progression of
  level resolutions between N_min and N_max (the printed formula is lost in the
  page's extraction; the reading used is N_l = floor(N_min * b^l),
  b = (N_max/N_min)^(1/(L-1)), evaluated exactly).

Every function here is pinned by ``tests/test_oracle_*.py`` against closed
forms, invariants, brute force and the pages' printed formulas; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from math import comb

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hg_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libhg_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile ``hg_oracle.c`` with gcc (no FMA contraction, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    # HG_ORACLE_LIB: load another build of hg_oracle.c instead (the mutation
    # tests point it at copies with planted mistakes)
    override = os.environ.get("HG_ORACLE_LIB")
    lib = ctypes.CDLL(override if override else build())
    P = ctypes.c_void_p
    i32, i64, u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    lib.oracle_basis_1d.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, P]
    lib.oracle_basis_1d.restype = None
    lib.oracle_eval_cell.argtypes = [ctypes.c_int, ctypes.c_int, i32, P, P, P, P, P, P, P]
    lib.oracle_hash_indices.argtypes = [ctypes.c_int, ctypes.c_int, P, P, i64, P, P, ctypes.c_int]
    lib.oracle_encode_fwd.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, u32, P,
                                      i64, P, P, P, P, P, P, P, ctypes.c_int]
    lib.oracle_encode_bwd_level.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            P, P, i64, P, P, P, P, P, P]
    lib.oracle_linear_fwd.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int, u32,
                                      P, i64, P, P, P, ctypes.c_int]
    lib.oracle_linear_bwd_level.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            P, ctypes.c_int, i64, P, P, P, P]
    lib.oracle_slot_in_bucket.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.oracle_hess_entries.argtypes = [ctypes.c_int]
    lib.oracle_eval_cell_hessian.argtypes = [ctypes.c_int, ctypes.c_int, i32, P, P, P, P, P, P, P]
    lib.oracle_encode_fwd_hessian.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, u32, P,
                                              i64, P, P, P, P, P, P, P, ctypes.c_int]
    lib.oracle_encode_bwd_hessian_level.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    P, P, i64, P, P, P, P, P, P]
    f32 = ctypes.c_float
    lib.oracle_linear_fd_fwd.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int, u32, P, i64,
                                         P, f32, P, P, P, P, P, P, P, P, ctypes.c_int]
    lib.oracle_linear_fd_bwd_level.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                               ctypes.c_int, i64, P, f32, P, P, P, P, P, P]
    lib.oracle_rbf_fwd.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int, u32, P, i64, P, f32,
                                   ctypes.c_int, P, P, P, P, P, P, ctypes.c_int]
    lib.oracle_rbf_bwd_level.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, ctypes.c_int,
                                         i64, P, f32, ctypes.c_int, P, P, P, P, P]
    for name in ("oracle_rbf_fwd", "oracle_rbf_bwd_level", "oracle_eval_cell", "oracle_hash_indices", "oracle_encode_fwd",
                 "oracle_encode_bwd_level", "oracle_linear_fwd", "oracle_linear_bwd_level",
                 "oracle_slot_in_bucket", "oracle_hess_entries", "oracle_eval_cell_hessian",
                 "oracle_encode_fwd_hessian", "oracle_encode_bwd_hessian_level", "oracle_linear_fd_fwd",
                 "oracle_linear_fd_bwd_level"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


# ---------------------------------------------------------------------------
# level schedule (exact)
# ---------------------------------------------------------------------------

def level_resolutions(L: int, n_min: int, n_max: int) -> list[int]:
    """N_l = floor(N_min * b^l), b = (N_max/N_min)^(1/(L-1)), exactly.

    N_l is the largest integer n with n^(L-1) * N_min^l <= N_max^l * N_min^(L-1)
    (both sides raised to the power L-1), found by bisection on Python's exact
    integers.  A single level (L = 1) sits at N_min.
    """
    if L < 1 or n_min < 1 or n_max < n_min:
        raise ValueError("need L >= 1 and 1 <= n_min <= n_max")
    if L == 1:
        return [n_min]
    out = []
    for l in range(L):
        rhs = n_max ** l * n_min ** (L - 1 - l)  # divide both sides by n_min^l
        lo, hi = n_min, n_max                      # N_min * b^l lies in [N_min, N_max]
        while lo < hi:
            mid = (lo + hi + 1) // 2
            if mid ** (L - 1) <= rhs:
                lo = mid
            else:
                hi = mid - 1
        out.append(lo)
    return out


# ---------------------------------------------------------------------------
# table layout helpers (storage only; no arithmetic of the method)
# ---------------------------------------------------------------------------

def slot_in_bucket(d: int, alpha: int) -> int:
    return _load().oracle_slot_in_bucket(d, alpha)


def order_table_shapes(d: int, L: int, F: int, log2T) -> list[tuple]:
    """Shapes of the d+1 order tables: table k is [L][T_k][C(d,k)][F]."""
    return [(L, 1 << int(log2T[k]), comb(d, k), F) for k in range(d + 1)]


# ---------------------------------------------------------------------------
# public oracle calls
# ---------------------------------------------------------------------------

def basis_1d(v: int, order: int, t: float) -> tuple[float, float, float]:
    """(value, d/dt, d2/dt2) of the cubic Hermite basis of the cell's vertex on
    side v (0 = low, 1 = high) for the value (order 0) or slope (order 1)."""
    out = np.zeros(3, np.float64)
    _load().oracle_basis_1d(int(v), int(order), float(t), _ptr(out))
    return float(out[0]), float(out[1]), float(out[2])


def eval_cell(d: int, F: int, N: int, log2T, level_tables, c, t):
    """Evaluate one cell (corner c, fp64 local coordinate t) of one level.

    ``level_tables[k]`` is that level's order-k table [T_k][C(d,k)][F].
    Returns (gamma[F], dgamma[d][F], lap[F]).
    """
    lib = _load()
    tabs = [np.ascontiguousarray(a, dtype=np.float64) for a in level_tables]
    lt = np.asarray(log2T, np.int32)
    cc = np.asarray(c, np.int64)
    tt = np.asarray(t, np.float64)
    g = np.zeros(F, np.float64)
    dg = np.zeros((d, F), np.float64)
    lp = np.zeros(F, np.float64)
    _check(lib.oracle_eval_cell(d, F, int(N), _ptr(lt), _ptr_array(tabs), _ptr(cc), _ptr(tt),
                                _ptr(g), _ptr(dg), _ptr(lp)), "eval_cell")
    return g, dg, lp


def hash_indices(d: int, res, log2T, coords: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    """uint32 [N][L][d+1][2^d]: the vertex index of every corner (bit i of the
    corner number = axis i) in every order table, at every level."""
    lib = _load()
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    L = len(res)
    r = np.asarray(res, np.int32)
    lt = np.asarray(log2T, np.int32)
    out = np.zeros((n, L, d + 1, 1 << d), np.uint32)
    _check(lib.oracle_hash_indices(d, L, _ptr(r), _ptr(lt), n, _ptr(coords), _ptr(out),
                                   nthreads or default_threads()), "hash_indices")
    return out


def _as_f64_tables(tables):
    # fp16 tables widen exactly to fp64 (every binary16 value is a binary64 value)
    return [np.ascontiguousarray(t, dtype=np.float64) for t in tables]


def encode_fwd(d: int, F: int, res, log2T, tables, coords: np.ndarray,
               level_mask: int | None = None, nthreads: int | None = None,
               with_mags: bool = True):
    """Hermite forward.  ``tables[k]`` is [L][T_k][C(d,k)][F] (any float dtype).

    Returns a dict with point-major fp64 arrays gamma [N][L][F],
    dgamma [N][d][L][F], lap [N][L][F] and, if ``with_mags``, their condition
    magnitudes mgamma, mdgamma, mlap.
    """
    lib = _load()
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    tabs = _as_f64_tables(tables)
    for k, tb in enumerate(tabs):
        want = (L, 1 << int(log2T[k]), comb(d, k), F)
        if tb.shape != want:
            raise ValueError(f"order table {k} has shape {tb.shape}, expected {want}")
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    lt = np.asarray(log2T, np.int32)
    out = {"gamma": np.zeros((n, L, F)), "dgamma": np.zeros((n, d, L, F)), "lap": np.zeros((n, L, F))}
    if with_mags:
        out.update(mgamma=np.zeros((n, L, F)), mdgamma=np.zeros((n, d, L, F)), mlap=np.zeros((n, L, F)))
    _check(lib.oracle_encode_fwd(d, L, F, _ptr(r), _ptr(lt), level_mask & 0xffffffff, _ptr_array(tabs),
                                 n, _ptr(coords), _ptr(out["gamma"]), _ptr(out["dgamma"]), _ptr(out["lap"]),
                                 _ptr(out.get("mgamma")), _ptr(out.get("mdgamma")), _ptr(out.get("mlap")),
                                 nthreads or default_threads()), "encode_fwd")
    return out


def encode_bwd_levels(d: int, F: int, res, log2T, coords: np.ndarray, g_gamma: np.ndarray | None,
                      g_dgamma: np.ndarray | None = None, g_lap: np.ndarray | None = None,
                      levels=None, with_mags: bool = True, nthreads: int | None = None):
    """Hermite backward for the listed levels: the transpose of
    :func:`encode_fwd` applied to the upstream gradients (float32,
    point-major layouts; any may be None).  Colliding vertices sum.

    Returns {level: (grads, mags)} with grads[k] / mags[k] fp64 arrays
    [T_k][C(d,k)][F] (mags None unless ``with_mags``).  Levels run in parallel
    threads, each on its own arrays, so the result does not depend on the
    thread count.
    """
    from concurrent.futures import ThreadPoolExecutor
    lib = _load()
    L = len(res)
    levels = list(range(L)) if levels is None else list(levels)
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    lt = np.asarray(log2T, np.int32)
    f32 = lambda a: None if a is None else np.ascontiguousarray(a, np.float32)
    gg, gd, gl = f32(g_gamma), f32(g_dgamma), f32(g_lap)
    shapes = [(1 << int(log2T[k]), comb(d, k), F) for k in range(d + 1)]
    out = {l: ([np.zeros(s) for s in shapes], [np.zeros(s) for s in shapes] if with_mags else None) for l in levels}

    def one(l):
        grads, mags = out[l]
        return lib.oracle_encode_bwd_level(d, L, F, l, _ptr(r), _ptr(lt), n, _ptr(coords), _ptr(gg), _ptr(gd),
                                           _ptr(gl), _ptr_array(grads), _ptr_array(mags) if with_mags else None)

    with ThreadPoolExecutor(max_workers=max(1, min(len(levels) or 1, nthreads or default_threads()))) as ex:
        for rc in ex.map(one, levels):
            _check(rc, "encode_bwd")
    return out


def encode_bwd(d: int, F: int, res, log2T, coords: np.ndarray, g_gamma: np.ndarray | None,
               g_dgamma: np.ndarray | None = None, g_lap: np.ndarray | None = None,
               level_mask: int | None = None, with_mags: bool = True, nthreads: int | None = None):
    """Hermite backward over all levels: (grads, mags), lists over order k of
    fp64 [L][T_k][C(d,k)][F] arrays; inactive levels stay zero."""
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    active = [l for l in range(L) if (level_mask >> l) & 1]
    per = encode_bwd_levels(d, F, res, log2T, coords, g_gamma, g_dgamma, g_lap, active, with_mags, nthreads)
    shapes = order_table_shapes(d, L, F, log2T)
    grads = [np.zeros(s) for s in shapes]
    mags = [np.zeros(s) for s in shapes] if with_mags else None
    for l, (g, m) in per.items():
        for k in range(d + 1):
            grads[k][l] = g[k]
            if with_mags:
                mags[k][l] = m[k]
    return grads, mags


def linear_fwd(d: int, F: int, res, log2T: int, table: np.ndarray, coords: np.ndarray,
               level_mask: int | None = None, nthreads: int | None = None, with_mags: bool = True):
    """d-linear forward: gamma [N][L][F] (and its magnitude) from table [L][T][F]."""
    lib = _load()
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    tb = np.ascontiguousarray(table, np.float64)
    if tb.shape != (L, 1 << int(log2T), F):
        raise ValueError("linear table must be [L][T][F]")
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    g = np.zeros((n, L, F))
    m = np.zeros((n, L, F)) if with_mags else None
    _check(lib.oracle_linear_fwd(d, L, F, _ptr(r), int(log2T), level_mask & 0xffffffff, _ptr(tb), n,
                                 _ptr(coords), _ptr(g), _ptr(m), nthreads or default_threads()), "linear_fwd")
    return (g, m) if with_mags else g


def linear_bwd_levels(d: int, F: int, res, log2T: int, coords: np.ndarray, g_gamma: np.ndarray,
                      levels=None, with_mags: bool = True, nthreads: int | None = None):
    """d-linear backward for the listed levels: {level: (grad [T][F], mag)}."""
    from concurrent.futures import ThreadPoolExecutor
    lib = _load()
    L = len(res)
    levels = list(range(L)) if levels is None else list(levels)
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    gg = np.ascontiguousarray(g_gamma, np.float32)
    out = {l: (np.zeros((1 << int(log2T), F)), np.zeros((1 << int(log2T), F)) if with_mags else None) for l in levels}

    def one(l):
        g, m = out[l]
        return lib.oracle_linear_bwd_level(d, L, F, l, _ptr(r), int(log2T), n, _ptr(coords), _ptr(gg), _ptr(g),
                                           _ptr(m))

    with ThreadPoolExecutor(max_workers=max(1, min(len(levels) or 1, nthreads or default_threads()))) as ex:
        for rc in ex.map(one, levels):
            _check(rc, "linear_bwd")
    return out


def linear_bwd(d: int, F: int, res, log2T: int, coords: np.ndarray, g_gamma: np.ndarray,
               level_mask: int | None = None, with_mags: bool = True, nthreads: int | None = None):
    """d-linear backward over all levels: fp64 grad [L][T][F] (and magnitude)."""
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    active = [l for l in range(L) if (level_mask >> l) & 1]
    per = linear_bwd_levels(d, F, res, log2T, coords, g_gamma, active, with_mags, nthreads)
    grad = np.zeros((L, 1 << int(log2T), F))
    mag = np.zeros_like(grad) if with_mags else None
    for l, (g, m) in per.items():
        grad[l] = g
        if with_mags:
            mag[l] = m
    return (grad, mag) if with_mags else grad


# ---------------------------------------------------------------------------
# INGP-FD: d-linear encoding with central finite differences
# ---------------------------------------------------------------------------

def linear_fd_fwd(d: int, F: int, res, log2T: int, table: np.ndarray, coords: np.ndarray, eps: float,
                  level_mask: int | None = None, nthreads: int | None = None, with_mags: bool = True):
    """INGP-FD forward: point-major fp64 gamma [N][L][F] at x, central-difference
    dgamma [N][d][L][F] and lap [N][L][F], and the stencil encodings
    [N][2d][L][F] (j = 2i: x + eps e_i, j = 2i+1: x - eps e_i), from the
    d-linear table [L][T][F]; eps is taken as float32 (the shift is one fp32 add)."""
    lib = _load()
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    tb = np.ascontiguousarray(table, np.float64)
    if tb.shape != (L, 1 << int(log2T), F):
        raise ValueError("linear table must be [L][T][F]")
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    out = {"gamma": np.zeros((n, L, F)), "dgamma": np.zeros((n, d, L, F)), "lap": np.zeros((n, L, F)),
           "stencil": np.zeros((n, 2 * d, L, F))}
    if with_mags:
        out.update({"m" + k: np.zeros_like(v) for k, v in list(out.items())})
    _check(lib.oracle_linear_fd_fwd(d, L, F, _ptr(r), int(log2T), level_mask & 0xffffffff, _ptr(tb), n, _ptr(coords),
                                    float(np.float32(eps)), _ptr(out["gamma"]), _ptr(out["dgamma"]),
                                    _ptr(out["lap"]), _ptr(out["stencil"]), _ptr(out.get("mgamma")),
                                    _ptr(out.get("mdgamma")), _ptr(out.get("mlap")), _ptr(out.get("mstencil")),
                                    nthreads or default_threads()), "linear_fd_fwd")
    return out


def linear_fd_bwd(d: int, F: int, res, log2T: int, coords: np.ndarray, eps: float, g_gamma=None, g_dgamma=None,
                  g_lap=None, g_stencil=None, level_mask: int | None = None, levels=None, with_mags: bool = True,
                  nthreads: int | None = None):
    """Backward of :func:`linear_fd_fwd` (float32 point-major upstream; any may
    be None): fp64 grad [L][T][F] and magnitude; levels outside ``levels`` /
    the mask stay zero."""
    from concurrent.futures import ThreadPoolExecutor
    lib = _load()
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    todo = [l for l in (range(L) if levels is None else levels) if (level_mask >> l) & 1]
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    f32 = lambda a: None if a is None else np.ascontiguousarray(a, np.float32)
    gg, gd, gl, gs = f32(g_gamma), f32(g_dgamma), f32(g_lap), f32(g_stencil)
    grad = np.zeros((L, 1 << int(log2T), F))
    mag = np.zeros_like(grad) if with_mags else None

    def one(l):
        return lib.oracle_linear_fd_bwd_level(d, L, F, l, _ptr(r), int(log2T), n, _ptr(coords),
                                              float(np.float32(eps)), _ptr(gg), _ptr(gd), _ptr(gl), _ptr(gs),
                                              _ptr(grad[l]), _ptr(mag[l]) if with_mags else None)

    with ThreadPoolExecutor(max_workers=max(1, min(len(todo) or 1, nthreads or default_threads()))) as ex:
        for rc in ex.map(one, todo):
            _check(rc, "linear_fd_bwd")
    return (grad, mag) if with_mags else grad


# ---------------------------------------------------------------------------
# Gaussian-RBF multi-resolution grid (DInf-Grid)
# ---------------------------------------------------------------------------

def rbf_fwd(d: int, F: int, res, log2T: int, table: np.ndarray, coords: np.ndarray, eps: float, rings: int,
            level_mask: int | None = None, nthreads: int | None = None, with_mags: bool = True):
    """Gaussian-RBF interpolation over the ring neighbourhood (distances in grid
    units): point-major fp64 gamma [N][L][F], dgamma [N][d][L][F], lap [N][L][F]
    (+ magnitudes) from the table [L][T][F]."""
    lib = _load()
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    tb = np.ascontiguousarray(table, np.float64)
    if tb.shape != (L, 1 << int(log2T), F):
        raise ValueError("RBF table must be [L][T][F]")
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    out = {"gamma": np.zeros((n, L, F)), "dgamma": np.zeros((n, d, L, F)), "lap": np.zeros((n, L, F))}
    if with_mags:
        out.update({"m" + k: np.zeros_like(v) for k, v in list(out.items())})
    _check(lib.oracle_rbf_fwd(d, L, F, _ptr(r), int(log2T), level_mask & 0xffffffff, _ptr(tb), n, _ptr(coords),
                              float(np.float32(eps)), int(rings), _ptr(out["gamma"]), _ptr(out["dgamma"]),
                              _ptr(out["lap"]), _ptr(out.get("mgamma")), _ptr(out.get("mdgamma")),
                              _ptr(out.get("mlap")), nthreads or default_threads()), "rbf_fwd")
    return out


def rbf_bwd(d: int, F: int, res, log2T: int, coords: np.ndarray, eps: float, rings: int, g_gamma=None,
            g_dgamma=None, g_lap=None, level_mask: int | None = None, levels=None, with_mags: bool = True,
            nthreads: int | None = None):
    """Backward of :func:`rbf_fwd` (float32 point-major upstream, any may be
    None): fp64 grad [L][T][F] and magnitude."""
    from concurrent.futures import ThreadPoolExecutor
    lib = _load()
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    todo = [l for l in (range(L) if levels is None else levels) if (level_mask >> l) & 1]
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    f32 = lambda a: None if a is None else np.ascontiguousarray(a, np.float32)
    gg, gd, gl = f32(g_gamma), f32(g_dgamma), f32(g_lap)
    grad = np.zeros((L, 1 << int(log2T), F))
    mag = np.zeros_like(grad) if with_mags else None

    def one(l):
        return lib.oracle_rbf_bwd_level(d, L, F, l, _ptr(r), int(log2T), n, _ptr(coords), float(np.float32(eps)),
                                        int(rings), _ptr(gg), _ptr(gd), _ptr(gl), _ptr(grad[l]),
                                        _ptr(mag[l]) if with_mags else None)

    with ThreadPoolExecutor(max_workers=max(1, min(len(todo) or 1, nthreads or default_threads()))) as ex:
        for rc in ex.map(one, todo):
            _check(rc, "rbf_bwd")
    return (grad, mag) if with_mags else grad


# ---------------------------------------------------------------------------
# full Hessian (upper triangle, row-major: 2D xx, xy, yy; 3D xx, xy, xz, yy, yz, zz)
# ---------------------------------------------------------------------------

def hess_entries(d: int) -> int:
    return int(_load().oracle_hess_entries(d))


def hess_pairs(d: int) -> list[tuple[int, int]]:
    """(i, j) of each Hessian entry, in storage order."""
    return [(i, j) for i in range(d) for j in range(i, d)]


def eval_cell_hessian(d: int, F: int, N: int, log2T, level_tables, c, t):
    """One cell at an fp64 local coordinate: (gamma[F], dgamma[d][F], hess[P][F])."""
    lib = _load()
    tabs = [np.ascontiguousarray(a, dtype=np.float64) for a in level_tables]
    lt = np.asarray(log2T, np.int32)
    cc = np.asarray(c, np.int64)
    tt = np.asarray(t, np.float64)
    P = hess_entries(d)
    g, dg, h = np.zeros(F), np.zeros((d, F)), np.zeros((P, F))
    _check(lib.oracle_eval_cell_hessian(d, F, int(N), _ptr(lt), _ptr_array(tabs), _ptr(cc), _ptr(tt), _ptr(g),
                                        _ptr(dg), _ptr(h)), "eval_cell_hessian")
    return g, dg, h


def encode_fwd_hessian(d: int, F: int, res, log2T, tables, coords: np.ndarray, level_mask: int | None = None,
                       nthreads: int | None = None, with_mags: bool = True):
    """Hermite forward with the full Hessian: point-major fp64 gamma [N][L][F],
    dgamma [N][d][L][F], hess [N][P][L][F] (+ magnitudes mgamma, mdgamma, mhess)."""
    lib = _load()
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    tabs = _as_f64_tables(tables)
    for k, tb in enumerate(tabs):
        if tb.shape != (L, 1 << int(log2T[k]), comb(d, k), F):
            raise ValueError(f"order table {k} has shape {tb.shape}")
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    P = hess_entries(d)
    r = np.asarray(res, np.int32)
    lt = np.asarray(log2T, np.int32)
    out = {"gamma": np.zeros((n, L, F)), "dgamma": np.zeros((n, d, L, F)), "hess": np.zeros((n, P, L, F))}
    if with_mags:
        out.update(mgamma=np.zeros((n, L, F)), mdgamma=np.zeros((n, d, L, F)), mhess=np.zeros((n, P, L, F)))
    _check(lib.oracle_encode_fwd_hessian(d, L, F, _ptr(r), _ptr(lt), level_mask & 0xffffffff, _ptr_array(tabs), n,
                                         _ptr(coords), _ptr(out["gamma"]), _ptr(out["dgamma"]), _ptr(out["hess"]),
                                         _ptr(out.get("mgamma")), _ptr(out.get("mdgamma")), _ptr(out.get("mhess")),
                                         nthreads or default_threads()), "encode_fwd_hessian")
    return out


def encode_bwd_hessian(d: int, F: int, res, log2T, coords: np.ndarray, g_gamma=None, g_dgamma=None, g_hess=None,
                       level_mask: int | None = None, levels=None, with_mags: bool = True,
                       nthreads: int | None = None):
    """Backward of :func:`encode_fwd_hessian` (float32 upstream, point-major;
    any may be None): (grads, mags) lists over order k of fp64
    [L][T_k][C(d,k)][F]; levels outside ``levels`` / the mask stay zero."""
    from concurrent.futures import ThreadPoolExecutor
    lib = _load()
    L = len(res)
    if level_mask is None:
        level_mask = (1 << L) - 1
    todo = [l for l in (range(L) if levels is None else levels) if (level_mask >> l) & 1]
    coords = np.ascontiguousarray(coords, np.float32)
    n = coords.shape[0]
    r = np.asarray(res, np.int32)
    lt = np.asarray(log2T, np.int32)
    f32 = lambda a: None if a is None else np.ascontiguousarray(a, np.float32)
    gg, gd, gh = f32(g_gamma), f32(g_dgamma), f32(g_hess)
    shapes = order_table_shapes(d, L, F, log2T)
    grads = [np.zeros(s) for s in shapes]
    mags = [np.zeros(s) for s in shapes] if with_mags else None

    def one(l):
        gs = _ptr_array([g[l] for g in grads])
        ms = _ptr_array([m[l] for m in mags]) if with_mags else None
        return lib.oracle_encode_bwd_hessian_level(d, L, F, l, _ptr(r), _ptr(lt), n, _ptr(coords), _ptr(gg),
                                                   _ptr(gd), _ptr(gh), gs, ms)

    with ThreadPoolExecutor(max_workers=max(1, min(len(todo) or 1, nthreads or default_threads()))) as ex:
        for rc in ex.map(one, todo):
            _check(rc, "encode_bwd_hessian")
    return grads, mags


# The SIREN consumer (numpy fp64).  HG_SIREN_ORACLE names a copy of siren.py with a
# planted mistake (tests/test_oracle_siren_mutants.py), as HG_ORACLE_LIB does for the C part.
if os.environ.get("HG_SIREN_ORACLE"):
    import importlib.util as _ilu

    _spec = _ilu.spec_from_file_location("oracle_siren_variant", os.environ["HG_SIREN_ORACLE"])
    _siren = _ilu.module_from_spec(_spec)
    _spec.loader.exec_module(_siren)
    siren_fwd, siren_bwd = _siren.siren_fwd, _siren.siren_bwd
else:
    from .siren import siren_bwd, siren_fwd  # noqa: E402,F401
