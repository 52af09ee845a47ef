"""Full-size GPU parity: the workloads at their published sizes, run exactly as
the benchmark launches them (packed table, feature-major outputs, every level
or the coarse-to-fine active-level masks), checked against the oracle on
every point and every level.

Forward: every output of every point at every level is compared.  The oracle
is called one level at a time on chunks of points (a one-level grid with
that level's explicit resolution and tables, widened to fp64 level by
level), which keeps host memory bounded and the oracle's table accesses
cache-local; its arithmetic is the same as a call over all levels.
Backward: every active level's whole gradient table is compared; the oracle
accumulates each level over all points (levels in parallel threads).  Inactive levels must be exactly zero.

Tolerance as in the small cases (1e-5 of the oracle's condition magnitude);
fp16 coefficients widen exactly, so the same bound applies to the fp16
workload.
"""
from math import comb

import numpy as np
import pytest

from _harness import check_close, host

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")

CHUNK = 1 << 20   # points per oracle forward call


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _mods():
    import multiresolution_hash_grid_02_b300 as m
    from multiresolution_hash_grid_02_b300 import hg, workloads as W
    import oracle
    return m, hg, W, oracle


# ---------------------------------------------------------------------------
# helpers: level slices of feature-major device outputs, per-level oracle calls
# ---------------------------------------------------------------------------

def _fm_level(t, l, has_axis):
    """Level l of a feature-major device output as host point-major:
    [L][F][n] -> [n][F]; [A][L][F][n] -> [n][A][F]."""
    if has_axis:
        return np.transpose(host(t[:, l]), (2, 0, 1))
    return host(t[l]).T


def _ref_level(a):
    """The single level of a one-level oracle output ([m][1][F] or [m][A][1][F])."""
    return a[:, 0] if a.ndim == 3 else a[:, :, 0]


def _level_orders(packed, d, l):
    """fp64 order tables [1][T][C(d,k)][F] of level l of an interleaved table."""
    _, _, W, _ = _mods()
    row = np.asarray(packed[l:l + 1], np.float64)
    return [np.ascontiguousarray(o) for o in W.split_orders(row, d)]


def _check_fwd_all_points(tag, n, levels, runs, oracle_level, keys):
    """Compare every point of every level.

    runs: [(label, mask, {key: (device tensor, has_axis)})] -- several GPU runs
    (e.g. the coarse-to-fine masks) against one oracle pass.
    oracle_level(l, lo, hi): one-level oracle outputs for points lo..hi.
    Inactive levels of a run must be exactly zero."""
    for l in levels:
        got = []
        for label, mask, outs in runs:
            if (mask >> l) & 1:
                got.append((label, {k: _fm_level(t, l, ax) for k, (t, ax) in outs.items()}))
            else:
                for k, (t, ax) in outs.items():
                    sl = t[:, l] if ax else t[l]
                    assert float(sl.abs().max()) == 0.0, f"{tag}{label}: inactive level {l} {k} not zero"
        if not got:
            continue
        for lo in range(0, n, CHUNK):
            hi = min(n, lo + CHUNK)
            ref = oracle_level(l, lo, hi)
            for label, outs in got:
                for k in keys:
                    check_close(f"{tag}{label} {k} level {l} points {lo}..{hi}", outs[k][lo:hi],
                                _ref_level(ref[k]), _ref_level(ref["m" + k]))


def _hermite_oracle_level(w, inp, res, hessian=False):
    m, hg, W, oracle = _mods()
    cache = {}

    def call(l, lo, hi):
        if cache.get("l") != l:
            cache.clear()
            cache["l"], cache["tabs"] = l, _level_orders(inp["table"], w.d, l)
        f = oracle.encode_fwd_hessian if hessian else oracle.encode_fwd
        return f(w.d, w.F, [res[l]], w.log2_T, cache["tabs"], inp["coords"][lo:hi])
    return call


def _hermite_desc(w, mask):
    m, hg, W, oracle = _mods()
    return m.GridDesc(d=w.d, L=w.L, F=w.F, n_min=w.n_min, n_max=w.n_max, log2_T=w.log2_T, level_mask=mask,
                      dtype=m.HG_F16 if w.dtype == "f16" else m.HG_F32, layout=m.HG_FEATURE_MAJOR)


def _run_hermite(w, dev_in, mask):
    """GPU forward + backward in the benchmark's launch configuration; the
    device inputs (coords, table, feature-major upstream) stay with the caller."""
    m, hg, W, oracle = _mods()
    n, d, L, F = w.n_points, w.d, w.L, w.F
    desc = _hermite_desc(w, mask)
    gamma = torch.full((L, F, n), float("nan"), device="cuda")
    dgamma = torch.full((d, L, F, n), float("nan"), device="cuda")
    lap = torch.full((L, F, n), float("nan"), device="cuda")
    hg.hg_encode_fwd(desc, n, dev_in["coords"], m.packed_views(dev_in["table"], d), gamma, dgamma, lap)
    grad = torch.zeros(dev_in["table"].shape, dtype=torch.float32, device="cuda")
    hg.hg_encode_bwd(desc, n, dev_in["coords"], dev_in["gg"], dev_in["gd"], dev_in["gl"], m.packed_views(grad, d))
    torch.cuda.synchronize()
    return {"gamma": (gamma, False), "dgamma": (dgamma, True), "lap": (lap, False)}, grad


def _hermite_device_inputs(w, inp):
    m, hg, W, oracle = _mods()
    return {"coords": torch.from_numpy(inp["coords"]).cuda(), "table": torch.from_numpy(inp["table"]).cuda(),
            "gg": torch.from_numpy(W.to_feature_major(inp["g_gamma"], False)).cuda(),
            "gd": torch.from_numpy(W.to_feature_major(inp["g_dgamma"], True)).cuda(),
            "gl": torch.from_numpy(W.to_feature_major(inp["g_lap"], False)).cuda()}


def _check_hermite_bwd_all_levels(tag, w, inp, res, grads_by_run, group, bwd=None):
    """Every active level of every run's packed gradient table against the
    oracle's level gradient (computed once per level, `group` levels at a time).
    grads_by_run: [(label, mask, device grad [L][T][2^d][F])]."""
    m, hg, W, oracle = _mods()
    d, F, T = w.d, w.F, 1 << w.log2_T[0]
    todo = [l for l in range(w.L) if any((mask >> l) & 1 for _, mask, _ in grads_by_run)]
    for label, mask, grad in grads_by_run:
        for l in range(w.L):
            if not (mask >> l) & 1:
                assert float(grad[l].abs().max()) == 0.0, f"{tag}{label}: inactive level {l} has gradients"
    for i in range(0, len(todo), group):
        levels = todo[i:i + group]
        if bwd is None:
            want = oracle.encode_bwd_levels(d, F, res, w.log2_T, inp["coords"], inp["g_gamma"], inp["g_dgamma"],
                                            inp["g_lap"], levels=levels)
        else:
            want = bwd(levels)
        for l in levels:
            gk, mk = want[l]
            for label, mask, grad in grads_by_run:
                if not (mask >> l) & 1:
                    continue
                got = W.split_orders(host(grad[l]).reshape(1, T, 1 << d, F), d)
                for k in range(d + 1):
                    check_close(f"{tag}{label} grad level {l} order {k}", got[k][0], gk[k], mk[k])
        del want


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def workload4():
    m, hg, W, oracle = _mods()
    return W.WORKLOADS[4], W.make(W.WORKLOADS[4])


def test_fullsize_2d_linear_ingp():
    """The d-linear Instant-NGP workload (2^20 points, 16 levels, T = 2^19):
    every point forward, the whole gradient table backward."""
    m, hg, W, oracle = _mods()
    w = W.WORKLOADS[2]
    inp = W.make(w)
    n, d, L, F = w.n_points, w.d, w.L, w.F
    res = oracle.level_resolutions(L, w.n_min, w.n_max)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=w.n_min, n_max=w.n_max, log2_T=w.log2_T * 3, layout=m.HG_FEATURE_MAJOR)
    coords = torch.from_numpy(inp["coords"]).cuda()
    table = torch.from_numpy(inp["table"]).cuda()
    gamma = torch.full((L, F, n), float("nan"), device="cuda")
    hg.hg_linear_fwd(desc, n, coords, m.linear_view(table), gamma)
    grad = torch.zeros_like(table)
    hg.hg_linear_bwd(desc, n, coords, torch.from_numpy(W.to_feature_major(inp["g_gamma"], False)).cuda(),
                     m.linear_view(grad))
    torch.cuda.synchronize()

    def level(l, lo, hi):
        g, mg = oracle.linear_fwd(d, F, [res[l]], w.log2_T[0], np.asarray(inp["table"][l:l + 1], np.float64),
                                  inp["coords"][lo:hi])
        return {"gamma": g, "mgamma": mg}

    _check_fwd_all_points("", n, range(L), [("", (1 << L) - 1, {"gamma": (gamma, False)})], level, ("gamma",))
    gw, gm = oracle.linear_bwd(d, F, res, w.log2_T[0], inp["coords"], inp["g_gamma"])
    check_close("linear grad", host(grad), gw, gm)


@pytest.mark.parametrize("cfg", [3, 10], ids=["stratum_order", "shuffled"])
def test_fullsize_2d_hermite_pinn(cfg):
    """The PINN-sized 2D Hermite workload (2^20 stratified points, 16
    levels, 14 one-to-one), in stratum order (consecutive points share cells:
    the backward sums their runs in the warp) and shuffled (no runs): every
    point and level forward, every level backward."""
    m, hg, W, oracle = _mods()
    w = W.WORKLOADS[cfg]
    inp = W.make(w)
    res = oracle.level_resolutions(w.L, w.n_min, w.n_max)
    full = (1 << w.L) - 1
    outs, grad = _run_hermite(w, _hermite_device_inputs(w, inp), full)
    _check_fwd_all_points("", w.n_points, range(w.L), [("", full, outs)], _hermite_oracle_level(w, inp, res),
                          ("gamma", "dgamma", "lap"))
    _check_hermite_bwd_all_levels("", w, inp, res, [("", full, grad)], group=16)


def test_fullsize_3d_hermite(workload4):
    """The 3D Hermite workload of the headline (2^21 points, 16 levels,
    levels 0-6 one-to-one, 7-15 hashed): every point and level forward,
    every level backward."""
    w, inp = workload4
    m, hg, W, oracle = _mods()
    res = oracle.level_resolutions(w.L, w.n_min, w.n_max)
    full = (1 << w.L) - 1
    dev_in = _hermite_device_inputs(w, inp)
    outs, grad = _run_hermite(w, dev_in, full)
    del dev_in
    _check_fwd_all_points("", w.n_points, range(w.L), [("", full, outs)], _hermite_oracle_level(w, inp, res),
                          ("gamma", "dgamma", "lap"))
    del outs
    _check_hermite_bwd_all_levels("", w, inp, res, [("", full, grad)], group=16)


def test_fullsize_3d_hermite_fp16_coarse_to_fine():
    """The large fp16 workload (2^23 points, 16 levels, T = 2^22) at the three
    coarse-to-fine masks L_active = 4, 10, 16: every point and active level
    forward and every active level backward of each run, against one oracle
    pass; inactive levels exactly zero."""
    m, hg, W, oracle = _mods()
    w = W.WORKLOADS[5]
    inp = W.make(w)
    res = oracle.level_resolutions(w.L, w.n_min, w.n_max)
    dev_in = _hermite_device_inputs(w, inp)
    runs, grads = [], []
    for active in (4, 10, 16):
        mask = (1 << active) - 1
        outs, grad = _run_hermite(w, dev_in, mask)
        runs.append((f" L_active={active}", mask, outs))
        grads.append((f" L_active={active}", mask, grad))
    del dev_in
    _check_fwd_all_points("", w.n_points, range(w.L), runs, _hermite_oracle_level(w, inp, res),
                          ("gamma", "dgamma", "lap"))
    del runs
    # 1 GB of oracle gradient and magnitude per level, all levels in parallel threads
    _check_hermite_bwd_all_levels("", w, inp, res, grads, group=16)


def test_fullsize_3d_hermite_hessian(workload4):
    """The full-Hessian forward and backward on the 3D workload (2^21 points,
    16 levels), packed table, feature-major outputs: every point and level
    forward, every level backward."""
    w, inp = workload4
    m, hg, W, oracle = _mods()
    n, d, L, F = w.n_points, w.d, w.L, w.F
    P = d * (d + 1) // 2
    res = oracle.level_resolutions(L, w.n_min, w.n_max)
    desc = _hermite_desc(w, (1 << L) - 1)
    coords = torch.from_numpy(inp["coords"]).cuda()
    table = torch.from_numpy(inp["table"]).cuda()
    gamma = torch.full((L, F, n), float("nan"), device="cuda")
    dgamma = torch.full((d, L, F, n), float("nan"), device="cuda")
    hess = torch.full((P, L, F, n), float("nan"), device="cuda")
    hg.hg_encode_fwd_hessian(desc, n, coords, m.packed_views(table, d), gamma, dgamma, hess)
    gh = W.draw_upstream_hessian(np.random.default_rng(61), w)
    grad = torch.zeros(table.shape, dtype=torch.float32, device="cuda")
    up = [torch.from_numpy(W.to_feature_major(a, ax)).cuda()
          for a, ax in ((inp["g_gamma"], False), (inp["g_dgamma"], True), (gh, True))]
    hg.hg_encode_bwd_hessian(desc, n, coords, up[0], up[1], up[2], m.packed_views(grad, d))
    torch.cuda.synchronize()
    del up, table
    outs = {"gamma": (gamma, False), "dgamma": (dgamma, True), "hess": (hess, True)}
    _check_fwd_all_points("", n, range(L), [("", (1 << L) - 1, outs)], _hermite_oracle_level(w, inp, res, True),
                          ("gamma", "dgamma", "hess"))
    del outs, gamma, dgamma, hess

    def bwd(levels):
        grads, mags = oracle.encode_bwd_hessian(d, F, res, w.log2_T, inp["coords"], inp["g_gamma"], inp["g_dgamma"],
                                                gh, levels=levels)
        return {l: ([g[l] for g in grads], [mm[l] for mm in mags]) for l in levels}

    _check_hermite_bwd_all_levels("hessian", w, inp, res, [("", (1 << L) - 1, grad)], group=16, bwd=bwd)


def test_fullsize_4d_hermite_spacetime():
    """The 4D space-time workload (2^20 points, 16 levels, 128-byte packed
    rows): lane-quad forward and lane-octet backward, benchmark launch
    configuration; dense levels 0-2 and hashed levels above; every point and
    level forward, every level backward."""
    m, hg, W, oracle = _mods()
    w = W.WORKLOADS[6]
    inp = W.make(w)
    res = oracle.level_resolutions(w.L, w.n_min, w.n_max)
    full = (1 << w.L) - 1
    dev_in = _hermite_device_inputs(w, inp)
    outs, grad = _run_hermite(w, dev_in, full)
    del dev_in
    _check_fwd_all_points("", w.n_points, range(w.L), [("", full, outs)], _hermite_oracle_level(w, inp, res),
                          ("gamma", "dgamma", "lap"))
    del outs
    _check_hermite_bwd_all_levels("", w, inp, res, [("", full, grad)], group=16)


def test_fullsize_3d_linear_fd():
    """INGP-FD on the 3D grid (2^21 points, 16 levels, T = 2^19): gamma and
    the six stencil encodings forward, their upstream backward, as the
    benchmark launches them; every point and level forward, every level
    backward (levels 0-6 one-to-one and privatised or direct, 7-15 hashed)."""
    m, hg, W, oracle = _mods()
    w = W.WORKLOADS[7]
    inp = W.make(w)
    n, d, L, F = w.n_points, w.d, w.L, w.F
    res = oracle.level_resolutions(L, w.n_min, w.n_max)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=w.n_min, n_max=w.n_max, log2_T=w.log2_T * (d + 1),
                      layout=m.HG_FEATURE_MAJOR)
    coords = torch.from_numpy(inp["coords"]).cuda()
    table = torch.from_numpy(inp["table"]).cuda()
    gamma = torch.full((L, F, n), float("nan"), device="cuda")
    stencil = torch.full((2 * d, L, F, n), float("nan"), device="cuda")
    hg.hg_linear_fd_fwd(desc, n, coords, w.eps, m.linear_view(table), gamma, None, None, stencil)
    grad = torch.zeros_like(table)
    hg.hg_linear_fd_bwd(desc, n, coords, w.eps, torch.from_numpy(W.to_feature_major(inp["g_gamma"], False)).cuda(),
                        None, None, torch.from_numpy(W.to_feature_major(inp["g_stencil"], True)).cuda(),
                        m.linear_view(grad))
    torch.cuda.synchronize()

    def level(l, lo, hi):
        return oracle.linear_fd_fwd(d, F, [res[l]], w.log2_T[0], np.asarray(inp["table"][l:l + 1], np.float64),
                                    inp["coords"][lo:hi], w.eps)

    _check_fwd_all_points("", n, range(L), [("", (1 << L) - 1, {"gamma": (gamma, False), "stencil": (stencil, True)})],
                          level, ("gamma", "stencil"))
    want, mag = oracle.linear_fd_bwd(d, F, res, w.log2_T[0], inp["coords"], w.eps, g_gamma=inp["g_gamma"],
                                     g_stencil=inp["g_stencil"])
    got = host(grad)
    for l in range(L):
        check_close(f"grad level {l}", got[l], want[l], mag[l])


@pytest.mark.parametrize("cfg", [8, 9])
def test_fullsize_dinf_rbf(cfg):
    """The DInf-Grid Gaussian-RBF workloads (2D: 2^20 stratified points, 4
    dense levels up to 512; 3D: 2^21 points, up to 56; eps = 1, 3 rings) as
    the benchmark launches them: every point and level forward, every level
    backward (the coarsest privatised, the finest direct)."""
    m, hg, W, oracle = _mods()
    w = W.WORKLOADS[cfg]
    inp = W.make(w)
    n, d, L, F = w.n_points, w.d, w.L, w.F
    res = oracle.level_resolutions(L, w.n_min, w.n_max)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=w.n_min, n_max=w.n_max, log2_T=w.log2_T * (d + 1),
                      layout=m.HG_FEATURE_MAJOR)
    coords = torch.from_numpy(inp["coords"]).cuda()
    table = torch.from_numpy(inp["table"]).cuda()
    gamma = torch.full((L, F, n), float("nan"), device="cuda")
    dgamma = torch.full((d, L, F, n), float("nan"), device="cuda")
    lap = torch.full((L, F, n), float("nan"), device="cuda")
    hg.hg_rbf_fwd(desc, n, coords, w.eps, w.rings, m.linear_view(table), gamma, dgamma, lap)
    grad = torch.zeros_like(table)
    up = [torch.from_numpy(W.to_feature_major(inp[k], k == "g_dgamma")).cuda() for k in ("g_gamma", "g_dgamma", "g_lap")]
    hg.hg_rbf_bwd(desc, n, coords, w.eps, w.rings, up[0], up[1], up[2], m.linear_view(grad))
    torch.cuda.synchronize()
    del up

    def level(l, lo, hi):
        return oracle.rbf_fwd(d, F, [res[l]], w.log2_T[0], np.asarray(inp["table"][l:l + 1], np.float64),
                              inp["coords"][lo:hi], w.eps, w.rings)

    outs = {"gamma": (gamma, False), "dgamma": (dgamma, True), "lap": (lap, False)}
    _check_fwd_all_points("", n, range(L), [("", (1 << L) - 1, outs)], level, ("gamma", "dgamma", "lap"))
    want, mag = oracle.rbf_bwd(d, F, res, w.log2_T[0], inp["coords"], w.eps, w.rings, g_gamma=inp["g_gamma"],
                               g_dgamma=inp["g_dgamma"], g_lap=inp["g_lap"])
    got = host(grad)
    for l in range(L):
        check_close(f"grad level {l}", got[l], want[l], mag[l])


def test_fullsize_siren_consumer():
    """The SIREN consumer in the benchmark's launch configuration: 2^21
    points, d = 3, K = L F = 32, H = 64, O = 1, omega = 30, inputs in the
    encoder's feature-major layout.  Every point's outputs (u, grad u, lap u
    and the input gradients) to 1e-5 of the oracle's magnitude; the weight
    gradients whole, against the oracle summed over chunks of points.  Those
    are sums over 2^21 points: a CTA accumulates its ~221 tiles in shared
    memory (about 8 adds per tile for the output-layer and bias gradients) and
    adds once to global memory, up to ~1900 fp32 roundings in a row, whose
    worst-case bound is ~1.1e-4 of the magnitude -- the test takes 2e-4 (the
    errors seen are far smaller)."""
    m, hg, W, oracle = _mods()
    n, d, L, F = 1 << 21, 3, 16, 2
    K, H, O = L * F, W.SIREN_H, W.SIREN_O
    rng = np.random.default_rng(44)
    f32 = np.float32
    feats = {"gamma": (rng.uniform(-1, 1, (n, K)) * 0.5).astype(f32),
             "dgamma": rng.normal(0, 5, (n, d, K)).astype(f32),
             "lap": rng.normal(0, 100, (n, K)).astype(f32)}
    sw, sup = W.siren_weights(rng, K, H, O), W.siren_upstream(rng, n, d, O)
    desc = m.SirenDesc(d=d, K=K, H=H, O=O, omega=W.SIREN_OMEGA)

    def fm(a):
        return torch.from_numpy(np.ascontiguousarray(np.moveaxis(a, 0, -1))).cuda()

    fin = [fm(feats[k]) for k in ("gamma", "dgamma", "lap")]
    wts = [torch.from_numpy(sw[k]).cuda() for k in ("W1", "b1", "W2", "b2")]
    ups = [fm(sup[k]) for k in ("g_u", "g_du", "g_lapu")]
    u, du, lu = (torch.full(sh, float("nan"), device="cuda") for sh in ((O, n), (d, O, n), (O, n)))
    hg.hg_siren_fwd(desc, n, *fin, *wts, u, du, lu)
    gin = [torch.full_like(t, float("nan")) for t in fin]
    wg = [torch.zeros(sh, device="cuda") for sh in ((H, K), (H,), (O, H), (O,))]
    hg.hg_siren_bwd(desc, n, *fin, *wts[:3], *ups, *gin, *wg)
    torch.cuda.synchronize()
    del fin, ups
    outs = {name: np.moveaxis(host(t), -1, 0) for name, t in (("u", u), ("du", du), ("lapu", lu))}
    gins = {name: np.moveaxis(host(t), -1, 0) for name, t in (("g_gamma", gin[0]), ("g_dgamma", gin[1]),
                                                              ("g_lap", gin[2]))}
    keys = ("gW1", "gb1", "gW2", "gb2")
    tot = {k: 0.0 for k in keys}
    mag = {k: 0.0 for k in keys}
    step = 1 << 17
    for lo in range(0, n, step):
        hi = lo + step
        sub = {k: v[lo:hi] for k, v in feats.items()}
        ref = oracle.siren_fwd(omega=W.SIREN_OMEGA, **sub, **sw)
        for name in ("u", "du", "lapu"):
            check_close(f"{name} points {lo}..{hi}", outs[name][lo:hi], ref[name], ref["m" + name])
        r = oracle.siren_bwd(omega=W.SIREN_OMEGA, **sub, **sw, **{k: v[lo:hi] for k, v in sup.items()})
        for name in ("g_gamma", "g_dgamma", "g_lap"):
            check_close(f"{name} points {lo}..{hi}", gins[name][lo:hi], r[name], r["m" + name])
        for k in keys:
            tot[k] = tot[k] + r[k]
            mag[k] = mag[k] + r["m" + k]
    for k, t in zip(keys, wg):
        check_close(k, host(t), tot[k], mag[k], rtol=2e-4)


def test_fullsize_fused_encoder_siren_pinn():
    """The fused encoder + SIREN forward on the PINN workload (2^20
    stratified points, 2D, 16 levels, T = 2^19, fp32; SIREN K = 32, H = 64,
    O = 1, omega = 30 with the benchmark's seeded weights): every point's u,
    grad u and lap u against the oracle's encoding followed by its SIREN (the
    encoder's magnitudes carried into the SIREN's), and bit for bit against
    the unfused chain on the GPU (encoder outputs through memory, then the
    SIREN)."""
    m, hg, W, oracle = _mods()
    w = W.WORKLOADS[3]
    inp = W.make(w)
    n, d, L, F = w.n_points, w.d, w.L, w.F
    K, H, O = L * F, W.SIREN_H, W.SIREN_O
    sw = W.siren_weights(np.random.default_rng(w.seed + 2000), K, H, O)
    res = oracle.level_resolutions(L, w.n_min, w.n_max)
    desc = _hermite_desc(w, (1 << L) - 1)
    sdesc = m.SirenDesc(d=d, K=K, H=H, O=O, omega=W.SIREN_OMEGA)
    coords = torch.from_numpy(inp["coords"]).cuda()
    table = torch.from_numpy(inp["table"]).cuda()
    wts = [torch.from_numpy(sw[k]).cuda() for k in ("W1", "b1", "W2", "b2")]
    u, du, lu = (torch.full(sh, float("nan"), device="cuda") for sh in ((O, n), (d, O, n), (O, n)))
    hg.hg_encode_siren_fwd(desc, n, coords, m.packed_views(table, d), sdesc, *wts, u, du, lu)
    g = torch.empty((L, F, n), device="cuda")
    dg = torch.empty((d, L, F, n), device="cuda")
    lp = torch.empty((L, F, n), device="cuda")
    hg.hg_encode_fwd(desc, n, coords, m.packed_views(table, d), g, dg, lp)
    u2, du2, lu2 = (torch.full(sh, float("nan"), device="cuda") for sh in ((O, n), (d, O, n), (O, n)))
    hg.hg_siren_fwd(sdesc, n, g, dg, lp, *wts, u2, du2, lu2)
    torch.cuda.synchronize()
    got = {k: np.moveaxis(host(t), -1, 0) for k, t in (("u", u), ("du", du), ("lapu", lu))}
    for a, b in ((u, u2), (du, du2), (lu, lu2)):
        assert np.array_equal(host(a), host(b))
    del g, dg, lp, u2, du2, lu2
    orders = [np.ascontiguousarray(o, np.float64) for o in W.split_orders(np.asarray(inp["table"], np.float64), d)]
    for lo in range(0, n, CHUNK // 4):
        hi = min(n, lo + CHUNK // 4)
        enc = oracle.encode_fwd(d, F, res, w.log2_T, orders, inp["coords"][lo:hi])
        m_ = hi - lo
        flat = {k: enc[k].reshape(m_, K) if k in ("gamma", "lap", "mgamma", "mlap") else enc[k].reshape(m_, d, K)
                for k in ("gamma", "dgamma", "lap", "mgamma", "mdgamma", "mlap")}
        ref = oracle.siren_fwd(flat["gamma"], flat["dgamma"], flat["lap"], sw["W1"], sw["b1"], sw["W2"], sw["b2"],
                               W.SIREN_OMEGA, mgamma=flat["mgamma"], mdgamma=flat["mdgamma"], mlap=flat["mlap"])
        for k in ("u", "du", "lapu"):
            check_close(f"{k} points {lo}..{hi}", got[k][lo:hi], ref[k], ref["m" + k])
