"""GPU parity of the SIREN chain-rule consumer (hg_siren_fwd / hg_siren_bwd:
"Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs", 整体框架
and 关键设计 2) against the oracle, element by element.

Cases: d = 1..4; K = 8..64; H = 16, 32, 64, 128 (1, 2, 4, 8 threads per
point, so 256 down to 32 points per tile); O = 1..4; omega = 30 (the page)
and others; several tiles with a ragged tail, and one point.  Tolerance: the
per-point outputs within 1e-5 of the oracle's first-order error magnitude
(omega times the magnitude of the sine's argument included).  The weight
gradients are sums over all points: an fp32 sum of m partial sums errs by at
most (m - 1) 2^-24 of its magnitude, and here m is about the number of
CTAs plus the adds inside a CTA (about 160 at these sizes), so they take 4e-5."""
import zlib

import numpy as np
import pytest

from _harness import check_close, dev, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

RTOL_W = 4e-5

# (id, d, K, H, O, n, omega)
CASES = [
    ("3d_K32_H64_workload_shape", 3, 32, 64, 1, 3000, 30.0),
    ("2d_K32_H32_O2", 2, 32, 32, 2, 1000, 30.0),
    ("1d_K8_H16_tp1", 1, 8, 16, 1, 700, 30.0),
    ("3d_K16_H128_O3", 3, 16, 128, 3, 500, 10.0),
    ("4d_K32_H64_O4", 4, 32, 64, 4, 900, 30.0),
    ("3d_K64_H64", 3, 64, 64, 1, 333, 1.0),
    ("2d_one_point", 2, 32, 64, 1, 1, 30.0),
    # the largest shape the ABI takes: the backward's tiles at their shared-memory peak (219 KB)
    ("4d_K64_H128_largest", 4, 64, 128, 1, 200, 30.0),
]


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _build(case, seed=0):
    import multiresolution_hash_grid_02_b300 as m
    import oracle
    cid, d, K, H, O, n, omega = case
    rng = np.random.default_rng(zlib.crc32(cid.encode()) + seed)
    f32 = np.float32
    inp = {"gamma": (rng.uniform(-1, 1, (n, K)) * 0.5).astype(f32),
           "dgamma": rng.normal(0, 5, (n, d, K)).astype(f32),
           "lap": rng.normal(0, 100, (n, K)).astype(f32),
           "W1": rng.uniform(-1 / K, 1 / K, (H, K)).astype(f32),
           "b1": rng.uniform(-1, 1, H).astype(f32) / np.sqrt(K).astype(f32),
           "W2": (rng.uniform(-1, 1, (O, H)) * np.sqrt(6 / H) / omega).astype(f32),
           "b2": rng.uniform(-0.1, 0.1, O).astype(f32)}
    up = {"g_u": rng.standard_normal((n, O)).astype(f32), "g_du": rng.standard_normal((n, d, O)).astype(f32),
          "g_lapu": rng.standard_normal((n, O)).astype(f32)}
    return m, oracle, m.SirenDesc(d=d, K=K, H=H, O=O, omega=omega), inp, up


def _fm(a):
    """Point-major [n][...] -> feature-major [...][n] (the encoder's layout)."""
    return np.ascontiguousarray(np.moveaxis(a, 0, -1))


def _pm(a):
    return np.moveaxis(a, -1, 0)


def _dev_inputs(inp):
    return [dev(_fm(inp[k])) for k in ("gamma", "dgamma", "lap")] + [dev(inp[k]) for k in ("W1", "b1", "W2", "b2")]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_siren_forward_parity(case):
    m, oracle, desc, inp, up = _build(case)
    n, d, O = inp["gamma"].shape[0], desc.d, desc.O
    g, dg, lp, W1, b1, W2, b2 = _dev_inputs(inp)
    u = torch.full((O, n), float("nan"), device="cuda")
    du = torch.full((d, O, n), float("nan"), device="cuda")
    lu = torch.full((O, n), float("nan"), device="cuda")
    m.hg.hg_siren_fwd(desc, n, g, dg, lp, W1, b1, W2, b2, u, du, lu)
    torch.cuda.synchronize()
    ref = oracle.siren_fwd(omega=desc.omega, **inp)
    check_close("u", _pm(host(u)), ref["u"], ref["mu"])
    check_close("du", _pm(host(du)), ref["du"], ref["mdu"])
    check_close("lapu", _pm(host(lu)), ref["lapu"], ref["mlapu"])
    # outputs not requested are not needed: u alone, without dgamma and lap
    u2 = torch.full((O, n), float("nan"), device="cuda")
    m.hg.hg_siren_fwd(desc, n, g, None, None, W1, b1, W2, b2, u2)
    torch.cuda.synchronize()
    assert np.array_equal(host(u2), host(u))


def _run_bwd(m, desc, inp, up, want=("g_gamma", "g_dgamma", "g_lap", "gW1", "gb1", "gW2", "gb2"), upstream=None):
    n, d, K, H, O = inp["gamma"].shape[0], desc.d, desc.K, desc.H, desc.O
    g, dg, lp, W1, b1, W2, _ = _dev_inputs(inp)
    upstream = upstream if upstream is not None else up
    ups = [None if upstream.get(k) is None else dev(_fm(upstream[k])) for k in ("g_u", "g_du", "g_lapu")]
    outs = {"g_gamma": torch.full((K, n), float("nan"), device="cuda"),
            "g_dgamma": torch.full((d, K, n), float("nan"), device="cuda"),
            "g_lap": torch.full((K, n), float("nan"), device="cuda"),
            "gW1": torch.zeros((H, K), device="cuda"), "gb1": torch.zeros(H, device="cuda"),
            "gW2": torch.zeros((O, H), device="cuda"), "gb2": torch.zeros(O, device="cuda")}
    args = {k: (outs[k] if k in want else None) for k in outs}
    m.hg.hg_siren_bwd(desc, n, g, dg, lp, W1, b1, W2, *ups, **args)
    torch.cuda.synchronize()
    got = {k: host(v) for k, v in outs.items() if k in want}
    for k in ("g_gamma", "g_dgamma", "g_lap"):
        if k in got:
            got[k] = _pm(got[k])
    return got


def _check_bwd(got, ref):
    for k, v in got.items():
        check_close(k, v, ref[k], ref["m" + k], rtol=RTOL_W if k[:2] in ("gW", "gb") else 1e-5)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_siren_backward_parity(case):
    m, oracle, desc, inp, up = _build(case, seed=1)
    got = _run_bwd(m, desc, inp, up)
    ref = oracle.siren_bwd(omega=desc.omega, **inp, **up)
    _check_bwd(got, ref)


@pytest.mark.parametrize("which", ["3d_K32_H64_workload_shape", "4d_K32_H64_O4"])
def test_siren_backward_partial_upstream(which):
    """One upstream output at a time (the others NULL), and weight gradients accumulated onto existing values."""
    case = next(c for c in CASES if c[0] == which)
    m, oracle, desc, inp, up = _build(case, seed=2)
    for keep in up:
        part = {k: (v if k == keep else None) for k, v in up.items()}
        got = _run_bwd(m, desc, inp, up, upstream=part)
        _check_bwd(got, oracle.siren_bwd(omega=desc.omega, **inp, **part))


def test_siren_weight_gradients_accumulate():
    case = CASES[0]
    m, oracle, desc, inp, up = _build(case, seed=3)
    n = inp["gamma"].shape[0]
    g, dg, lp, W1, b1, W2, _ = _dev_inputs(inp)
    ups = [dev(_fm(up[k])) for k in ("g_u", "g_du", "g_lapu")]
    gW1 = torch.ones((desc.H, desc.K), device="cuda")
    for _ in range(2):
        m.hg.hg_siren_bwd(desc, n, g, dg, lp, W1, b1, W2, *ups, gW1=gW1)
    torch.cuda.synchronize()
    ref = oracle.siren_bwd(omega=desc.omega, **inp, **up)
    check_close("gW1 (1 + 2 calls)", host(gW1), 1 + 2 * ref["gW1"], 1 + 2 * ref["mgW1"], rtol=RTOL_W)


# Fused encoder + SIREN forward (hg_encode_siren_fwd): the Hermite encoding of
# each point formed on chip and fed to the first layer.
# (id, d, L, n_min, n_max, log2T, dtype, n, level_mask, H, O, omega)
FUSED = [
    ("2d_pinn_grid", 2, 16, 16, 1024, 19, "f32", 3000, None, 64, 1, 30.0),
    ("2d_f16_mask", 2, 8, 4, 200, 12, "f16", 2049, 0b10110101, 32, 2, 30.0),
    ("2d_H128_O3", 2, 8, 4, 90, 10, "f32", 700, None, 128, 3, 10.0),
    ("3d_f32", 3, 8, 4, 64, 12, "f32", 1500, None, 64, 1, 30.0),
    ("3d_f16_mask", 3, 4, 4, 40, 10, "f16", 777, 0b1011, 64, 1, 30.0),
    ("2d_one_point", 2, 4, 4, 32, 12, "f32", 1, None, 64, 1, 30.0),
    # shapes that keep the first layer on the CUDA cores (H < 32; (d + 2) H > 512 TMEM columns)
    ("2d_H16_cuda_cores", 2, 8, 4, 60, 10, "f32", 900, None, 16, 1, 30.0),
    ("3d_H128_cuda_cores", 3, 4, 4, 40, 10, "f32", 500, None, 128, 1, 30.0),
]


def _oracle_chain(oracle, d, F, res, log2T, orders, coords, mask, sw, omega):
    """The oracle's encoding, then its SIREN, with the encoder's magnitudes
    carried into the SIREN's (the condition magnitude of the composed
    evaluation)."""
    L = len(res)
    n = coords.shape[0]
    enc = oracle.encode_fwd(d, F, res, log2T, orders, coords, level_mask=mask)
    K = L * F
    flat = {k: enc[k].reshape(n, K) if k in ("gamma", "lap", "mgamma", "mlap") else enc[k].reshape(n, d, K)
            for k in ("gamma", "dgamma", "lap", "mgamma", "mdgamma", "mlap")}
    return oracle.siren_fwd(flat["gamma"], flat["dgamma"], flat["lap"], sw["W1"], sw["b1"], sw["W2"], sw["b2"],
                            omega, mgamma=flat["mgamma"], mdgamma=flat["mdgamma"], mlap=flat["mlap"])


@pytest.mark.parametrize("case", FUSED, ids=[c[0] for c in FUSED])
def test_fused_encoder_siren_forward_parity(case):
    import multiresolution_hash_grid_02_b300 as m
    from multiresolution_hash_grid_02_b300 import workloads as W
    import oracle
    from test_parity_gpu import _coords
    cid, d, L, nmin, nmax, log2T, dt, n, mask, H, O, omega = case
    F, K = 2, L * 2
    rng = np.random.default_rng(zlib.crc32(cid.encode()))
    res = oracle.level_resolutions(L, nmin, nmax)
    coords = _coords(rng, n, d, res)
    npdt = np.float16 if dt == "f16" else np.float32
    table = (rng.uniform(-1, 1, (L, 1 << log2T, 1 << d, F)) * 0.05).astype(npdt)
    sw = W.siren_weights(rng, K, H, O, omega)
    desc = m.GridDesc(d=d, L=L, F=F, n_min=nmin, n_max=nmax, log2_T=(log2T,) * (d + 1), level_mask=mask,
                      dtype=m.HG_F16 if dt == "f16" else m.HG_F32, layout=m.HG_FEATURE_MAJOR)
    sdesc = m.SirenDesc(d=d, K=K, H=H, O=O, omega=omega)
    t_dev, c_dev = dev(table), dev(coords)
    wts = [dev(sw[k]) for k in ("W1", "b1", "W2", "b2")]
    u, du, lu = (torch.full(sh, float("nan"), device="cuda") for sh in ((O, n), (d, O, n), (O, n)))
    m.hg.hg_encode_siren_fwd(desc, n, c_dev, m.packed_views(t_dev, d), sdesc, *wts, u, du, lu)
    torch.cuda.synchronize()
    ref = _oracle_chain(oracle, d, F, res, (log2T,) * (d + 1), W.split_orders(table, d), coords, mask, sw, omega)
    check_close("u", _pm(host(u)), ref["u"], ref["mu"])
    check_close("du", _pm(host(du)), ref["du"], ref["mdu"])
    check_close("lapu", _pm(host(lu)), ref["lapu"], ref["mlapu"])
    # against the unfused chain on the GPU: the encoder's outputs through memory, then the SIREN
    g = torch.empty((L, F, n), device="cuda")
    dg = torch.empty((d, L, F, n), device="cuda")
    lp = torch.empty((L, F, n), device="cuda")
    m.hg.hg_encode_fwd(desc, n, c_dev, m.packed_views(t_dev, d), g, dg, lp)
    u2, du2, lu2 = (torch.full(sh, float("nan"), device="cuda") for sh in ((O, n), (d, O, n), (O, n)))
    m.hg.hg_siren_fwd(sdesc, n, g, dg, lp, *wts, u2, du2, lu2)
    torch.cuda.synchronize()
    if d == 2:
        # the same 2D encoder arithmetic (one thread per item) and the same SIREN tile: bit for bit
        for a, b in ((u, u2), (du, du2), (lu, lu2)):
            assert np.array_equal(host(a), host(b))
    # outputs not requested are not written
    u3 = torch.full((O, n), float("nan"), device="cuda")
    m.hg.hg_encode_siren_fwd(desc, n, c_dev, m.packed_views(t_dev, d), sdesc, *wts, u3)
    torch.cuda.synchronize()
    assert np.array_equal(host(u3), host(u))
