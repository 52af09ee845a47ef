"""Pins of the oracle's SIREN chain-rule consumer ("Hermite-NGP: Gradient-
Augmented Hash Encoding for Learning PDEs", 整体框架 and 关键设计 2), tied to
the network's plain definition u(x) = W2 sin(omega (W1 gamma(x) + b1)) + b2
rather than to the chain-rule formulas:

- with an analytic encoding gamma(x) (known gradient and Laplacian), the
  oracle's u, grad u and lap u equal the composed field and its fourth-order
  central differences in x -- a dropped term of the one-layer Laplacian, a
  sign or a missing omega fails;
- the backward is the transpose of the forward's derivative: the adjoint
  identity along random directions (finite differences of the forward) and
  the brute-force Jacobian of a tiny network;
- every magnitude bounds its value."""
import numpy as np
import pytest

OMEGA = 30.0


def _net(rng, K, H, O):
    """SIREN-style initialisation: first layer U(-1/K, 1/K), the rest of order 1/sqrt(H)."""
    return (rng.uniform(-1 / K, 1 / K, (H, K)), rng.uniform(-0.5, 0.5, H),
            rng.uniform(-1, 1, (O, H)) / np.sqrt(H), rng.uniform(-0.5, 0.5, O))


def _field(rng, d, K):
    """gamma_k(x) = r_k sin(p_k . x + q_k): value, gradient [d][K], Laplacian."""
    p = rng.uniform(-2, 2, (K, d))
    q = rng.uniform(-np.pi, np.pi, K)
    r = rng.uniform(0.5, 1.5, K)

    def at(x):
        ph = p @ x + q
        return r * np.sin(ph), (r * np.cos(ph))[None, :] * p.T, -r * np.sin(ph) * (p ** 2).sum(axis=1)
    return at


def _u(x, at, W1, b1, W2, b2):
    return W2 @ np.sin(OMEGA * (W1 @ at(x)[0] + b1)) + b2


@pytest.mark.parametrize("d,K,H,O", [(2, 8, 16, 1), (3, 32, 64, 1), (3, 12, 20, 3), (4, 6, 10, 2), (1, 5, 7, 1)])
def test_chain_rule_matches_the_composed_field(oracle_mod, d, K, H, O):
    rng = np.random.default_rng(40 + d + K)
    W1, b1, W2, b2 = _net(rng, K, H, O)
    at = _field(rng, d, K)
    h = 1e-3
    for _ in range(6):
        x = rng.uniform(-1, 1, d)
        g, dg, lg = at(x)
        out = oracle_mod.siren_fwd(g[None], dg[None], lg[None], W1, b1, W2, b2, OMEGA)
        u0 = _u(x, at, W1, b1, W2, b2)
        assert np.allclose(out["u"][0], u0, rtol=0, atol=1e-12)
        lap = np.zeros(O)
        for i in range(d):
            e = np.zeros(d)
            e[i] = h
            f = [_u(x + k * e, at, W1, b1, W2, b2) for k in (-2, -1, 1, 2)]
            grad = (f[0] - 8 * f[1] + 8 * f[2] - f[3]) / (12 * h)
            lap += (-f[0] + 16 * f[1] - 30 * u0 + 16 * f[2] - f[3]) / (12 * h * h)
            assert np.allclose(out["du"][0, i], grad, rtol=0, atol=1e-7 * max(1.0, np.abs(grad).max()))
        assert np.allclose(out["lapu"][0], lap, rtol=0, atol=1e-5 * max(1.0, np.abs(lap).max()))


def _inputs(rng, n, d, K, H, O):
    W1, b1, W2, b2 = _net(rng, K, H, O)
    return {"gamma": rng.standard_normal((n, K)) * 0.3, "dgamma": rng.standard_normal((n, d, K)) * 3,
            "lap": rng.standard_normal((n, K)) * 30, "W1": W1, "b1": b1, "W2": W2, "b2": b2}


def _upstream(rng, n, d, O):
    return {"g_u": rng.standard_normal((n, O)), "g_du": rng.standard_normal((n, d, O)),
            "g_lapu": rng.standard_normal((n, O))}


_GRADS = {"gamma": "g_gamma", "dgamma": "g_dgamma", "lap": "g_lap", "W1": "gW1", "b1": "gb1", "W2": "gW2",
          "b2": "gb2"}


def _pairing(oracle_mod, inp, up):
    """<g, f(inputs)>: the scalar whose gradient the backward returns."""
    o = oracle_mod.siren_fwd(omega=OMEGA, with_mags=False, **inp)
    return sum(float((up["g_" + k] * o[k]).sum()) for k in ("u", "du", "lapu"))


@pytest.mark.parametrize("d,K,H,O", [(2, 8, 16, 1), (3, 10, 12, 2), (4, 6, 8, 1)])
def test_siren_backward_adjoint_identity(oracle_mod, d, K, H, O):
    rng = np.random.default_rng(50 + d)
    n = 7
    inp = _inputs(rng, n, d, K, H, O)
    up = _upstream(rng, n, d, O)
    grads = oracle_mod.siren_bwd(omega=OMEGA, with_mags=False, **inp, **up)
    for _ in range(3):
        v = {k: rng.standard_normal(np.shape(a)) for k, a in inp.items()}
        h = 1e-6
        plus = _pairing(oracle_mod, {k: inp[k] + h * v[k] for k in inp}, up)
        minus = _pairing(oracle_mod, {k: inp[k] - h * v[k] for k in inp}, up)
        fd = (plus - minus) / (2 * h)
        vjp = sum(float((grads[_GRADS[k]] * v[k]).sum()) for k in inp)
        assert abs(fd - vjp) <= 1e-6 * max(1.0, abs(vjp))


def test_siren_backward_equals_bruteforce_jacobian(oracle_mod):
    rng = np.random.default_rng(55)
    n, d, K, H, O = 3, 2, 4, 5, 2
    inp = _inputs(rng, n, d, K, H, O)
    up = _upstream(rng, n, d, O)
    grads = oracle_mod.siren_bwd(omega=OMEGA, with_mags=False, **inp, **up)
    h = 1e-6
    for k, a in inp.items():
        want = np.zeros(np.shape(a))
        for idx in np.ndindex(*np.shape(a)):
            p, m = {kk: np.array(vv, copy=True) for kk, vv in inp.items()}, {kk: np.array(vv, copy=True) for kk, vv in inp.items()}
            p[k][idx] += h
            m[k][idx] -= h
            want[idx] = (_pairing(oracle_mod, p, up) - _pairing(oracle_mod, m, up)) / (2 * h)
        assert np.allclose(grads[_GRADS[k]], want, rtol=1e-6, atol=1e-6), k


def test_siren_partial_upstream_is_linear(oracle_mod):
    """A missing upstream output counts as zero, and the backward is linear in the upstream."""
    rng = np.random.default_rng(56)
    n, d, K, H, O = 9, 3, 8, 10, 1
    inp = _inputs(rng, n, d, K, H, O)
    up = _upstream(rng, n, d, O)
    full = oracle_mod.siren_bwd(omega=OMEGA, with_mags=False, **inp, **up)
    parts = [oracle_mod.siren_bwd(omega=OMEGA, with_mags=False, **inp,
                                  **{k: (v if k == keep else None) for k, v in up.items()}) for keep in up]
    for g in _GRADS.values():
        assert np.allclose(full[g], sum(p[g] for p in parts), rtol=1e-12, atol=1e-12)


def test_siren_magnitudes_bound_values(oracle_mod):
    rng = np.random.default_rng(57)
    n, d, K, H, O = 20, 3, 16, 24, 2
    inp = _inputs(rng, n, d, K, H, O)
    up = _upstream(rng, n, d, O)
    f = oracle_mod.siren_fwd(omega=OMEGA, **inp)
    for k in ("u", "du", "lapu"):
        assert np.all(np.abs(f[k]) <= f["m" + k] * (1 + 1e-12))
    b = oracle_mod.siren_bwd(omega=OMEGA, **inp, **up)
    for k in ("g_gamma", "g_dgamma", "g_lap", "gW1", "gb1", "gW2", "gb2"):
        assert np.all(np.abs(b[k]) <= b["m" + k] * (1 + 1e-12)), k


def test_siren_input_magnitudes_bound_input_perturbations(oracle_mod):
    """Given condition magnitudes of its inputs (the encoder's), the forward's
    magnitudes bound, to first order, the change of u, grad u and lap u when
    every input moves by up to eta times its magnitude.  The worst move is
    along the sign of each output's gradient (from the backward with a unit
    upstream); the input magnitudes are taken ten times the inputs' size, so
    a magnitude that ignored them is exceeded (one hidden unit, so the bound
    is nearly reached).  With |inputs| as magnitudes
    the defaults come back."""
    rng = np.random.default_rng(77)
    # few hidden units: the magnitude's sum of absolute values over units is
    # then close to the largest reachable change (no cancellation to hide in)
    n, d, K, H = 256, 2, 16, 1
    W1, b1, W2, b2 = _net(rng, K, H, 1)
    g = rng.uniform(-0.5, 0.5, (n, K))
    dg = rng.normal(0, 3, (n, d, K))
    lg = rng.normal(0, 30, (n, K))
    mags = [np.abs(a) + 10 * np.abs(a).mean() * rng.uniform(0.5, 1.0, a.shape) for a in (g, dg, lg)]
    base = oracle_mod.siren_fwd(g, dg, lg, W1, b1, W2, b2, OMEGA, mgamma=mags[0], mdgamma=mags[1], mlap=mags[2])
    eta = 1e-9
    one, zero = np.ones((n, 1)), np.zeros((n, 1))
    ups = {"u": (one, None, None), "lapu": (None, None, one)}
    for i in range(d):
        e = np.zeros((n, d, 1))
        e[:, i] = 1.0
        ups[f"du{i}"] = (None, e, None)
    for key, (gu, gdu, glu) in ups.items():
        grad = oracle_mod.siren_bwd(g, dg, lg, W1, b1, W2, b2, OMEGA, gu, gdu, glu, with_mags=False)
        moved = [a + eta * m * np.sign(grad[k]) for a, m, k in zip((g, dg, lg), mags, ("g_gamma", "g_dgamma", "g_lap"))]
        out = oracle_mod.siren_fwd(*moved, W1, b1, W2, b2, OMEGA, with_mags=False)
        name = key[:2] if key.startswith("du") else key
        sel = (slice(None), int(key[2]), 0) if key.startswith("du") else (slice(None), 0)
        ratio = np.abs(out[name] - base[name])[sel] / (eta * base["m" + name][sel])
        assert ratio.max() <= 1.0 + 1e-3, f"{key}: a move within the input magnitudes exceeds the output magnitude"
        assert ratio.max() > 0.05, f"{key}: the magnitude is far above any reachable change ({ratio.max()})"
    plain = oracle_mod.siren_fwd(g, dg, lg, W1, b1, W2, b2, OMEGA)
    same = oracle_mod.siren_fwd(g, dg, lg, W1, b1, W2, b2, OMEGA, mgamma=np.abs(g), mdgamma=np.abs(dg),
                                mlap=np.abs(lg))
    for k in ("mu", "mdu", "mlapu"):
        assert np.array_equal(plain[k], same[k])
