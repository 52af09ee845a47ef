"""Oracle for the SIREN chain-rule consumer of the encoding -- TEST INFRASTRUCTURE.

Plain fp64 numpy (matrix products as library steps, nothing fused or
reordered), used only by ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm.

Source: "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs",
section "整体框架" (the chain rule: grad u = (du/dgamma) grad gamma and
lap u = (d2u/dgamma2)(grad gamma)^2 + (du/dgamma) lap gamma) and section
"关键设计 2" (SIREN, sigma(x) = sin(omega x), whose identity
sigma'' = -omega^2 sigma gives the one-layer Laplacian
lap u = W2 [ -omega^2 a * sum_i (W1 gamma_{x_i})^2 + omega cos(omega z) * W1 lap gamma ],
a = sin(omega z), z = W1 gamma + b1); section "损失函数 / 训练策略" fixes
omega_0 = 30.  The network is the one of that formula -- one sine layer and a
linear output layer, u = W2 sin(omega (W1 gamma + b1)) + b2 -- which is the
depth the section "关键发现" calls sufficient.

Layouts here are point-major: gamma [n][K], dgamma [n][d][K], lap [n][K]
(K = L * F, the levels' features concatenated), W1 [H][K], b1 [H],
W2 [O][H], b2 [O]; u [n][O], du [n][d][O], lapu [n][O].

Magnitudes (``m*``) bound the rounding error of an fp32 evaluation: every
quantity carries the sum of the absolute values of its terms, products and
sums propagate them to first order, and the sine layer adds omega times the
magnitude of its argument (d sin(omega z) = omega cos(omega z) dz).  Pinned by
``tests/test_oracle_siren_pins.py`` (finite differences of the composed
field, the adjoint identity, brute-force Jacobians); not "parity unpinned".
"""
from __future__ import annotations

import numpy as np


def _f64(*arrays):
    return [None if a is None else np.asarray(a, np.float64) for a in arrays]


def siren_fwd(gamma, dgamma, lap, W1, b1, W2, b2, omega, with_mags=True, mgamma=None, mdgamma=None, mlap=None):
    """u, grad u and lap u of the SIREN at the encoder outputs ("关键设计 2").

    The magnitudes treat the inputs as exact unless their own condition
    magnitudes are given (mgamma, mdgamma, mlap: same shapes, e.g. the
    encoder oracle's), in which case those replace |gamma|, |dgamma|, |lap|
    and the returned magnitudes are those of the composed evaluation."""
    gamma, dgamma, lap, W1, b1, W2, b2 = _f64(gamma, dgamma, lap, W1, b1, W2, b2)
    z = gamma @ W1.T + b1                      # [n][H]
    a = np.sin(omega * z)
    c = np.cos(omega * z)
    y = dgamma @ W1.T                          # [n][d][H]: W1 gamma_{x_i}
    s = lap @ W1.T                             # [n][H]: W1 lap gamma
    u = a @ W2.T + b2                          # [n][O]
    du = (omega * c[:, None, :] * y) @ W2.T    # [n][d][O]
    lapu = (-omega ** 2 * a * (y ** 2).sum(axis=1) + omega * c * s) @ W2.T
    out = {"u": u, "du": du, "lapu": lapu}
    if with_mags:
        A = np.abs
        mg = A(gamma) if mgamma is None else np.asarray(mgamma, np.float64)
        mdg = A(dgamma) if mdgamma is None else np.asarray(mdgamma, np.float64)
        ml = A(lap) if mlap is None else np.asarray(mlap, np.float64)
        mz = mg @ A(W1).T + A(b1)
        my = mdg @ A(W1).T
        ms = ml @ A(W1).T
        ma = A(a) + omega * mz
        mc = A(c) + omega * mz
        y2 = (y ** 2).sum(axis=1)
        my2 = (2 * A(y) * my).sum(axis=1)
        out["mu"] = ma @ A(W2).T + A(b2)
        out["mdu"] = (omega * (mc[:, None, :] * A(y) + A(c)[:, None, :] * my)) @ A(W2).T
        out["mlapu"] = (omega ** 2 * (ma * y2 + A(a) * my2) + omega * (mc * A(s) + A(c) * ms)) @ A(W2).T
    return out


def siren_bwd(gamma, dgamma, lap, W1, b1, W2, b2, omega, g_u, g_du, g_lapu, with_mags=True):
    """Vector-Jacobian product of :func:`siren_fwd` with upstream gradients
    g_u [n][O], g_du [n][d][O], g_lapu [n][O] (None = zero): the gradients of
    the encoder outputs (g_gamma [n][K], g_dgamma [n][d][K], g_lap [n][K]) and
    of the weights (gW1 [H][K], gb1 [H], gW2 [O][H], gb2 [O])."""
    gamma, dgamma, lap, W1, b1, W2, b2 = _f64(gamma, dgamma, lap, W1, b1, W2, b2)
    n, d = dgamma.shape[0], dgamma.shape[1]
    O = W2.shape[0]
    gu = np.zeros((n, O)) if g_u is None else np.asarray(g_u, np.float64)
    gdu = np.zeros((n, d, O)) if g_du is None else np.asarray(g_du, np.float64)
    glu = np.zeros((n, O)) if g_lapu is None else np.asarray(g_lapu, np.float64)
    # the forward's intermediates
    z = gamma @ W1.T + b1
    a = np.sin(omega * z)
    c = np.cos(omega * z)
    y = dgamma @ W1.T
    s = lap @ W1.T
    y2 = (y ** 2).sum(axis=1)
    # adjoints of the hidden layer's outputs (the forward read backwards)
    U = gu @ W2                                # d/da of W2 a
    D = gdu @ W2                               # [n][d][H]
    P = glu @ W2
    g_a = U - omega ** 2 * P * y2
    g_c = omega * (D * y).sum(axis=1) + omega * P * s
    g_y = omega * c[:, None, :] * D - 2 * omega ** 2 * (a * P)[:, None, :] * y
    g_s = omega * c * P
    g_z = omega * c * g_a - omega * a * g_c    # a = sin(omega z), c = cos(omega z)
    out = {
        "g_gamma": g_z @ W1,
        "g_dgamma": g_y @ W1,
        "g_lap": g_s @ W1,
        "gW1": g_z.T @ gamma + np.einsum("nih,nik->hk", g_y, dgamma) + g_s.T @ lap,
        "gb1": g_z.sum(axis=0),
        "gW2": gu.T @ a + np.einsum("nio,nih->oh", gdu, omega * c[:, None, :] * y)
        + glu.T @ (-omega ** 2 * a * y2 + omega * c * s),
        "gb2": gu.sum(axis=0),
    }
    if with_mags:
        A = np.abs
        mz = A(gamma) @ A(W1).T + A(b1)
        my = A(dgamma) @ A(W1).T
        ms = A(lap) @ A(W1).T
        ma = A(a) + omega * mz
        mc = A(c) + omega * mz
        my2 = (2 * A(y) * my).sum(axis=1)
        mU = A(gu) @ A(W2)
        mD = A(gdu) @ A(W2)
        mP = A(glu) @ A(W2)
        mga = mU + omega ** 2 * (mP * y2 + A(P) * my2)
        mgc = omega * (mD * A(y) + A(D) * my).sum(axis=1) + omega * (mP * A(s) + A(P) * ms)
        mgy = (omega * (mc[:, None, :] * A(D) + A(c)[:, None, :] * mD)
               + 2 * omega ** 2 * ((ma * A(P) + A(a) * mP)[:, None, :] * A(y) + (A(a) * A(P))[:, None, :] * my))
        mgs = omega * (mc * A(P) + A(c) * mP)
        mgz = omega * (mc * A(g_a) + A(c) * mga) + omega * (ma * A(g_c) + A(a) * mgc)
        out["mg_gamma"] = mgz @ A(W1)
        out["mg_dgamma"] = mgy @ A(W1)
        out["mg_lap"] = mgs @ A(W1)
        out["mgW1"] = mgz.T @ A(gamma) + np.einsum("nih,nik->hk", mgy, A(dgamma)) + mgs.T @ A(lap)
        out["mgb1"] = mgz.sum(axis=0)
        out["mgW2"] = (A(gu).T @ ma
                       + np.einsum("nio,nih->oh", A(gdu), omega * (mc[:, None, :] * A(y) + A(c)[:, None, :] * my))
                       + A(glu).T @ (omega ** 2 * (ma * y2 + A(a) * my2) + omega * (mc * A(s) + A(c) * ms)))
        out["mgb2"] = A(gu).sum(axis=0)
    return out
