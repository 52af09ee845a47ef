"""Test harness: run the CUDA library (through its C ABI) and the oracle on the
same seeded inputs, and compare them.

Tolerance: a float result r with oracle value o and oracle condition
magnitude m (the same sum with every factor replaced by its absolute value)
passes when |r - o| <= rtol * m.  With fp32 arithmetic the blend's rounding
error is a small multiple of 2^-24 * m (a few dozen roundings per sum), so
rtol = 1e-5 holds with room to spare; cancellation in the Laplacian (which
carries N^2) cannot cause false failures because m carries the same factor.
fp16 tables are widened exactly, so the same bound applies to them.
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-5


def torch_mod():
    import torch
    return torch


def dev(a: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def check_close(name: str, got: np.ndarray, want: np.ndarray, mag: np.ndarray, rtol: float = RTOL):
    got = np.asarray(got, np.float64)
    err = np.abs(got - want)
    bound = rtol * mag
    bad = ~(err <= bound)          # a NaN (an output never written) fails too
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, np.nan_to_num(err / np.maximum(mag, 1e-300), nan=np.inf), 0)),
                             err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} elements outside {rtol:g} * magnitude; "
                             f"worst at {i}: got {got[i]!r}, oracle {want[i]!r}, magnitude {mag[i]!r}")
    nz = mag > 0
    return float((err[nz] / mag[nz]).max()) if nz.any() else 0.0


def gpu_hermite_fwd(desc, coords: np.ndarray, views, want_d=True, want_l=True, torch_tables=None):
    """Run hg_encode_fwd; returns point-major numpy (gamma, dgamma, lap)."""
    from multiresolution_hash_grid_02_b300 import hg, HG_FEATURE_MAJOR
    from multiresolution_hash_grid_02_b300.workloads import from_feature_major
    torch = torch_mod()
    n, d, L, F = coords.shape[0], desc.d, desc.L, desc.F
    c = dev(coords)
    fm = desc.layout == HG_FEATURE_MAJOR
    shape_g = (L, F, n) if fm else (n, L, F)
    shape_d = (d, L, F, n) if fm else (n, d, L, F)
    g = torch.full(shape_g, float("nan"), device="cuda")
    dg = torch.full(shape_d, float("nan"), device="cuda") if want_d else None
    lp = torch.full(shape_g, float("nan"), device="cuda") if want_l else None
    hg.hg_encode_fwd(desc, n, c, views, g, dg, lp)
    torch.cuda.synchronize()
    g = host(g)
    dg = host(dg) if want_d else None
    lp = host(lp) if want_l else None
    if fm:
        g = from_feature_major(g, False)
        dg = from_feature_major(dg, True) if want_d else None
        lp = from_feature_major(lp, False) if want_l else None
    return g, dg, lp


def gpu_hermite_bwd(desc, coords, gg, gd, gl, grad_tensors, grad_views):
    """Run hg_encode_bwd on point-major numpy upstream grads (converted to
    desc.layout); grad_tensors are zeroed device tensors, returned as numpy."""
    from multiresolution_hash_grid_02_b300 import hg, HG_FEATURE_MAJOR
    from multiresolution_hash_grid_02_b300.workloads import to_feature_major
    torch = torch_mod()
    fm = desc.layout == HG_FEATURE_MAJOR
    conv = (lambda a, ax: to_feature_major(a, ax)) if fm else (lambda a, ax: a)
    n = coords.shape[0]
    g1 = dev(conv(gg, False)) if gg is not None else None
    g2 = dev(conv(gd, True)) if gd is not None else None
    g3 = dev(conv(gl, False)) if gl is not None else None
    hg.hg_encode_bwd(desc, n, dev(coords), g1, g2, g3, grad_views)
    torch.cuda.synchronize()
    return [host(t) for t in grad_tensors]


def packed_to_orders(packed: np.ndarray, d: int):
    from multiresolution_hash_grid_02_b300.workloads import split_orders
    return split_orders(packed, d)
