"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/hg.h declares, computes the level schedule on the
host, and rejects bad arguments with a status code before touching the GPU.

Every call here either fails argument checking or has n = 0, so no kernel
is ever launched.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    import multiresolution_hash_grid_02_b300 as pkg
    from multiresolution_hash_grid_02_b300 import build
    build.build()
    return pkg


def _declared(header):
    with open(os.path.join(ROOT, "include", header)) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hg_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(m):
    lib = m.hg.lib()
    names = _declared("hg.h") + _declared("hg_probe.h")
    assert {"hg_encode_fwd", "hg_encode_bwd", "hg_linear_fwd", "hg_linear_bwd", "hg_level_resolutions",
            "hg_hash_indices", "hg_status_string", "hg_last_error", "hg_abi_version", "hg_encode_fwd_hessian",
            "hg_encode_bwd_hessian"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_abi_version_matches_header(m):
    with open(os.path.join(ROOT, "include", "hg.h")) as f:
        v = int(re.search(r"#define HG_ABI_VERSION (\d+)", f.read()).group(1))
    assert m.hg.hg_abi_version() == v


def test_status_strings(m):
    assert [m.hg.hg_status_string(s) for s in range(4)] == ["HG_OK", "HG_ERR_INVALID_ARG", "HG_ERR_UNSUPPORTED",
                                                            "HG_ERR_CUDA"]


@pytest.mark.parametrize("L,n_min,n_max", [(4, 4, 32), (16, 16, 2048), (16, 16, 1024), (16, 16, 512),
                                           (1, 7, 7), (2, 1, 1), (32, 2, 1 << 22), (9, 3, 1000), (31, 5, 4000000),
                                           (16, 1, 65536), (24, 16, 1 << 19)])
def test_level_schedule_equals_oracle(m, oracle_mod, L, n_min, n_max):
    got = m.hg.hg_level_resolutions(m.GridDesc(d=2, L=L, F=2, n_min=n_min, n_max=n_max))
    assert got == oracle_mod.level_resolutions(L, n_min, n_max)


def test_level_schedule_sweep(m, oracle_mod):
    import random
    rnd = random.Random(3)
    for _ in range(300):
        L = rnd.randint(1, 32)
        a = rnd.randint(1, 5000)
        b = rnd.randint(a, 1 << 22)
        got = m.hg.hg_level_resolutions(m.GridDesc(d=3, L=L, F=1, n_min=a, n_max=b))
        assert got == oracle_mod.level_resolutions(L, a, b), (L, a, b)


def test_explicit_resolutions(m):
    assert m.hg.hg_level_resolutions(m.GridDesc(d=2, L=3, F=2, res=[5, 9, 700])) == [5, 9, 700]
    with pytest.raises(m.HGError):
        m.hg.hg_level_resolutions(m.GridDesc(d=2, L=2, F=2, res=[0, 9]))


def _fwd_status(m, desc, n=5, coords=16, tables=None, gamma=16):
    if tables is None:
        tables = m.hg.packed_views(_FakeTable((desc.L, 1 << desc.log2_T[0], 1 << desc.d, desc.F)), desc.d)
    return m.hg.hg_encode_fwd(desc, n, coords, tables, gamma, None, None, stream=0, check=False)


class _FakeTable:
    """Shape-only stand-in for a tensor: address 0 (so every call that gets
    past the shape checks fails on the NULL pointer, before any launch)."""

    def __init__(self, shape, addr=0, esize=4):
        self.shape = shape
        self._addr = addr
        self._esize = esize

    def data_ptr(self):
        return self._addr

    def element_size(self):
        return self._esize


@pytest.mark.parametrize("field,value", [("d", 1), ("d", 5), ("L", 0), ("L", 33), ("F", 3), ("F", 16),
                                         ("dtype", 2), ("layout", 7), ("n_min", 0), ("n_max", 1 << 23)])
def test_bad_descriptor_is_rejected(m, field, value):
    desc = m.GridDesc(d=3, L=4, F=2, n_min=4, n_max=32, log2_T=(8, 8, 8, 8))
    setattr(desc, field, value)
    assert m.hg.hg_abi_version() == m.hg.HG_ABI_VERSION
    t = _FakeTable((4, 256, 8, 2), addr=1 << 20)
    views = m.hg.packed_views(t, 3) if field != "d" else []
    st = m.hg.hg_encode_fwd(desc, 5, 16, views or m.hg.packed_views(t, 3), 1 << 21, None, None, stream=0,
                            check=False)
    assert st == m.hg.HG_ERR_INVALID_ARG
    assert m.hg.hg_last_error() != ""


def test_bad_arguments_are_rejected(m):
    hg = m.hg
    ok_desc = lambda: m.GridDesc(d=3, L=4, F=2, n_min=4, n_max=32, log2_T=(8, 8, 8, 8))
    t = _FakeTable((4, 256, 8, 2), addr=1 << 20)
    views = hg.packed_views(t, 3)
    E = hg.HG_ERR_INVALID_ARG
    # level mask above L, table size out of range
    d = ok_desc(); d.level_mask = 1 << 4
    assert hg.hg_encode_fwd(d, 5, 16, views, 32, stream=0, check=False) == E
    d = ok_desc(); d.log2_T = (31, 8, 8, 8)
    assert hg.hg_encode_fwd(d, 5, 16, views, 32, stream=0, check=False) == E
    # n out of range
    assert hg.hg_encode_fwd(ok_desc(), -1, 16, views, 32, stream=0, check=False) == E
    assert hg.hg_encode_fwd(ok_desc(), 1 << 31, 16, views, 32, stream=0, check=False) == E
    # NULL coords / gamma with n > 0
    assert hg.hg_encode_fwd(ok_desc(), 5, 0, views, 32, stream=0, check=False) == E
    assert hg.hg_encode_fwd(ok_desc(), 5, 16, views, 0, stream=0, check=False) == E
    # NULL and misaligned table pointers
    nul = hg.packed_views(_FakeTable((4, 256, 8, 2), addr=0), 3)
    assert hg.hg_encode_fwd(ok_desc(), 5, 16, nul, 32, stream=0, check=False) == E
    odd = hg.packed_views(_FakeTable((4, 256, 8, 2), addr=(1 << 20) + 1), 3)
    assert hg.hg_encode_fwd(ok_desc(), 5, 16, odd, 32, stream=0, check=False) == E
    # rows that overlap: row stride below the values per entry, level stride below T * row stride
    bad = [hg.TableView(t, 256 * 8 * 2, 1, 0)] + views[1:]
    assert hg.hg_encode_fwd(ok_desc(), 5, 16, bad, 32, stream=0, check=False) == E
    bad = [hg.TableView(t, 100, 16, 0)] + views[1:]
    assert hg.hg_encode_fwd(ok_desc(), 5, 16, bad, 32, stream=0, check=False) == E
    # misaligned coordinates / outputs
    assert hg.hg_encode_fwd(ok_desc(), 5, 18, views, 32, stream=0, check=False) == E
    assert hg.hg_encode_fwd(ok_desc(), 5, 16, views, 33, stream=0, check=False) == E
    # backward: misaligned upstream gradient, NULL coords
    assert hg.hg_encode_bwd(ok_desc(), 5, 16, 18, None, None, views, stream=0, check=False) == E
    assert hg.hg_encode_bwd(ok_desc(), 5, 0, 16, None, None, views, stream=0, check=False) == E
    # full Hessian: NULL or misaligned hess, misaligned upstream g_hess
    assert hg.hg_encode_fwd_hessian(ok_desc(), 5, 16, views, 32, None, None, stream=0, check=False) == E
    assert hg.hg_encode_fwd_hessian(ok_desc(), 5, 16, views, 32, None, 34, stream=0, check=False) == E
    assert hg.hg_encode_fwd_hessian(ok_desc(), 5, 16, views, 0, None, 64, stream=0, check=False) == E
    assert hg.hg_encode_bwd_hessian(ok_desc(), 5, 16, None, None, 18, views, stream=0, check=False) == E
    assert hg.hg_encode_bwd_hessian(ok_desc(), 5, 0, None, None, 16, views, stream=0, check=False) == E
    # d-linear and indices
    lv = hg.linear_view(_FakeTable((4, 256, 2), addr=1 << 20))
    assert hg.hg_linear_fwd(ok_desc(), 5, 0, lv, 32, stream=0, check=False) == E
    assert hg.hg_linear_bwd(ok_desc(), 5, 0, 16, lv, stream=0, check=False) == E
    assert hg.hg_hash_indices(ok_desc(), 5, 16, 0, stream=0, check=False) == E
    # NULL descriptor / table array at the C level
    lib = hg.lib()
    assert lib.hg_encode_fwd(None, 5, 16, None, 32, None, None, None) == E
    assert lib.hg_level_resolutions(None, None) == E


def test_four_dimensional_descriptor_is_accepted(m):
    """d = 4 (space-time) passes argument checking; n = 0 launches nothing."""
    hg = m.hg
    desc = m.GridDesc(d=4, L=3, F=2, n_min=4, n_max=16, log2_T=(8, 8, 8, 8, 8))
    t = _FakeTable((3, 256, 16, 2), addr=1 << 20)
    views = hg.packed_views(t, 4)
    assert len(views) == 5
    assert hg.hg_encode_fwd(desc, 0, 0, views, 0, stream=0, check=False) == hg.HG_OK
    assert hg.hg_encode_bwd_hessian(desc, 0, 0, 0, 0, 0, views, stream=0, check=False) == hg.HG_OK
    # the fifth table's size is checked too
    desc.log2_T = (8, 8, 8, 8, 31)
    assert hg.hg_encode_fwd(desc, 5, 16, views, 32, stream=0, check=False) == hg.HG_ERR_INVALID_ARG
    # a level mask, schedule and index query in 4D pass checking as well
    assert hg.hg_level_resolutions(m.GridDesc(d=4, L=3, F=2, n_min=4, n_max=16)) == [4, 8, 16]


def test_replay_probe_arguments_are_checked(m):
    """The replay probes reject unsupported chunks, short strides and NULL
    pointers before any launch; n = 0 is a no-op."""
    hg = m.hg
    desc = m.GridDesc(d=3, L=4, F=2, n_min=4, n_max=32, log2_T=(8, 8, 8, 8))
    E, buf = hg.HG_ERR_INVALID_ARG, 1 << 20
    stride = 256 * 64
    assert hg.hg_probe_replay_gather(desc, 5, 16, buf, stride, 64, 1, 32, stream=0, check=False) == E   # 64-B chunk
    assert hg.hg_probe_replay_red(desc, 5, 16, buf, stride, 64, 2, stream=0, check=False) == E          # 32-B RED
    assert hg.hg_probe_replay_red(desc, 5, 16, buf, stride, 64, 3, stream=0, check=False) == E          # 64 % 3
    assert hg.hg_probe_replay_red(desc, 5, 16, buf, stride - 64, 64, 4, stream=0, check=False) == E     # overlap
    assert hg.hg_probe_replay_red(desc, 5, 0, buf, stride, 64, 4, stream=0, check=False) == E           # NULL coords
    assert hg.hg_probe_replay_gather(desc, 5, 16, buf, stride, 64, 2, 0, stream=0, check=False) == E    # NULL sink
    assert hg.hg_probe_replay_red(desc, 5, 16, buf + 4, stride, 64, 4, stream=0, check=False) == E      # misaligned
    assert hg.hg_probe_replay_red(desc, 0, 0, 0, stride, 64, 4, stream=0, check=False) == hg.HG_OK


def test_finite_difference_step_is_checked(m):
    hg = m.hg
    desc = m.GridDesc(d=3, L=4, F=2, n_min=4, n_max=32, log2_T=(8,))
    lv = hg.linear_view(_FakeTable((4, 256, 2), addr=1 << 20))
    E = hg.HG_ERR_INVALID_ARG
    for eps in (0.0, -1e-3, float("nan"), float("inf"), 1e-30):
        assert hg.hg_linear_fd_fwd(desc, 5, 16, eps, lv, 32, stream=0, check=False) == E, eps
        assert hg.hg_linear_fd_bwd(desc, 5, 16, eps, 32, None, None, None, lv, stream=0, check=False) == E, eps
    assert hg.hg_linear_fd_fwd(desc, 5, 0, 1e-3, lv, 32, stream=0, check=False) == E          # NULL coords
    assert hg.hg_linear_fd_fwd(desc, 0, 0, 1e-3, lv, 0, stream=0, check=False) == hg.HG_OK     # n = 0
    assert hg.hg_linear_fd_bwd(desc, 0, 0, 1e-3, 0, 0, 0, 0, lv, stream=0, check=False) == hg.HG_OK


def test_rbf_arguments_are_checked(m):
    hg = m.hg
    desc = m.GridDesc(d=3, L=4, F=2, n_min=4, n_max=32, log2_T=(8,))
    lv = hg.linear_view(_FakeTable((4, 256, 2), addr=1 << 20))
    E = hg.HG_ERR_INVALID_ARG
    for eps, rings in ((0.0, 3), (-1.0, 3), (float("nan"), 3), (1.0, 0), (1.0, 5)):
        assert hg.hg_rbf_fwd(desc, 5, 16, eps, rings, lv, 32, stream=0, check=False) == E, (eps, rings)
        assert hg.hg_rbf_bwd(desc, 5, 16, eps, rings, 32, None, None, lv, stream=0, check=False) == E, (eps, rings)
    d4 = m.GridDesc(d=4, L=4, F=2, n_min=4, n_max=32, log2_T=(8,))
    assert hg.hg_rbf_fwd(d4, 5, 16, 1.0, 3, lv, 32, stream=0, check=False) == hg.HG_ERR_UNSUPPORTED
    assert hg.hg_rbf_fwd(desc, 0, 0, 1.0, 3, lv, 0, stream=0, check=False) == hg.HG_OK


def test_zero_points_touch_nothing(m):
    """n = 0 with a valid descriptor succeeds without a launch (no GPU here)."""
    hg = m.hg
    desc = m.GridDesc(d=2, L=3, F=2, n_min=4, n_max=16, log2_T=(8, 8, 8))
    t = _FakeTable((3, 256, 4, 2), addr=1 << 20)
    assert hg.hg_encode_fwd(desc, 0, 0, hg.packed_views(t, 2), 0, stream=0, check=False) == hg.HG_OK
    assert hg.hg_encode_bwd(desc, 0, 0, 0, 0, 0, hg.packed_views(t, 2), stream=0, check=False) == hg.HG_OK
    assert hg.hg_encode_fwd_hessian(desc, 0, 0, hg.packed_views(t, 2), 0, 0, 0, stream=0, check=False) == hg.HG_OK
    assert hg.hg_encode_bwd_hessian(desc, 0, 0, 0, 0, 0, hg.packed_views(t, 2), stream=0, check=False) == hg.HG_OK
    assert hg.hg_last_error() == ""


def test_siren_arguments_are_checked(m):
    """Descriptor and pointer checks of the SIREN consumer, before any launch."""
    hg = m.hg
    E, A = hg.HG_ERR_INVALID_ARG, 1 << 20
    good = m.SirenDesc(d=3, K=32, H=64, O=1, omega=30.0)
    bad = [m.SirenDesc(d=0, K=32, H=64), m.SirenDesc(d=5, K=32, H=64), m.SirenDesc(d=3, K=12, H=64),
           m.SirenDesc(d=3, K=72, H=64), m.SirenDesc(d=3, K=32, H=48), m.SirenDesc(d=3, K=32, H=256),
           m.SirenDesc(d=3, K=32, H=64, O=0), m.SirenDesc(d=3, K=32, H=64, O=5),
           m.SirenDesc(d=3, K=32, H=64, omega=float("inf"))]
    for desc in bad:
        assert hg.hg_siren_fwd(desc, 5, A, A, A, A, A, A, A, A, stream=0, check=False) == E, desc
        assert hg.hg_siren_bwd(desc, 5, A, A, A, A, A, A, A, None, None, A, stream=0, check=False) == E, desc
    # required pointers, and what the requested outputs need
    assert hg.hg_siren_fwd(good, 5, 0, A, A, A, A, A, A, A, stream=0, check=False) == E            # gamma
    assert hg.hg_siren_fwd(good, 5, A, 0, A, A, A, A, A, A, du=A, stream=0, check=False) == E      # du needs dgamma
    assert hg.hg_siren_fwd(good, 5, A, A, 0, A, A, A, A, A, lapu=A, stream=0, check=False) == E    # lapu needs lap
    assert hg.hg_siren_fwd(good, 5, A + 2, A, A, A, A, A, A, A, stream=0, check=False) == E        # alignment
    assert hg.hg_siren_bwd(good, 5, A, 0, A, A, A, A, A, None, None, A, stream=0, check=False) == E  # dgamma
    assert hg.hg_siren_fwd(good, -1, A, A, A, A, A, A, A, A, stream=0, check=False) == E
    # n = 0, or nothing requested: no launch
    assert hg.hg_siren_fwd(good, 0, 0, 0, 0, 0, 0, 0, 0, 0, stream=0, check=False) == E             # still NULL
    assert hg.hg_siren_fwd(good, 0, A, A, A, A, A, A, A, A, stream=0, check=False) == hg.HG_OK
    assert hg.hg_siren_bwd(good, 5, A, A, A, A, A, A, A, A, A, stream=0, check=False) == hg.HG_OK


def test_fused_encoder_siren_arguments_are_checked(m):
    """Grid, SIREN and table checks of the fused encoder + SIREN forward,
    before any launch."""
    hg = m.hg
    E, U, A = hg.HG_ERR_INVALID_ARG, hg.HG_ERR_UNSUPPORTED, 1 << 20
    desc = m.GridDesc(d=2, L=4, F=2, n_min=4, n_max=32, log2_T=(8, 8, 8))
    views = hg.packed_views(_FakeTable((4, 256, 4, 2), addr=A), 2)
    sd = m.SirenDesc(d=2, K=8, H=64)

    def call(desc=desc, n=5, views=views, sd=sd, W1=A, u=A):
        return hg.hg_encode_siren_fwd(desc, n, A, views, sd, W1, A, A, 0, u, stream=0, check=False)

    assert call(n=0) == hg.HG_OK                                       # nothing to do: no launch
    assert call(u=0) == hg.HG_OK                                       # no output requested
    assert call(sd=m.SirenDesc(d=2, K=16, H=64)) == E                  # K must be L * F
    assert call(sd=m.SirenDesc(d=3, K=8, H=64)) == E                   # d must match the grid
    assert call(sd=m.SirenDesc(d=2, K=8, H=48)) == E                   # bad SIREN width
    assert call(W1=0) == E
    assert call(n=-1) == E
    d1 = m.GridDesc(d=2, L=8, F=1, n_min=4, n_max=32, log2_T=(8, 8, 8))
    assert call(desc=d1, views=hg.packed_views(_FakeTable((8, 256, 4, 1), addr=A), 2)) == U   # F = 2 only
    d4 = m.GridDesc(d=4, L=4, F=2, n_min=2, n_max=8, log2_T=(8, 8, 8, 8, 8))
    assert call(desc=d4, views=hg.packed_views(_FakeTable((4, 256, 16, 2), addr=A), 4),
                sd=m.SirenDesc(d=4, K=8, H=64)) == U                   # d = 2 or 3 only
    sep = m.order_views([_FakeTable((4, 256, k, 2), addr=A + i * (1 << 16)) for i, k in enumerate((1, 2, 1))])
    assert call(views=sep) == U                                        # packed layout only
    assert call(views=hg.packed_views(_FakeTable((4, 256, 4, 2), addr=A + 16), 2)) == U   # 32-byte rows unaligned
    assert hg.hg_last_error() != ""
