"""ctypes binding of libhg.so (include/hg.h), with the same entry-point names.

Argument marshalling only: tensors become device pointers, table views become
``hg_table`` structs, the stream defaults to torch's current stream.  Every
step of the encoding runs in the library's CUDA kernels; there is no fallback.
If ``libhg.so`` is missing or cannot be loaded, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from math import comb
from typing import Optional, Sequence

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libhg.so")

HG_OK, HG_ERR_INVALID_ARG, HG_ERR_UNSUPPORTED, HG_ERR_CUDA = 0, 1, 2, 3
HG_F32, HG_F16 = 0, 1
HG_POINT_MAJOR, HG_FEATURE_MAJOR = 0, 1
HG_MAX_LEVELS = 32
HG_ABI_VERSION = 4        # the include/hg.h layout this binding marshals

c_i32, c_i64, c_u32, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_void_p


class hg_grid_desc(ctypes.Structure):
    _fields_ = [("d", c_i32), ("L", c_i32), ("F", c_i32), ("n_min", c_i32), ("n_max", c_i32),
                ("res", ctypes.POINTER(c_i32)), ("log2_T", c_i32 * 5), ("level_mask", c_u32),
                ("dtype", c_i32), ("layout", c_i32)]


class hg_siren_desc(ctypes.Structure):
    _fields_ = [("d", c_i32), ("K", c_i32), ("H", c_i32), ("O", c_i32), ("omega", ctypes.c_float)]


class hg_table(ctypes.Structure):
    _fields_ = [("ptr", c_vp), ("level_stride", c_i64), ("row_stride", c_i64)]


class hg_grad_table(ctypes.Structure):
    _fields_ = [("ptr", c_vp), ("level_stride", c_i64), ("row_stride", c_i64)]


class HGError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {hg_status_string(status)}: {hg_last_error()}")


_lib = None


def lib() -> ctypes.CDLL:
    """Load libhg.so (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"libhg.so not found at {_LIB_PATH}; build it with "
                          "`python -m multiresolution_hash_grid_02_b300.build`")
    L = ctypes.CDLL(_LIB_PATH)
    D, T, G = ctypes.POINTER(hg_grid_desc), ctypes.POINTER(hg_table), ctypes.POINTER(hg_grad_table)
    S = ctypes.POINTER(hg_siren_desc)
    sig = {
        "hg_level_resolutions": [D, ctypes.POINTER(c_i32)],
        "hg_encode_fwd": [D, c_i64, c_vp, T, c_vp, c_vp, c_vp, c_vp],
        "hg_encode_bwd": [D, c_i64, c_vp, c_vp, c_vp, c_vp, G, c_vp],
        "hg_encode_fwd_hessian": [D, c_i64, c_vp, T, c_vp, c_vp, c_vp, c_vp],
        "hg_encode_bwd_hessian": [D, c_i64, c_vp, c_vp, c_vp, c_vp, G, c_vp],
        "hg_linear_fwd": [D, c_i64, c_vp, T, c_vp, c_vp],
        "hg_linear_bwd": [D, c_i64, c_vp, c_vp, G, c_vp],
        "hg_hash_indices": [D, c_i64, c_vp, c_vp, c_vp],
        "hg_linear_fd_fwd": [D, c_i64, c_vp, ctypes.c_float, T, c_vp, c_vp, c_vp, c_vp, c_vp],
        "hg_linear_fd_bwd": [D, c_i64, c_vp, ctypes.c_float, c_vp, c_vp, c_vp, c_vp, G, c_vp],
        "hg_rbf_fwd": [D, c_i64, c_vp, ctypes.c_float, c_i32, T, c_vp, c_vp, c_vp, c_vp],
        "hg_rbf_bwd": [D, c_i64, c_vp, ctypes.c_float, c_i32, c_vp, c_vp, c_vp, G, c_vp],
        "hg_siren_fwd": [S] + [c_i64] + [c_vp] * 11,
        "hg_encode_siren_fwd": [D, c_i64, c_vp, T, S] + [c_vp] * 8,
        "hg_siren_bwd": [S] + [c_i64] + [c_vp] * 17,
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.hg_status_string.argtypes = [ctypes.c_int]
    L.hg_status_string.restype = ctypes.c_char_p
    L.hg_last_error.argtypes = []
    L.hg_last_error.restype = ctypes.c_char_p
    L.hg_abi_version.argtypes = []
    L.hg_abi_version.restype = c_i32
    if L.hg_abi_version() != HG_ABI_VERSION:
        raise ImportError(f"{_LIB_PATH} has ABI version {L.hg_abi_version()}, this binding marshals version "
                          f"{HG_ABI_VERSION}; rebuild it with `python -m multiresolution_hash_grid_02_b300.build`")
    _lib = L
    return L


# ---------------------------------------------------------------------------
# descriptors and views
# ---------------------------------------------------------------------------

@dataclass
class GridDesc:
    """Python mirror of ``hg_grid_desc``."""
    d: int
    L: int
    F: int
    n_min: int = 16
    n_max: int = 512
    log2_T: Sequence[int] = (19, 19, 19, 19, 19)
    level_mask: Optional[int] = None          # None = all levels active
    dtype: int = HG_F32
    layout: int = HG_FEATURE_MAJOR
    res: Optional[Sequence[int]] = None
    _keep: list = field(default_factory=list, repr=False)

    def as_c(self) -> hg_grid_desc:
        c = hg_grid_desc()
        c.d, c.L, c.F, c.n_min, c.n_max = self.d, self.L, self.F, self.n_min, self.n_max
        lt = list(self.log2_T)
        lt += [lt[-1]] * (5 - len(lt))          # unlisted orders repeat the last size
        for k in range(5):
            c.log2_T[k] = int(lt[k])
        mask = ((1 << self.L) - 1) if self.level_mask is None else self.level_mask
        c.level_mask = mask & 0xffffffff
        c.dtype, c.layout = self.dtype, self.layout
        if self.res is not None:
            arr = (c_i32 * len(self.res))(*[int(r) for r in self.res])
            self._keep.append(arr)
            c.res = ctypes.cast(arr, ctypes.POINTER(c_i32))
        return c


@dataclass
class TableView:
    """A strided table view; ``base`` is a tensor (or raw address), ``offset``
    and the strides are in elements of the table's dtype."""
    base: object
    level_stride: int
    row_stride: int
    offset: int = 0
    elem_size: int = 4

    def address(self) -> int:
        return _addr(self.base) + self.offset * self.elem_size


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _esize(t) -> int:
    return int(t.element_size()) if hasattr(t, "element_size") else 4


def packed_views(table, d: int) -> list[TableView]:
    """Order-k views of an interleaved table [L][T][2^d][F] (see hg.h)."""
    L, T, V, F = table.shape
    assert V == 1 << d
    out, off = [], 0
    for k in range(d + 1):
        out.append(TableView(table, T * V * F, V * F, off * F, _esize(table)))
        off += comb(d, k)
    return out


def order_views(tables) -> list[TableView]:
    """Views of separate contiguous order tables [L][T_k][C(d,k)][F]."""
    return [TableView(t, t.shape[1] * t.shape[2] * t.shape[3], t.shape[2] * t.shape[3], 0, _esize(t)) for t in tables]


def linear_view(table) -> TableView:
    """View of a d-linear table [L][T][F]."""
    L, T, F = table.shape
    return TableView(table, T * F, F, 0, _esize(table))


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int, where: str):
    if status != HG_OK:
        raise HGError(status, where)


def _tables_c(views: Sequence[TableView], cls):
    arr = (cls * max(1, len(views)))()
    for i, v in enumerate(views):
        arr[i].ptr = v.address()
        arr[i].level_stride = int(v.level_stride)
        arr[i].row_stride = int(v.row_stride)
    return arr


# ---------------------------------------------------------------------------
# entry points (same names as include/hg.h)
# ---------------------------------------------------------------------------

def hg_abi_version() -> int:
    return int(lib().hg_abi_version())


def hg_status_string(status: int) -> str:
    return lib().hg_status_string(int(status)).decode()


def hg_last_error() -> str:
    return lib().hg_last_error().decode()


def hg_level_resolutions(desc: GridDesc) -> list[int]:
    out = (c_i32 * desc.L)()
    c = desc.as_c()
    _check(lib().hg_level_resolutions(ctypes.byref(c), out), "hg_level_resolutions")
    return list(out)


def hg_encode_fwd(desc: GridDesc, n: int, coords, tables: Sequence[TableView], gamma, dgamma=None, lap=None,
                  stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_encode_fwd(ctypes.byref(c), int(n), _addr(coords), _tables_c(tables, hg_table), _addr(gamma),
                             _addr(dgamma), _addr(lap), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_encode_fwd")
    return st


def hg_encode_bwd(desc: GridDesc, n: int, coords, g_gamma, g_dgamma, g_lap, grads: Sequence[TableView],
                  stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_encode_bwd(ctypes.byref(c), int(n), _addr(coords), _addr(g_gamma), _addr(g_dgamma), _addr(g_lap),
                             _tables_c(grads, hg_grad_table), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_encode_bwd")
    return st


def hg_encode_fwd_hessian(desc: GridDesc, n: int, coords, tables: Sequence[TableView], gamma, dgamma=None,
                          hess=None, stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_encode_fwd_hessian(ctypes.byref(c), int(n), _addr(coords), _tables_c(tables, hg_table),
                                     _addr(gamma), _addr(dgamma), _addr(hess), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_encode_fwd_hessian")
    return st


def hg_encode_bwd_hessian(desc: GridDesc, n: int, coords, g_gamma, g_dgamma, g_hess, grads: Sequence[TableView],
                          stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_encode_bwd_hessian(ctypes.byref(c), int(n), _addr(coords), _addr(g_gamma), _addr(g_dgamma),
                                     _addr(g_hess), _tables_c(grads, hg_grad_table), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_encode_bwd_hessian")
    return st


def hg_linear_fwd(desc: GridDesc, n: int, coords, table: TableView, gamma, stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_linear_fwd(ctypes.byref(c), int(n), _addr(coords), _tables_c([table], hg_table), _addr(gamma),
                             _stream(stream) if n else 0)
    if check:
        _check(st, "hg_linear_fwd")
    return st


def hg_linear_bwd(desc: GridDesc, n: int, coords, g_gamma, grad: TableView, stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_linear_bwd(ctypes.byref(c), int(n), _addr(coords), _addr(g_gamma), _tables_c([grad], hg_grad_table),
                             _stream(stream) if n else 0)
    if check:
        _check(st, "hg_linear_bwd")
    return st


def hg_linear_fd_fwd(desc: GridDesc, n: int, coords, eps: float, table: TableView, gamma, dgamma=None, lap=None,
                     stencil=None, stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_linear_fd_fwd(ctypes.byref(c), int(n), _addr(coords), float(eps), _tables_c([table], hg_table),
                                _addr(gamma), _addr(dgamma), _addr(lap), _addr(stencil), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_linear_fd_fwd")
    return st


def hg_linear_fd_bwd(desc: GridDesc, n: int, coords, eps: float, g_gamma, g_dgamma, g_lap, g_stencil,
                     grad: TableView, stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_linear_fd_bwd(ctypes.byref(c), int(n), _addr(coords), float(eps), _addr(g_gamma), _addr(g_dgamma),
                                _addr(g_lap), _addr(g_stencil), _tables_c([grad], hg_grad_table),
                                _stream(stream) if n else 0)
    if check:
        _check(st, "hg_linear_fd_bwd")
    return st


def hg_rbf_fwd(desc: GridDesc, n: int, coords, eps: float, rings: int, table: TableView, gamma, dgamma=None,
               lap=None, stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_rbf_fwd(ctypes.byref(c), int(n), _addr(coords), float(eps), int(rings), _tables_c([table], hg_table),
                          _addr(gamma), _addr(dgamma), _addr(lap), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_rbf_fwd")
    return st


def hg_rbf_bwd(desc: GridDesc, n: int, coords, eps: float, rings: int, g_gamma, g_dgamma, g_lap, grad: TableView,
               stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_rbf_bwd(ctypes.byref(c), int(n), _addr(coords), float(eps), int(rings), _addr(g_gamma),
                          _addr(g_dgamma), _addr(g_lap), _tables_c([grad], hg_grad_table), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_rbf_bwd")
    return st


@dataclass
class SirenDesc:
    """The SIREN consumer's shape: d spatial dimensions, K = L F inputs, H
    hidden units, O outputs and the sine frequency omega (hg_siren_desc)."""
    d: int
    K: int
    H: int
    O: int = 1
    omega: float = 30.0

    def as_c(self) -> hg_siren_desc:
        return hg_siren_desc(self.d, self.K, self.H, self.O, self.omega)


def hg_siren_fwd(desc: SirenDesc, n: int, gamma, dgamma, lap, W1, b1, W2, b2, u, du=None, lapu=None, stream=None,
                 check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_siren_fwd(ctypes.byref(c), int(n), *[_addr(a) for a in (gamma, dgamma, lap, W1, b1, W2, b2, u, du,
                                                                           lapu)], _stream(stream) if n else 0)
    if check:
        _check(st, "hg_siren_fwd")
    return st


def hg_encode_siren_fwd(desc: GridDesc, n: int, coords, tables: Sequence[TableView], sdesc: SirenDesc, W1, b1, W2,
                        b2, u, du=None, lapu=None, stream=None, check: bool = True) -> int:
    c, sc = desc.as_c(), sdesc.as_c()
    st = lib().hg_encode_siren_fwd(ctypes.byref(c), int(n), _addr(coords), _tables_c(tables, hg_table),
                                   ctypes.byref(sc), *[_addr(a) for a in (W1, b1, W2, b2, u, du, lapu)],
                                   _stream(stream) if n else 0)
    if check:
        _check(st, "hg_encode_siren_fwd")
    return st


def hg_siren_bwd(desc: SirenDesc, n: int, gamma, dgamma, lap, W1, b1, W2, g_u, g_du, g_lapu, g_gamma=None,
                 g_dgamma=None, g_lap=None, gW1=None, gb1=None, gW2=None, gb2=None, stream=None,
                 check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_siren_bwd(ctypes.byref(c), int(n), *[_addr(a) for a in (gamma, dgamma, lap, W1, b1, W2, g_u, g_du,
                                                                           g_lapu, g_gamma, g_dgamma, g_lap, gW1,
                                                                           gb1, gW2, gb2)],
                            _stream(stream) if n else 0)
    if check:
        _check(st, "hg_siren_bwd")
    return st


def hg_hash_indices(desc: GridDesc, n: int, coords, idx, stream=None, check: bool = True) -> int:
    c = desc.as_c()
    st = lib().hg_hash_indices(ctypes.byref(c), int(n), _addr(coords), _addr(idx), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_hash_indices")
    return st


# ---------------------------------------------------------------------------
# hardware probes (include/hg_probe.h)
# ---------------------------------------------------------------------------

def hg_probe_l2_gather(buf, log2_rows: int, row_bytes: int, lanes_per_row: int, n_threads: int,
                       rows_per_group: int, seed: int, sink, stream=None) -> None:
    L = lib()
    L.hg_probe_l2_gather.argtypes = [c_vp, c_i32, c_i32, c_i32, c_i64, c_i32, c_u32, c_vp, c_vp]
    L.hg_probe_l2_gather.restype = ctypes.c_int
    _check(L.hg_probe_l2_gather(_addr(buf), log2_rows, row_bytes, lanes_per_row, n_threads, rows_per_group,
                                seed & 0xffffffff, _addr(sink), _stream(stream)), "hg_probe_l2_gather")


def hg_probe_l2_red(buf, log2_rows: int, row_bytes: int, lanes_per_row: int, n_threads: int, rows_per_group: int,
                    seed: int, stream=None) -> None:
    L = lib()
    L.hg_probe_l2_red.argtypes = [c_vp, c_i32, c_i32, c_i32, c_i64, c_i32, c_u32, c_vp]
    L.hg_probe_l2_red.restype = ctypes.c_int
    _check(L.hg_probe_l2_red(_addr(buf), log2_rows, row_bytes, lanes_per_row, n_threads, rows_per_group,
                             seed & 0xffffffff, _stream(stream)), "hg_probe_l2_red")


def hg_probe_replay_gather(desc: GridDesc, n: int, coords, table, level_stride_bytes: int, row_bytes: int,
                           lanes_per_row: int, sink, stream=None, check: bool = True) -> int:
    L = lib()
    L.hg_probe_replay_gather.argtypes = [ctypes.POINTER(hg_grid_desc), c_i64, c_vp, c_vp, c_i64, c_i32, c_i32, c_vp,
                                         c_vp]
    L.hg_probe_replay_gather.restype = ctypes.c_int
    c = desc.as_c()
    st = L.hg_probe_replay_gather(ctypes.byref(c), int(n), _addr(coords), _addr(table), int(level_stride_bytes),
                                  row_bytes, lanes_per_row, _addr(sink), _stream(stream) if n else 0)
    if check:
        _check(st, "hg_probe_replay_gather")
    return st


def hg_probe_replay_red(desc: GridDesc, n: int, coords, grad, level_stride_bytes: int, row_bytes: int,
                        lanes_per_row: int, stream=None, check: bool = True) -> int:
    L = lib()
    L.hg_probe_replay_red.argtypes = [ctypes.POINTER(hg_grid_desc), c_i64, c_vp, c_vp, c_i64, c_i32, c_i32, c_vp]
    L.hg_probe_replay_red.restype = ctypes.c_int
    c = desc.as_c()
    st = L.hg_probe_replay_red(ctypes.byref(c), int(n), _addr(coords), _addr(grad), int(level_stride_bytes),
                               row_bytes, lanes_per_row, _stream(stream) if n else 0)
    if check:
        _check(st, "hg_probe_replay_red")
    return st
