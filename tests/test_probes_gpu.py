"""The roofline probes on the GPU.  The replay probes must touch exactly the
rows the encoding touches: after hg_probe_replay_red every float of a row
holds the number of (point, active level, corner) hits on that row, which
the oracle's vertex indices count independently (exact small integers)."""
import zlib

import numpy as np
import pytest

from _harness import dev, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


# (id, d, L, F, n_min, n_max, log2T, lanes per row, n, level mask)
CASES = [
    ("3d_quads", 3, 4, 2, 4, 64, 12, 4, 3000, None),
    ("3d_pairs_mask", 3, 4, 1, 4, 40, 11, 2, 2000, 0b0110),
    ("4d_octets", 4, 3, 2, 2, 10, 12, 8, 1500, None),
    ("2d_pairs", 2, 5, 2, 4, 100, 10, 2, 4000, None),
    ("2d_one_lane_per_row", 2, 3, 1, 4, 30, 9, 1, 999, None),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_replay_red_touches_exactly_the_encoding_rows(case):
    import multiresolution_hash_grid_02_b300 as m
    import oracle
    cid, d, L, F, nmin, nmax, log2T, lanes, n, mask = case
    rng = np.random.default_rng(zlib.crc32(cid.encode()))
    coords = rng.random((n, d), dtype=np.float32)
    coords[:8] = np.array([0.0, 1.0, 0.5, -1.0, 2.0, np.nan, 1.0 - 2 ** -24, 0.25], np.float32)[:, None]
    res = oracle.level_resolutions(L, nmin, nmax)
    T, V = 1 << log2T, 1 << d
    idx = oracle.hash_indices(d, res, [log2T] * (d + 1), coords)       # [n][L][d+1][2^d]
    want = np.zeros((L, T))
    for l in range(L):
        if mask is None or (mask >> l) & 1:
            np.add.at(want[l], idx[:, l, 0, :].ravel(), 1.0)
    row = V * F                                                       # floats per row
    grad = torch.zeros((L, T, row), device="cuda")
    desc = m.GridDesc(d=d, L=L, F=F, n_min=nmin, n_max=nmax, log2_T=(log2T,) * (d + 1), level_mask=mask)
    m.hg.hg_probe_replay_red(desc, n, dev(coords), grad, T * row * 4, row * 4, lanes)
    torch.cuda.synchronize()
    got = host(grad)
    assert np.array_equal(got, np.broadcast_to(want[:, :, None], got.shape))


def test_replay_gather_runs_on_every_chunk_size():
    import multiresolution_hash_grid_02_b300 as m
    d, L, F, log2T, n = 3, 3, 2, 10, 2048
    desc = m.GridDesc(d=d, L=L, F=F, n_min=4, n_max=32, log2_T=(log2T,) * 4)
    coords = dev(np.random.default_rng(3).random((n, d), dtype=np.float32))
    table = torch.rand((L, 1 << log2T, 16), device="cuda")               # 64-byte rows
    for lanes in (2, 4, 8, 16):
        sink = torch.full((n * lanes,), float("nan"), device="cuda")
        m.hg.hg_probe_replay_gather(desc, n, coords, table, table.stride(0) * 4, 64, lanes, sink)
        torch.cuda.synchronize()
        assert bool(torch.isfinite(sink).all())
