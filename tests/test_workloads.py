"""The seeded input generators (host only): the shuffled PINN workload is the
stratified workload's points in a seeded random order, with every other draw
unchanged."""
import numpy as np


def test_shuffled_pinn_is_a_permutation_of_the_stratified_points():
    from multiresolution_hash_grid_02_b300 import workloads as W
    a, b = W.WORKLOADS[3].scaled(4096), W.WORKLOADS[10].scaled(4096)
    ia, ib = W.make(a), W.make(b)
    # same strata, same draws, a different order
    assert not np.array_equal(ia["coords"], ib["coords"])
    order_a = np.lexsort(ia["coords"].T)
    order_b = np.lexsort(ib["coords"].T)
    assert np.array_equal(ia["coords"][order_a], ib["coords"][order_b])
    for k in ("table", "g_gamma", "g_dgamma", "g_lap"):
        assert np.array_equal(ia[k], ib[k])
    # consecutive points of the shuffled order are rarely in neighbouring strata
    side = 64
    cell = np.floor(ib["coords"] * side).astype(int)
    assert np.mean(np.abs(np.diff(cell[:, 0])) <= 1) < 0.2
