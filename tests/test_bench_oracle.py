"""bench.py's CPU baselines run the oracle unchanged: each call's columns split
over host threads must give the same bits as one thread (CPU only)."""

from concurrent.futures import ThreadPoolExecutor

import numpy as np

import bench
import oracle
from int4_group_quantized_quant_gb300 import inputs as I


def test_threaded_oracle_layer_is_bit_identical():
    orc = oracle.load()
    L = I.stack_layer(0)
    h = I.stack_input(1)
    one = bench.oracle_layer(orc, L, h, 1)
    with ThreadPoolExecutor(max_workers=3) as pool:
        par = bench.oracle_layer_parallel(orc, L, h, 1, pool, 3)
    assert one.shape == par.shape == (1, bench.HIDDEN)
    assert np.array_equal(one.view(np.uint32), par.view(np.uint32))


def test_time_oracle_splits_every_column():
    seen = []
    one, par, cores = bench.time_oracle(lambda c0, c1: seen.append((c0, c1)), 10, reps=1)
    assert one >= 0 and par >= 0 and cores >= 1
    # one call over all columns, then the parallel split covers 0..10 exactly once
    assert seen[0] == (0, 10)
    parts = sorted(seen[1:])
    assert parts[0][0] == 0 and parts[-1][1] == 10
    assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
