"""The EPLB replica planner: the oracle's rule pinned by brute force and
invariants, and the library's host planner (mm_plan_replicas, no GPU needed)
checked against it exactly."""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _max_ratio(load, rc):
    return max(Fraction(int(l), int(r)) for l, r in zip(load, rc))


@pytest.mark.parametrize("seed", range(40))
def test_greedy_plan_minimises_peak_load_per_replica(seed):
    # brute force over every way to place the redundant slots (small cases)
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 5))
    R = int(rng.integers(1, 4))
    extra = int(rng.integers(0, E * (R - 1) + 1))
    load = rng.integers(0, 50, E)
    pol, rc = oracle.plan_replicas(load, E + extra, R)
    best = None
    for combo in itertools.product(range(R), repeat=E):
        if sum(combo) != extra:
            continue
        m = _max_ratio(load, [1 + c for c in combo])
        best = m if best is None or m < best else best
    assert _max_ratio(load, rc) == best


@pytest.mark.parametrize("E,P,R", [(8, 12, 2), (256, 320, 2), (256, 320, 4), (16, 16, 1), (5, 9, 3)])
def test_plan_is_a_valid_map(E, P, R):
    rng = np.random.default_rng(E + P)
    load = (rng.pareto(1.2, E) * 100).astype(np.int64)
    pol, rc = oracle.plan_replicas(load, P, R)
    used = [pol[e, r] for e in range(E) for r in range(rc[e])]
    assert sorted(used) == list(range(P))               # every physical slot exactly once
    assert np.all(pol[:, 0] == np.arange(E))            # each expert keeps its own slot
    assert np.all((rc >= 1) & (rc <= R))
    assert np.all(pol[np.arange(R)[None, :] >= rc[:, None]] == -1)
    # the hottest expert never ends with fewer replicas than a cooler one
    order = np.argsort(-load, kind="stable")
    assert np.all(np.diff(rc[order]) <= 0) or _max_ratio(load, rc) <= _max_ratio(load, np.ones(E))


@pytest.fixture(scope="module")
def lib():
    from moe_layer_serving_gb300 import build
    build.build()
    import moe_layer_serving_gb300 as mm
    return mm


@pytest.mark.parametrize("E,P,R,seed", [(8, 12, 2, 0), (256, 320, 2, 1), (256, 320, 4, 2), (16, 16, 1, 3),
                                        (64, 100, 3, 4), (10, 28, 3, 5)])
def test_library_planner_matches_oracle(lib, E, P, R, seed):
    rng = np.random.default_rng(seed)
    load = (rng.pareto(1.1, E) * 1000).astype(np.int64)
    load[::7] = load[0]                                 # ties
    pol, rc = lib.plan_replicas(load, P, R)
    opol, orc = oracle.plan_replicas(load, P, R)
    assert np.array_equal(rc, orc)
    assert np.array_equal(pol, opol)


def test_library_planner_rejects_impossible_plans(lib):
    with pytest.raises(lib.MegaMoEError):
        lib.plan_replicas(np.ones(4, np.int64), 13, 3)   # 9 extra slots, room for 8
