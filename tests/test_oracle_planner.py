"""Pins of the oracle's fragment planner.

The Decoupled DiLoCo note (architecture item 4) packs whole tensors into P
balanced fragments in the manner of greedy bin-packing. The oracle reads this
as Graham's longest-processing-time rule; these tests pin it to facts from
scheduling theory (R. L. Graham, "Bounds on multiprocessing timing
anomalies", SIAM J. Appl. Math. 17, 1969), not to its own code.
"""
import itertools

import numpy as np
import pytest

import oracle
import synthetic


def _opt_makespan(sizes, P):
    best = None
    for assign in itertools.product(range(P), repeat=len(sizes)):
        loads = [0] * P
        for s, a in zip(sizes, assign):
            loads[a] += s
        m = max(loads)
        best = m if best is None else min(best, m)
    return best


def test_partition_invariants():
    rng = np.random.default_rng(1)
    for _ in range(50):
        T = int(rng.integers(0, 40))
        P = int(rng.integers(1, 9))
        sizes = rng.integers(0, 10**6, T)
        frag, load = oracle.plan_fragments(sizes, P)
        assert frag.shape == (T,) and ((frag >= 0) & (frag < P)).all()
        for p in range(P):
            assert load[p] == sizes[frag == p].sum()
        assert load.sum() == sizes.sum()


@pytest.mark.parametrize("P", [2, 3, 4])
def test_lpt_bound_against_brute_force_optimum(P):
    rng = np.random.default_rng(P)
    for _ in range(25):
        T = int(rng.integers(1, 9 if P < 4 else 8))
        sizes = [int(x) for x in rng.integers(1, 100, T)]
        _, load = oracle.plan_fragments(sizes, P)
        opt = _opt_makespan(sizes, P)
        assert opt <= load.max() <= (4 / 3 - 1 / (3 * P)) * opt + 1e-9


@pytest.mark.parametrize("m", [2, 3, 4, 5])
def test_graham_tight_instance(m):
    # 2m+1 jobs: 2m-1, 2m-1, 2m-2, 2m-2, ..., m+1, m+1, m, m, m. LPT reaches
    # 4m-1 while the optimum is 3m, the worst case of the 4/3 - 1/(3m) bound.
    sizes = []
    for v in range(2 * m - 1, m, -1):
        sizes += [v, v]
    sizes += [m, m, m]
    _, load = oracle.plan_fragments(sizes, m)
    assert load.max() == 4 * m - 1
    if m <= 3:
        assert _opt_makespan(sizes, m) == 3 * m


def test_tie_rules():
    # equal sizes: index order decides who goes first; equal loads: lowest
    # fragment index wins
    frag, load = oracle.plan_fragments([5, 5, 5, 5, 5], 2)
    assert list(frag) == [0, 1, 0, 1, 0] and list(load) == [15, 10]
    frag, load = oracle.plan_fragments([1, 7, 3, 7], 3)
    assert list(frag) == [2, 0, 2, 1] and list(load) == [7, 7, 4]


def test_oversized_tensor_gets_its_own_fragment():
    sizes = synthetic.decoder_1b_numels()
    frag, load = oracle.plan_fragments(sizes, 24)
    big = max(sizes)
    assert big > sum(sizes) / 24
    for t, s in enumerate(sizes):
        if s == big:
            assert (frag == frag[t]).sum() == 1 and load[frag[t]] == big


def test_errors():
    with pytest.raises(ValueError):
        oracle.plan_fragments([1, 2], 0)
    with pytest.raises(ValueError):
        oracle.plan_fragments([1, -2], 2)
