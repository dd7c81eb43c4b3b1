"""CUDA path vs oracle on seeded inputs, element by element (needs a GPU).

Sizes span several 8192-element chunks, ragged tensor boundaries, a ragged
tail and the degenerate cases the method has (sigma = 0, empty tensors,
non-finite values, |mu| >> sigma, a single learner, the largest K).
"""
import os

import numpy as np
import pytest

import synthetic
from parity import compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import pseudo_grad_sync_gb300 as dl
    dl.lib()


def _make(numels, K, seed, scales=None, theta_std=0.02, dist="normal", mean_shift=None):
    rng = np.random.default_rng(seed)
    n = int(sum(numels))
    g = (rng.standard_normal(n) * theta_std).astype(np.float32)
    if scales is None:
        scales = [1.2e-3] * len(numels)
    sc = np.repeat(np.asarray(scales, dtype=np.float64), numels)
    reps = []
    for k in range(K):
        if dist == "t3":
            z = rng.standard_normal(n)
            chi = rng.chisquare(3, n)
            x = z / np.sqrt(chi / 3)
        else:
            x = rng.standard_normal(n)
        d = sc * x
        if mean_shift is not None:
            d = d + np.repeat(np.asarray(mean_shift, dtype=np.float64), numels)
        reps.append((g - d).astype(np.float32))
    return g, reps


RAGGED = [1, 3, 4095, 4096, 4097, 8191, 8192, 8193, 12345, 0, 70000, 64, 5, 16384, 2]


def test_worked_example_full_size():
    w = synthetic.worked_example(K=3)
    g = w.theta_global(0)
    reps = [w.replica(k, 0, g) for k in range(3)]
    rep, o, gp = compare(g, reps, w.numels)
    print("worked example:", rep)
    assert rep["boundary_exceptions"] <= 20


@pytest.mark.parametrize("K", [1, 3, 5])
def test_ragged_fragment(K):
    scales = [10 ** (-4 + 2 * (i % 3) / 2) for i in range(len(RAGGED))]
    g, reps = _make(RAGGED, K, seed=K, scales=scales)
    m = (np.random.default_rng(99).standard_normal(g.size) * 1e-3).astype(np.float32)
    rep, _, _ = compare(g, reps, RAGGED, m=m)
    print(K, rep)


def test_max_learners_and_weights():
    K = 32
    sizes = [9000, 33, 20000]
    g, reps = _make(sizes, K, seed=7)
    rng = np.random.default_rng(8)
    w = (0.5 + rng.random(K)).astype(np.float32)
    present = (rng.random(K) < 0.7).astype(np.uint8)
    present[3] = 1
    rep, _, _ = compare(g, reps, sizes, weights=w, present=present, min_quorum=4)
    print(rep)


@pytest.mark.parametrize("np_", [1, 4, 5, 8, 9, 16, 17])
def test_present_subsets(np_):
    K = 17
    sizes = [8192 * 3 + 100]
    g, reps = _make(sizes, K, seed=np_)
    present = np.zeros(K, dtype=np.uint8)
    present[np.random.default_rng(np_).permutation(K)[:np_]] = 1
    w = np.linspace(0.5, 1.5, K).astype(np.float32)
    compare(g, reps, sizes, weights=w, present=present)


def test_unquantised_mode_and_identity():
    sizes = [8192 * 2 + 3, 77]
    g, reps = _make(sizes, 4, seed=11)
    compare(g, reps, sizes, quantized=False)
    # K=1, no quantisation, lr=1, mu=0 returns theta_k exactly
    g1 = (1.0 + np.random.default_rng(1).random(30001)).astype(np.float32)
    r1 = (g1 - np.random.default_rng(2).standard_normal(30001) * 1e-3).astype(np.float32)
    from parity import gpu_outer_step
    out = gpu_outer_step(g1, [r1], [30001], lr=1.0, mu=0.0, quantized=False)
    assert np.array_equal(out["theta_g"], r1)


def test_degenerate_segments():
    # sigma = 0 (constant Delta), |mu| >> sigma (fp64 guard path for every
    # element), sigma far below the fp32 bucket-width range (fp64 residuals),
    # |mu| ~ 100 sigma (fast path with a wide guard)
    sizes = [10000, 9000, 5000, 7000, 300]
    n = sum(sizes)
    rng = np.random.default_rng(5)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g[:10000] = 1.0
    g[19000:24000] = 0.0
    reps = []
    for k in range(2):
        d = np.empty(n)
        d[:10000] = 0.25 * k
        d[10000:19000] = 3.0 + rng.standard_normal(9000) * 1e-6
        d[19000:24000] = rng.standard_normal(5000) * 1e-30
        d[24000:31000] = 0.1 + rng.standard_normal(7000) * 1e-3
        d[31000:] = rng.standard_normal(300) * 1e-3
        reps.append((g - d).astype(np.float32))
    rep, o, gp = compare(g, reps, sizes)
    assert o["stats"].std[0, 0] == 0.0 and o["stats"].std[1, 0] == 0.0
    assert (gp["codes"][:, :10000] == 0).all()
    assert gp["codebook"][1, 0, 7] == np.float32(0.25)


def test_nonfinite_segment_is_invalid():
    sizes = [5000, 9000]
    g, reps = _make(sizes, 2, seed=3)
    reps[1][6000] = np.float32(np.inf)
    reps[0][9321] = np.float32(np.nan)  # NaN must be counted like Inf
    rep, o, gp = compare(g, reps, sizes, nan_ok=True)
    assert gp["stats"]["nonfinite"][1, 1] == 1 and gp["stats"]["nonfinite"][0, 1] == 1
    assert (gp["codes"][1, 5000:] == 0).all()
    assert np.isnan(gp["theta_g"][5000:]).all() and np.isfinite(gp["theta_g"][:5000]).all()


def test_heavy_tail_clipping():
    sizes = [50000, 4096, 130000]
    g, reps = _make(sizes, 3, seed=21, scales=[1e-3] * 3, dist="t3")
    rep, o, gp = compare(g, reps, sizes)
    clipped = (o["counts"][:, :, 0] + o["counts"][:, :, 255]).sum()
    assert clipped > 100  # Student-t(3) puts ~2e-3 of the mass beyond 6 sigma


def test_flush_path_with_one_block(monkeypatch):
    # one block covers every chunk: the histogram must flush on capacity
    monkeypatch.setenv("DL_GRID_LIMIT", "1")
    sizes = [8192 * 20 + 5, 3000]
    g, reps = _make(sizes, 2, seed=31)
    compare(g, reps, sizes)


@pytest.mark.parametrize("grid,K", [(1, 5), (3, 14), (7, 9), (2, 17), (5, 1)])
def test_small_grids_learner_groups_and_batches(grid, K, monkeypatch):
    """A capped grid makes the quantiser's blocks take multi-chunk batches from
    their group's counter (and, for K > 8, serve unequal learner groups with
    fewer blocks than chunks); the statistics blocks take long chunk runs.
    Ragged tensors across chunk edges, a tail, a tensor under 4096 elements."""
    monkeypatch.setenv("DL_GRID_LIMIT", str(grid))
    sizes = [8192 * 40 + 3, 5000, 8192 * 7 + 100, 64, 8192 * 25]
    g, reps = _make(sizes, K, seed=40 + K)
    compare(g, reps, sizes)


@pytest.mark.parametrize("grid,K", [(0, 7), (0, 8), (6, 15), (0, 22)])
def test_learner_group_boundaries(grid, K, monkeypatch):
    """The quantiser serves at most 7 learners per block: K = 7, 8, 15 and 22
    give one to four groups of near-equal size."""
    if grid:
        monkeypatch.setenv("DL_GRID_LIMIT", str(grid))
    sizes = [8192 * 12 + 9, 700, 8192 * 5, 4100]
    g, reps = _make(sizes, K, seed=70 + K)
    compare(g, reps, sizes)


@pytest.mark.parametrize("grid", [1, 3])
def test_one_learner_histogram_copies(grid, monkeypatch):
    """One learner: the quantiser's histogram copies are folded every 8
    pieces and at tensor changes. Tensors of exactly 8, 9, 16 and 17 chunks
    (the last one starting mid-chunk) put folds on and just past that
    boundary; a capped grid gives each block a long run of pieces."""
    monkeypatch.setenv("DL_GRID_LIMIT", str(grid))
    sizes = [8192 * 8, 8192 * 9, 8192 * 16 + 7, 8192 * 17, 100]
    g, reps = _make(sizes, 1, seed=80 + grid)
    compare(g, reps, sizes)


def test_tail_not_multiple_of_four():
    for n in (1, 2, 3, 5, 8191, 8193, 24579):
        g, reps = _make([n], 2, seed=n)
        compare(g, reps, [n])


def test_empty_fragment_and_empty_tensors():
    g, reps = _make([0, 0, 10, 0], 2, seed=1)
    compare(g, reps, [0, 0, 10, 0])


def test_large_mean_offset():
    """Pseudo-gradients with |mu| thousands of sigma (a shared drift plus
    small noise): the fp32 bucket edges then carry rounding errors of several
    hundredths of a bucket width, and the fixed-point residuals must still be
    in range. |mu|/sigma of 1e4 and 2e4 take the fp32 path, 1e5 the fp64 path."""
    sizes = [60000, 4096, 20000, 9000]
    g, reps = _make(sizes, 3, seed=31, scales=[1e-7, 1e-7, 3e-8, 1e-8],
                    mean_shift=[1e-3, -2e-3, 5e-4, 1e-3])
    rep, o, gp = compare(g, reps, sizes)
    st = o["stats"]
    ratio = np.abs(st.mean) / st.std
    assert ratio.min() > 5e3 and ratio.max() > 5e4, ratio


@pytest.mark.parametrize("seed,K", [(60, 2), (63, 2), (63, 4)])
def test_mean_offset_straddling_a_power_of_two(seed, K):
    """mu just inside -2^-10 (and -2^-8, -2^-12) with sigma ~1e-7 and theta
    near 0, so Delta sits on the fine fp32 grid of the bucket edges: lo lies
    one binade above most edges, its fp32 rounding is a whole ulp of an edge,
    and an element can sit up to ~w/30 below its fp32 edge. Its residual must
    still be carried exactly into the bucket mean."""
    sizes = [60000, 60000, 60000]
    mu = [-2.0**-10, -2.0**-8 + 2e-7, -2.0**-12]
    g, reps = _make(sizes, K, seed=seed, scales=[1e-7, 1e-7, 1e-8], theta_std=1e-6,
                    mean_shift=mu)
    compare(g, reps, sizes)


def test_unrepresentative_leading_values():
    """Tensors whose first values differ from the rest: a large-spread head
    (1000x sigma) followed by small values, a constant head, and a head of
    exact zeros. Neither the shift nor the square offsets may depend on the
    head being typical."""
    sizes = [70000, 50000, 30000]
    K = 3
    g, reps = _make(sizes, K, seed=41, scales=[1e-6, 1e-4, 3e-5])
    rng = np.random.default_rng(42)
    off = np.concatenate([[0], np.cumsum(sizes)])
    for k in range(K):
        d = (g - reps[k]).astype(np.float64)
        d[off[0]:off[0] + 64] = rng.standard_normal(64) * 1e-3      # 1000x spread head
        d[off[1]:off[1] + 100] = 2.5e-4                            # constant head
        d[off[2]:off[2] + 200] = 0.0                               # zero head
        reps[k] = (g - d).astype(np.float32)
    compare(g, reps, sizes)


@pytest.mark.parametrize("K", [1, 4, 5, 8, 9, 14, 16, 17, 32])
def test_staged_merge_equals_the_unstaged_one(K, monkeypatch):
    """The merge staged through shared memory (one instance per bound on the
    number of present learners: 4, 8, 16, 32) and the unstaged k_merge_q
    (DL_MERGE_UNSTAGED=1) must give the same theta, momentum and D bit for
    bit, on ragged tensors (tails of 1-3 elements and of under 16 bytes of
    codes, chunk-crossing tensors, an empty tensor), with unequal weights and
    one absent learner when K > 1."""
    import pseudo_grad_sync_gb300 as dl
    sizes = RAGGED
    g, reps = _make(sizes, K, seed=21 + K)
    m = (np.random.default_rng(22).standard_normal(g.size) * 1e-3).astype(np.float32)
    F = dl.Fragment(sizes)
    gd = torch.from_numpy(g).cuda()
    reps_d = [torch.from_numpy(r).cuda() for r in reps]
    st = dl.pseudograd_stats(gd, reps_d, F)
    codes, cb = dl.quantize(gd, reps_d, F, st)
    w = (0.5 + np.random.default_rng(23).random(K)).astype(np.float32)
    present = np.ones(K, np.uint8)
    if K > 1:
        present[K // 2] = 0
    outs = []
    for unstaged in (False, True):
        if unstaged:
            monkeypatch.setenv("DL_MERGE_UNSTAGED", "1")
        else:
            monkeypatch.delenv("DL_MERGE_UNSTAGED", raising=False)
        ga, ma = gd.clone(), torch.from_numpy(m).cuda()
        da = torch.empty_like(ga)
        dl.merge_outer_step(ga, ma, F, codes, cb, weights=w, present=present, delta_bar=da, K=K)
        torch.cuda.synchronize()
        outs.append([x.cpu().numpy() for x in (ga, ma, da)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)  # == on floats: +0 and -0 count as equal
    assert dl.read_device_status(None) == 0
