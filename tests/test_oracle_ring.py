"""Pins of the oracle's ring accumulation (INTELLECT-1 notes, section 4.2: a
node dequantises what it receives, adds in fp32, and quantises again before
sending on), checked against what the mathematics fixes rather than against
a retyped copy of the ring:

* one present learner: no hop, so the result is the unquantised merge;
* constant tensors: every partial sum is a constant, its quantiser is
  degenerate and decodes exactly, so the sum is exact;
* uniform pseudo-gradients (never clipped at 6 sigma): every element's error
  against the exact weighted sum lies within the sum of the hops' bucket
  widths, and reaches a sizeable part of the last one (the hops really
  re-quantise);
* many learners: the error grows like sqrt((S-1)/2) times the one-shot
  quantiser's (each hop adds the variance of one quantisation of a partial
  sum whose spread grows with the hop), while the one-shot error stays flat;
* a present learner of weight 0 is still a hop, which re-quantises an
  already decoded sum (nearly idempotent); weights and quorum follow the
  merge's rules.
"""
import numpy as np
import pytest

import oracle


def _replicas(rng, g, K, scale=1e-3, dist="normal"):
    reps = []
    for _ in range(K):
        x = rng.standard_normal(g.size) if dist == "normal" else rng.uniform(-1, 1, g.size)
        reps.append((g - scale * x).astype(np.float32))
    return reps


def _deltas(g, reps):
    return [(g - r).astype(np.float32) for r in reps]  # fp32 subtraction, as the method


def test_single_learner_is_the_unquantised_merge():
    rng = np.random.default_rng(1)
    g = (rng.standard_normal(20000) * 0.02).astype(np.float32)
    m = (rng.standard_normal(20000) * 1e-3).astype(np.float32)
    reps = _replicas(rng, g, 3)
    off = [0, 7000, 20000]
    present = [0, 1, 0]
    st, g1, m1, db = oracle.ring_outer_step(g, m, reps, offsets=off, present=present)
    assert st == 0
    assert np.array_equal(db, _deltas(g, reps)[1])  # D = Delta of the only learner
    st2, g2, m2, _ = oracle.merge_outer_step(g, m, replicas=reps, offsets=off, present=present)
    assert st2 == 0
    assert np.array_equal(g1, g2) and np.array_equal(m1, m2)


def test_constant_tensors_sum_exactly():
    # theta_g = 1/2 and dyadic constants: every Delta and every partial sum is
    # exact, each quantiser sees a constant (sigma = 0) and decodes it exactly
    consts = np.array([[1 / 8, -3 / 16, 5 / 32, 1 / 4],
                       [-1 / 64, 3 / 128, 1 / 32, -1 / 16]])
    sizes = [3000, 5000]
    off = np.concatenate([[0], np.cumsum(sizes)])
    g = np.full(off[-1], 0.5, dtype=np.float32)
    reps = []
    for k in range(4):
        r = np.empty_like(g)
        for t in range(2):
            r[off[t]:off[t + 1]] = 0.5 - consts[t, k]
        reps.append(r)
    st, g1, m1, db = oracle.ring_outer_step(g, np.zeros_like(g), reps, offsets=off)
    assert st == 0
    for t in range(2):
        assert np.all(db[off[t]:off[t + 1]] == np.float32(consts[t].sum() / 4))


def _hop_widths(deltas, w_hat, S):
    """Bucket widths 12 sigma / 256 of the exact partial sums P_0 .. P_{S-2}."""
    acc = np.zeros_like(deltas[0], dtype=np.float64)
    widths = []
    for s in range(S - 1):
        acc = acc + w_hat[s] * deltas[s].astype(np.float64)
        widths.append(12.0 * acc.std() / 256.0)
    return np.array(widths)


@pytest.mark.parametrize("S", [2, 3, 5, 8])
def test_error_within_the_hops_bucket_widths(S):
    rng = np.random.default_rng(10 + S)
    n = 60000
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = _replicas(rng, g, S, dist="uniform")
    d = _deltas(g, reps)
    st, _, _, db = oracle.ring_outer_step(g, np.zeros_like(g), reps)
    assert st == 0
    w_hat = oracle.merge_weights(None, None, S)[1]
    exact = sum(float(w_hat[s]) * d[s].astype(np.float64) for s in range(S))
    err = np.abs(db.astype(np.float64) - exact)
    widths = _hop_widths(d, w_hat, S)
    # the quantised partial sums' spreads differ from the exact ones by the
    # earlier hops' errors (< 2% here); fp32 rounding adds a few ulps
    bound = 1.02 * widths.sum() + 8 * np.spacing(np.float32(np.abs(exact).max()))
    assert err.max() <= bound, (err.max(), bound)
    assert err.max() >= 0.25 * widths[-1], (err.max(), widths[-1])


def test_error_grows_with_the_ring_while_one_shot_stays_flat():
    rng = np.random.default_rng(7)
    n = 200000
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    ratios = {}
    for S in (2, 4, 8, 16):
        reps = _replicas(rng, g, S)
        d = _deltas(g, reps)
        exact = np.mean([x.astype(np.float64) for x in d], axis=0)
        _, _, _, db_ring = oracle.ring_outer_step(g, np.zeros_like(g), reps)
        o = oracle.outer_step(g, np.zeros_like(g), reps)
        e_ring = np.linalg.norm(db_ring - exact) / np.linalg.norm(exact)
        e_one = np.linalg.norm(o["delta_bar"] - exact) / np.linalg.norm(exact)
        ratios[S] = e_ring / e_one
        # one quantisation per learner: about w / (sqrt(12) sigma) = 1.35%
        assert 0.011 < e_one < 0.016, (S, e_one)
        # ring: one quantisation per hop of a growing partial sum
        predicted = np.sqrt((S - 1) / 2.0)
        assert 0.85 * predicted < ratios[S] < 1.15 * predicted, (S, ratios[S], predicted)
    print("ring / one-shot error ratio:", {S: round(r, 3) for S, r in ratios.items()})


def test_zero_weight_hop_requantises_a_decoded_sum():
    """A present learner of weight 0 passes the decoded partial sum on after
    quantising it again. Those values are at most 256 codebook values about a
    bucket width apart, so the new quantiser puts (almost always) one of them
    per bucket and decodes it back exactly: the hop may change an element by
    at most one bucket width, and changes few."""
    rng = np.random.default_rng(3)
    n = 30000
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = _replicas(rng, g, 3)
    w = np.array([1.0, 0.0, 1.0], dtype=np.float32)
    _, _, _, db_hop = oracle.ring_outer_step(g, np.zeros_like(g), reps, weights=w)
    _, _, _, db_absent = oracle.ring_outer_step(g, np.zeros_like(g), reps, weights=w,
                                                present=[1, 0, 1])
    diff = np.abs(db_hop.astype(np.float64) - db_absent)
    d = _deltas(g, reps)
    width = 12.0 * (0.5 * d[0].astype(np.float64)).std() / 256.0
    assert diff.max() <= 1.05 * width
    assert (diff > 0).mean() < 0.05


def test_weights_and_quorum_follow_the_merge_rules():
    rng = np.random.default_rng(4)
    n = 5000
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = _replicas(rng, g, 4)
    w = np.array([0.5, 1.5, 1.0, 0.75], dtype=np.float32)
    a = oracle.ring_outer_step(g, np.zeros_like(g), reps, weights=w)
    b = oracle.ring_outer_step(g, np.zeros_like(g), reps, weights=4 * w)  # exact rescale
    assert a[0] == 0 and all(np.array_equal(x, y) for x, y in zip(a[1:], b[1:]))
    for weights, present, q in (([1, 1, 1, 1], [1, 0, 0, 0], 2), ([0, 0, 0, 0], None, 1),
                                ([1, -1, 1, 1], None, 1), ([1, 1, 1, 1], [0, 0, 0, 0], 1)):
        wf = np.asarray(weights, dtype=np.float32)
        st_ring = oracle.ring_outer_step(g, np.zeros_like(g), reps, weights=wf, present=present,
                                         min_quorum=q)[0]
        st_merge = oracle.merge_weights(wf, present, 4, q)[0]
        assert st_ring == st_merge < 0
