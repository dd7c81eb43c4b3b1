"""Properties of the oracle's Radial-Directional Averaging merge.

The Decoupled DiLoCo note (architecture item 4) only says that the outer
gradients' norms and directions are averaged apart; it gives no formula, so
this merge is "parity unpinned": the reading (per tensor: D = r u / ||u||
with r the weighted mean of the learners' norms and u the weighted mean of
their unit vectors) is checked against the properties that define it, not
against the pages:

* one learner, or identical learners: D is their decoded values;
* ||D|| per tensor is the weighted mean of the learners' norms;
* two orthogonal learners of equal norm: the plain mean shrinks the norm by
  sqrt(2), RDA keeps it (closed form);
* D points along the weighted mean of unit vectors;
* scaling one learner changes the length of D only through r;
* a learner whose values are all zero has no direction;
* weights and quorum follow the merge's rules.
"""
import numpy as np

import oracle

NB = 256


def _quantised(rng, n_per_t, K, scale=1e-3):
    """Codes, codebooks and counts of K learners (from the oracle quantiser)."""
    n = sum(n_per_t)
    off = np.concatenate([[0], np.cumsum(n_per_t)]).astype(np.int64)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = [(g - scale * (1 + 0.3 * k) * rng.standard_normal(n)).astype(np.float32)
            for k in range(K)]
    st = oracle.stats(g, reps, off)
    codes, cb, cnt = oracle.quantize(g, reps, st, off)
    return g, off, codes, cb, cnt


def _decoded(codes, cb, off, k):
    T = len(off) - 1
    v = np.empty(codes.shape[1], dtype=np.float32)
    for t in range(T):
        v[off[t]:off[t + 1]] = cb[k, t][codes[k, off[t]:off[t + 1]]]
    return v


def _rda(g, codes, cb, cnt, off, **kw):
    st, g1, m1, db = oracle.rda_merge_outer_step(g, np.zeros_like(g), list(codes), cb, cnt,
                                                 offsets=off, **kw)
    assert st == 0
    return db


def test_single_and_identical_learners_give_the_decoded_values():
    rng = np.random.default_rng(1)
    g, off, codes, cb, cnt = _quantised(rng, [5000, 3000], 3)
    v1 = _decoded(codes, cb, off, 1)
    db = _rda(g, codes, cb, cnt, off, present=[0, 1, 0])
    assert np.array_equal(db, v1)
    # three copies of learner 1 with unequal weights
    c3 = np.stack([codes[1]] * 3)
    cb3 = np.stack([cb[1]] * 3)
    cnt3 = np.stack([cnt[1]] * 3)
    db3 = _rda(g, c3, cb3, cnt3, off, weights=np.array([0.5, 2.0, 1.0], np.float32))
    assert np.allclose(db3, v1, rtol=4e-7, atol=0)


def test_norm_is_the_weighted_mean_norm_and_direction_the_mean_unit_vector():
    rng = np.random.default_rng(2)
    g, off, codes, cb, cnt = _quantised(rng, [20000, 7000, 4096], 4)
    w = np.array([0.7, 1.3, 1.0, 0.4], np.float32)
    w_hat = oracle.merge_weights(w, None, 4)[1].astype(np.float64)
    db = _rda(g, codes, cb, cnt, off, weights=w).astype(np.float64)
    for t in range(3):
        sl = slice(off[t], off[t + 1])
        vs = [_decoded(codes, cb, off, k)[sl].astype(np.float64) for k in range(4)]
        norms = [np.linalg.norm(v) for v in vs]
        r = sum(w_hat[k] * norms[k] for k in range(4))
        assert abs(np.linalg.norm(db[sl]) - r) <= 1e-6 * r
        u = sum(w_hat[k] * vs[k] / norms[k] for k in range(4))
        cos = db[sl] @ u / (np.linalg.norm(db[sl]) * np.linalg.norm(u))
        assert cos > 1 - 1e-11
        # the plain weighted mean is shorter whenever the directions differ
        mean = sum(w_hat[k] * vs[k] for k in range(4))
        assert np.linalg.norm(mean) < r


def test_orthogonal_learners_of_equal_norm_closed_form():
    n = 1000
    codes = np.zeros((2, n), dtype=np.uint8)
    codes[0, :500] = 1
    codes[1, 500:] = 1
    cb = np.zeros((2, 1, NB), dtype=np.float32)
    cb[:, 0, 1] = 1.0
    cnt = np.zeros((2, 1, NB), dtype=np.uint32)
    cnt[:, 0, 0] = 500
    cnt[:, 0, 1] = 500
    g = np.zeros(n, dtype=np.float32)
    db = _rda(g, codes, cb, cnt, None)
    # norms sqrt(500) each; the mean is 0.5 everywhere (norm sqrt(250));
    # RDA keeps the norm sqrt(500): every element sqrt(1/2)
    assert np.allclose(db, np.sqrt(0.5), rtol=2e-7, atol=0)
    st, _, _, dmean = oracle.merge_outer_step(g, np.zeros_like(g), codes=list(codes), codebook=cb,
                                              want_delta_bar=True)
    assert np.all(dmean == 0.5)


def test_scaling_one_learner_changes_only_the_radial_part():
    rng = np.random.default_rng(3)
    g, off, codes, cb, cnt = _quantised(rng, [12000], 3)
    db = _rda(g, codes, cb, cnt, off).astype(np.float64)
    cb2 = cb.copy()
    cb2[2] *= 4.0  # exact: a power of two
    db2 = _rda(g, codes, cb2, cnt, off).astype(np.float64)
    vs = [_decoded(codes, cb, off, k).astype(np.float64) for k in range(3)]
    norms = np.array([np.linalg.norm(v) for v in vs])
    r1 = norms.sum() / 3
    r2 = (norms[0] + norms[1] + 4 * norms[2]) / 3
    # fp32 sums of differently scaled terms: a few ulps of the tensor's scale
    assert np.allclose(db2, db * (r2 / r1), rtol=2e-6, atol=1e-6 * np.abs(db2).max())


def test_zero_learner_has_no_direction():
    rng = np.random.default_rng(4)
    g, off, codes, cb, cnt = _quantised(rng, [8000], 3)
    cb0 = cb.copy()
    cb0[1] = 0.0
    db = _rda(g, codes, cb0, cnt, off).astype(np.float64)
    vs = [_decoded(codes, cb0, off, k).astype(np.float64) for k in (0, 2)]
    norms = [np.linalg.norm(v) for v in vs]
    r = sum(norms) / 3  # the zero learner still counts in the mean norm
    u = sum(v / nv for v, nv in zip(vs, norms)) / 3
    expect = r * u / np.linalg.norm(u)
    assert np.allclose(db, expect, rtol=1e-5, atol=1e-5 * np.abs(expect).max())


def test_weights_and_quorum_follow_the_merge_rules():
    rng = np.random.default_rng(5)
    g, off, codes, cb, cnt = _quantised(rng, [3000], 4)
    for weights, present, q in (([1, 1, 1, 1], [1, 0, 0, 0], 2), ([0, 0, 0, 0], None, 1),
                                ([1, -1, 1, 1], None, 1)):
        wf = np.asarray(weights, dtype=np.float32)
        st = oracle.rda_merge_outer_step(g, np.zeros_like(g), list(codes), cb, cnt, offsets=off,
                                         weights=wf, present=present, min_quorum=q)[0]
        assert st == oracle.merge_weights(wf, present, 4, q)[0] < 0
