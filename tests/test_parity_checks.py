"""The checkers of the GPU parity tests, on the CPU.

`parity.check_merge_elementwise` holds one side's merge and outer step to
fp64 recomputed from that side's own decoded values. Here it must accept the
oracle's own outputs (several tensors, weights, an absent learner, carried
momentum with cancellations, the unquantised mode) and reject the oracle's
outputs with a mistake planted in them: one element off, a learner's weight
dropped, momentum or Nesterov terms changed.

The checkers that compare the GPU with the oracle (statistics, codes,
codebooks and counts, the merge's relative L2) must pass the oracle's
outputs against themselves and fail when one value in a copy of them is
planted wrong by a few times the bar.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic
from parity import check_codebook, check_codes, check_merge, check_merge_elementwise, check_stats

NUMELS = [1, 257, 4096, 9000]


def _case(K=5, seed=11, quantized=True, present=None, weights=None):
    rng = np.random.default_rng(seed)
    n = sum(NUMELS)
    off = synthetic.offsets_of(NUMELS)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = [(g - rng.standard_normal(n).astype(np.float32) * 1e-3).astype(np.float32)
            for _ in range(K)]
    # momentum of the same size as the pseudo-gradients and either sign, so
    # that mu m + delta_bar cancels at many elements
    m0 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    o = oracle.outer_step(g, m0, reps, offsets=off, weights=weights, present=present,
                          quantized=quantized)
    assert o["status"] == 0
    pres = np.ones(K, bool) if present is None else np.asarray(present, bool)
    w = np.ones(K, np.float32) if weights is None else np.asarray(weights, np.float32)
    if quantized:
        t_of = np.searchsorted(off, np.arange(n), side="right") - 1
        vals = [o["codebook"][k][t_of, o["codes"][k]] for k in np.nonzero(pres)[0]]
    else:
        vals = [(g - reps[k]).astype(np.float32) for k in np.nonzero(pres)[0]]
    return g, m0, vals, w[pres], o


CASES = {
    "plain": {},
    "weights_and_absent": {"present": [1, 0, 1, 1, 1], "weights": [0.5, 9.0, 1.25, 0.0, 2.0]},
    "unquantised": {"quantized": False, "weights": [1.0, 2.0, 3.0, 4.0, 5.0]},
}


@pytest.mark.parametrize("name", list(CASES))
def test_oracle_outputs_pass(name):
    g, m0, vals, w, o = _case(**CASES[name])
    worst = check_merge_elementwise(g, m0, vals, w, o)
    print(name, worst)
    assert all(v <= 1.0 for v in worst.values())


def _planted(name, what):
    g, m0, vals, w, o = _case(**CASES[name])
    bad = {k: np.array(o[k], copy=True) for k in ("delta_bar", "momentum", "theta_g")}
    i = 4096 + 300  # an element of the third tensor
    if what == "one_delta_bar":
        # one element's merged value off by 8 ulps, carried on through m and theta
        d = np.float32(bad["delta_bar"][i])
        bad["delta_bar"][i] = np.float32(d + 8 * np.spacing(np.abs(d)))
    elif what == "one_theta":
        t = np.float32(bad["theta_g"][i])
        bad["theta_g"][i] = np.float32(t + 4 * np.spacing(np.abs(t)))
    elif what == "momentum_mu":
        # momentum decayed with 0.8 in place of 0.9
        bad["momentum"] = (np.float32(0.8) * m0 + bad["delta_bar"]).astype(np.float32)
    elif what == "heavy_ball":
        # theta stepped along momentum alone (no Nesterov look-ahead)
        bad["theta_g"] = (g - np.float32(0.7) * bad["momentum"]).astype(np.float32)
    elif what == "dropped_learner":
        # the merge leaves the last learner out but normalises over all
        ww = w.astype(np.float64) / w.astype(np.float64).sum()
        bad["delta_bar"] = sum(ww[k] * vals[k].astype(np.float64)
                               for k in range(len(vals) - 1)).astype(np.float32)
    return g, m0, vals, w, bad


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("what", ["one_delta_bar", "one_theta", "momentum_mu", "heavy_ball",
                                  "dropped_learner"])
def test_planted_mistakes_fail(name, what):
    g, m0, vals, w, bad = _planted(name, what)
    with pytest.raises(AssertionError):
        check_merge_elementwise(g, m0, vals, w, bad)


# --- the other checkers of the GPU parity tests, against planted mistakes ----

def _full_case(K=4, seed=5):
    """The oracle's outputs, and a copy of them in the form the GPU side
    takes (`gp`), for several tensors of one fragment."""
    rng = np.random.default_rng(seed)
    n = sum(NUMELS)
    off = synthetic.offsets_of(NUMELS)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = [(g - rng.standard_normal(n).astype(np.float32) * 1e-3).astype(np.float32)
            for _ in range(K)]
    m0 = np.zeros(n, np.float32)
    o = oracle.outer_step(g, m0, reps, offsets=off)
    assert o["status"] == 0
    st = o["stats"]
    gp = {"stats": {k: np.array(getattr(st, k), copy=True)
                    for k in ("count", "nonfinite", "mean", "std", "lo", "hi")}}
    for k in ("codes", "codebook", "counts", "delta_bar", "theta_g", "momentum"):
        gp[k] = np.array(o[k], copy=True)
    return g, reps, off, o, gp


def _run_checks(g, reps, off, o, gp):
    K = len(reps)
    check_stats(o["stats"], gp["stats"], K, len(NUMELS))
    exc, moved = check_codes(o, gp, g, reps, off)
    check_codebook(o, gp, moved)
    w_hat = oracle.merge_weights(None, None, K)[1]
    t_of = np.searchsorted(off, np.arange(g.size), side="right") - 1
    check_merge(gp, o, gp["codes"], o["codes"], gp["codebook"], o["codebook"], w_hat, t_of)
    return exc


def test_identical_outputs_pass_every_checker():
    assert _run_checks(*_full_case()) == 0


def _far_from_edges(g, reps, off, o, k, t):
    """An element of tensor t whose bucket coordinate for learner k sits
    mid-bucket, far from either edge."""
    a, b = int(off[t]), int(off[t + 1])
    idx = np.arange(a, b)
    u = oracle.bucket_coord(g, reps[k], idx, o["stats"].lo[k, t], o["stats"].hi[k, t])
    frac = u - np.floor(u)
    pick = idx[(frac > 0.3) & (frac < 0.7) & (u > 1) & (u < 254)]
    assert pick.size
    return int(pick[0])


@pytest.mark.parametrize("what", ["mean", "std", "count", "code", "code_by_two", "codebook",
                                  "counts", "theta_far"])
def test_planted_mistakes_fail_a_checker(what):
    g, reps, off, o, gp = _full_case()
    k, t = 2, 3  # learner 2, the 9000-element tensor
    s = o["stats"].std[k, t]
    if what == "mean":
        gp["stats"]["mean"][k, t] += 2e-8 * s  # 4x the statistics bar
    elif what == "std":
        gp["stats"]["std"][k, t] *= 1 + 2e-8
    elif what == "count":
        gp["stats"]["count"][k, t] -= 1
    elif what in ("code", "code_by_two"):
        i = _far_from_edges(g, reps, off, o, k, t)
        gp["codes"][k, i] += 1 if what == "code" else 2
    elif what == "codebook":
        # an occupied entry off by 4x the bar derived from the Delta_bar contract
        from parity import codebook_tolerance
        b = int(np.argmax(gp["counts"][k, t]))
        bar = codebook_tolerance(o["stats"].std[:, t])
        gp["codebook"][k, t, b] += np.float32(4 * bar)
    elif what == "counts":
        b = int(np.argmax(gp["counts"][k, t]))
        gp["counts"][k, t, b] -= 1
        gp["counts"][k, t, b + 1] += 1
    elif what == "theta_far":
        # one element's theta off by 1e-3 of itself: the relative L2 catches this
        i = int(off[t]) + 17
        gp["theta_g"][i] *= np.float32(1 + 1e-3)
    with pytest.raises(AssertionError):
        _run_checks(g, reps, off, o, gp)


def test_relative_l2_alone_misses_one_element_that_the_elementwise_check_catches():
    """Why the element-wise check exists: one theta' element off by 1e-5 of
    itself stays under the 1e-6 relative L2 of its 13,354-element fragment,
    and fails the element-wise bound."""
    g, reps, off, o, gp = _full_case()
    i = int(off[3]) + 17
    gp["theta_g"][i] *= np.float32(1 + 1e-5)
    _run_checks(g, reps, off, o, gp)  # passes: hidden in the L2 norm
    t_of = np.searchsorted(off, np.arange(g.size), side="right") - 1
    vals = [gp["codebook"][k][t_of, gp["codes"][k]] for k in range(len(reps))]
    with pytest.raises(AssertionError):
        check_merge_elementwise(g, np.zeros_like(g), vals, np.ones(len(reps), np.float32), gp)
