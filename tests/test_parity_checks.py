"""The element-wise merge check of the GPU parity tests, on the CPU.

`parity.check_merge_elementwise` holds one side's merge and outer step to
fp64 recomputed from that side's own decoded values. Here it must accept the
oracle's own outputs (several tensors, weights, an absent learner, carried
momentum with cancellations, the unquantised mode) and reject the oracle's
outputs with a mistake planted in them: one element off, a learner's weight
dropped, momentum or Nesterov terms changed.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synthetic
from parity import check_merge_elementwise

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
