"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the pages or mathematics fix:
the INTELLECT-1 worked example's printed numbers (section 3.2), closed-form
statistics, exact-rational brute force of the bucket rule, the bucket-mean
optimality property (section 4.1 step 4), the code-space counterexample
(section 4.2), PyTorch's own SGD-with-Nesterov routine, and the quorum /
weighting semantics of the Decoupled DiLoCo note (fault-tolerance items 1, 3).
"""
from fractions import Fraction
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic
from conftest import read_golden

NB = 256


def _stats_obj(K, T, mean, lo, hi, std=None):
    s = oracle.Stats(K, T)
    s.mean[:] = mean
    s.lo[:] = lo
    s.hi[:] = hi
    s.std[:] = (hi - lo) / 12 if std is None else std
    return s


# ---------------------------------------------------------------------------
# worked example (INTELLECT-1 notes, section 3.2)


@pytest.fixture(scope="module")
def worked():
    gold = read_golden("intellect1_worked_example.txt")
    w = synthetic.worked_example(K=gold["workers"])
    g = w.theta_global(0)
    reps = [w.replica(k, 0, g) for k in range(w.K)]
    m0 = np.zeros_like(g)
    out = oracle.outer_step(g, m0, reps, lr=gold["outer_lr"], mu=gold["outer_momentum"])
    return gold, w, g, reps, out


def test_worked_example_quant_parameters(worked):
    gold, w, g, reps, out = worked
    st = out["stats"]
    n = gold["rows"] * gold["cols"]
    assert st.count[0, 0] == n
    # the synthetic Delta has std 1.2e-3 by construction; the sampling error of
    # a population std over n values is sigma / sqrt(2n) ~ 2e-7
    tol_sigma = 6 * gold["sigma"] / math.sqrt(2 * n) + 1e-8
    for k in range(w.K):
        assert abs(st.std[k, 0] - gold["sigma"]) < tol_sigma
        assert abs(st.mean[k, 0] - gold["mu"]) < 6 * gold["sigma"] / math.sqrt(n)
        # range printed as [-7.2e-3, 7.2e-3]
        assert abs(st.lo[k, 0] - gold["range_lo"]) < 1e-5
        assert abs(st.hi[k, 0] - gold["range_hi"]) < 1e-5
        width = (st.hi[k, 0] - st.lo[k, 0]) / gold["buckets"]
        # printed as ~5.6e-5 (exact value for sigma=1.2e-3 is 5.625e-5)
        assert abs(width - gold["bucket_width"]) < 0.05e-5
    codes = out["codes"]
    assert codes.dtype == np.uint8
    assert codes[0].nbytes == gold["uint8_megabytes"] * 2**20
    assert g.nbytes == gold["fp32_megabytes"] * 2**20


def test_worked_example_coverage_and_decode(worked):
    gold, w, g, reps, out = worked
    cnt = out["counts"]
    n = g.size
    # +-6 sigma covers ~99.9999% of near-Gaussian data (section 4.1 step 2);
    # buckets 0 and 255 hold at most the clipped values plus their own share
    for k in range(w.K):
        assert cnt[k, 0].sum() == n
        edge_share = (cnt[k, 0, 0] + cnt[k, 0, 255]) / n
        assert edge_share < 1 - gold["gaussian_coverage"]
    # decode error is at most one bucket width for every element
    st = out["stats"]
    for k in range(w.K):
        d = (g - reps[k]).astype(np.float64)
        d = np.clip(d, st.lo[k, 0], st.hi[k, 0])
        dec = out["codebook"][k, 0][out["codes"][k]].astype(np.float64)
        width = (st.hi[k, 0] - st.lo[k, 0]) / NB
        assert np.max(np.abs(dec - d)) <= width * (1 + 1e-6)


def test_worked_example_mean_over_workers(worked):
    gold, w, g, reps, out = worked
    # section 3.2 step 6: the merged pseudo-gradient is the mean of the three
    # workers'. Bucket-mean quantisation error per element is at most the
    # uniform-quantiser error w/sqrt(12) in rms, so the relative L2 error of
    # the merged mean is far below 2%.
    exact = np.mean([(g - r).astype(np.float64) for r in reps], axis=0)
    db = out["delta_bar"].astype(np.float64)
    rel = np.linalg.norm(db - exact) / np.linalg.norm(exact)
    assert rel < 0.02
    # step 7 with momentum starting at 0: theta' = theta - lr (1 + mu) Delta_bar
    expect = g.astype(np.float64) - gold["outer_lr"] * (1 + gold["outer_momentum"]) * db
    np.testing.assert_allclose(out["theta_g"], expect, rtol=0, atol=4e-9)
    np.testing.assert_allclose(out["momentum"], db, rtol=0, atol=0)


# ---------------------------------------------------------------------------
# statistics: closed forms (section 4.1 step 1)


def _stats_of_values(values, offsets=None, clip=6.0):
    d = np.asarray(values, dtype=np.float32)
    # theta_k = 0 so that the pseudo-gradient is theta_g itself, exactly
    return oracle.stats(d, [np.zeros_like(d)], offsets, clip)


def test_stats_alternating_pm_a():
    a = 0.375
    st = _stats_of_values([a, -a] * 50)
    assert st.mean[0, 0] == 0.0 and st.std[0, 0] == a
    assert st.lo[0, 0] == -6 * a and st.hi[0, 0] == 6 * a


def test_stats_ramp_population_sigma():
    n = 1001
    st = _stats_of_values(np.arange(n))
    assert st.mean[0, 0] == (n - 1) / 2
    # population variance of 0..n-1 is (n^2 - 1) / 12 (the sample one differs)
    assert st.std[0, 0] == pytest.approx(math.sqrt((n * n - 1) / 12), rel=1e-14)
    st4 = _stats_of_values([0, 1, 2, 3])
    assert st4.std[0, 0] == pytest.approx(math.sqrt(1.25), rel=1e-15)


def test_stats_large_offset_two_pass():
    # mu >> sigma: a one-pass E[x^2]-E[x]^2 in fp64 loses digits here; the
    # pages' per-tensor sigma must still come out as 0.5
    st = _stats_of_values([4096.5, 4095.5] * 512)
    assert st.mean[0, 0] == 4096.0 and st.std[0, 0] == 0.5


def test_stats_constant_and_empty_and_nonfinite():
    st = _stats_of_values([0.125] * 33 + [1.0, 2.0] + [np.inf] + [], offsets=[0, 33, 33, 35, 36])
    assert st.std[0, 0] == 0.0 and st.mean[0, 0] == 0.125 and st.lo[0, 0] == 0.125
    assert st.count[0, 1] == 0 and st.mean[0, 1] == 0.0
    assert st.count[0, 2] == 2 and st.std[0, 2] == 0.5
    assert st.nonfinite[0, 3] == 1 and math.isnan(st.mean[0, 3])


def test_stats_clip_multiplier_and_pseudo_grad_sign():
    # Delta = theta_g - theta_k (start point minus learner, section 3.2 step 4)
    g = np.full(8, 1.0, dtype=np.float32)
    r = np.array([0.5, 0.75] * 4, dtype=np.float32)
    st = oracle.stats(g, [r], None, clip_sigmas=3.0)
    assert st.mean[0, 0] == 0.375 and st.std[0, 0] == 0.125
    assert st.lo[0, 0] == 0.375 - 3 * 0.125 and st.hi[0, 0] == 0.375 + 3 * 0.125


# ---------------------------------------------------------------------------
# bucket rule (section 4.1 steps 2-3)


def _exact_bucket(d, lo, hi):
    """Membership search over the 256 exact rational intervals."""
    D, L, H = Fraction(float(d)), Fraction(lo), Fraction(hi)
    if D < L:
        return 0
    if D >= H:
        return NB - 1
    W = (H - L) / NB
    for j in range(NB):
        if L + j * W <= D < L + (j + 1) * W:
            return j
    raise AssertionError


def _quantize_values(values, lo, hi, mean=0.0):
    d = np.asarray(values, dtype=np.float32)
    st = _stats_obj(1, 1, mean, lo, hi)
    return oracle.quantize(d, [np.zeros_like(d)], st)


def test_bucket_rule_brute_force_random():
    rng = np.random.default_rng(7)
    for lo, hi in [(-6.0, 6.0), (-7.3e-3, 7.1e-3), (0.25, 0.3125), (-1e-30, 3e-30)]:
        span = hi - lo
        vals = (lo + rng.uniform(-0.1, 1.1, 64) * span).astype(np.float32)
        codes, _, _ = _quantize_values(vals, lo, hi)
        for v, c in zip(vals, codes[0]):
            e = _exact_bucket(v, lo, hi)
            if c != e:
                # only an element within 1e-12 bucket widths of an edge may differ
                u = (Fraction(float(v)) - Fraction(lo)) * NB / (Fraction(hi) - Fraction(lo))
                assert abs(u - round(u)) < Fraction(1, 10**12) and abs(int(c) - e) == 1


def test_bucket_rule_exact_edges_go_up():
    # lo=-6, hi=6: width 3/64, every edge is exact in binary
    lo, hi = -6.0, 6.0
    w = 12.0 / 256
    edges = [lo + j * w for j in range(257)]
    codes, _, _ = _quantize_values(edges + [-7.0, 7.0, 1e30, -1e30], lo, hi)
    c = codes[0]
    assert list(c[:256]) == list(range(256))      # on an edge -> upper bucket
    assert c[256] == 255                           # x == hi -> last bucket
    assert list(c[257:]) == [0, 255, 255, 0]       # clipped


# ---------------------------------------------------------------------------
# bucket-mean codebook (section 4.1 step 4)


def test_codebook_empty_buckets_are_midpoints_and_singletons_exact():
    lo, hi = -6.0, 6.0
    w = 12.0 / 256
    vals = [lo + 10.3 * w, lo + 10.6 * w, lo + 200.25 * w]
    codes, cb, cnt = _quantize_values(vals, lo, hi)
    assert list(codes[0]) == [10, 10, 200]
    v32 = np.asarray(vals, dtype=np.float32).astype(np.float64)
    assert cb[0, 0, 10] == np.float32((v32[0] + v32[1]) / 2)
    assert cb[0, 0, 200] == np.float32(v32[2])
    for j in range(NB):
        if j not in (10, 200):
            assert cb[0, 0, j] == np.float32(lo + (j + 0.5) * w)
            assert cnt[0, 0, j] == 0
    assert cnt[0, 0, 10] == 2 and cnt[0, 0, 200] == 1


def test_codebook_minimises_bucket_sse():
    rng = np.random.default_rng(11)
    d = (rng.standard_normal(20000) * 1e-3).astype(np.float32)
    d[:40] *= 12  # some clipped values
    z = np.zeros_like(d)
    st = oracle.stats(d, [z])
    codes, cb, cnt = oracle.quantize(d, [z], st)
    lo, hi = st.lo[0, 0], st.hi[0, 0]
    width = (hi - lo) / NB
    v = np.clip(d.astype(np.float64), lo, hi)
    prev = -np.inf
    for j in range(NB):
        members = v[codes[0] == j]
        assert members.size == cnt[0, 0, j]
        c = float(cb[0, 0, j])
        left, right = lo + j * width, lo + (j + 1) * width
        if members.size == 0:
            continue
        ulp = float(np.spacing(np.float32(abs(c))))   # fp32 rounding of the mean
        assert left - ulp <= c <= right + ulp
        assert c >= prev  # non-decreasing over non-empty buckets
        prev = c

        def sse(x):
            return float(np.sum((members - x) ** 2))

        eps = width * 1e-3
        base = sse(c)
        tol = 1e-9 * max(base, 1e-30) + members.size * abs(c) * 1.2e-7 * eps
        assert base <= sse(c + eps) + tol and base <= sse(c - eps) + tol
        assert base <= sse(lo + (j + 0.5) * width) + tol


def test_clipped_values_enter_their_edge_bucket_mean():
    lo, hi = -6.0, 6.0
    codes, cb, cnt = _quantize_values([-100.0, 100.0], lo, hi)
    assert cb[0, 0, 0] == np.float32(lo) and cb[0, 0, 255] == np.float32(hi)


def test_degenerate_and_invalid_segments():
    d = np.full(10, 0.3, dtype=np.float32)
    z = np.zeros_like(d)
    st = oracle.stats(d, [z])
    codes, cb, cnt = oracle.quantize(d, [z], st)
    assert (codes == 0).all() and (cb == np.float32(0.3)).all()
    assert cnt[0, 0, 0] == 10 and cnt[0, 0, 1:].sum() == 0
    d2 = d.copy()
    d2[3] = np.nan
    st2 = oracle.stats(d2, [z])
    codes2, cb2, cnt2 = oracle.quantize(d2, [z], st2)
    assert st2.nonfinite[0, 0] == 1 and (codes2 == 0).all() and np.isnan(cb2).all()


# ---------------------------------------------------------------------------
# fp32 accumulation, never in code space (section 4.2)


def test_code_space_addition_counterexample():
    rng = np.random.default_rng(3)
    n = 4096
    g = (1.0 + rng.standard_normal(n) * 0.01).astype(np.float32)
    d0 = rng.standard_normal(n) * 1e-3
    d1 = 5e-4 + rng.standard_normal(n) * 3e-3
    reps = [(g - d0).astype(np.float32), (g - d1).astype(np.float32)]
    out = oracle.outer_step(g, np.zeros_like(g), reps)
    codes, cb = out["codes"].astype(np.int64), out["codebook"]
    dec0 = cb[0, 0][codes[0]].astype(np.float64)
    dec1 = cb[1, 0][codes[1]].astype(np.float64)
    fp32_sum = 0.5 * dec0 + 0.5 * dec1
    # the merge equals the fp32 sum of per-learner decodes (to one rounding)
    db = out["delta_bar"].astype(np.float64)
    assert np.max(np.abs(db - fp32_sum) / np.maximum(np.abs(fp32_sum), 1e-30)) < 1.2e-7
    # adding codes first and decoding the (clamped) sum through either codebook
    # is far from it: Q(a) + Q(b) != Q(a + b)
    csum = np.clip(codes[0] + codes[1] - 128, 0, 255)
    for k in range(2):
        wrong = 0.5 * cb[k, 0][csum].astype(np.float64)
        assert np.linalg.norm(wrong - fp32_sum) > 0.3 * np.linalg.norm(fp32_sum)


# ---------------------------------------------------------------------------
# outer Nesterov (section 3.2 step 7: lr 0.7, momentum 0.9)


def test_identity_k1_unquantised_lr1_mu0():
    rng = np.random.default_rng(5)
    g = (1.0 + 0.4 * rng.random(1000)).astype(np.float32)
    r = (g - rng.standard_normal(1000) * 1e-3).astype(np.float32)
    st, g2, m2, _ = oracle.merge_outer_step(g, np.zeros_like(g), replicas=[r], lr=1.0, mu=0.0)
    assert st == 0 and np.array_equal(g2, r)


def test_nesterov_matches_torch_sgd():
    # torch.optim.SGD(nesterov=True, dampening=0) is the textbook outer step;
    # each step starts torch from the oracle's own fp32 theta and momentum so
    # that one step's rounding is compared, not an accumulated drift.
    rng = np.random.default_rng(9)
    n = 2048
    g0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g, m = g0.copy(), np.zeros_like(g0)
    p = torch.nn.Parameter(torch.from_numpy(g0.astype(np.float64)))
    opt = torch.optim.SGD([p], lr=0.7, momentum=0.9, nesterov=True, dampening=0.0)
    for step in range(4):
        r = (g - rng.standard_normal(n) * 1e-3).astype(np.float32)
        st, g_new, m_new, db = oracle.merge_outer_step(g, m, replicas=[r], want_delta_bar=True)
        assert st == 0
        p.data = torch.from_numpy(g.astype(np.float64))
        if step > 0:
            opt.state[p]["momentum_buffer"] = torch.from_numpy(m.astype(np.float64))
        opt.zero_grad()
        p.grad = torch.from_numpy(db.astype(np.float64))
        opt.step()
        buf = opt.state[p]["momentum_buffer"].numpy()
        # fp32 evaluation against the fp64 reference: a few units of 2^-24
        # relative to the operands of each update
        m_scale = 0.9 * np.abs(m) + np.abs(db)
        assert np.all(np.abs(m_new - buf) <= 2 * 2.0**-24 * m_scale)
        scale = np.abs(g) + 0.7 * (np.abs(db) + 0.9 * np.abs(m_new))
        assert np.all(np.abs(g_new - p.data.numpy()) <= 4 * 2.0**-24 * scale)
        g, m = g_new, m_new


def test_momentum_closed_form_constant_delta():
    # lr=0 keeps theta fixed, so every step sees the same Delta_bar:
    # m_t = Delta_bar (1 - mu^t) / (1 - mu)
    g = np.full(16, 0.5, dtype=np.float32)
    r = np.full(16, 0.5 - 0.001, dtype=np.float32)
    d = float(np.float32(0.5) - np.float32(0.5 - 0.001))
    m = np.zeros_like(g)
    for t in range(1, 21):
        st, g2, m, _ = oracle.merge_outer_step(g, m, replicas=[r], lr=0.0, mu=0.9)
        assert np.array_equal(g2, g)
        np.testing.assert_allclose(m, d * (1 - 0.9**t) / 0.1, rtol=2e-6)


# ---------------------------------------------------------------------------
# quorum and weights (Decoupled DiLoCo note, fault-tolerance items 1 and 3)


def _four_learners(n=3000, seed=13):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = [(g - rng.standard_normal(n) * 1e-3 * (k + 1)).astype(np.float32) for k in range(4)]
    return g, reps


def test_equal_weights_is_plain_mean_and_scale_invariant():
    g, reps = _four_learners()
    out = oracle.outer_step(g, np.zeros_like(g), reps)
    dec = [out["codebook"][k, 0][out["codes"][k]].astype(np.float64) for k in range(4)]
    # K fp32 fused multiply-adds: error within (K+1) 2^-24 sum |terms|
    bound = 5 * 2.0**-24 * np.sum(np.abs(dec), axis=0) / 4
    assert np.all(np.abs(out["delta_bar"] - np.mean(dec, axis=0)) <= bound)
    out2 = oracle.outer_step(g, np.zeros_like(g), reps, weights=np.full(4, 8.0, np.float32))
    assert np.array_equal(out2["theta_g"], out["theta_g"])
    out3 = oracle.outer_step(g, np.zeros_like(g), reps, weights=np.full(4, 3.7, np.float32))
    np.testing.assert_allclose(out3["theta_g"], out["theta_g"], rtol=0, atol=1e-9)


def test_zero_weight_equals_absent_and_absent_never_read():
    g, reps = _four_learners()
    w = np.array([1.0, 0.0, 2.0, 0.5], dtype=np.float32)
    a = oracle.outer_step(g, np.zeros_like(g), reps, weights=w)
    pres = np.array([1, 0, 1, 1], dtype=np.uint8)
    reps_bad = list(reps)
    reps_bad[1] = np.full_like(g, np.nan)   # an absent learner's buffer is garbage
    st = oracle.stats(g, [reps[0], reps[2], reps[3]])
    codes, cb, _ = oracle.quantize(g, [reps[0], reps[2], reps[3]], st)
    full_codes = [codes[0], np.zeros_like(codes[0]), codes[1], codes[2]]
    full_cb = np.stack([cb[0], np.full_like(cb[0], np.nan), cb[1], cb[2]])
    s, g2, m2, db = oracle.merge_outer_step(g, np.zeros_like(g), codes=full_codes,
                                            codebook=full_cb, weights=w, present=pres,
                                            want_delta_bar=True)
    assert s == 0 and np.array_equal(g2, a["theta_g"]) and np.isfinite(db).all()
    s, g3, _, _ = oracle.merge_outer_step(g, np.zeros_like(g), replicas=reps_bad,
                                          weights=w, present=pres)
    assert s == 0 and np.isfinite(g3).all()


def test_weighted_mean_closed_form():
    g, reps = _four_learners()
    w = np.array([0.6, 1.4, 0.9, 1.1], dtype=np.float32)
    pres = np.array([1, 1, 0, 1], dtype=np.uint8)
    s, _, _, db = oracle.merge_outer_step(g, np.zeros_like(g), replicas=reps, weights=w,
                                          present=pres, want_delta_bar=True)
    d = [(g - r).astype(np.float64) for r in reps]
    ww = w.astype(np.float64) * pres
    expect = sum(ww[k] * d[k] for k in range(4)) / ww.sum()
    # fp32 weights (one rounding each) and K fp32 fused multiply-adds
    bound = 8 * 2.0**-24 * sum(ww[k] * np.abs(d[k]) for k in range(4)) / ww.sum()
    assert np.all(np.abs(db - expect) <= bound)


def test_quorum_errors_leave_state_untouched():
    g, reps = _four_learners(64)
    m = np.full_like(g, 0.25)
    s, g2, m2, _ = oracle.merge_outer_step(g, m, replicas=reps, present=np.zeros(4, np.uint8))
    assert s == oracle.ERR_QUORUM and np.array_equal(g2, g) and np.array_equal(m2, m)
    s, g2, m2, _ = oracle.merge_outer_step(g, m, replicas=reps,
                                           present=np.array([1, 0, 1, 0], np.uint8), min_quorum=3)
    assert s == oracle.ERR_QUORUM and np.array_equal(g2, g)
    s, *_ = oracle.merge_outer_step(g, m, replicas=reps, weights=np.zeros(4, np.float32))
    assert s == oracle.ERR_ARG
    s, *_ = oracle.merge_outer_step(g, m, replicas=reps,
                                    weights=np.array([1, -1, 1, 1], np.float32))
    assert s == oracle.ERR_ARG


# ---------------------------------------------------------------------------
# multi-tensor fragments: per-tensor statistics and codebooks


def test_fragment_equals_tensor_by_tensor():
    rng = np.random.default_rng(21)
    sizes = [5, 1, 300, 0, 4097, 64]
    off = synthetic.offsets_of(sizes)
    n = int(off[-1])
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    scales = np.repeat([1e-3, 2e-2, 5e-4, 1.0, 3e-3, 1e-4], sizes)
    reps = [(g - rng.standard_normal(n) * scales * (k + 1)).astype(np.float32) for k in range(3)]
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    whole = oracle.outer_step(g, m, reps, offsets=off)
    for t in range(len(sizes)):
        a, b = off[t], off[t + 1]
        part = oracle.outer_step(g[a:b], m[a:b], [r[a:b] for r in reps])
        assert np.array_equal(whole["codes"][:, a:b], part["codes"])
        assert np.array_equal(whole["theta_g"][a:b], part["theta_g"])
        assert np.array_equal(whole["momentum"][a:b], part["momentum"])
        np.testing.assert_array_equal(whole["codebook"][:, t], part["codebook"][:, 0])
