"""Ring accumulation with re-quantisation at every hop (dl_ring_outer_step)
and the values mode it quantises partial sums with, against the oracle
(needs a GPU).

Values mode: dl_pseudograd_stats / dl_quantize with no replica quantise
theta_g itself; the oracle does the same with an all-zero replica (x - 0 is
x exactly). Bars as for the pseudo-gradient quantiser.

Ring: every hop quantises the partial sum, so a boundary exception at one
hop (an element within 1e-6 of a bucket edge, allowed) moves that element's
partial sum by one bucket and carries into every later hop. The bars: the
relative L2 of D, theta and momentum over all other elements is <= 1e-6,
such elements are rare (<= 1e-4 of them), and each differs by at most one
bucket width of the widest hop.
"""
import numpy as np
import pytest

import oracle
from parity import TOL_REL_L2, check_codebook, check_codes, check_stats, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import pseudo_grad_sync_gb300 as dl
    dl.lib()
    return dl


RAGGED = [70000, 3, 4095, 4096, 8193, 0, 12345, 65536 * 2 + 5, 1000]


def _inputs(seed, numels, K, scale=1.2e-3):
    rng = np.random.default_rng(seed)
    n = int(sum(numels))
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    sc = np.repeat(scale * 10 ** rng.uniform(-0.5, 0.5, len(numels)), numels)
    reps = [(g - sc * rng.standard_normal(n)).astype(np.float32) for _ in range(K)]
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    return g, reps, m


def test_values_mode_matches_the_oracle(dl):
    rng = np.random.default_rng(2)
    numels = RAGGED
    n = sum(numels)
    x = (rng.standard_normal(n) * 3e-3 + 1e-4).astype(np.float32)
    off = np.concatenate([[0], np.cumsum(numels)]).astype(np.int64)
    zero = np.zeros_like(x)
    st_o = oracle.stats(x, [zero], off)
    codes_o, cb_o, cnt_o = oracle.quantize(x, [zero], st_o, off)
    F = dl.Fragment(numels)
    xd = torch.from_numpy(x).cuda()
    st = dl.pseudograd_stats(xd, None, F)
    counts = torch.empty((1, F.T, 256), dtype=torch.int32, device="cuda")
    codes, cb = dl.quantize(xd, None, F, st, counts=counts)
    torch.cuda.synchronize()
    o = {"stats": st_o, "codes": codes_o, "codebook": cb_o, "counts": cnt_o}
    gp = {"stats": dl.stats_to_host(st), "codes": codes[0].cpu().numpy()[None, :],
          "codebook": cb.cpu().numpy(), "counts": counts.cpu().numpy().view(np.uint32)}
    check_stats(st_o, gp["stats"], 1, len(numels))
    exc, moved = check_codes(o, gp, x, [zero], off)
    check_codebook(o, gp, moved)


def _hop_width_max(g, reps, w_hat):
    acc = np.zeros(g.size)
    wmax = 0.0
    for s in range(len(reps) - 1):
        acc = acc + float(w_hat[s]) * (g - reps[s]).astype(np.float32).astype(np.float64)
        wmax = max(wmax, 12.0 * acc.std() / 256.0)
    return wmax


def _ring_compare(dl, g, reps, m, numels, weights=None, present=None):
    off = np.concatenate([[0], np.cumsum(numels)]).astype(np.int64)
    st_o, g_o, m_o, d_o = oracle.ring_outer_step(g, m, reps, offsets=off, weights=weights,
                                                 present=present)
    assert st_o == 0
    F = dl.Fragment(numels)
    gd, md = torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda()
    dd = torch.full_like(gd, float("nan"))
    ws = dl.ring_outer_step(gd, md, F, [torch.from_numpy(r).cuda() for r in reps],
                            weights=weights, present=present, delta_bar=dd)
    torch.cuda.synchronize()
    assert dl.read_device_status(ws) == 0
    out = {"delta_bar": dd.cpu().numpy(), "theta_g": gd.cpu().numpy(), "momentum": md.cpu().numpy()}
    ref = {"delta_bar": d_o, "theta_g": g_o, "momentum": m_o}
    idx = [k for k in range(len(reps)) if present is None or present[k]]
    w_hat = oracle.merge_weights(weights, present, len(reps))[1][idx]
    width = _hop_width_max(g, [reps[k] for k in idx], w_hat)
    diff = np.abs(out["delta_bar"].astype(np.float64) - d_o)
    # a flipped code moves a partial sum by about a bucket width; codebook
    # differences within the quantiser's bar are some 2^-21 widths
    far = diff > 1e-3 * width
    assert far.mean() <= 1e-4, far.sum()
    assert np.all(diff[far] <= 1.1 * width), (diff[far].max(), width)
    keep = ~far
    res = {key: rel_l2(out[key][keep], ref[key][keep]) for key in out}
    assert all(v <= TOL_REL_L2 for v in res.values()), res
    res["moved_elements"] = int(far.sum())
    return res, out, ref


@pytest.mark.parametrize("K", [2, 3, 5])
def test_ring_matches_the_oracle(dl, K):
    g, reps, m = _inputs(10 + K, RAGGED, K)
    rng = np.random.default_rng(K)
    weights = rng.uniform(0.5, 1.5, K).astype(np.float32)
    res, _, _ = _ring_compare(dl, g, reps, m, RAGGED, weights=weights)
    print(K, res)


def test_ring_with_present_subset_and_zero_weight(dl):
    K = 6
    g, reps, m = _inputs(31, RAGGED, K)
    weights = np.array([1.0, 0.0, 2.0, 1.0, 0.5, 1.0], dtype=np.float32)
    present = np.array([1, 1, 0, 1, 1, 0], dtype=np.uint8)
    reps[2] = np.full_like(reps[2], np.nan)  # absent: must never be read
    reps[5] = np.full_like(reps[5], np.nan)
    _ring_compare(dl, g, reps, m, RAGGED, weights=weights, present=present)


def test_single_learner_ring_is_the_unquantised_merge(dl):
    K = 3
    g, reps, m = _inputs(41, RAGGED, K)
    present = np.array([0, 0, 1], dtype=np.uint8)
    F = dl.Fragment(RAGGED)
    a_g, a_m = torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda()
    b_g, b_m = a_g.clone(), a_m.clone()
    reps_d = [torch.from_numpy(r).cuda() for r in reps]
    dl.ring_outer_step(a_g, a_m, F, reps_d, present=present)
    dl.merge_outer_step(b_g, b_m, F, replicas=reps_d, present=present)
    torch.cuda.synchronize()
    assert torch.equal(a_g, b_g) and torch.equal(a_m, b_m)


def test_ring_error_growth_matches_the_oracle(dl):
    """The measurement the ring exists for: D's error against the exact mean
    grows with the number of hops; GPU and oracle agree on it."""
    n = 400000
    rng = np.random.default_rng(5)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    F = dl.Fragment([n])
    table = {}
    for S in (2, 4, 8, 16):
        reps = [(g - 1e-3 * rng.standard_normal(n)).astype(np.float32) for _ in range(S)]
        exact = np.mean([(g - r).astype(np.float32).astype(np.float64) for r in reps], axis=0)
        gd = torch.from_numpy(g).cuda()
        md = torch.zeros_like(gd)
        dd = torch.empty_like(gd)
        dl.ring_outer_step(gd, md, F, [torch.from_numpy(r).cuda() for r in reps], delta_bar=dd)
        torch.cuda.synchronize()
        e_gpu = rel_l2(dd.cpu().numpy(), exact)
        e_or = rel_l2(oracle.ring_outer_step(g, np.zeros_like(g), reps)[3], exact)
        assert abs(e_gpu - e_or) <= 1e-3 * e_or, (S, e_gpu, e_or)
        table[S] = e_gpu
    print("ring relative L2 error of D vs the exact mean:", table)
    assert table[2] < table[4] < table[8] < table[16]


def test_ring_quorum_failure_leaves_state_untouched(dl):
    g, reps, m = _inputs(51, [5000], 3)
    F = dl.Fragment([5000])
    gd, md = torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda()
    with pytest.raises(dl.DLError) as e:
        dl.ring_outer_step(gd, md, F, [torch.from_numpy(r).cuda() for r in reps],
                           present=[1, 0, 0], min_quorum=2)
    assert e.value.status == -3
    torch.cuda.synchronize()
    assert np.array_equal(gd.cpu().numpy(), g) and np.array_equal(md.cpu().numpy(), m)


def test_hop_statistics_match_the_oracle(dl):
    """The hops accumulate the statistics of the partial sums they write
    (no separate pass). Checked against the oracle's statistics of the same
    fp32 values, to the statistics bar: P_0 = w_0 Delta_0 is formed exactly as
    the oracle forms it, and P_1 is read back as D of a two-learner ring (a
    third learner of weight 0 keeps both rings' first two hops identical)."""
    K = 3
    g, reps, m = _inputs(61, RAGGED, K)
    off = np.concatenate([[0], np.cumsum(RAGGED)]).astype(np.int64)
    F = dl.Fragment(RAGGED)
    reps_d = [torch.from_numpy(r).cuda() for r in reps]
    hs = dl.new_stats(2, F.T)
    gd, md = torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda()
    ws = dl.ring_outer_step(gd, md, F, reps_d, weights=[1.0, 1.0, 0.0], hop_stats=hs)
    g2, m2 = torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda()
    p1 = torch.empty_like(g2)
    dl.ring_outer_step(g2, m2, F, reps_d[:2], delta_bar=p1)
    torch.cuda.synchronize()
    assert dl.read_device_status(ws) == 0
    got = dl.stats_to_host(hs)
    zero = np.zeros_like(g)
    p0 = (np.float32(0.5) * (g - reps[0])).astype(np.float32)  # w_hat = 1/2 exactly
    for row, vals in ((0, p0), (1, p1.cpu().numpy())):
        st_o = oracle.stats(vals, [zero], off)
        check_stats(st_o, {key: v[row:row + 1] for key, v in got.items()}, 1, len(RAGGED))


def test_hop_statistics_of_a_long_ring(dl):
    """Every row of the hop statistics is written, with counts and a spread
    that grows with the partial sum."""
    K = 6
    g, reps, m = _inputs(62, RAGGED, K)
    F = dl.Fragment(RAGGED)
    hs = dl.new_stats(K - 1, F.T)
    hs.fill_(-1)
    dl.ring_outer_step(torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda(), F,
                       [torch.from_numpy(r).cuda() for r in reps], hop_stats=hs,
                       weights=np.ones(K, np.float32))
    torch.cuda.synchronize()
    got = dl.stats_to_host(hs)
    assert np.array_equal(got["count"], np.tile(np.asarray(RAGGED), (K - 1, 1)))
    assert np.all(got["nonfinite"] == 0)
    big = np.asarray(RAGGED) >= 1000
    # P_s sums s + 1 independent pseudo-gradients of weight 1/K: sigma ~ sqrt(s + 1)
    ratio = got["std"][-1, big] / got["std"][0, big]
    assert np.all((ratio > 0.8 * np.sqrt(K - 1)) & (ratio < 1.25 * np.sqrt(K - 1))), ratio


def test_nonfinite_value_poisons_its_tensor_only(dl):
    """A NaN in one learner's replica makes that tensor's partial sum invalid
    at the first hop (counted in the hop statistics, NaN codebook), so D is
    NaN over that tensor; every other tensor matches the oracle."""
    K = 3
    numels = [9000, 20000, 5000]
    g, reps, m = _inputs(71, numels, K)
    reps[0][9000 + 123] = np.nan  # tensor 1
    off = np.concatenate([[0], np.cumsum(numels)]).astype(np.int64)
    st_o, g_o, m_o, d_o = oracle.ring_outer_step(g, m, reps, offsets=off)
    assert st_o == 0
    F = dl.Fragment(numels)
    hs = dl.new_stats(K - 1, F.T)
    gd, md = torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda()
    dd = torch.empty_like(gd)
    dl.ring_outer_step(gd, md, F, [torch.from_numpy(r).cuda() for r in reps], delta_bar=dd,
                       hop_stats=hs)
    torch.cuda.synchronize()
    got = dl.stats_to_host(hs)
    assert list(got["nonfinite"][0]) == [0, 1, 0]
    d = dd.cpu().numpy()
    t1 = slice(9000, 29000)
    assert np.isnan(d[t1]).all() and np.isnan(d_o[t1]).all()
    w_hat = oracle.merge_weights(None, None, K)[1]
    for sl in (slice(0, 9000), slice(29000, 34000)):
        width = _hop_width_max(g[sl], [r[sl] for r in reps], w_hat)
        diff = np.abs(d[sl].astype(np.float64) - d_o[sl])
        far = diff > 1e-3 * width  # a boundary exception at a hop moves one element
        assert far.sum() <= 1 and np.all(diff[far] <= 1.1 * width)
        assert rel_l2(d[sl][~far], d_o[sl][~far]) <= TOL_REL_L2
