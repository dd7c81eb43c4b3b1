"""GPU path vs oracle on identical inputs: run both and check every output.

Bars (per the outer-step tolerance contract):
  * codes bit-exact, except elements whose oracle bucket coordinate u lies
    within 1e-6 bucket widths of an integer (boundary exceptions, counted);
  * mu within 5e-9 sigma and sigma within 5e-9 relative (fp64-grade stats:
    the bucket rule is shifted by about 128 * dsigma/sigma + 21 * dmu/sigma
    bucket widths, which must stay well below the 1e-6 exception band);
  * codebook values within the share of the Delta_bar bar that codebooks may
    take (TOL_CB_SHARE, derived below) plus 2 fp32 ulps of the value (the
    final rounding on each side), bucket counts exact (both only where no
    boundary exception moved an element);
  * relative L2 <= 1e-6 on Delta_bar, theta' and momentum' over the elements
    whose codes match; at a counted boundary exception the decoded value of
    that learner moves by one bucket, so there the difference must be exactly
    what the flipped code explains (sum over learners of w_hat_k times the
    difference of the two decoded values). Without this split a handful of
    permitted exceptions in a 500M-element tensor would alone move the
    relative L2 of Delta_bar by ~1e-6 each.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import pseudo_grad_sync_gb300 as dl

TOL_REL_L2 = 1e-6
TOL_BOUNDARY = 1e-6
TOL_STATS = 5e-9

# Codebook bar, from the contract on Delta_bar (relative L2 <= TOL_REL_L2).
# Where codes match, Delta_bar(i) - Delta_bar'(i) = sum_k w_k (cb_k - cb'_k)
# at the element's codes, and the normalised weights sum to 1, so the
# difference is at most max |cb - cb'| and its relative L2 at most
# max |cb - cb'| / rms(Delta_bar). Delta_bar is a weighted mean of K learners'
# pseudo-gradients; for learners whose Delta are independent with spreads
# sigma_k (the workloads' case; a component they share only raises it),
# rms(Delta_bar)^2 >= sum_k w_k^2 sigma_k^2, which over all weights summing to
# 1 is smallest at w_k ~ sigma_k^-2: rms(Delta_bar) >= S = (sum_k
# sigma_k^-2)^(-1/2) (= sigma / sqrt(K) for equal spreads). The codebooks get
# half of the budget (the merge's own fp32 rounding and the statistics take
# the rest): |cb - cb'| <= TOL_CB_SHARE * TOL_REL_L2 * S. In bucket widths
# (w = 12 sigma / 256) and equal spreads that is 1.07e-5 w / sqrt(K):
# 2.8e-6 w at K=14, 1.9e-6 w at K=32.
TOL_CB_SHARE = 0.5


def codebook_tolerance(sigmas, K=None):
    """Largest codebook difference the Delta_bar bar allows for a tensor whose
    learners' spreads are `sigmas` (see TOL_CB_SHARE); learners with sigma = 0
    (a constant Delta, decoded exactly) are left out."""
    s = np.asarray(sigmas, dtype=np.float64)
    s = s[s > 0]
    if s.size == 0:
        return 0.0
    return TOL_CB_SHARE * TOL_REL_L2 / float(np.sqrt(np.sum(s ** -2.0)))


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    num = np.linalg.norm(a - b)
    return float(num / den) if den > 0 else float(num)


def gpu_outer_step(g, reps, numels, m=None, weights=None, present=None, min_quorum=1, lr=0.7,
                   mu=0.9, clip_sigmas=6.0, quantized=True):
    dev = "cuda"
    frag = dl.Fragment(numels, dev)
    g_d = torch.from_numpy(np.ascontiguousarray(g)).to(dev)
    reps_d = [torch.from_numpy(np.ascontiguousarray(r)).to(dev) for r in reps]
    m_d = (torch.zeros_like(g_d) if m is None else torch.from_numpy(np.ascontiguousarray(m)).to(dev))
    K = len(reps)
    out = {}
    db = torch.empty_like(g_d)
    if quantized:
        stats = dl.pseudograd_stats(g_d, reps_d, frag, clip_sigmas)
        counts = torch.empty((K, frag.T, 256), dtype=torch.int32, device=dev)
        codes, cb = dl.quantize(g_d, reps_d, frag, stats, counts=counts)
        dl.merge_outer_step(g_d, m_d, frag, codes, cb, weights=weights, present=present,
                            min_quorum=min_quorum, lr=lr, mu=mu, delta_bar=db)
        torch.cuda.synchronize()
        out["stats"] = dl.stats_to_host(stats)
        out["codes"] = np.stack([c.cpu().numpy() for c in codes]) if K else None
        out["codebook"] = cb.cpu().numpy()
        out["counts"] = counts.cpu().numpy().view(np.uint32)
    else:
        dl.merge_outer_step(g_d, m_d, frag, replicas=reps_d, weights=weights, present=present,
                            min_quorum=min_quorum, lr=lr, mu=mu, delta_bar=db)
        torch.cuda.synchronize()
    out["theta_g"] = g_d.cpu().numpy()
    out["momentum"] = m_d.cpu().numpy()
    out["delta_bar"] = db.cpu().numpy()
    return out


def check_stats(o_st, g_st, K, T, tol=TOL_STATS):
    assert np.array_equal(g_st["count"], o_st.count)
    assert np.array_equal(g_st["nonfinite"], o_st.nonfinite)
    for k in range(K):
        for t in range(T):
            if o_st.nonfinite[k, t] > 0:
                assert np.isnan(g_st["mean"][k, t]) and np.isnan(g_st["lo"][k, t])
                continue
            s_o, s_g = o_st.std[k, t], g_st["std"][k, t]
            m_o, m_g = o_st.mean[k, t], g_st["mean"][k, t]
            if s_o == 0.0:
                assert s_g == 0.0 and m_g == m_o, (k, t, m_o, m_g, s_g)
                continue
            assert abs(s_g - s_o) <= tol * s_o, (k, t, s_o, s_g)
            assert abs(m_g - m_o) <= tol * s_o + 1e-15 * abs(m_o), (k, t, m_o, m_g, s_o)


def check_codes(o, gp, g, reps, offsets):
    """Returns the number of boundary exceptions; asserts there are no others."""
    K = len(reps)
    st = o["stats"]
    exceptions = 0
    moved = np.zeros((K, len(offsets) - 1, 256), dtype=bool)
    for k in range(K):
        diff = np.nonzero(gp["codes"][k] != o["codes"][k])[0]
        if diff.size == 0:
            continue
        t_of = np.searchsorted(offsets, diff, side="right") - 1
        for t in np.unique(t_of):
            idx = diff[t_of == t]
            u = oracle.bucket_coord(g, reps[k], idx, st.lo[k, t], st.hi[k, t])
            dist = np.abs(u - np.round(u))
            assert np.all(dist < TOL_BOUNDARY), (k, t, idx[dist >= TOL_BOUNDARY][:5],
                                                 u[dist >= TOL_BOUNDARY][:5])
            assert np.all(np.abs(gp["codes"][k][idx].astype(int) - o["codes"][k][idx]) == 1)
            moved[k, t, gp["codes"][k][idx]] = True
            moved[k, t, o["codes"][k][idx]] = True
        exceptions += diff.size
    return exceptions, moved


def check_codebook(o, gp, moved):
    st = o["stats"]
    cb_o, cb_g = o["codebook"], gp["codebook"]
    cnt_o, cnt_g = o["counts"], gp["counts"]
    K, T, _ = cb_o.shape
    worst = 0.0  # largest difference seen, in bucket widths
    for t in range(T):
        finite = st.nonfinite[:, t] == 0
        bar = codebook_tolerance(st.std[finite, t]) if finite.any() else 0.0
        for k in range(K):
            keep = ~moved[k, t]
            assert np.array_equal(cnt_g[k, t][keep], cnt_o[k, t][keep]), (k, t)
            if st.nonfinite[k, t] > 0:
                assert np.isnan(cb_g[k, t]).all()
                continue
            a = cb_g[k, t][keep].astype(np.float64)
            b = cb_o[k, t][keep].astype(np.float64)
            tol = 2 * np.spacing(np.abs(cb_o[k, t][keep])).astype(np.float64) + bar
            assert np.all(np.abs(a - b) <= tol), (k, t, np.max(np.abs(a - b) - tol))
            w = (st.hi[k, t] - st.lo[k, t]) / 256
            if w > 0 and a.size:
                worst = max(worst, float(np.max(np.abs(a - b))) / w)
    return worst


def check_merge(gp_vals, o_vals, codes_g, codes_o, cb_g, cb_o, w_hat, t_of=None, tol=TOL_REL_L2,
                exclude=None, carried=0.0):
    """Relative L2 of (delta_bar, theta_g, momentum) over elements whose codes
    match, and the explained-difference check at boundary exceptions.

    gp_vals / o_vals: dicts of 1-D arrays; codes_*: [K, n]; cb_*: [K, T, 256];
    w_hat: [K] fp32 weights of the learners in codes order; t_of: tensor index
    of every element (None = one tensor). exclude: elements already moved by an
    exception at an earlier outer step (their momentum and parameters carry
    that difference); they are checked against `carried`, the largest
    explained difference seen so far, instead of the relative-L2 bar.
    Returns (report, exception mask, largest explained difference)."""
    n = codes_g.shape[1]
    t_of = np.zeros(n, dtype=np.int64) if t_of is None else t_of
    diff = (codes_g != codes_o).any(axis=0)
    keep = ~diff if exclude is None else ~(diff | exclude)
    out = {"exception_elems": int(diff.sum())}
    for key in ("delta_bar", "theta_g", "momentum"):
        a, b = gp_vals[key], o_vals[key]
        r = rel_l2(a[keep], b[keep])
        out[key] = r
        assert r <= tol, (key, r)
    expl_max = 0.0
    if diff.any():
        idx = np.nonzero(diff)[0]
        expl = np.zeros(idx.size)
        for k in range(codes_g.shape[0]):
            vg = cb_g[k, t_of[idx], codes_g[k, idx]].astype(np.float64)
            vo = cb_o[k, t_of[idx], codes_o[k, idx]].astype(np.float64)
            expl += float(w_hat[k]) * np.abs(vg - vo)
        expl_max = float(expl.max())
        if exclude is None or not exclude[idx].any():
            for key in ("delta_bar", "momentum"):
                d = np.abs(gp_vals[key][idx].astype(np.float64) - o_vals[key][idx])
                scale = np.abs(o_vals[key][idx]).astype(np.float64)
                assert np.all(d <= expl * (1 + 1e-5) + 4e-7 * scale + 1e-30), key
    if exclude is not None and exclude.any():
        # a carried difference decays with mu and is re-injected at most by
        # lr (1 + mu) through theta: bounded by a few times the largest one
        bound = 4.0 * max(carried, expl_max)
        for key in ("delta_bar", "momentum"):
            d = np.abs(gp_vals[key][exclude].astype(np.float64) - o_vals[key][exclude])
            assert np.all(d <= bound + 4e-7 * np.abs(o_vals[key][exclude]) + 1e-30), key
    return out, diff, expl_max


def check_merge_elementwise(g0, m0, values, w, out, lr=0.7, mu=0.9):
    """Every element, from one side's own inputs to its merge: `values` holds
    one fp32 array per learner taking part (its decoded values, or its
    pseudo-gradients when unquantised) and `w` their weights as given (fp32,
    normalised here in fp64). delta_bar lies within the error of K fp32
    multiply-adds and of the fp32 normalised weights, (K + 3) u sum |w v|, of
    the fp64 weighted sum; momentum' = mu m + delta_bar and theta' = theta -
    lr (mu momentum' + delta_bar) lie within the rounding of their fp32
    results (with that of the intermediate for theta') of fp64 from the side's
    own delta_bar and momentum'. A relative L2 over a tensor can hide one
    wrong element; this cannot. Returns the largest error seen as a fraction
    of its bound, per output."""
    u = 2.0 ** -24
    floor = 1e-43  # a few fp32 subnormal spacings
    w = np.asarray(w, np.float32).astype(np.float64)
    w = w / w.sum()
    mu, lr = float(np.float32(mu)), float(np.float32(lr))
    acc = np.zeros(np.size(g0))
    mag = np.zeros_like(acc)
    for wk, v in zip(w, values):
        x = wk * np.asarray(v, np.float32).astype(np.float64)
        acc += x
        mag += np.abs(x)
    worst = {}
    d = out["delta_bar"].astype(np.float64)
    for key, got, ref, tol in _merge_terms(d, acc, mag, len(values), g0, m0, out, lr, mu, u, floor):
        r = np.abs(got - ref) / tol
        bad = np.nonzero(r > 1.0)[0]
        assert bad.size == 0, (key, bad[:5], got[bad[:5]], ref[bad[:5]])
        worst[key] = float(r.max()) if r.size else 0.0
    return worst


def _merge_terms(d, acc, mag, K, g0, m0, out, lr, mu, u, floor):
    yield "delta_bar", d, acc, (K + 3) * u * mag + floor
    mn = out["momentum"].astype(np.float64)
    ref = mu * np.asarray(m0, np.float64) + d
    yield "momentum", mn, ref, 2 * u * np.abs(ref) + floor
    gn = mu * mn + d
    ref = np.asarray(g0, np.float64) - lr * gn
    tol = 2 * u * (np.abs(ref) + lr * np.abs(gn)) + floor
    yield "theta_g", out["theta_g"].astype(np.float64), ref, tol


def compare(g, reps, numels, m=None, weights=None, present=None, min_quorum=1, lr=0.7, mu=0.9,
            clip_sigmas=6.0, quantized=True, nan_ok=False):
    offsets = np.zeros(len(numels) + 1, dtype=np.int64)
    np.cumsum(numels, out=offsets[1:])
    m0 = np.zeros_like(g) if m is None else m
    o = oracle.outer_step(g, m0, reps, offsets=offsets, weights=weights, present=present,
                          min_quorum=min_quorum, lr=lr, mu=mu, clip_sigmas=clip_sigmas,
                          quantized=quantized)
    assert o["status"] == 0
    gp = gpu_outer_step(g, reps, numels, m0, weights, present, min_quorum, lr, mu, clip_sigmas,
                        quantized)
    report = {}
    if quantized:
        check_stats(o["stats"], gp["stats"], len(reps), len(numels))
        exc, moved = check_codes(o, gp, g, reps, offsets)
        check_codebook(o, gp, moved)
        report["boundary_exceptions"] = exc
    if quantized and not nan_ok:
        K = len(reps)
        st_w, w_hat = oracle.merge_weights(weights, present, K, min_quorum)
        pres = np.ones(K, bool) if present is None else np.asarray(present, bool)
        t_of = np.searchsorted(offsets, np.arange(g.size), side="right") - 1
        res, _, _ = check_merge(gp, o, gp["codes"][pres], o["codes"][pres], gp["codebook"][pres],
                                o["codebook"][pres], w_hat[pres], t_of)
        report.update(res)
        w = np.ones(K, np.float32) if weights is None else np.asarray(weights, np.float32)
        vals = [gp["codebook"][k][t_of, gp["codes"][k]] for k in np.nonzero(pres)[0]]
        report["elementwise"] = check_merge_elementwise(g, m0, vals, w[pres], gp, lr, mu)
    else:
        if not nan_ok:
            K = len(reps)
            pres = np.ones(K, bool) if present is None else np.asarray(present, bool)
            w = np.ones(K, np.float32) if weights is None else np.asarray(weights, np.float32)
            vals = [(g - reps[k]).astype(np.float32) for k in np.nonzero(pres)[0]]
            report["elementwise"] = check_merge_elementwise(g, m0, vals, w[pres], gp, lr, mu)
        for key in ("delta_bar", "theta_g", "momentum"):
            a, b = gp[key], o[key]
            if nan_ok:
                nan = np.isnan(b)
                assert np.array_equal(np.isnan(a), nan), key
                a, b = a[~nan], b[~nan]
            r = rel_l2(a, b)
            report[key] = r
            assert r <= TOL_REL_L2, (key, r)
    upd_o = (o["theta_g"].astype(np.float64) - g)
    upd_g = (gp["theta_g"].astype(np.float64) - g)
    if nan_ok:
        keep = ~np.isnan(upd_o)
        upd_o, upd_g = upd_o[keep], upd_g[keep]
    report["update"] = rel_l2(upd_g, upd_o)
    return report, o, gp
