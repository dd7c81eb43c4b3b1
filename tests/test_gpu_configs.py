"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (one dl_pseudograd_stats / dl_quantize / dl_merge_outer_step sequence per
fragment), on sampled tensors (needs a GPU; minutes).

Statistics, codebooks and the merge are per tensor, so a sampled tensor can be
checked against the oracle run on that tensor alone. Sampled tensors come from
the seeded host generator (identical bits on both sides); the rest of each
fragment is filled on the device with the same distributions from torch's
generator, which only the GPU sees. Every checked fragment samples its
smallest tensor, its smallest matrix and its largest matrix.

Multi-step workloads: before every step after the first, the oracle chain's
theta and momentum of each sampled tensor are copied into the GPU buffers
(values flow from the oracle to the GPU only, never back), and both sides
build that step's learner replicas from that common theta. Every step is
therefore compared on identical inputs and held to the same bar as the first:
codes bit-exact except counted boundary exceptions, statistics within 5e-9,
relative L2 <= 1e-6 on Delta_bar, theta and momentum.
"""
import numpy as np
import pytest

import oracle
import synthetic
from parity import (TOL_REL_L2, TOL_STATS, check_codebook, check_codes, check_merge, check_stats,
                    rel_l2)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import pseudo_grad_sync_gb300 as dl
    dl.lib()


def _delta_host(wl, t, k, step):
    """Delta of learner k, tensor t, outer step `step` (fp32, host generator)."""
    z = np.zeros(wl.numels[t], dtype=np.float32)
    return -synthetic.replica_f32(synthetic.key(wl.seed, 2, step, t, k), 0, z, wl.tensor_scale(t),
                                  wl.delta_dist)


def _delta_device(wl, t, m, gen):
    x = torch.randn(m, device="cuda", generator=gen)
    if wl.delta_dist == 1:  # Student-t(3)
        c = torch.randn(3, m, device="cuda", generator=gen).square_().sum(0).div_(3.0)
        x.div_(c.sqrt_())
    return x.mul_(wl.tensor_scale(t))


def _decode_bound_everywhere(run, g_before, reps, idx):
    """Every element of every present learner, the whole fragment: the decoded
    value cb_k[t][code] lies within one bucket width of clamp(Delta, lo, hi).
    A correct code puts both in the same bucket, a counted boundary exception
    puts the value in the neighbouring one, still within a width. This holds
    at any size, so it covers what the oracle cannot run on: a wrong code,
    codebook entry or tensor mapping anywhere in the fragment fails it."""
    st = run.dl.stats_to_host(run.sync.stats[:len(idx)])
    ends = torch.tensor(run.off[1:], device="cuda")
    step = 1 << 27  # elements per slice: bounds the temporaries at a few GB
    for s, k in enumerate(idx):
        lo = torch.tensor(st["lo"][s], device="cuda", dtype=torch.float64)
        hi = torch.tensor(st["hi"][s], device="cuda", dtype=torch.float64)
        for a in range(0, run.n, step):
            b = min(run.n, a + step)
            t_of = torch.searchsorted(ends, torch.arange(a, b, device="cuda"), right=True)
            d = (g_before[a:b] - reps[k][a:b]).double()  # Delta as the kernels form it (fp32)
            dc = torch.clamp(d, lo[t_of], hi[t_of])
            v = run.sync.codebook[s][t_of, run.sync.codes[s][a:b].long()].double()
            bound = (hi - lo)[t_of] / 256.0 * (1 + 1e-5) + 1e-7 * v.abs()
            bad = int(((v - dc).abs() > bound).sum())
            assert bad == 0, (k, a, bad)
            del t_of, d, dc, v, bound


def _stats_everywhere(run, g_before, reps, idx, clip=6.0):
    """Every tensor of every present learner: count, non-finite count, mean,
    std (population), lo and hi against torch fp64 two-pass sums over the same
    fp32 Delta, at the oracle's bar (std within TOL_STATS relative, mean
    within TOL_STATS std, lo and hi within that of mean -/+ 6 std)."""
    st = run.dl.stats_to_host(run.sync.stats[:len(idx)])
    T = len(run.numels)
    assert (st["count"] == np.asarray(run.numels)[None, :]).all()
    assert (st["nonfinite"] == 0).all()
    for s, k in enumerate(idx):
        mus, sds = [], []
        for i in range(T):
            a, b = int(run.off[i]), int(run.off[i + 1])
            if b == a:
                mus.append(torch.zeros((), dtype=torch.float64, device="cuda"))
                sds.append(mus[-1])
                continue
            d = (g_before[a:b] - reps[k][a:b]).double()
            mu = d.mean()
            mus.append(mu)
            sds.append((d - mu).square_().mean().sqrt())
            del d
        mu = torch.stack(mus).cpu().numpy()
        sd = torch.stack(sds).cpu().numpy()
        assert (np.abs(st["std"][s] - sd) <= TOL_STATS * sd).all(), k
        assert (np.abs(st["mean"][s] - mu) <= TOL_STATS * sd + 1e-15 * np.abs(mu)).all(), k
        for key, ref in (("lo", mu - clip * sd), ("hi", mu + clip * sd)):
            tol = (1 + clip) * TOL_STATS * sd + 1e-15 * np.abs(ref)
            assert (np.abs(st[key][s] - ref) <= tol).all(), (k, key)


def _merge_everywhere(run, g_before, m_before, db, idx, weights, lr=0.7, mu=0.9):
    """Every element of the fragment, from the kernel's own codes and codebooks:
    delta_bar against their fp64 weighted sum, within the error of K fp32
    multiply-adds and of the fp32 normalised weights, (K + 3) u sum|w v|; then
    m' = mu m + D and theta' = theta - lr (mu m' + D) against fp64 from the
    kernel's own D and m', each within the rounding of its fp32 result (with
    the rounding of the intermediate fp32 mu m' + D for theta'). A wrong
    codebook row, weight, absent learner read or update term anywhere in the
    fragment fails it; the oracle holds the sampled tensors to the bits."""
    u = 2.0 ** -24
    w = np.ones(len(idx)) if weights is None else np.asarray(weights, np.float32)[idx]
    w = w.astype(np.float64)
    w_hat = w / w.sum()
    mu, lr = float(np.float32(mu)), float(np.float32(lr))  # the fp32 constants the kernels get
    ends = torch.tensor(run.off[1:], device="cuda")
    step = 1 << 27
    for a in range(0, run.n, step):
        b = min(run.n, a + step)
        t_of = torch.searchsorted(ends, torch.arange(a, b, device="cuda"), right=True)
        acc = torch.zeros(b - a, dtype=torch.float64, device="cuda")
        mag = torch.zeros_like(acc)
        for s in range(len(idx)):
            v = run.sync.codebook[s][t_of, run.sync.codes[s][a:b].long()].double() * w_hat[s]
            acc += v
            mag += v.abs()
            del v
        d = db[a:b].double()
        bad = int(((d - acc).abs() > (len(idx) + 3) * u * mag + 1e-44).sum())
        assert bad == 0, ("delta_bar", a, bad)
        del acc, mag, t_of
        m_new = run.m[a:b].double()
        ref = mu * m_before[a:b].double() + d
        bad = int(((m_new - ref).abs() > 2 * u * ref.abs() + 1e-44).sum())
        assert bad == 0, ("momentum", a, bad)
        gn = mu * m_new + d
        ref = g_before[a:b].double() - lr * gn
        tol = 2 * u * (ref.abs() + lr * gn.abs()) + 1e-44
        bad = int(((run.g[a:b].double() - ref).abs() > tol).sum())
        assert bad == 0, ("theta", a, bad)
        del d, m_new, ref, gn, tol


class FragmentRun:
    """Device state of one fragment and host copies of its sampled tensors."""

    def __init__(self, wl, tensors, sampled, K=None, gen_seed=0):
        import pseudo_grad_sync_gb300 as dl

        self.dl, self.wl, self.tensors = dl, wl, tensors
        self.K = wl.K if K is None else K
        self.numels = [wl.numels[t] for t in tensors]
        self.off = synthetic.offsets_of(self.numels)
        self.n = int(self.off[-1])
        self.frag = dl.Fragment(self.numels)
        self.gen = torch.Generator(device="cuda")
        self.gen.manual_seed(gen_seed)
        self.g = torch.empty(self.n, device="cuda")
        self.m = torch.zeros(self.n, device="cuda")
        self.host = {}  # t -> dict(a, b, g, m) oracle chain of a sampled tensor
        for i, t in enumerate(tensors):
            a, b = int(self.off[i]), int(self.off[i + 1])
            if t in sampled:
                gh = wl.theta_global(t)
                self.g[a:b].copy_(torch.from_numpy(gh))
                self.host[t] = {"i": i, "a": a, "b": b, "g": gh, "m": np.zeros_like(gh)}
            else:
                self.g[a:b].normal_(0.0, wl.theta_std, generator=self.gen)
        self.sync = dl.OuterSync(self.frag, self.K)

    def replicas(self, step):
        reps = []
        for k in range(self.K):
            r = torch.empty(self.n, device="cuda")
            for i, t in enumerate(self.tensors):
                a, b = int(self.off[i]), int(self.off[i + 1])
                if t in self.host:
                    d = torch.from_numpy(_delta_host(self.wl, t, k, step)).cuda()
                else:
                    d = _delta_device(self.wl, t, b - a, self.gen)
                torch.sub(self.g[a:b], d, out=r[a:b])
            reps.append(r)
        return reps

    def step(self, step, present=None, weights=None, twin=None, everywhere=False):
        """One outer step through the per-call sequence. With `twin` (a
        ModelSync over this fragment) the same step also runs through
        dl_outer_sync, the call bench.py times, on copies of theta and m, and
        both must give the same bits. With `everywhere`, every element of the
        fragment is held to the decode bound (_decode_bound_everywhere), its
        statistics to torch fp64 (_stats_everywhere), and its merge and update
        to fp64 from the kernel's codes (_merge_everywhere)."""
        # the oracle chain's state of the sampled tensors goes into the GPU
        # buffers (a no-op at step 0, where both hold the initial theta and 0)
        for h in self.host.values():
            self.g[h["a"]:h["b"]].copy_(torch.from_numpy(h["g"]))
            self.m[h["a"]:h["b"]].copy_(torch.from_numpy(h["m"]))
        reps = self.replicas(step)
        if twin is not None:
            g2, m2, db2 = self.g.clone(), self.m.clone(), torch.empty_like(self.g)
            twin.step([g2], [m2], [reps], weights=None if weights is None else [weights],
                      present=None if present is None else [present], delta_bar=[db2])
        db = torch.empty_like(self.g)
        counts = torch.empty((self.K, self.frag.T, 256), dtype=torch.int32, device="cuda")
        g_before = self.g.clone() if everywhere else None
        m_before = self.m.clone() if everywhere else None
        idx = self.sync.step(self.g, self.m, reps, weights=weights, present=present, delta_bar=db,
                             counts=counts)
        torch.cuda.synchronize()
        if everywhere:
            _stats_everywhere(self, g_before, reps, idx)
            _decode_bound_everywhere(self, g_before, reps, idx)
            _merge_everywhere(self, g_before, m_before, db, idx, weights)
            del g_before, m_before
        del reps
        if twin is not None:
            for a, b in ((g2, self.g), (m2, self.m), (db2, db)):
                assert torch.equal(a.view(torch.int32), b.view(torch.int32))
            assert self.dl.read_device_status(twin.workspace) == 0
            del g2, m2, db2
        return idx, db, counts

    def check(self, step, idx, db, counts, present=None, weights=None):
        """Oracle on every sampled tensor from the same inputs; returns the
        number of boundary exceptions."""
        dl = self.dl
        st_all = dl.stats_to_host(self.sync.stats[:len(idx)])
        cb_all = self.sync.codebook[:len(idx)].cpu().numpy()
        cnt_all = counts[:len(idx)].cpu().numpy().view(np.uint32)
        exc = 0
        for t, h in self.host.items():
            i, a, b = h["i"], h["a"], h["b"]
            # the oracle learners are the present ones, in order, with their weights
            d = [_delta_host(self.wl, t, k, step) for k in idx]
            reps = [(h["g"] - dk).astype(np.float32) for dk in d]
            w = None if weights is None else np.asarray(weights, np.float32)[idx]
            o = oracle.outer_step(h["g"], h["m"], reps, weights=w)
            assert o["status"] == 0
            gp = {
                "stats": {key: v[:, i:i + 1] for key, v in st_all.items()},
                "codes": np.stack([self.sync.codes[s][a:b].cpu().numpy() for s in range(len(idx))]),
                "codebook": cb_all[:, i:i + 1], "counts": cnt_all[:, i:i + 1],
            }
            check_stats(o["stats"], gp["stats"], len(idx), 1)
            n_exc, moved = check_codes(o, gp, h["g"], reps, np.array([0, b - a]))
            check_codebook(o, gp, moved)
            exc += n_exc
            w_hat = oracle.merge_weights(w, None, len(idx))[1]
            gvals = {key: dev[a:b].cpu().numpy() for key, dev in
                     (("delta_bar", db), ("theta_g", self.g), ("momentum", self.m))}
            res, _, _ = check_merge(gvals, o, gp["codes"], o["codes"], gp["codebook"],
                                    o["codebook"], w_hat)
            print(f"step {step} tensor {t} n={b - a} K={len(idx)} {res}")
            # the oracle chain carries on from its own outputs
            h["g"], h["m"] = o["theta_g"], o["momentum"]
        return exc


def _plan(wl):
    frag_of, load = oracle.plan_fragments(wl.numels, wl.n_frags)
    return [[t for t in range(wl.n_tensors) if frag_of[t] == f] for f in range(wl.n_frags)], load


def _smallest(wl, ts, kind="any"):
    cand = [t for t in ts if kind == "any" or wl.numels[t] > 65536]
    return min(cand, key=lambda t: wl.numels[t]) if cand else None


def _largest(wl, ts):
    return max(ts, key=lambda t: (wl.numels[t], -t))


def _sampled(wl, ts):
    """Smallest tensor, smallest matrix and largest matrix of a fragment."""
    return {_smallest(wl, ts), _smallest(wl, ts, "matrix"), _largest(wl, ts)} - {None}


def test_decoder_1b_every_fragment():
    """1.1B set, K=4, P=24: every fragment synced; its smallest tensor, smallest
    matrix and largest matrix checked against the oracle."""
    wl = synthetic.decoder_1b()
    frags, load = _plan(wl)
    assert load.max() == 65536000 and load.sum() == wl.n_elems
    total_exc = 0
    for f, ts in enumerate(frags):
        sampled = _sampled(wl, ts)
        run = FragmentRun(wl, ts, sampled, gen_seed=f)
        idx, db, counts = run.step(0, everywhere=True)
        assert torch.isfinite(run.g).all() and torch.isfinite(run.m).all()
        total_exc += run.check(0, idx, db, counts)
        del run
        torch.cuda.empty_cache()
    print("decoder_1b boundary exceptions:", total_exc)


def test_decoder_10b_fragment_three_steps():
    """10B set, K=14: the median (~415M-element) fragment over 3 outer steps
    with momentum carried; each step also through dl_outer_sync (bitwise the
    same), and every element of every learner held to the decode bound."""
    wl = synthetic.decoder_10b()
    frags, load = _plan(wl)
    f = int(np.argsort(load, kind="stable")[len(load) // 2])  # bench.py's fragment
    ts = frags[f]
    sampled = _sampled(wl, ts)
    run = FragmentRun(wl, ts, sampled, gen_seed=3)
    assert 4e8 < run.n < 4.3e8
    # the same steps through dl_outer_sync, as bench.py runs them: bitwise equal
    twin = run.dl.ModelSync([run.frag], run.K)
    for step in range(wl.steps):
        idx, db, counts = run.step(step, twin=twin, everywhere=True)
        run.check(step, idx, db, counts)
    assert torch.isfinite(run.g).all()


def test_ragged_heavy_single_batch():
    """2000 ragged tensors (64..16Mi, every 10th a 4096 norm), K=8, Student-t(3)
    pseudo-gradients, all in one launch per kernel."""
    wl = synthetic.ragged_heavy()
    ts = list(range(wl.n_tensors))
    sizes = np.array(wl.numels)
    order = np.argsort(sizes)
    sampled = {int(order[0]), 9, int(order[len(order) // 2]), int(order[-200]), int(order[-1])}
    run = FragmentRun(wl, ts, sampled, gen_seed=4)
    idx, db, counts = run.step(0, everywhere=True)
    exc = run.check(0, idx, db, counts)
    st = run.dl.stats_to_host(run.sync.stats)
    assert (st["nonfinite"] == 0).all() and (st["count"] == sizes[None, :]).all()
    # heavy tails: Student-t(3) puts ~1.9e-3 of the mass beyond 6 sigma
    cnt = counts.cpu().numpy().view(np.uint32).astype(np.int64)
    clipped = (cnt[:, :, 0] + cnt[:, :, 255]).sum() / (wl.K * wl.n_elems)
    assert 5e-4 < clipped < 5e-3, clipped
    print("ragged boundary exceptions:", exc, "edge-bucket fraction:", clipped)


def test_quorum_10b_fragments_and_steps():
    """10B shapes, K=16, random present subsets of size 1..16 and weights
    U[0.5, 1.5] per (fragment, step), 4 outer steps with per-fragment momentum;
    three multi-tensor fragments checked against the oracle at every step."""
    wl = synthetic.quorum_10b()
    frags, load = _plan(wl)
    mixed = [f for f, ts in enumerate(frags) if len(ts) > 1]  # not the embedding / lm_head alone
    for f in (mixed[0], mixed[len(mixed) // 2], mixed[-1]):
        ts = frags[f]
        sampled = _sampled(wl, ts)
        run = FragmentRun(wl, ts, sampled, gen_seed=5 + f)
        for step in range(wl.steps):
            present = wl.present(f, step)
            weights = wl.weights(f, step)
            idx, db, counts = run.step(step, present=present, weights=weights, everywhere=True)
            assert idx == [k for k in range(wl.K) if present[k]]
            run.check(step, idx, db, counts, present=present, weights=weights)
        assert torch.isfinite(run.g).all()
        del run
        torch.cuda.empty_cache()


def test_quorum_10b_embedding_fragment():
    """The 525M-element embedding, a fragment of its own, first outer step:
    the largest single tensor of the workloads (boundary exceptions appear
    here and must be fully explained by their flipped codes)."""
    wl = synthetic.quorum_10b()
    frags, load = _plan(wl)
    f = int(np.argmax(load))
    ts = frags[f]
    assert len(ts) == 1 and wl.numels[ts[0]] == 525336576
    run = FragmentRun(wl, ts, {ts[0]}, gen_seed=7)
    present, weights = wl.present(f, 0), wl.weights(f, 0)
    idx, db, counts = run.step(0, present=present, weights=weights, everywhere=True)
    run.check(0, idx, db, counts, present=present, weights=weights)


def _learner_whole_model(wl, sampled):
    """Stats + quantise of one learner's whole model as one ragged batch (the
    learner-side quantiser); sampled tensors checked against the oracle."""
    run = FragmentRun(wl, list(range(wl.n_tensors)), sampled, K=1, gen_seed=11)
    dl = run.dl
    reps = run.replicas(0)
    counts = torch.empty((1, run.frag.T, 256), dtype=torch.int32, device="cuda")
    dl.pseudograd_stats(run.g, reps, run.frag, 6.0, run.sync.stats, run.sync.ws_stats)
    dl.quantize(run.g, reps, run.frag, run.sync.stats, run.sync.codes, run.sync.codebook, counts,
                run.sync.ws_quant)
    torch.cuda.synchronize()
    del reps
    st_all = dl.stats_to_host(run.sync.stats)
    cb_all = run.sync.codebook.cpu().numpy()
    cnt_all = counts.cpu().numpy().view(np.uint32)
    assert (st_all["count"][0] == np.asarray(wl.numels)).all()
    assert (st_all["nonfinite"] == 0).all()
    exc = 0
    for t, h in run.host.items():
        i, a, b = h["i"], h["a"], h["b"]
        rep = (h["g"] - _delta_host(wl, t, 0, 0)).astype(np.float32)
        st = oracle.stats(h["g"], [rep])
        codes_o, cb_o, cnt_o = oracle.quantize(h["g"], [rep], st)
        o = {"stats": st, "codes": codes_o, "codebook": cb_o, "counts": cnt_o}
        gp = {"stats": {key: v[:, i:i + 1] for key, v in st_all.items()},
              "codes": run.sync.codes[0][a:b].cpu().numpy()[None, :],
              "codebook": cb_all[:, i:i + 1], "counts": cnt_all[:, i:i + 1]}
        check_stats(st, gp["stats"], 1, 1)
        n_exc, moved = check_codes(o, gp, h["g"], [rep], np.array([0, b - a]))
        check_codebook(o, gp, moved)
        exc += n_exc
        print(f"learner tensor {t} n={b - a} boundary exceptions {n_exc}")
    return exc


def test_learner_1b_whole_model():
    """One learner, the whole 1.1B set (201 tensors, 1.1G elements) in one
    launch per kernel: smallest tensor, a norm vector, a 2048x2048 and the
    embedding checked against the oracle."""
    wl = synthetic.learner_1b()
    sizes = np.asarray(wl.numels)
    sampled = {int(np.argmin(sizes)), int(np.nonzero(sizes == 2048)[0][0]),
               int(np.nonzero(sizes == 2048 * 2048)[0][0]), 0}
    _learner_whole_model(wl, sampled)


def test_learner_10b_whole_model():
    """One learner, the whole 10B set (381 tensors, 10.2G elements: element
    indices far past 2^32) in one launch per kernel; the lm_head, the final
    norm and the last layer's down projection (all starting past 9.6G) and
    the first layer's q projection are checked against the oracle."""
    wl = synthetic.learner_10b()
    T = wl.n_tensors
    assert wl.numels[T - 5] == 4096 * 14336 and wl.numels[T - 2] == 4096
    _learner_whole_model(wl, {T - 1, T - 2, T - 5, 1})


def _rda_coefficients(cb, cnt, codes, w_hat):
    """Per-learner scale c_k of the RDA reading for one tensor (fp64, from one
    side's quantisation): D = sum_k c_k v_k with n_k = ||v_k||,
    r = sum_k w_k n_k, u = sum_k (w_k / n_k) v_k, c_k = (w_k / n_k) r / ||u||.
    Used only to bound the difference a flipped code makes to D."""
    K = len(codes)
    cbd = cb.astype(np.float64)
    n = np.sqrt([(cnt[k].astype(np.float64) * cbd[k] ** 2).sum() for k in range(K)])
    r = float((w_hat * n).sum())
    u = np.zeros(codes[0].size)
    for k in range(K):
        if n[k] > 0:
            u += (w_hat[k] / n[k]) * cbd[k][codes[k]]
    nu = float(np.linalg.norm(u))
    return np.array([(w_hat[k] / n[k]) * r / nu if n[k] > 0 and nu > 0 else 0.0
                     for k in range(K)])


def test_ring_and_rda_on_a_full_decoder_1b_fragment():
    """The largest multi-tensor 1.1B fragment (K=4) through the ring and the RDA
    merge, as bench.py --mode ring / rda run it. Both work tensor by tensor,
    so the sampled tensors are checked against the oracle on their own, end
    to end from the same host data: the ring's D within one bucket width of
    its last quantiser at a few elements and to 1e-6 elsewhere; RDA's
    statistics, codes (boundary exceptions counted) and codebooks, then D,
    theta and momentum to 1e-6 where every learner's code matches and,
    where one differs, by exactly what the flipped codes explain (the page
    gives RDA no formula: it is held to the oracle's reading)."""
    import pseudo_grad_sync_gb300 as dl

    wl = synthetic.decoder_1b()
    frags, load = _plan(wl)
    f = max((f for f, ts in enumerate(frags) if len(ts) > 1), key=lambda f: load[f])
    ts = frags[f]
    sampled = _sampled(wl, ts)
    run = FragmentRun(wl, ts, sampled, gen_seed=9)
    reps = run.replicas(0)
    g0 = run.g.clone()
    # ring
    db = torch.empty_like(run.g)
    dl.ring_outer_step(run.g, run.m, run.frag, reps, delta_bar=db)
    torch.cuda.synchronize()
    for t, h in run.host.items():
        a, b = h["a"], h["b"]
        rh = [(h["g"] - _delta_host(wl, t, k, 0)).astype(np.float32) for k in range(wl.K)]
        st, g_o, m_o, d_o = oracle.ring_outer_step(h["g"], h["m"], rh)
        d_g = db[a:b].cpu().numpy()
        acc = np.zeros(b - a)
        width = 0.0
        for k in range(wl.K - 1):
            acc = acc + 0.25 * (h["g"] - rh[k]).astype(np.float32).astype(np.float64)
            width = max(width, 12.0 * acc.std() / 256.0)
        diff = np.abs(d_g.astype(np.float64) - d_o)
        far = diff > 1e-3 * width
        assert far.mean() <= 1e-4 and np.all(diff[far] <= 1.1 * width), (t, far.sum())
        assert rel_l2(d_g[~far], d_o[~far]) <= TOL_REL_L2, t
        print(f"ring tensor {t} n={b - a} moved elements {int(far.sum())}")
    # RDA from a fresh copy of theta_g: both sides from the same host data
    run.g.copy_(g0)
    run.m.zero_()
    counts = torch.empty((wl.K, run.frag.T, 256), dtype=torch.int32, device="cuda")
    dl.pseudograd_stats(run.g, reps, run.frag, 6.0, run.sync.stats, run.sync.ws_stats)
    dl.quantize(run.g, reps, run.frag, run.sync.stats, run.sync.codes, run.sync.codebook, counts,
                run.sync.ws_quant)
    db.fill_(float("nan"))
    dl.rda_merge_outer_step(run.g, run.m, run.frag, run.sync.codes, run.sync.codebook, counts,
                            delta_bar=db)
    torch.cuda.synchronize()
    st_all = dl.stats_to_host(run.sync.stats)
    cb_all = run.sync.codebook.cpu().numpy()
    cnt_all = counts.cpu().numpy().view(np.uint32)
    w_hat = np.full(wl.K, 1.0 / wl.K)
    total_exc = 0
    for t, h in run.host.items():
        i, a, b = h["i"], h["a"], h["b"]
        rh = [(h["g"] - _delta_host(wl, t, k, 0)).astype(np.float32) for k in range(wl.K)]
        st = oracle.stats(h["g"], rh)
        codes_o, cb_o, cnt_o = oracle.quantize(h["g"], rh, st)
        stat, g_o, m_o, d_o = oracle.rda_merge_outer_step(h["g"], h["m"], list(codes_o), cb_o,
                                                          cnt_o)
        assert stat == 0
        o = {"stats": st, "codes": codes_o, "codebook": cb_o, "counts": cnt_o,
             "delta_bar": d_o, "theta_g": g_o, "momentum": m_o}
        gp = {"stats": {key: v[:, i:i + 1] for key, v in st_all.items()},
              "codes": np.stack([run.sync.codes[k][a:b].cpu().numpy() for k in range(wl.K)]),
              "codebook": cb_all[:, i:i + 1], "counts": cnt_all[:, i:i + 1]}
        check_stats(st, gp["stats"], wl.K, 1)
        n_exc, moved = check_codes(o, gp, h["g"], rh, np.array([0, b - a]))
        check_codebook(o, gp, moved)
        total_exc += n_exc
        c = _rda_coefficients(cb_o[:, 0], cnt_o[:, 0], list(codes_o), w_hat)
        gvals = {key: dev[a:b].cpu().numpy() for key, dev in
                 (("delta_bar", db), ("theta_g", run.g), ("momentum", run.m))}
        res, _, _ = check_merge(gvals, o, gp["codes"], codes_o, gp["codebook"], cb_o, c)
        print(f"rda tensor {t} n={b - a} {res}")
    print("rda boundary exceptions:", total_exc)
