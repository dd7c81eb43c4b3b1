"""dl_outer_sync, the whole-model outer step with consecutive fragments
overlapped on two streams (needs a GPU).

Its results must be bitwise those of the per-fragment call sequence
(dl_pseudograd_stats -> dl_quantize -> dl_merge_outer_step over the present
learners), whichever schedule runs: the two-stream pipeline or
DL_SYNC_SERIAL. The per-fragment sequence itself is checked against the
oracle here on the first step and in the other GPU parity tests. The same
holds for the RDA merge (DL_SYNC_RDA: stats -> quantize with counts ->
dl_rda_merge_outer_step) and the ring (DL_SYNC_RING: dl_ring_outer_step per
fragment), whose per-call results the RDA and ring tests check further.
"""
import numpy as np
import pytest

import oracle
from parity import TOL_REL_L2, check_merge, rel_l2

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import pseudo_grad_sync_gb300 as dl
    dl.lib()
    return dl


# fragments of a small ragged model: tiny tensors (fp64 path), chunk tails,
# multi-chunk tensors, an empty tensor, a one-element and an empty fragment
LAYOUT = [
    [8192 * 3 + 5, 77, 4096],
    [100000],
    [1, 0, 3000, 8192],
    [8192 * 20],
    [65536, 65536 + 12],
    [1],
    [12345, 54321, 7],
    [0, 0],
]


def _model(seed, K, layout=LAYOUT):
    rng = np.random.default_rng(seed)
    g, sig = [], []
    for numels in layout:
        n = sum(numels)
        g.append((rng.standard_normal(n) * 0.02).astype(np.float32))
        s = np.concatenate([np.full(m, 10 ** rng.uniform(-3.5, -2.5)) for m in numels]) \
            if n else np.zeros(0)
        sig.append(s)
    return rng, g, sig


def _replicas(rng, g, sig, K):
    return [[(gf - rng.standard_normal(gf.size) * sf).astype(np.float32) for _ in range(K)]
            for gf, sf in zip(g, sig)]


def _dev(arrs):
    return [torch.from_numpy(a).cuda() for a in arrs]


class Run:
    """Device state of the whole model for one schedule."""

    def __init__(self, dl, g, layout=LAYOUT):
        self.frags = [dl.Fragment(numels) for numels in layout]
        self.g = _dev(g)
        self.m = [torch.zeros_like(x) for x in self.g]
        self.db = [torch.full_like(x, float("nan")) for x in self.g]

    def host(self):
        return ([x.cpu().numpy() for x in self.g], [x.cpu().numpy() for x in self.m],
                [x.cpu().numpy() for x in self.db])


def _per_call(dl, run, reps_d, K, weights, present):
    syncs = []
    for j, F in enumerate(run.frags):
        sync = dl.OuterSync(F, K)
        sync.step(run.g[j], run.m[j], reps_d[j], weights=weights[j], present=present[j],
                  delta_bar=run.db[j])
        syncs.append(sync)
    return syncs


def _assert_same(a, b):
    for xa, xb in zip(a, b):
        for ya, yb in zip(xa, xb):
            assert np.array_equal(ya.view(np.uint32), yb.view(np.uint32))


def test_pipeline_bitwise_equals_serial_and_per_call(dl):
    K, steps = 5, 3
    rng, g, sig = _model(1, K)
    P = len(LAYOUT)
    runs = {name: Run(dl, g) for name in ("pipe", "serial", "calls")}
    ms = dl.ModelSync(runs["pipe"].frags, K)
    ms_serial = dl.ModelSync(runs["serial"].frags, K)
    host_g = [x.copy() for x in g]
    host_m = [np.zeros_like(x) for x in g]
    for step in range(steps):
        present = [(rng.random(K) < 0.7).astype(np.uint8) for _ in range(P)]
        for p in present:
            p[rng.integers(K)] = 1
        weights = [rng.uniform(0.5, 1.5, K).astype(np.float32) for _ in range(P)]
        # every schedule sees the same Delta, applied to its own theta_g
        deltas = [[(rng.standard_normal(gf.size) * sf).astype(np.float32) for _ in range(K)]
                  for gf, sf in zip(g, sig)]

        def reps_of(run):
            return [[run.g[j] - torch.from_numpy(d).cuda() for d in deltas[j]] for j in range(P)]

        ms.step(runs["pipe"].g, runs["pipe"].m, reps_of(runs["pipe"]), weights=weights,
                present=present, delta_bar=runs["pipe"].db)
        ms_serial.step(runs["serial"].g, runs["serial"].m, reps_of(runs["serial"]),
                       weights=weights, present=present, delta_bar=runs["serial"].db,
                       flags=dl.DL_SYNC_SERIAL)
        syncs = _per_call(dl, runs["calls"], reps_of(runs["calls"]), K, weights, present)
        torch.cuda.synchronize()
        out = {k: r.host() for k, r in runs.items()}
        _assert_same(out["pipe"], out["serial"])
        _assert_same(out["pipe"], out["calls"])
        assert dl.read_device_status(ms.workspace) == 0
        if step == 0:
            # the oracle on every fragment, present learners in order
            for j in range(P):
                if sum(LAYOUT[j]) == 0:
                    continue
                idx = [k for k in range(K) if present[j][k]]
                reps = [(host_g[j] - deltas[j][k]).astype(np.float32) for k in idx]
                off = np.concatenate([[0], np.cumsum(LAYOUT[j])]).astype(np.int64)
                o = oracle.outer_step(host_g[j], host_m[j], reps, offsets=off,
                                      weights=weights[j][idx])
                assert o["status"] == 0
                gg, mm, db = (x[j] for x in out["pipe"])
                n = gg.size
                # codes and codebooks of the per-call run (whose outputs the
                # pipeline matched bit for bit); boundary exceptions explained
                sy = syncs[j]
                codes_g = np.stack([sy.codes[i][:n].cpu().numpy() for i in range(len(idx))])
                cb_g = sy.codebook[:len(idx)].cpu().numpy()
                t_of = np.searchsorted(off, np.arange(n), side="right") - 1
                w_hat = oracle.merge_weights(weights[j][idx], None, len(idx))[1]
                check_merge({"delta_bar": db, "theta_g": gg, "momentum": mm}, o, codes_g,
                            o["codes"], cb_g, o["codebook"], w_hat, t_of)


def test_unquantized_mode_matches_oracle_and_merge(dl):
    K = 3
    rng, g, sig = _model(2, K)
    reps = _replicas(rng, g, sig, K)
    a, b = Run(dl, g), Run(dl, g)
    reps_d = [_dev(r) for r in reps]
    dl.outer_sync(a.frags, a.g, a.m, reps_d, K, flags=dl.DL_SYNC_UNQUANTIZED, delta_bar=a.db)
    for j, F in enumerate(b.frags):
        dl.merge_outer_step(b.g[j], b.m[j], F, replicas=reps_d[j], delta_bar=b.db[j])
    torch.cuda.synchronize()
    _assert_same(a.host(), b.host())
    for j, numels in enumerate(LAYOUT):
        if sum(numels) == 0:
            continue
        off = np.concatenate([[0], np.cumsum(numels)]).astype(np.int64)
        o = oracle.outer_step(g[j], np.zeros_like(g[j]), reps[j], offsets=off, quantized=False)
        gg, mm, db = (x[j] for x in a.host())
        for key, v in (("delta_bar", db), ("theta_g", gg), ("momentum", mm)):
            assert rel_l2(v, o[key]) <= TOL_REL_L2, (j, key)


def test_quorum_failure_leaves_every_fragment_untouched(dl):
    K = 4
    rng, g, sig = _model(3, K)
    reps_d = [_dev(r) for r in _replicas(rng, g, sig, K)]
    run = Run(dl, g)
    ms = dl.ModelSync(run.frags, K)
    present = [np.ones(K, np.uint8) for _ in LAYOUT]
    present[-1][:] = [1, 0, 0, 0]  # the last fragment alone misses the quorum
    before = run.host()
    with pytest.raises(dl.DLError) as e:
        ms.step(run.g, run.m, reps_d, present=present, min_quorum=2, delta_bar=run.db)
    assert e.value.status == -3
    torch.cuda.synchronize()
    _assert_same(run.host(), before)


def test_many_fragments_single_learner(dl):
    """K = 1 over 40 small fragments: the event ring is reused many times."""
    layout = [[int(n)] for n in np.random.default_rng(5).integers(1, 30000, 40)]
    rng, g, sig = _model(4, 1, layout)
    reps_d = [_dev(r) for r in _replicas(rng, g, sig, 1)]
    a, b = Run(dl, g, layout), Run(dl, g, layout)
    dl.ModelSync(a.frags, 1).step(a.g, a.m, reps_d, delta_bar=a.db)
    _per_call(dl, b, reps_d, 1, [None] * len(layout), [None] * len(layout))
    torch.cuda.synchronize()
    _assert_same(a.host(), b.host())


def _per_call_mode(dl, mode, run, reps_d, K, weights, present):
    """The per-fragment calls that DL_SYNC_RDA / DL_SYNC_RING stand for, over
    the present learners in ascending order."""
    for j, F in enumerate(run.frags):
        if mode == "ring":
            dl.ring_outer_step(run.g[j], run.m[j], F, reps_d[j], weights=weights[j],
                               present=present[j], delta_bar=run.db[j])
            continue
        idx = [k for k in range(K) if present[j][k]]
        reps = [reps_d[j][k] for k in idx]
        st = dl.pseudograd_stats(run.g[j], reps, F)
        counts = torch.empty((len(idx), F.T, 256), dtype=torch.int32, device="cuda")
        codes, cb = dl.quantize(run.g[j], reps, F, st, counts=counts)
        dl.rda_merge_outer_step(run.g[j], run.m[j], F, codes, cb, counts,
                                weights=weights[j][idx], delta_bar=run.db[j])


@pytest.mark.parametrize("mode", ["rda", "ring"])
def test_rda_and_ring_modes_bitwise_equal_per_call(dl, mode):
    K, steps = 4, 2
    flag = dl.DL_SYNC_RDA if mode == "rda" else dl.DL_SYNC_RING
    rng, g, sig = _model(6 if mode == "rda" else 7, K)
    P = len(LAYOUT)
    runs = {name: Run(dl, g) for name in ("pipe", "serial", "calls")}
    ms = dl.ModelSync(runs["pipe"].frags, K, mode=flag)
    ms_serial = dl.ModelSync(runs["serial"].frags, K, mode=flag)
    for _step in range(steps):
        present = [(rng.random(K) < 0.75).astype(np.uint8) for _ in range(P)]
        for p in present:
            p[rng.integers(K)] = 1
        weights = [rng.uniform(0.5, 1.5, K).astype(np.float32) for _ in range(P)]
        deltas = [[(rng.standard_normal(gf.size) * sf).astype(np.float32) for _ in range(K)]
                  for gf, sf in zip(g, sig)]

        def reps_of(run):
            return [[run.g[j] - torch.from_numpy(d).cuda() for d in deltas[j]] for j in range(P)]

        ms.step(runs["pipe"].g, runs["pipe"].m, reps_of(runs["pipe"]), weights=weights,
                present=present, delta_bar=runs["pipe"].db)
        ms_serial.step(runs["serial"].g, runs["serial"].m, reps_of(runs["serial"]),
                       weights=weights, present=present, delta_bar=runs["serial"].db,
                       flags=dl.DL_SYNC_SERIAL)
        _per_call_mode(dl, mode, runs["calls"], reps_of(runs["calls"]), K, weights, present)
        torch.cuda.synchronize()
        out = {k: r.host() for k, r in runs.items()}
        _assert_same(out["pipe"], out["serial"])
        _assert_same(out["pipe"], out["calls"])
        assert dl.read_device_status(ms.workspace) == 0
        assert all(np.isfinite(x).all() for x in out["pipe"][0])


def test_shutdown_releases_and_the_next_call_recreates(dl):
    """dl_shutdown drops the side stream and events; the next pipelined call
    creates them again and gives the same bits."""
    K = 3
    rng, g, sig = _model(8, K)
    reps_d = [_dev(r) for r in _replicas(rng, g, sig, K)]
    a, b = Run(dl, g), Run(dl, g)
    ms = dl.ModelSync(a.frags, K)
    ms.step(a.g, a.m, reps_d, delta_bar=a.db)
    dl.shutdown()  # with a's work possibly still in flight
    dl.shutdown()
    ms.step(b.g, b.m, reps_d, delta_bar=b.db)
    torch.cuda.synchronize()
    _assert_same(a.host(), b.host())
    assert dl.read_device_status(ms.workspace) == 0
