"""Radial-Directional Averaging merge on the GPU (dl_rda_merge_outer_step)
against the oracle's reading (needs a GPU).

The page names the method without a formula, so the oracle's RDA is parity
unpinned (it is checked against the reading's defining properties in
test_oracle_rda.py); here the GPU is held to that oracle on identical
inputs - the oracle's own codes, codebooks and counts - with the merge's
bar (relative L2 <= 1e-6 on D, theta and momentum), and to the same
properties on its own.
"""
import numpy as np
import pytest

import oracle
from parity import TOL_REL_L2, rel_l2

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


def _oracle_quantised(seed, numels, K):
    rng = np.random.default_rng(seed)
    n = sum(numels)
    off = np.concatenate([[0], np.cumsum(numels)]).astype(np.int64)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = [(g - 1e-3 * (1 + 0.4 * k) * rng.standard_normal(n)).astype(np.float32)
            for k in range(K)]
    st = oracle.stats(g, reps, off)
    codes, cb, cnt = oracle.quantize(g, reps, st, off)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    return g, m, off, codes, cb, cnt


def _gpu_rda(dl, g, m, numels, codes, cb, cnt, **kw):
    F = dl.Fragment(numels)
    gd, md = torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda()
    dd = torch.full_like(gd, float("nan"))
    codes_d = [torch.from_numpy(np.ascontiguousarray(c)).cuda() for c in codes]
    ws = dl.rda_merge_outer_step(gd, md, F, codes_d, torch.from_numpy(cb).cuda(),
                                 torch.from_numpy(cnt.view(np.int32)).cuda(), delta_bar=dd, **kw)
    torch.cuda.synchronize()
    assert dl.read_device_status(ws) == 0
    return gd.cpu().numpy(), md.cpu().numpy(), dd.cpu().numpy()


@pytest.mark.parametrize("K", [1, 3, 5])
def test_rda_matches_the_oracle_on_the_same_codes(dl, K):
    g, m, off, codes, cb, cnt = _oracle_quantised(20 + K, RAGGED, K)
    w = np.random.default_rng(K).uniform(0.5, 1.5, K).astype(np.float32)
    st, g_o, m_o, d_o = oracle.rda_merge_outer_step(g, m, list(codes), cb, cnt, offsets=off,
                                                    weights=w)
    assert st == 0
    g1, m1, d1 = _gpu_rda(dl, g, m, RAGGED, codes, cb, cnt, weights=w)
    for key, a, b in (("delta_bar", d1, d_o), ("theta_g", g1, g_o), ("momentum", m1, m_o)):
        assert rel_l2(a, b) <= TOL_REL_L2, (key, rel_l2(a, b))


def test_rda_with_present_subset(dl):
    K = 6
    g, m, off, codes, cb, cnt = _oracle_quantised(31, RAGGED, K)
    present = np.array([1, 0, 1, 1, 0, 1], dtype=np.uint8)
    w = np.array([1.0, 5.0, 0.5, 2.0, 1.0, 1.0], dtype=np.float32)
    st, g_o, m_o, d_o = oracle.rda_merge_outer_step(g, m, list(codes), cb, cnt, offsets=off,
                                                    weights=w, present=present)
    g1, m1, d1 = _gpu_rda(dl, g, m, RAGGED, codes, cb, cnt, weights=w, present=present)
    assert rel_l2(d1, d_o) <= TOL_REL_L2 and rel_l2(g1, g_o) <= TOL_REL_L2


def test_rda_norm_and_direction_on_the_gpu(dl):
    K = 4
    g, m, off, codes, cb, cnt = _oracle_quantised(41, RAGGED, K)
    _, _, d1 = _gpu_rda(dl, g, m, RAGGED, codes, cb, cnt)
    d1 = d1.astype(np.float64)  # norms and dot products in fp64
    T = len(RAGGED)
    for t in range(T):
        sl = slice(off[t], off[t + 1])
        if off[t + 1] == off[t]:
            continue
        vs = [cb[k, t][codes[k, sl]].astype(np.float64) for k in range(K)]
        norms = [np.linalg.norm(v) for v in vs]
        r = sum(norms) / K
        u = sum(v / nv for v, nv in zip(vs, norms) if nv > 0) / K
        assert abs(np.linalg.norm(d1[sl]) - r) <= 2e-6 * r + 1e-30, t
        if np.linalg.norm(u) > 0:
            cos = d1[sl] @ u / (np.linalg.norm(d1[sl]) * np.linalg.norm(u))
            assert cos > 1 - 1e-10, t


def test_rda_quorum_failure_leaves_state_untouched(dl):
    K = 3
    g, m, off, codes, cb, cnt = _oracle_quantised(51, [5000], K)
    F = dl.Fragment([5000])
    gd, md = torch.from_numpy(g).cuda(), torch.from_numpy(m).cuda()
    with pytest.raises(dl.DLError) as e:
        dl.rda_merge_outer_step(gd, md, F, [torch.from_numpy(c).cuda() for c in codes],
                                torch.from_numpy(cb).cuda(),
                                torch.from_numpy(cnt.view(np.int32)).cuda(),
                                present=[0, 1, 0], min_quorum=2)
    assert e.value.status == -3
    torch.cuda.synchronize()
    assert np.array_equal(gd.cpu().numpy(), g) and np.array_equal(md.cpu().numpy(), m)


@pytest.mark.parametrize("K", [3, 5, 14, 16, 32])
def test_staged_rda_merge_equals_the_unstaged_one(dl, K, monkeypatch):
    """The staged merge (any number of present learners) and the unstaged
    kernels (DL_MERGE_UNSTAGED=1) give the same D, theta and momentum bit for
    bit in the RDA merge, with unequal weights."""
    g, m, off, codes, cb, cnt = _oracle_quantised(41 + K, RAGGED, K)
    w = (0.5 + np.random.default_rng(42).random(K)).astype(np.float32)
    monkeypatch.delenv("DL_MERGE_UNSTAGED", raising=False)
    a = _gpu_rda(dl, g, m, RAGGED, codes, cb, cnt, weights=w)
    monkeypatch.setenv("DL_MERGE_UNSTAGED", "1")
    b = _gpu_rda(dl, g, m, RAGGED, codes, cb, cnt, weights=w)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)  # == on floats: +0 and -0 count as equal
