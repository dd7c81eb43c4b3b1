"""Host-only checks of the C ABI: the library loads, exports every declared
symbol, and its host logic (planner, argument validation, quorum) behaves -
all without a GPU. Calls that would launch work are not made here; every
case below returns during host-side validation."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import pseudo_grad_sync_gb300 as dl
from pseudo_grad_sync_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return dl.lib()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^\s*(?:[\w\s\*]+?)\b(dl_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert {"dl_plan_fragments", "dl_pseudograd_stats", "dl_quantize",
            "dl_merge_outer_step"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    assert L.dl_version() == 200


def test_read_device_status_arguments(L):
    out = ctypes.c_uint32(0)
    assert L.dl_read_device_status(FAKE, None, None) == -1  # no place for the word
    # NULL workspace: the library's own word, which needs a device (none here)
    assert L.dl_read_device_status(None, ctypes.byref(out), None) == -4


def test_selftests_validate_before_launch(L):
    f = L.dl_selftest_pipeline
    assert f(None, FAKE, 4, 2, 100, FAKE, None) == -1          # no workspace
    assert f(FAKE, FAKE, 0, 0, 100, FAKE, None) == -1          # no tiles
    assert f(FAKE, FAKE, 4, 5, 100, FAKE, None) == -1          # stall past the end
    assert f(FAKE, FAKE, 4, 2, 0, FAKE, None) == -1            # no polls
    assert f(FAKE, FAKE, 4, 2, (1 << 22) + 1, FAKE, None) == -1
    assert f(FAKE + 16, FAKE, 4, 2, 100, FAKE, None) == -2     # workspace not 256-aligned
    assert f(FAKE, FAKE + 4, 4, 2, 100, FAKE, None) == -2      # source not 16-aligned
    assert L.dl_selftest_wait_timeout(FAKE, 0, None) == -1


def test_shutdown_without_resources_is_a_no_op(L):
    # nothing was created on this host (no GPU): no CUDA call is made
    assert L.dl_shutdown() == 0
    assert L.dl_shutdown() == 0


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6, -7, 12345):
        assert dl.status_string(code)


def test_planner_matches_oracle(L):
    rng = np.random.default_rng(0)
    for _ in range(100):
        T = int(rng.integers(0, 300))
        P = int(rng.integers(1, 30))
        sizes = rng.integers(0, 1 << 40, T) if rng.random() < 0.5 else rng.integers(0, 5, T)
        f1, l1 = dl.plan_fragments(sizes, P)
        f2, l2 = oracle.plan_fragments(sizes, P)
        assert np.array_equal(f1, f2) and np.array_equal(l1, l2)


def test_planner_rejects_bad_args(L):
    with pytest.raises(dl.DLError):
        dl.plan_fragments([1, 2, 3], 0)
    with pytest.raises(dl.DLError):
        dl.plan_fragments([1, -2, 3], 2)


def _frag(offsets, dptr=16):
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    f = dl._Fragment(off.ctypes.data, dptr, len(off) - 1)
    return f, off


FAKE = 1 << 20  # a 16-byte aligned, never dereferenced device address


def _ptrs(*vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_validation_errors_before_any_launch(L):
    f, off = _frag([0, 10, 30])
    fb = ctypes.byref(f)
    ws = L.dl_stats_workspace_bytes(fb, 2)
    assert ws > 0
    # bad K, null arrays, misaligned pointers, short or misaligned workspace
    assert L.dl_pseudograd_stats(FAKE, _ptrs(FAKE, FAKE), 0, fb, 6.0, FAKE, FAKE, ws, None) == -1
    assert L.dl_pseudograd_stats(FAKE, _ptrs(FAKE, FAKE), 33, fb, 6.0, FAKE, FAKE, ws, None) == -1
    assert L.dl_pseudograd_stats(FAKE, _ptrs(FAKE, None), 2, fb, 6.0, FAKE, FAKE, ws, None) == -1
    assert L.dl_pseudograd_stats(FAKE + 4, _ptrs(FAKE, FAKE), 2, fb, 6.0, FAKE, FAKE, ws, None) == -2
    assert L.dl_pseudograd_stats(FAKE, _ptrs(FAKE, FAKE), 2, fb, 0.0, FAKE, FAKE, ws, None) == -1
    assert L.dl_pseudograd_stats(FAKE, _ptrs(FAKE, FAKE), 2, fb, 6.0, FAKE, FAKE, ws - 1, None) == -6
    assert L.dl_pseudograd_stats(FAKE, _ptrs(FAKE, FAKE), 2, fb, 6.0, FAKE, FAKE + 16, ws, None) == -2
    # offsets must start at 0 and not decrease
    g, _o = _frag([1, 10, 30])
    assert L.dl_pseudograd_stats(FAKE, _ptrs(FAKE), 1, ctypes.byref(g), 6.0, FAKE, FAKE, ws, None) == -5
    h, _o2 = _frag([0, 10, 5])
    assert L.dl_quantize(FAKE, _ptrs(FAKE), 1, ctypes.byref(h), FAKE, _ptrs(FAKE), FAKE, None,
                         FAKE, 1 << 30, None) == -5
    # quantize: misaligned codes buffer, short workspace
    wq = L.dl_quantize_workspace_bytes(fb, 1)
    assert L.dl_quantize(FAKE, _ptrs(FAKE), 1, fb, FAKE, _ptrs(FAKE + 1), FAKE, None, FAKE, wq,
                         None) == -2
    assert L.dl_quantize(FAKE, _ptrs(FAKE), 1, fb, FAKE, _ptrs(FAKE), FAKE, None, FAKE, wq - 8,
                         None) == -6


def _merge(L, fb, K, weights=None, present=None, min_quorum=1, codes=True):
    c = _ptrs(*([FAKE] * K))
    w = None if weights is None else np.ascontiguousarray(weights, np.float32)
    p = None if present is None else np.ascontiguousarray(present, np.uint8)
    return L.dl_merge_outer_step(
        FAKE, FAKE, c if codes else None, FAKE, None if codes else c, K, fb,
        None if w is None else w.ctypes.data, None if p is None else p.ctypes.data,
        min_quorum, 0.7, 0.9, None, None)


def test_merge_quorum_and_weight_rules_match_oracle(L):
    # empty fragment (n = 0): validation still runs, nothing is launched
    f, off = _frag([0, 0])
    fb = ctypes.byref(f)
    rng = np.random.default_rng(4)
    for _ in range(200):
        K = int(rng.integers(1, 9))
        w = rng.choice([0.0, 0.5, 1.0, 2.0, -1.0, np.inf], K, p=[.2, .3, .2, .2, .05, .05])
        p = (rng.random(K) < 0.6).astype(np.uint8)
        q = int(rng.integers(0, 5))
        st_or, _ = oracle.merge_weights(w.astype(np.float32), p, K, q)
        st_dl = _merge(L, fb, K, w, p, q)
        expect = st_or if st_or < 0 else 0
        assert st_dl == expect, (w, p, q, st_or, st_dl)
    assert _merge(L, fb, 33) == -1
    assert _merge(L, fb, 0) == -1


def _sync_jobs(frags, K, weights=None, present=None, theta_k=True):
    """dl_fragment_job array with fake device pointers (never dereferenced)."""
    arr = (dl._FragmentJob * len(frags))()
    keep = []
    for j, f in enumerate(frags):
        arr[j].frag = ctypes.pointer(f)
        arr[j].theta_g = FAKE
        arr[j].momentum = FAKE
        if theta_k:
            ra = _ptrs(*([FAKE] * K))
            keep.append(ra)
            arr[j].theta_k = ctypes.cast(ra, ctypes.c_void_p)
        if weights is not None and weights[j] is not None:
            w = np.ascontiguousarray(weights[j], np.float32)
            keep.append(w)
            arr[j].weights = w.ctypes.data
        if present is not None and present[j] is not None:
            p = np.ascontiguousarray(present[j], np.uint8)
            keep.append(p)
            arr[j].present = p.ctypes.data
    return arr, keep


def _outer_sync(L, arr, n, K, min_quorum=1, flags=0, ws=FAKE, nbytes=0):
    return L.dl_outer_sync(arr, n, K, 6.0, min_quorum, 0.7, 0.9, flags, ws, nbytes, None)


def test_outer_sync_validates_every_job_before_any_launch(L):
    fs = [_frag([0, 10, 30]), _frag([0, 5]), _frag([0, 0, 0])]
    frags = [f for f, _ in fs]
    K = 3
    arr, keep = _sync_jobs(frags, K)
    need = L.dl_outer_sync_workspace_bytes(arr, 3, K, 0)
    assert need > 0
    # quantised mode: every job valid, so the short workspace is what fails
    assert _outer_sync(L, arr, 3, K, nbytes=need - 1) == -6
    assert _outer_sync(L, arr, 3, K, ws=FAKE + 16, nbytes=need) == -2
    # unknown flags and combinations that mean nothing
    for fl in (16, 1 | 4, 1 | 8, 4 | 8, 1 | 4 | 8, -1):
        assert _outer_sync(L, arr, 3, K, flags=fl) == -1, fl
        assert L.dl_outer_sync_workspace_bytes(arr, 3, K, fl) == 0, fl
    for fl in (4, 8, 4 | 2, 8 | 2):
        need_m = L.dl_outer_sync_workspace_bytes(arr, 3, K, fl)
        assert need_m > 0, fl
        assert _outer_sync(L, arr, 3, K, flags=fl, nbytes=need_m - 1) == -6, fl
        assert _outer_sync(L, arr, 3, K, flags=fl, ws=FAKE + 16, nbytes=need_m) == -2, fl
        assert _outer_sync(L, arr, 3, K, flags=fl, min_quorum=4) == -3, fl
    assert _outer_sync(L, arr, 3, 0) == -1 and _outer_sync(L, arr, 3, 33) == -1
    assert L.dl_outer_sync(arr, 3, K, 0.0, 1, 0.7, 0.9, 0, FAKE, need, None) == -1
    assert _outer_sync(L, arr, 3, K, min_quorum=4) == -3
    # a later job's bad layout, missing replica array or misaligned buffer
    bad, _ = _frag([0, 10, 5])
    arr2, keep2 = _sync_jobs(frags[:2] + [bad], K)
    assert _outer_sync(L, arr2, 3, K) == -5
    arr3, keep3 = _sync_jobs(frags, K, theta_k=False)
    assert _outer_sync(L, arr3, 3, K) == -1
    arr[1].momentum = FAKE + 4
    assert _outer_sync(L, arr, 3, K, nbytes=need) == -2
    assert L.dl_outer_sync_workspace_bytes(arr, 3, 0, 0) == 0


def test_outer_sync_quorum_and_weights_per_job_match_oracle(L):
    """Each job's present set and weights are checked like the merge's; the
    first failing job (in order) decides the status. All-valid calls stop at
    the (deliberately) short workspace, so nothing is launched."""
    rng = np.random.default_rng(11)
    f, _o = _frag([0, 40, 100])
    for _ in range(150):
        K = int(rng.integers(1, 9))
        P = int(rng.integers(1, 5))
        q = int(rng.integers(0, 4))
        ws, ps, expect = [], [], 0
        for _j in range(P):
            w = rng.choice([0.0, 0.5, 1.0, 2.0, -1.0, np.inf], K, p=[.2, .3, .2, .2, .05, .05])
            p = (rng.random(K) < 0.7).astype(np.uint8)
            ws.append(w)
            ps.append(p)
            st_or, _ = oracle.merge_weights(w.astype(np.float32), p, K, q)
            if expect == 0 and st_or < 0:
                expect = st_or
        arr, keep = _sync_jobs([f] * P, K, ws, ps)
        st = _outer_sync(L, arr, P, K, min_quorum=q, nbytes=0)
        assert st == (expect if expect < 0 else -6), (st, expect)


def test_outer_sync_workspace_covers_every_quorum(L):
    f, _o = _frag(np.cumsum([0, 4096, 77, 8192 * 9 + 3]))
    for K in (1, 3, 4, 7, 16, 32):
        arr, keep = _sync_jobs([f, f], K)
        need = L.dl_outer_sync_workspace_bytes(arr, 2, K, 0)
        need_rda = L.dl_outer_sync_workspace_bytes(arr, 2, K, 4)
        fb = ctypes.byref(f)
        for np_ in range(1, K + 1):
            parts = (L.dl_stats_workspace_bytes(fb, np_) + 2 * 48 * K * 3
                     + L.dl_quantize_workspace_bytes(fb, np_) + 4 * K * 3 * 256 + K * (8192 * 9 + 4174))
            assert need >= parts, (K, np_)
            # RDA adds the bucket counts and the RDA merge's own scratch
            assert need_rda >= parts + 4 * K * 3 * 256 + L.dl_rda_workspace_bytes(fb, np_)
        # the ring needs its own workspace, whatever K
        assert L.dl_outer_sync_workspace_bytes(arr, 2, K, 8) >= L.dl_ring_workspace_bytes(fb)


def test_workspace_needs_never_decrease_with_K(L):
    """A workspace sized for K must serve any subset of present learners."""
    for offs in ([0, 10, 30], list(np.cumsum([0, 4096, 77, 8192 * 9 + 3])), [0] + [1] * 50):
        f, _o = _frag(np.asarray(offs))
        fb = ctypes.byref(f)
        s = [L.dl_stats_workspace_bytes(fb, k) for k in range(1, 33)]
        q = [L.dl_quantize_workspace_bytes(fb, k) for k in range(1, 33)]
        assert all(a <= b for a, b in zip(s, s[1:])), s
        assert all(a <= b for a, b in zip(q, q[1:])), q


def test_values_mode_needs_one_learner(L):
    f, _o = _frag([0, 10, 30])
    fb = ctypes.byref(f)
    ws = L.dl_stats_workspace_bytes(fb, 2)
    # theta_k NULL selects values mode, which is defined for K = 1 only
    assert L.dl_pseudograd_stats(FAKE, None, 2, fb, 6.0, FAKE, FAKE, ws, None) == -1
    wq = L.dl_quantize_workspace_bytes(fb, 2)
    assert L.dl_quantize(FAKE, None, 2, fb, FAKE, _ptrs(FAKE, FAKE), FAKE, None, FAKE, wq,
                         None) == -1
    # K = 1 in values mode passes validation and stops at the short workspace
    assert L.dl_pseudograd_stats(FAKE, None, 1, fb, 6.0, FAKE, FAKE, 0, None) == -6


def _ring(L, fb, K, weights=None, present=None, min_quorum=1, ws=FAKE, nbytes=0, hop_stats=None):
    w = None if weights is None else np.ascontiguousarray(weights, np.float32)
    p = None if present is None else np.ascontiguousarray(present, np.uint8)
    return L.dl_ring_outer_step(FAKE, FAKE, _ptrs(*([FAKE] * K)), K, fb,
                                None if w is None else w.ctypes.data,
                                None if p is None else p.ctypes.data, min_quorum, 6.0, 0.7, 0.9,
                                None, hop_stats, ws, nbytes, None)


def test_ring_validation_and_quorum_rules(L):
    f, _o = _frag([0, 100, 4000])
    fb = ctypes.byref(f)
    need = L.dl_ring_workspace_bytes(fb)
    assert need >= 4000 * 5
    assert _ring(L, fb, 0) == -1 and _ring(L, fb, 33) == -1
    assert _ring(L, fb, 3, nbytes=need - 1) == -6       # valid otherwise: short workspace
    assert _ring(L, fb, 3, ws=FAKE + 16, nbytes=need) == -2
    assert _ring(L, fb, 3, nbytes=need, hop_stats=FAKE + 4) == -2  # stats need 8-byte alignment
    assert _ring(L, fb, 3, nbytes=need - 1, hop_stats=FAKE + 8) == -6
    rng = np.random.default_rng(8)
    for _ in range(150):
        K = int(rng.integers(1, 9))
        w = rng.choice([0.0, 0.5, 1.0, 2.0, -1.0, np.inf], K, p=[.2, .3, .2, .2, .05, .05])
        p = (rng.random(K) < 0.6).astype(np.uint8)
        q = int(rng.integers(0, 5))
        st_or, _ = oracle.merge_weights(w.astype(np.float32), p, K, q)
        st = _ring(L, fb, K, w, p, q)
        assert st == (st_or if st_or < 0 else -6), (w, p, q, st_or, st)


def test_rda_validation_and_quorum_rules(L):
    f, _o = _frag([0, 100, 4000])
    fb = ctypes.byref(f)
    K = 3
    need = L.dl_rda_workspace_bytes(fb, K)
    assert need > 0 and L.dl_rda_workspace_bytes(fb, 0) == 0

    def rda(K, weights=None, present=None, q=1, counts=FAKE, ws=FAKE, nbytes=0, codes=True):
        w = None if weights is None else np.ascontiguousarray(weights, np.float32)
        p = None if present is None else np.ascontiguousarray(present, np.uint8)
        return L.dl_rda_merge_outer_step(FAKE, FAKE, _ptrs(*([FAKE] * K)) if codes else None,
                                         FAKE, counts, K, fb,
                                         None if w is None else w.ctypes.data,
                                         None if p is None else p.ctypes.data, q, 0.7, 0.9,
                                         None, ws, nbytes, None)

    assert rda(K, codes=False) == -1           # quantised mode only
    assert rda(K, counts=None, nbytes=need) == -1
    assert rda(K, counts=FAKE + 4, nbytes=need) == -2
    assert rda(K, nbytes=need - 1) == -6
    rng = np.random.default_rng(9)
    for _ in range(100):
        Kr = int(rng.integers(1, 9))
        w = rng.choice([0.0, 0.5, 1.0, -1.0], Kr, p=[.2, .5, .25, .05])
        p = (rng.random(Kr) < 0.6).astype(np.uint8)
        q = int(rng.integers(0, 4))
        st_or, _ = oracle.merge_weights(w.astype(np.float32), p, Kr, q)
        assert rda(Kr, w, p, q) == (st_or if st_or < 0 else -6)


def test_quantize_noalloc_limits_before_any_device_call(L):
    """dl_quantize_noalloc refuses on the host, before it looks up its static
    scratch: K outside 1..32 (DL_ERR_ARG), and a fragment whose K * n_tensors
    exceeds the scratch's segment limit (DL_ERR_WORKSPACE), from just past
    the limit. Only refusals are called here: an accepted call would go on to
    the device. The binding's constant matches the header's."""
    hdr = open(os.path.join(ROOT, "include", "diloco_sync.h")).read()
    lim = int(re.search(r"#define DL_QUANTIZE_NOALLOC_MAX_SEGMENTS (\d+)", hdr).group(1))
    assert lim == dl.DL_QUANTIZE_NOALLOC_MAX_SEGMENTS
    f, off = _frag(np.arange(lim // 2 + 2))  # lim/2 + 1 one-element tensors
    fb = ctypes.byref(f)
    q = L.dl_quantize_noalloc
    assert q(FAKE, _ptrs(FAKE, FAKE), 2, fb, FAKE, _ptrs(FAKE, FAKE), FAKE, None, None) == -6
    assert q(FAKE, _ptrs(*[FAKE] * 4), 4, fb, FAKE, _ptrs(*[FAKE] * 4), FAKE, None, None) == -6
    assert q(FAKE, _ptrs(FAKE), 0, fb, FAKE, _ptrs(FAKE), FAKE, None, None) == -1
    assert q(FAKE, _ptrs(*[FAKE] * 33), 33, fb, FAKE, _ptrs(*[FAKE] * 33), FAKE, None,
             None) == -1
    h, _o = _frag([0, 10, 5])
    assert q(FAKE, _ptrs(FAKE), 1, ctypes.byref(h), FAKE, _ptrs(FAKE), FAKE, None, None) == -5


def test_binding_has_every_entry_point_under_its_name(L):
    """Every dl_* function the header declares has a binding function of the
    same name without the prefix, so a user of the C ABI finds each call in
    Python under its own name."""
    missing = [n for n in _declared_functions() if not callable(getattr(dl, n[3:], None))]
    assert not missing, missing
    assert dl.version() == L.dl_version()
