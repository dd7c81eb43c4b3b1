"""CPU oracle of the outer synchronisation step - TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never loads it and the
two share no code. See ``oracle.c`` for the page passages each function
follows and for the readings taken where the pages are silent.

Every function here is pinned by tests that do not retype its formulas:
closed forms, the INTELLECT-1 worked example (section 3.2), brute force on
tiny inputs, the bucket-mean optimality property (section 4.1 step 4), the
code-space counterexample (section 4.2), the planner's LPT bound, and for the
ring accumulation its reductions to the plain merge and its per-hop error
bound. One exception: ``rda_merge_outer_step`` is PARITY UNPINNED - the page
names Radial-Directional Averaging without a formula, so its reading is
checked only against the properties that define that reading.
"""
from __future__ import annotations

import ctypes
import fcntl
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
OUT = os.path.join(HERE, "liboracle.so")

OK, ERR_ARG, ERR_QUORUM = 0, -1, -3
NB = 256


def build(force: bool = False) -> str:
    with open(os.path.join(HERE, ".build.lock"), "w") as fh:
        fcntl.flock(fh, fcntl.LOCK_EX)
        if force or not os.path.exists(OUT) or os.path.getmtime(OUT) < os.path.getmtime(SRC):
            tmp = OUT + f".tmp{os.getpid()}"
            subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                            "-fno-fast-math", "-o", tmp, SRC, "-lm"], check=True)
            os.replace(tmp, OUT)
    return OUT


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, i32, i64, f32, f64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_float, ctypes.c_double)
        L.oracle_threads.restype = ctypes.c_int
        L.oracle_plan_fragments.restype = ctypes.c_int
        L.oracle_plan_fragments.argtypes = [vp, i32, i32, vp, vp]
        L.oracle_stats.restype = None
        L.oracle_stats.argtypes = [vp, vp, i32, vp, i32, f64, vp, vp, vp, vp, vp, vp]
        L.oracle_bucket_coord.restype = None
        L.oracle_bucket_coord.argtypes = [vp, vp, vp, i64, f64, f64, vp]
        L.oracle_quantize.restype = None
        L.oracle_quantize.argtypes = [vp, vp, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp]
        L.oracle_merge_weights.restype = ctypes.c_int
        L.oracle_merge_weights.argtypes = [vp, vp, i32, i32, vp]
        L.oracle_merge_outer_step.restype = ctypes.c_int
        L.oracle_merge_outer_step.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, vp, vp, i32,
                                              f32, f32, vp]
        L.oracle_rda_merge_outer_step.restype = ctypes.c_int
        L.oracle_rda_merge_outer_step.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, vp, vp, i32,
                                                  f32, f32, vp]
        L.oracle_set_threads.restype = None
        L.oracle_set_threads.argtypes = [ctypes.c_int]
        L.oracle_ring_outer_step.restype = ctypes.c_int
        L.oracle_ring_outer_step.argtypes = [vp, vp, vp, i32, vp, i32, vp, vp, i32, f64, f32,
                                             f32, vp]
        _lib = L
    return _lib


def threads() -> int:
    return int(lib().oracle_threads())


def set_threads(n: int) -> None:
    """Threads of the oracle's later parallel loops (timing only)."""
    lib().oracle_set_threads(int(n))


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _ptrs(arrays):
    arr = (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])
    return arr


def _offsets(offsets, n):
    if offsets is None:
        offsets = [0, n]
    return np.ascontiguousarray(offsets, dtype=np.int64)


def plan_fragments(numel, n_frags):
    numel = np.ascontiguousarray(numel, dtype=np.int64)
    frag = np.empty(len(numel), dtype=np.int32)
    load = np.empty(n_frags, dtype=np.int64)
    st = lib().oracle_plan_fragments(numel.ctypes.data, len(numel), n_frags, frag.ctypes.data,
                                     load.ctypes.data)
    if st != OK:
        raise ValueError(f"oracle_plan_fragments: status {st}")
    return frag, load


class Stats:
    """Per (k, t) statistics, arrays of shape [K, T]."""

    def __init__(self, K, T):
        self.count = np.zeros((K, T), dtype=np.int64)
        self.nonfinite = np.zeros((K, T), dtype=np.int64)
        self.mean = np.zeros((K, T))
        self.std = np.zeros((K, T))
        self.lo = np.zeros((K, T))
        self.hi = np.zeros((K, T))


def stats(theta_g, replicas, offsets=None, clip_sigmas=6.0) -> Stats:
    g = _f32(theta_g)
    rs = [_f32(r) for r in replicas]
    K = len(rs)
    off = _offsets(offsets, g.size)
    T = len(off) - 1
    s = Stats(K, T)
    lib().oracle_stats(g.ctypes.data, _ptrs(rs), K, off.ctypes.data, T, clip_sigmas,
                       s.count.ctypes.data, s.nonfinite.ctypes.data, s.mean.ctypes.data,
                       s.std.ctypes.data, s.lo.ctypes.data, s.hi.ctypes.data)
    return s


def bucket_coord(theta_g, replica, idx, lo, hi):
    g, r = _f32(theta_g), _f32(replica)
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    u = np.empty(idx.size)
    lib().oracle_bucket_coord(g.ctypes.data, r.ctypes.data, idx.ctypes.data, idx.size, lo, hi,
                              u.ctypes.data)
    return u


def quantize(theta_g, replicas, st: Stats, offsets=None):
    """Returns (codes [K, n] uint8, codebook [K, T, 256] f32, counts [K, T, 256] u32)."""
    g = _f32(theta_g)
    rs = [_f32(r) for r in replicas]
    K = len(rs)
    off = _offsets(offsets, g.size)
    T = len(off) - 1
    codes = np.empty((K, g.size), dtype=np.uint8)
    cb = np.empty((K, T, NB), dtype=np.float32)
    cnt = np.empty((K, T, NB), dtype=np.uint32)
    mean = np.ascontiguousarray(st.mean)
    lo, hi = np.ascontiguousarray(st.lo), np.ascontiguousarray(st.hi)
    nf = np.ascontiguousarray(st.nonfinite)
    lib().oracle_quantize(g.ctypes.data, _ptrs(rs), K, off.ctypes.data, T, mean.ctypes.data,
                          lo.ctypes.data, hi.ctypes.data, nf.ctypes.data,
                          _ptrs([codes[k] for k in range(K)]), cb.ctypes.data, cnt.ctypes.data)
    return codes, cb, cnt


def merge_weights(weights, present, K, min_quorum=1):
    w = None if weights is None else _f32(weights)
    p = None if present is None else np.ascontiguousarray(present, dtype=np.uint8)
    out = np.zeros(K, dtype=np.float32)
    st = lib().oracle_merge_weights(None if w is None else w.ctypes.data,
                                    None if p is None else p.ctypes.data, K, min_quorum,
                                    out.ctypes.data)
    return st, out


def merge_outer_step(theta_g, momentum, codes=None, codebook=None, replicas=None,
                     offsets=None, weights=None, present=None, min_quorum=1, lr=0.7, mu=0.9,
                     want_delta_bar=False):
    """Returns (status, theta_g', momentum', delta_bar or None); inputs untouched."""
    g = np.array(theta_g, dtype=np.float32, copy=True)
    m = np.array(momentum, dtype=np.float32, copy=True)
    off = _offsets(offsets, g.size)
    T = len(off) - 1
    if codes is not None:
        codes = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes]
        K = len(codes)
        cb = np.ascontiguousarray(codebook, dtype=np.float32)
        assert cb.size == K * T * NB
        cptr, cbptr, rptr = _ptrs(codes), cb.ctypes.data, None
    else:
        reps = [_f32(r) for r in replicas]
        K = len(reps)
        cptr, cbptr, rptr = None, None, _ptrs(reps)
    w = None if weights is None else _f32(weights)
    p = None if present is None else np.ascontiguousarray(present, dtype=np.uint8)
    db = np.empty_like(g) if want_delta_bar else None
    st = lib().oracle_merge_outer_step(
        g.ctypes.data, m.ctypes.data, cptr, cbptr, rptr, K, off.ctypes.data, T,
        None if w is None else w.ctypes.data, None if p is None else p.ctypes.data,
        min_quorum, lr, mu, None if db is None else db.ctypes.data)
    return st, g, m, db


def outer_step(theta_g, momentum, replicas, offsets=None, weights=None, present=None,
               min_quorum=1, lr=0.7, mu=0.9, clip_sigmas=6.0, quantized=True):
    """The whole step for one fragment: stats -> quantise -> merge + Nesterov.

    Returns a dict with every intermediate (stats, codes, codebook, counts,
    delta_bar) and the new theta_g / momentum.
    """
    st = stats(theta_g, replicas, offsets, clip_sigmas)
    out = {"stats": st}
    if quantized:
        codes, cb, cnt = quantize(theta_g, replicas, st, offsets)
        out.update(codes=codes, codebook=cb, counts=cnt)
        status, g, m, db = merge_outer_step(theta_g, momentum, codes=list(codes), codebook=cb,
                                            offsets=offsets, weights=weights, present=present,
                                            min_quorum=min_quorum, lr=lr, mu=mu,
                                            want_delta_bar=True)
    else:
        status, g, m, db = merge_outer_step(theta_g, momentum, replicas=replicas,
                                            offsets=offsets, weights=weights, present=present,
                                            min_quorum=min_quorum, lr=lr, mu=mu,
                                            want_delta_bar=True)
    out.update(status=status, theta_g=g, momentum=m, delta_bar=db)
    return out


def ring_outer_step(theta_g, momentum, replicas, offsets=None, weights=None, present=None,
                    min_quorum=1, lr=0.7, mu=0.9, clip_sigmas=6.0):
    """Ring accumulation with re-quantisation at every hop (INTELLECT-1 notes,
    section 4.2), then the outer Nesterov step. Returns (status, theta_g',
    momentum', delta_bar); inputs untouched."""
    g = np.array(theta_g, dtype=np.float32, copy=True)
    m = np.array(momentum, dtype=np.float32, copy=True)
    off = _offsets(offsets, g.size)
    T = len(off) - 1
    reps = [_f32(r) for r in replicas]
    w = None if weights is None else _f32(weights)
    p = None if present is None else np.ascontiguousarray(present, dtype=np.uint8)
    db = np.empty_like(g)
    st = lib().oracle_ring_outer_step(
        g.ctypes.data, m.ctypes.data, _ptrs(reps), len(reps), off.ctypes.data, T,
        None if w is None else w.ctypes.data, None if p is None else p.ctypes.data, min_quorum,
        clip_sigmas, lr, mu, db.ctypes.data)
    return st, g, m, db


def rda_merge_outer_step(theta_g, momentum, codes, codebook, counts, offsets=None, weights=None,
                         present=None, min_quorum=1, lr=0.7, mu=0.9):
    """Radial-Directional Averaging merge of decoded values, then the outer
    step (see oracle.c for the reading: no formula on the page; parity
    unpinned). Returns (status, theta_g', momentum', delta_bar)."""
    g = np.array(theta_g, dtype=np.float32, copy=True)
    m = np.array(momentum, dtype=np.float32, copy=True)
    off = _offsets(offsets, g.size)
    T = len(off) - 1
    codes = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes]
    K = len(codes)
    cb = np.ascontiguousarray(codebook, dtype=np.float32)
    cnt = np.ascontiguousarray(counts, dtype=np.uint32)
    assert cb.size == K * T * NB and cnt.size == K * T * NB
    w = None if weights is None else _f32(weights)
    p = None if present is None else np.ascontiguousarray(present, dtype=np.uint8)
    db = np.empty_like(g)
    st = lib().oracle_rda_merge_outer_step(
        g.ctypes.data, m.ctypes.data, _ptrs(codes), cb.ctypes.data, cnt.ctypes.data, K,
        off.ctypes.data, T, None if w is None else w.ctypes.data,
        None if p is None else p.ctypes.data, min_quorum, lr, mu, db.ctypes.data)
    return st, g, m, db
