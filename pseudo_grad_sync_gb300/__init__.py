"""Python binding of libdiloco_sync.so, the GB300 DiLoCo outer-sync library.

Argument marshalling only: every step of the outer synchronisation runs in
the library's CUDA kernels. PyTorch provides device memory and streams. The
C entry points (see include/diloco_sync.h) keep their names here:

    plan_fragments       balanced tensor -> fragment assignment (host)
    pseudograd_stats     per-(learner, tensor) mu / sigma / clip range
    quantize             uint8 codes + bucket-mean codebooks
    quantize_noalloc     quantize with the library's static scratch (no workspace)
    merge_outer_step     decode, weighted fp32 mean, outer Nesterov (in place)
    rda_merge_outer_step Radial-Directional Averaging merge, then the outer step
    ring_outer_step      ring accumulation re-quantised at every hop, then the
                         outer step (measures the error growth of a ring)
    outer_sync           the three calls over every fragment of a model, with
                         consecutive fragments overlapped on two streams

``OuterSync`` bundles the three device calls of one fragment with their
workspaces; ``ModelSync`` holds the workspace of ``outer_sync`` for a fixed
list of fragments.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import _build

DL_OK = 0
DL_NBUCKETS = 256
DL_MAX_LEARNERS = 32
DL_SYNC_UNQUANTIZED = 1
DL_SYNC_SERIAL = 2
DL_SYNC_RDA = 4
DL_SYNC_RING = 8
DL_ERR_WORKSPACE = -6
DL_QUANTIZE_NOALLOC_MAX_SEGMENTS = 2000
STATS_FIELDS = ("count", "nonfinite", "mean", "std", "lo", "hi")

_lib = None


class _Fragment(ctypes.Structure):
    _fields_ = [("offsets", ctypes.c_void_p), ("d_offsets", ctypes.c_void_p),
                ("n_tensors", ctypes.c_int32)]


class _FragmentJob(ctypes.Structure):
    _fields_ = [("frag", ctypes.POINTER(_Fragment)), ("theta_g", ctypes.c_void_p),
                ("momentum", ctypes.c_void_p), ("theta_k", ctypes.c_void_p),
                ("weights", ctypes.c_void_p), ("present", ctypes.c_void_p),
                ("delta_bar_out", ctypes.c_void_p)]


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise ImportError(f"{_build.LIB} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(_build.LIB)
        vp, i32, i64, f32, f64, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                      ctypes.c_float, ctypes.c_double, ctypes.c_size_t)
        fr = ctypes.POINTER(_Fragment)
        L.dl_version.restype = ctypes.c_int
        L.dl_status_string.restype = ctypes.c_char_p
        L.dl_status_string.argtypes = [ctypes.c_int]
        L.dl_plan_fragments.restype = ctypes.c_int
        L.dl_plan_fragments.argtypes = [vp, i32, i32, vp, vp]
        L.dl_stats_workspace_bytes.restype = sz
        L.dl_stats_workspace_bytes.argtypes = [fr, i32]
        L.dl_pseudograd_stats.restype = ctypes.c_int
        L.dl_pseudograd_stats.argtypes = [vp, vp, i32, fr, f64, vp, vp, sz, vp]
        L.dl_quantize_workspace_bytes.restype = sz
        L.dl_quantize_workspace_bytes.argtypes = [fr, i32]
        L.dl_quantize.restype = ctypes.c_int
        L.dl_quantize.argtypes = [vp, vp, i32, fr, vp, vp, vp, vp, vp, sz, vp]
        L.dl_quantize_noalloc.restype = ctypes.c_int
        L.dl_quantize_noalloc.argtypes = [vp, vp, i32, fr, vp, vp, vp, vp, vp]
        L.dl_merge_outer_step.restype = ctypes.c_int
        L.dl_merge_outer_step.argtypes = [vp, vp, vp, vp, vp, i32, fr, vp, vp, i32, f32, f32, vp,
                                          vp]
        jb = ctypes.POINTER(_FragmentJob)
        L.dl_outer_sync_workspace_bytes.restype = sz
        L.dl_outer_sync_workspace_bytes.argtypes = [jb, i32, i32, i32]
        L.dl_outer_sync.restype = ctypes.c_int
        L.dl_outer_sync.argtypes = [jb, i32, i32, f64, i32, f32, f32, i32, vp, sz, vp]
        L.dl_shutdown.restype = ctypes.c_int
        L.dl_shutdown.argtypes = []
        L.dl_rda_workspace_bytes.restype = sz
        L.dl_rda_workspace_bytes.argtypes = [fr, i32]
        L.dl_rda_merge_outer_step.restype = ctypes.c_int
        L.dl_rda_merge_outer_step.argtypes = [vp, vp, vp, vp, vp, i32, fr, vp, vp, i32, f32, f32,
                                              vp, vp, sz, vp]
        L.dl_ring_workspace_bytes.restype = sz
        L.dl_ring_workspace_bytes.argtypes = [fr]
        L.dl_ring_outer_step.restype = ctypes.c_int
        L.dl_ring_outer_step.argtypes = [vp, vp, vp, i32, fr, vp, vp, i32, f64, f32, f32, vp, vp,
                                         vp, sz, vp]
        L.dl_selftest_wait_timeout.restype = ctypes.c_int
        L.dl_selftest_wait_timeout.argtypes = [vp, i32, vp]
        L.dl_selftest_pipeline.restype = ctypes.c_int
        L.dl_selftest_pipeline.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        L.dl_read_device_status.restype = ctypes.c_int
        L.dl_read_device_status.argtypes = [vp, vp, vp]
        _lib = L
    return _lib


class DLError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {lib().dl_status_string(status).decode()} (status {status})")


def _check(fn, status):
    if status != DL_OK:
        raise DLError(fn, status)


def status_string(status: int) -> str:
    return lib().dl_status_string(status).decode()


def version() -> int:
    """The library's ABI version (dl_version)."""
    return int(lib().dl_version())


_F32 = (torch.float32,)
_U8 = (torch.uint8,)
_I64 = (torch.int64,)
_U32 = tuple(d for d in (torch.int32, getattr(torch, "uint32", None)) if d is not None)


def _need(t, dtypes, n, name):
    """The C ABI takes raw pointers and sizes from the fragment layout; check
    here what it cannot: a contiguous tensor of the right element type with at
    least n elements (None passes: the ABI decides whether NULL is allowed).
    The device is checked by _cuda once all of a call's tensors passed."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {' or '.join(map(str, dtypes))}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < n:
        raise ValueError(f"{name}: {t.numel()} elements, need at least {n}")


def _cuda(*items):
    """After the per-tensor checks: every tensor given (or in a list given)
    lives on a CUDA device."""
    for it in items:
        for t in (it if isinstance(it, (list, tuple)) else [it]):
            if t is not None and t.device.type != "cuda":
                raise ValueError(f"tensors must be on a CUDA device, found one on {t.device}")


def _need_all(ts, dtypes, n, name):
    for i, t in enumerate(ts):
        _need(t, dtypes, n, f"{name}[{i}]")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _ptr_array(tensors):
    return (ctypes.c_void_p * len(tensors))(*[None if t is None else t.data_ptr() for t in tensors])


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Fragment:
    """Tensor layout of one fragment: offsets on the host and on the device."""

    def __init__(self, numels, device="cuda"):
        numels = [int(x) for x in numels]
        self.numels = numels
        self.offsets = np.zeros(len(numels) + 1, dtype=np.int64)
        np.cumsum(np.asarray(numels, dtype=np.int64), out=self.offsets[1:])
        self.d_offsets = torch.from_numpy(self.offsets).to(device)
        self.n = int(self.offsets[-1])
        self.T = len(numels)
        self._c = _Fragment(self.offsets.ctypes.data, self.d_offsets.data_ptr(), self.T)

    @property
    def c(self):
        return ctypes.byref(self._c)


def plan_fragments(numel, n_frags: int):
    numel = np.ascontiguousarray(numel, dtype=np.int64)
    frag = np.empty(len(numel), dtype=np.int32)
    load = np.empty(n_frags, dtype=np.int64)
    _check("dl_plan_fragments", lib().dl_plan_fragments(
        numel.ctypes.data, len(numel), n_frags, frag.ctypes.data, load.ctypes.data))
    return frag, load


def stats_workspace_bytes(frag: Fragment, K: int) -> int:
    return int(lib().dl_stats_workspace_bytes(frag.c, K))


def quantize_workspace_bytes(frag: Fragment, K: int) -> int:
    return int(lib().dl_quantize_workspace_bytes(frag.c, K))


def new_workspace(nbytes: int, device="cuda"):
    """A zeroed workspace (its first word is the device status word, which
    must start at 0). torch's caching allocator returns 512-byte aligned
    blocks."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def new_stats(K: int, T: int, device="cuda"):
    """Device array of dl_stats, shape [K, T, 6] int64 (fields as raw 8-byte words)."""
    return torch.zeros((K, T, 6), dtype=torch.int64, device=device)


def stats_to_host(stats: torch.Tensor) -> dict:
    """dl_stats array -> dict of numpy arrays [K, T] (count, nonfinite, mean, std, lo, hi)."""
    raw = stats.detach().cpu().numpy()
    f = raw.view(np.float64)
    return {"count": raw[..., 0].copy(), "nonfinite": raw[..., 1].copy(), "mean": f[..., 2].copy(),
            "std": f[..., 3].copy(), "lo": f[..., 4].copy(), "hi": f[..., 5].copy()}


def pseudograd_stats(theta_g, replicas, frag: Fragment, clip_sigmas=6.0, stats=None,
                     workspace=None, stream=None):
    """replicas=None: values mode (statistics of theta_g itself, K = 1)."""
    K = 1 if replicas is None else len(replicas)
    if stats is None:
        stats = new_stats(K, frag.T, theta_g.device)
    need = stats_workspace_bytes(frag, K)
    if workspace is None:
        workspace = new_workspace(need, theta_g.device)
    _need(theta_g, _F32, frag.n, "theta_g")
    _need_all(replicas or [], _F32, frag.n, "replicas")
    _need(stats, _I64, K * frag.T * 6, "stats")
    _need(workspace, _U8, 0, "workspace")
    _cuda(theta_g, replicas or [], stats, workspace)
    _check("dl_pseudograd_stats", lib().dl_pseudograd_stats(
        _ptr(theta_g), None if replicas is None else _ptr_array(replicas), K, frag.c,
        float(clip_sigmas), _ptr(stats),
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return stats


def quantize(theta_g, replicas, frag: Fragment, stats, codes=None, codebook=None, counts=None,
             workspace=None, stream=None):
    """replicas=None: values mode (quantise theta_g itself, K = 1)."""
    K = 1 if replicas is None else len(replicas)
    dev = theta_g.device
    if codes is None:
        codes = [torch.empty(frag.n, dtype=torch.uint8, device=dev) for _ in range(K)]
    if codebook is None:
        codebook = torch.empty((K, frag.T, DL_NBUCKETS), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_workspace(quantize_workspace_bytes(frag, K), dev)
    _need(theta_g, _F32, frag.n, "theta_g")
    _need_all(replicas or [], _F32, frag.n, "replicas")
    _need(stats, _I64, K * frag.T * 6, "stats")
    _need_all(codes, _U8, frag.n, "codes")
    _need(codebook, _F32, K * frag.T * DL_NBUCKETS, "codebook")
    _need(counts, _U32, K * frag.T * DL_NBUCKETS, "counts")
    _need(workspace, _U8, 0, "workspace")
    _cuda(theta_g, replicas or [], stats, codes, codebook, counts, workspace)
    _check("dl_quantize", lib().dl_quantize(
        _ptr(theta_g), None if replicas is None else _ptr_array(replicas), K, frag.c,
        _ptr(stats), _ptr_array(codes),
        _ptr(codebook), _ptr(counts), _ptr(workspace), workspace.numel(), _stream(stream)))
    return codes, codebook


def quantize_noalloc(theta_g, replicas, frag: Fragment, stats, codes, codebook, counts=None,
                     stream=None):
    """quantize() for callers that cannot allocate (dl_quantize_noalloc): the
    scratch is one static device array inside the library, so the caller
    passes every output and nothing is allocated on the device, here or in
    the library. Calls share that array: order calls whose GPU work could
    overlap on one stream. K * frag.T above DL_QUANTIZE_NOALLOC_MAX_SEGMENTS
    raises DLError with status DL_ERR_WORKSPACE, before any launch.
    replicas=None: values mode (quantise theta_g itself, K = 1)."""
    K = 1 if replicas is None else len(replicas)
    if codes is None or codebook is None:
        raise ValueError("quantize_noalloc: codes and codebook are the caller's (no allocation)")
    _need(theta_g, _F32, frag.n, "theta_g")
    _need_all(replicas or [], _F32, frag.n, "replicas")
    _need(stats, _I64, K * frag.T * 6, "stats")
    if len(codes) < K:
        raise ValueError(f"codes: {len(codes)} buffers, need {K}")
    _need_all(codes, _U8, frag.n, "codes")
    _need(codebook, _F32, K * frag.T * DL_NBUCKETS, "codebook")
    _need(counts, _U32, K * frag.T * DL_NBUCKETS, "counts")
    _cuda(theta_g, replicas or [], stats, codes, codebook, counts)
    _check("dl_quantize_noalloc", lib().dl_quantize_noalloc(
        _ptr(theta_g), None if replicas is None else _ptr_array(replicas), K, frag.c,
        _ptr(stats), _ptr_array(codes), _ptr(codebook), _ptr(counts), _stream(stream)))
    return codes, codebook


def merge_outer_step(theta_g, momentum, frag: Fragment, codes=None, codebook=None,
                     replicas=None, weights=None, present=None, min_quorum=1, lr=0.7, mu=0.9,
                     delta_bar=None, stream=None, K=None):
    if K is None:
        K = len(codes) if codes is not None else len(replicas)
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32)
    p = None if present is None else np.ascontiguousarray(present, dtype=np.uint8)
    _need(theta_g, _F32, frag.n, "theta_g")
    _need(momentum, _F32, frag.n, "momentum")
    _need_all(codes or [], _U8, frag.n, "codes")
    _need(codebook, _F32, K * frag.T * DL_NBUCKETS, "codebook")
    _need_all(replicas or [], _F32, frag.n, "replicas")
    _need(delta_bar, _F32, frag.n, "delta_bar")
    _host_k(w, p, K)
    _cuda(theta_g, momentum, codes or [], codebook, replicas or [], delta_bar)
    _check("dl_merge_outer_step", lib().dl_merge_outer_step(
        _ptr(theta_g), _ptr(momentum), None if codes is None else _ptr_array(codes),
        _ptr(codebook), None if replicas is None else _ptr_array(replicas), K, frag.c,
        None if w is None else w.ctypes.data, None if p is None else p.ctypes.data,
        int(min_quorum), float(lr), float(mu), _ptr(delta_bar), _stream(stream)))


def _host_k(weights, present, K):
    """Host arrays the ABI reads K entries of."""
    for name, arr in (("weights", weights), ("present", present)):
        if arr is not None and arr.size < K:
            raise ValueError(f"{name}: {arr.size} entries, need {K}")


def _jobs(frags, theta_g=None, momentum=None, replicas=None, weights=None, present=None,
          delta_bar=None):
    """ctypes array of dl_fragment_job plus the host arrays it points into
    (returned together so that they stay alive for the call)."""
    P = len(frags)
    arr = (_FragmentJob * max(P, 1))()
    keep = []
    for j, F in enumerate(frags):
        job = arr[j]
        job.frag = ctypes.pointer(F._c)
        if theta_g is not None:
            _need(theta_g[j], _F32, F.n, f"theta_g[{j}]")
            _need(momentum[j], _F32, F.n, f"momentum[{j}]")
            job.theta_g = theta_g[j].data_ptr()
            job.momentum = momentum[j].data_ptr()
        if replicas is not None:
            _need_all(replicas[j], _F32, F.n, f"replicas[{j}]")
            ra = _ptr_array(replicas[j])
            keep.append(ra)
            job.theta_k = ctypes.cast(ra, ctypes.c_void_p)
        if weights is not None and weights[j] is not None:
            w = np.ascontiguousarray(weights[j], dtype=np.float32)
            keep.append(w)
            job.weights = w.ctypes.data
        if present is not None and present[j] is not None:
            pr = np.ascontiguousarray(present[j], dtype=np.uint8)
            keep.append(pr)
            job.present = pr.ctypes.data
        if delta_bar is not None and delta_bar[j] is not None:
            _need(delta_bar[j], _F32, F.n, f"delta_bar[{j}]")
            job.delta_bar_out = delta_bar[j].data_ptr()
    return arr, keep


def outer_sync_workspace_bytes(frags, K: int, flags: int = 0) -> int:
    arr, _ = _jobs(frags)
    return int(lib().dl_outer_sync_workspace_bytes(arr, len(frags), K, int(flags)))


def outer_sync(frags, theta_g, momentum, replicas, K, workspace=None, weights=None, present=None,
               min_quorum=1, clip_sigmas=6.0, lr=0.7, mu=0.9, flags=0, delta_bar=None,
               stream=None):
    """One outer step over every fragment (dl_outer_sync). Per-fragment lists:
    theta_g[j], momentum[j], replicas[j] (K tensors), and optionally
    weights[j] / present[j] (length-K host arrays) and delta_bar[j]. flags:
    DL_SYNC_UNQUANTIZED, DL_SYNC_RDA or DL_SYNC_RING, each optionally with
    DL_SYNC_SERIAL."""
    arr, keep = _jobs(frags, theta_g, momentum, replicas, weights, present, delta_bar)
    if workspace is None and not flags & DL_SYNC_UNQUANTIZED:
        workspace = new_workspace(outer_sync_workspace_bytes(frags, K, flags), theta_g[0].device)
    _need(workspace, _U8, 0, "workspace")
    _cuda(workspace, list(theta_g), list(momentum), [r for rs in replicas for r in rs],
          [d for d in (delta_bar or [])])
    nbytes = 0 if workspace is None else workspace.numel()
    _check("dl_outer_sync", lib().dl_outer_sync(
        arr, len(frags), K, float(clip_sigmas), int(min_quorum), float(lr), float(mu), int(flags),
        _ptr(workspace), nbytes, _stream(stream)))
    del keep
    return workspace


def shutdown():
    """Release the side stream and events dl_outer_sync created (dl_shutdown)."""
    _check("dl_shutdown", lib().dl_shutdown())


def rda_workspace_bytes(frag: Fragment, K: int) -> int:
    return int(lib().dl_rda_workspace_bytes(frag.c, K))


def rda_merge_outer_step(theta_g, momentum, frag: Fragment, codes, codebook, counts, weights=None,
                         present=None, min_quorum=1, lr=0.7, mu=0.9, delta_bar=None,
                         workspace=None, stream=None, K=None):
    """Radial-Directional Averaging merge of decoded values, then the outer
    step (dl_rda_merge_outer_step); counts as written by quantize()."""
    if K is None:
        K = len(codes)
    if workspace is None:
        workspace = new_workspace(rda_workspace_bytes(frag, K), theta_g.device)
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32)
    p = None if present is None else np.ascontiguousarray(present, dtype=np.uint8)
    _need(theta_g, _F32, frag.n, "theta_g")
    _need(momentum, _F32, frag.n, "momentum")
    _need_all(codes, _U8, frag.n, "codes")
    _need(codebook, _F32, K * frag.T * DL_NBUCKETS, "codebook")
    _need(counts, _U32, K * frag.T * DL_NBUCKETS, "counts")
    _need(delta_bar, _F32, frag.n, "delta_bar")
    _need(workspace, _U8, 0, "workspace")
    _host_k(w, p, K)
    _cuda(theta_g, momentum, codes, codebook, counts, delta_bar, workspace)
    _check("dl_rda_merge_outer_step", lib().dl_rda_merge_outer_step(
        _ptr(theta_g), _ptr(momentum), _ptr_array(codes), _ptr(codebook), _ptr(counts), K,
        frag.c, None if w is None else w.ctypes.data, None if p is None else p.ctypes.data,
        int(min_quorum), float(lr), float(mu), _ptr(delta_bar), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return workspace


def ring_workspace_bytes(frag: Fragment) -> int:
    return int(lib().dl_ring_workspace_bytes(frag.c))


def ring_outer_step(theta_g, momentum, frag: Fragment, replicas, weights=None, present=None,
                    min_quorum=1, clip_sigmas=6.0, lr=0.7, mu=0.9, delta_bar=None,
                    workspace=None, stream=None, hop_stats=None):
    """Ring accumulation with re-quantisation at every hop, then the outer
    step (dl_ring_outer_step); theta_g and momentum are updated in place.
    hop_stats: optional device int64 tensor of (S-1) * T * 6 words (as
    new_stats(S - 1, T)) that receives the statistics of each quantised
    partial sum."""
    if workspace is None:
        workspace = new_workspace(ring_workspace_bytes(frag), theta_g.device)
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32)
    p = None if present is None else np.ascontiguousarray(present, dtype=np.uint8)
    K = len(replicas)
    _host_k(w, p, K)
    S = K if p is None else int(np.count_nonzero(p[:K]))
    _need(theta_g, _F32, frag.n, "theta_g")
    _need(momentum, _F32, frag.n, "momentum")
    _need_all([r for k, r in enumerate(replicas) if p is None or p[k]], _F32, frag.n, "replicas")
    _need(delta_bar, _F32, frag.n, "delta_bar")
    _need(hop_stats, _I64, max(S - 1, 0) * frag.T * 6, "hop_stats")
    _need(workspace, _U8, 0, "workspace")
    _cuda(theta_g, momentum, [r for k, r in enumerate(replicas) if p is None or p[k]], delta_bar,
          hop_stats, workspace)
    _check("dl_ring_outer_step", lib().dl_ring_outer_step(
        _ptr(theta_g), _ptr(momentum), _ptr_array(replicas), len(replicas), frag.c,
        None if w is None else w.ctypes.data, None if p is None else p.ctypes.data,
        int(min_quorum), float(clip_sigmas), float(lr), float(mu), _ptr(delta_bar),
        _ptr(hop_stats), _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


def selftest_wait_timeout(workspace, polls=1000, stream=None):
    """Run one bounded wait that nothing completes (dl_selftest_wait_timeout);
    the workspace's status word then reports it."""
    _need(workspace, _U8, 4, "workspace")
    _cuda(workspace)
    _check("dl_selftest_wait_timeout",
           lib().dl_selftest_wait_timeout(_ptr(workspace), int(polls), _stream(stream)))


def selftest_pipeline(workspace, src, stall_tile, polls=1000, out=None, stream=None):
    """Run the tile pipeline's abort self-test (dl_selftest_pipeline): src is a
    device float32 tensor of n_tiles * 1024 elements; returns the per-tile
    sums (NaN from stall_tile on when the pipeline aborted)."""
    n_tiles = src.numel() // 1024
    if out is None:
        out = torch.empty(n_tiles, dtype=torch.float32, device=src.device)
    _need(workspace, _U8, 4, "workspace")
    _need(src, _F32, n_tiles * 1024, "src")
    _need(out, _F32, n_tiles, "out")
    _cuda(workspace, src, out)
    _check("dl_selftest_pipeline",
           lib().dl_selftest_pipeline(_ptr(workspace), _ptr(src), n_tiles, int(stall_tile),
                                      int(polls), _ptr(out), _stream(stream)))
    return out


def read_device_status(workspace, stream=None) -> int:
    _need(workspace, _U8, 4, "workspace")
    _cuda(workspace)
    v = ctypes.c_uint32(0)
    _check("dl_read_device_status",
           lib().dl_read_device_status(_ptr(workspace), ctypes.byref(v), _stream(stream)))
    return int(v.value)


class OuterSync:
    """The three device calls of one fragment with preallocated buffers.

    ``step`` computes stats, codes and codebooks of the K replicas, then merges
    them into theta_g / momentum in place. Buffers are reused across calls.
    """

    def __init__(self, frag: Fragment, K: int, device="cuda", clip_sigmas=6.0, lr=0.7, mu=0.9):
        self.frag, self.K, self.clip, self.lr, self.mu = frag, K, clip_sigmas, lr, mu
        self.stats = new_stats(K, frag.T, device)
        self.ws_stats = new_workspace(stats_workspace_bytes(frag, K), device)
        self.ws_quant = new_workspace(quantize_workspace_bytes(frag, K), device)
        self.codes = [torch.empty(max(frag.n, 1), dtype=torch.uint8, device=device)
                      for _ in range(K)]
        self.codebook = torch.empty((K, max(frag.T, 1), DL_NBUCKETS), dtype=torch.float32,
                                    device=device)

    def step(self, theta_g, momentum, replicas, weights=None, present=None, min_quorum=1,
             delta_bar=None, stream=None, counts=None):
        """One outer step; only present learners' replicas are read (others may be None)."""
        idx = [k for k in range(len(replicas)) if present is None or present[k]]
        if len(idx) < max(1, int(min_quorum)):
            raise DLError("OuterSync.step", -3)
        reps = [replicas[k] for k in idx]
        kp = len(idx)
        w = None if weights is None else np.asarray(weights, dtype=np.float32)[idx]
        pseudograd_stats(theta_g, reps, self.frag, self.clip, self.stats[:kp], self.ws_stats,
                         stream)
        quantize(theta_g, reps, self.frag, self.stats[:kp], self.codes[:kp], self.codebook[:kp],
                 counts, self.ws_quant, stream)
        merge_outer_step(theta_g, momentum, self.frag, self.codes[:kp], self.codebook[:kp],
                         weights=w, min_quorum=min_quorum, lr=self.lr, mu=self.mu,
                         delta_bar=delta_bar, stream=stream)
        return idx


class ModelSync:
    """Whole-model outer step (dl_outer_sync) over a fixed list of fragments,
    with its workspace allocated once."""

    def __init__(self, frags, K: int, device="cuda", clip_sigmas=6.0, lr=0.7, mu=0.9, mode=0):
        """mode: 0 (mean merge), DL_SYNC_RDA or DL_SYNC_RING; the workspace is
        sized for it (and serves the unquantised and serial variants)."""
        self.frags, self.K, self.clip, self.lr, self.mu = list(frags), K, clip_sigmas, lr, mu
        self.mode = int(mode)
        self.workspace = new_workspace(outer_sync_workspace_bytes(self.frags, K, self.mode),
                                       device)

    def step(self, theta_g, momentum, replicas, weights=None, present=None, min_quorum=1,
             delta_bar=None, flags=0, stream=None):
        if not flags & DL_SYNC_UNQUANTIZED:
            flags |= self.mode
        outer_sync(self.frags, theta_g, momentum, replicas, self.K, self.workspace, weights,
                   present, min_quorum, self.clip, self.lr, self.mu, flags, delta_bar, stream)
