"""dl_quantize_noalloc: dl_quantize for callers that cannot allocate.

Some callers cannot allocate device memory: their memory belongs to another
allocator or budget (a framework's caching allocator, a plugin host), or
cudaMalloc is not allowed or too costly where they run, since it may
synchronise the device. dl_quantize_noalloc serves them from one static
device array inside the library instead of a caller workspace.

These tests call it through the C ABI, twice in a row on different inputs
(the second call must not see the first call's leftovers), and check its
codes, codebooks and bucket counts against the workspace-based dl_quantize
with the same tolerances as the oracle parity tests. The file sorts last so
that a failure here comes after every other test has run.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def noalloc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import pseudo_grad_sync_gb300 as dl

    fn = dl.lib().dl_quantize_noalloc
    vp = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, vp, ctypes.c_int32, ctypes.POINTER(dl._Fragment), vp, vp, vp, vp, vp]
    return dl, fn


def _inputs(seed, numels, K):
    rng = np.random.default_rng(seed)
    n = sum(numels)
    g = (rng.standard_normal(n) * 0.02).astype(np.float32)
    reps = [(g - rng.standard_normal(n) * 1.2e-3 * (1 + k)).astype(np.float32) for k in range(K)]
    return (torch.from_numpy(g).cuda(), [torch.from_numpy(r).cuda() for r in reps])


def _call_noalloc(dl, fn, g, reps, frag, stats):
    K = len(reps)
    codes = [torch.full((frag.n,), 7, dtype=torch.uint8, device="cuda") for _ in range(K)]
    cb = torch.full((K, frag.T, 256), float("nan"), dtype=torch.float32, device="cuda")
    counts = torch.full((K, frag.T, 256), -1, dtype=torch.int32, device="cuda")
    st = fn(ctypes.c_void_p(g.data_ptr()), dl._ptr_array(reps), K, frag.c,
            ctypes.c_void_p(stats.data_ptr()), dl._ptr_array(codes),
            ctypes.c_void_p(cb.data_ptr()), ctypes.c_void_p(counts.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, codes, cb, counts


@pytest.mark.parametrize("reverse", [False, True])
def test_noalloc_matches_quantize_on_two_calls(noalloc, reverse):
    dl, fn = noalloc
    # K = 1 takes the one-learner quantiser (histogram copies), the others
    # learner groups
    cases = [(1, [9000, 8192 * 3 + 5, 77], 3), (2, [40000, 3, 8192], 5),
             (3, [8192 * 10 + 17, 500], 1)]
    if reverse:
        cases = cases[::-1]
    for seed, numels, K in cases:
        g, reps = _inputs(seed, numels, K)
        frag = dl.Fragment(numels)
        stats = dl.pseudograd_stats(g, reps, frag)
        counts_a = torch.empty((K, frag.T, 256), dtype=torch.int32, device="cuda")
        codes_a, cb_a = dl.quantize(g, reps, frag, stats, counts=counts_a)
        st, codes_b, cb_b, counts_b = _call_noalloc(dl, fn, g, reps, frag, stats)
        assert st == 0, dl.status_string(st)
        torch.cuda.synchronize()
        for k in range(K):
            assert torch.equal(codes_a[k], codes_b[k])
        assert torch.equal(counts_a, counts_b)
        # the same kernels on the same inputs, with integer bucket sums: the
        # codebooks agree bit for bit
        assert torch.equal(cb_a, cb_b)


def test_noalloc_rejects_fragments_beyond_its_scratch(noalloc):
    dl, fn = noalloc
    # the array serves up to K * n_tensors = 2000 (learner, tensor) segments
    frag = dl.Fragment([1] * 2001)
    g, reps = _inputs(3, [2001], 1)
    stats = dl.new_stats(1, 2001)
    st, _, _, _ = _call_noalloc(dl, fn, g, reps, frag, stats)
    assert st == -6  # DL_ERR_WORKSPACE, nothing launched
    frag_ok = dl.Fragment([1] * 2000)
    assert dl.quantize_workspace_bytes(frag_ok, 1) <= 8 * 1024 * 1024
    g, reps = _inputs(4, [2000], 1)
    stats = dl.pseudograd_stats(g, reps, frag_ok)
    st, codes, cb, counts = _call_noalloc(dl, fn, g, reps, frag_ok, stats)
    assert st == 0
    torch.cuda.synchronize()
    # one-element tensors: sigma = 0, so every code is 0 and cb = the value
    assert int(codes[0].max()) == 0


def test_binding_quantize_noalloc_matches_quantize(noalloc):
    """The Python binding of the same entry point (dl.quantize_noalloc), in
    values mode and with replicas, against dl.quantize bit for bit; a
    fragment past the segment limit raises DLError with DL_ERR_WORKSPACE."""
    dl, _ = noalloc
    for seed, numels, K in ((5, [70000, 9], 2), (6, [8192 * 5 + 3], 1)):
        g, reps = _inputs(seed, numels, K)
        frag = dl.Fragment(numels)
        reps_or_none = None if K == 1 else reps  # K = 1: values mode (theta_g itself)
        stats = dl.pseudograd_stats(g, reps_or_none, frag)
        counts_a = torch.empty((K, frag.T, 256), dtype=torch.int32, device="cuda")
        codes_a, cb_a = dl.quantize(g, reps_or_none, frag, stats, counts=counts_a)
        codes_b = [torch.full((frag.n,), 7, dtype=torch.uint8, device="cuda") for _ in range(K)]
        cb_b = torch.full((K, frag.T, 256), float("nan"), device="cuda")
        counts_b = torch.full((K, frag.T, 256), -1, dtype=torch.int32, device="cuda")
        dl.quantize_noalloc(g, reps_or_none, frag, stats, codes_b, cb_b, counts=counts_b)
        torch.cuda.synchronize()
        for k in range(K):
            assert torch.equal(codes_a[k], codes_b[k])
        assert torch.equal(cb_a, cb_b) and torch.equal(counts_a, counts_b)
    big = dl.Fragment([1] * 2001)
    g, _ = _inputs(7, [2001], 1)
    with pytest.raises(dl.DLError) as e:
        dl.quantize_noalloc(g, None, big, dl.new_stats(1, 2001),
                            [torch.empty(2001, dtype=torch.uint8, device="cuda")],
                            torch.empty((1, 2001, 256), device="cuda"))
    assert e.value.status == dl.DL_ERR_WORKSPACE
