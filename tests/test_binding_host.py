"""The Python binding's own checks, on the host (no GPU): the C ABI takes raw
pointers and sizes, so the binding refuses tensors whose element type,
layout, size or device would make those pointers wrong, before any call."""
import numpy as np
import pytest
import torch

import pseudo_grad_sync_gb300 as dl
from pseudo_grad_sync_gb300 import _build


@pytest.fixture(scope="module")
def F():
    _build.build()  # in-tree, and only when its sources are newer
    dl.lib()
    return dl.Fragment([100, 28], device="cpu")


def _f32(n):
    return torch.zeros(n, dtype=torch.float32)


def test_wrong_dtype_size_layout_and_device_are_refused(F):
    g = _f32(F.n)
    reps = [_f32(F.n), _f32(F.n)]
    with pytest.raises(TypeError, match="theta_g: dtype"):
        dl.pseudograd_stats(g.double(), reps, F)
    with pytest.raises(ValueError, match=r"replicas\[1\]: 127 elements"):
        dl.pseudograd_stats(g, [reps[0], _f32(F.n - 1)], F)
    with pytest.raises(ValueError, match="must be contiguous"):
        dl.pseudograd_stats(torch.zeros(2 * F.n)[::2], reps, F)
    with pytest.raises(ValueError, match="CUDA device"):
        dl.pseudograd_stats(g, reps, F)
    with pytest.raises(TypeError, match="expected a torch.Tensor"):
        dl.pseudograd_stats(np.zeros(F.n, np.float32), reps, F)


def test_quantize_checks_every_output(F):
    g = _f32(F.n)
    reps = [_f32(F.n)] * 3
    st = dl.new_stats(3, F.T, "cpu")
    codes = [torch.zeros(F.n, dtype=torch.uint8) for _ in range(3)]
    cb = torch.zeros((3, F.T, 256))
    with pytest.raises(TypeError, match="stats: dtype"):
        dl.quantize(g, reps, F, st.double(), codes, cb)
    with pytest.raises(ValueError, match="stats: .* need at least"):
        dl.quantize(g, reps, F, dl.new_stats(2, F.T, "cpu"), codes, cb)
    with pytest.raises(TypeError, match=r"codes\[2\]: dtype"):
        dl.quantize(g, reps, F, st, codes[:2] + [torch.zeros(F.n, dtype=torch.int8)], cb)
    with pytest.raises(ValueError, match="codebook: .* need at least"):
        dl.quantize(g, reps, F, st, codes, torch.zeros((2, F.T, 256)))
    with pytest.raises(TypeError, match="counts: dtype"):
        dl.quantize(g, reps, F, st, codes, cb, counts=torch.zeros((3, F.T, 256)))


def test_merge_ring_and_rda_check_their_host_arrays(F):
    g, m = _f32(F.n), _f32(F.n)
    codes = [torch.zeros(F.n, dtype=torch.uint8) for _ in range(3)]
    cb = torch.zeros((3, F.T, 256))
    with pytest.raises(ValueError, match="weights: 2 entries, need 3"):
        dl.merge_outer_step(g, m, F, codes, cb, weights=[1.0, 1.0])
    with pytest.raises(ValueError, match="present: 2 entries, need 3"):
        dl.ring_outer_step(g, m, F, [_f32(F.n)] * 3, present=[1, 1], workspace=torch.zeros(
            dl.ring_workspace_bytes(F), dtype=torch.uint8))
    with pytest.raises(ValueError, match="hop_stats: .* need at least"):
        dl.ring_outer_step(g, m, F, [_f32(F.n)] * 3, hop_stats=dl.new_stats(1, F.T, "cpu"),
                           workspace=torch.zeros(dl.ring_workspace_bytes(F), dtype=torch.uint8))
    counts = torch.zeros((3, F.T, 256), dtype=torch.int32)
    with pytest.raises(ValueError, match="momentum: .* need at least"):
        dl.rda_merge_outer_step(g, _f32(3), F, codes, cb, counts,
                                workspace=torch.zeros(16, dtype=torch.uint8))


def test_outer_sync_checks_every_job(F):
    frags = [F, dl.Fragment([64], device="cpu")]
    g = [_f32(F.n), _f32(64)]
    m = [_f32(F.n), _f32(63)]
    reps = [[_f32(F.n)] * 2, [_f32(64)] * 2]
    with pytest.raises(ValueError, match=r"momentum\[1\]: 63 elements"):
        dl.outer_sync(frags, g, m, reps, 2, workspace=torch.zeros(16, dtype=torch.uint8))


def test_quantize_noalloc_takes_caller_outputs_and_checks_them(F):
    g = _f32(F.n)
    reps = [_f32(F.n)] * 2
    st = dl.new_stats(2, F.T, "cpu")
    codes = [torch.zeros(F.n, dtype=torch.uint8) for _ in range(2)]
    cb = torch.zeros((2, F.T, 256))
    with pytest.raises(ValueError, match="caller's"):
        dl.quantize_noalloc(g, reps, F, st, None, cb)
    with pytest.raises(ValueError, match="codes: 1 buffers, need 2"):
        dl.quantize_noalloc(g, reps, F, st, codes[:1], cb)
    with pytest.raises(ValueError, match="codebook: .* need at least"):
        dl.quantize_noalloc(g, reps, F, st, codes, torch.zeros((1, F.T, 256)))
    with pytest.raises(TypeError, match="counts: dtype"):
        dl.quantize_noalloc(g, reps, F, st, codes, cb, counts=torch.zeros((2, F.T, 256)))
    with pytest.raises(ValueError, match="CUDA device"):
        dl.quantize_noalloc(g, reps, F, st, codes, cb)
