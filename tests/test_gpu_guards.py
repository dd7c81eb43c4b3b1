"""Failure path and memory hygiene of the device calls (needs a GPU).

* A bounded wait that nothing completes gives up, reports its failure in the
  workspace's status word and returns; the context stays usable (no trap,
  no hang). The staged kernels' tile pipeline, its producer stalled on
  purpose (it stops issuing copies; nothing faults), aborts, drains its
  issued copies and reports the same way.
* Canary bytes around every output buffer and every workspace of every entry
  point are untouched after the calls, on ragged sizes (tails of 1-3
  elements, a tensor of 3, an empty tensor, chunk-crossing tensors).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dl():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import pseudo_grad_sync_gb300 as dl
    dl.lib()
    return dl


def test_bounded_wait_reports_and_returns(dl):
    ws = dl.new_workspace(256)
    dl.selftest_wait_timeout(ws, polls=1000)
    assert dl.read_device_status(ws) == 1  # the copy-timeout bit
    assert dl.read_device_status(ws) == 0  # read clears it
    dl.selftest_wait_timeout(ws, polls=200000)
    assert dl.read_device_status(ws) == 1
    # the context still works: a small quantisation runs and is clean
    F = dl.Fragment([5000, 70])
    g = torch.randn(F.n, device="cuda") * 0.02
    reps = [g - torch.randn(F.n, device="cuda") * 1e-3 for _ in range(2)]
    st = dl.pseudograd_stats(g, reps, F)
    codes, cb = dl.quantize(g, reps, F, st)
    torch.cuda.synchronize()
    assert torch.isfinite(cb).all()
    with pytest.raises(dl.DLError):
        dl.selftest_wait_timeout(ws, polls=0)


def test_pipeline_abort_drains_and_reports(dl):
    """The staged kernels' tile pipeline with a producer that stops issuing at
    tile 5 of 12 (a stalled copy engine, simulated without any fault): the
    consumers' bounded waits run out, the block aborts - no further copy, no
    further stage read - waits for its issued copies and ends; the status
    word reports the timeout and the context keeps working. With no stall the
    same kernel sums every tile and reports nothing."""
    ws = dl.new_workspace(256)
    src = torch.arange(12 * 1024, dtype=torch.float32, device="cuda").remainder_(4096)
    want = src.view(12, 1024).double().sum(1).float().cpu().numpy()
    got = dl.selftest_pipeline(ws, src, stall_tile=12, polls=1 << 20).cpu().numpy()
    assert np.array_equal(got, want)
    assert dl.read_device_status(ws) == 0
    for stall in (0, 1, 5):
        got = dl.selftest_pipeline(ws, src, stall_tile=stall, polls=2000).cpu().numpy()
        assert np.array_equal(got[:stall], want[:stall])
        assert np.isnan(got[stall:]).all()
        assert dl.read_device_status(ws) == 1  # the copy-timeout bit, cleared by the read
    got = dl.selftest_pipeline(ws, src, stall_tile=12, polls=1 << 20).cpu().numpy()
    assert np.array_equal(got, want) and dl.read_device_status(ws) == 0
    with pytest.raises(dl.DLError):
        dl.selftest_pipeline(ws, src, stall_tile=13)


PAD = 256  # elements of guard on each side: keeps workspaces 256-byte aligned
CANARY = {torch.float32: np.array([0x7FC0DEAD], dtype=np.uint32).view(np.float32)[0],
          torch.uint8: 0xA5, torch.int32: 0x5A5A5A5A, torch.int64: 0x5A5A5A5A5A5A5A5A}


class Guarded:
    """A device buffer with canary padding on both sides; .t is the inside."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) if shape else 1
        self.raw = torch.empty(n + 2 * PAD, dtype=dtype, device="cuda")
        self.raw.view(torch.uint8 if dtype != torch.float32 else torch.int32).fill_(0)
        self._canary(dtype)
        self.t = self.raw[PAD:PAD + n].view(shape)
        if fill is not None:
            self.t.copy_(fill)
        self.dtype = dtype

    def _canary(self, dtype):
        if dtype == torch.float32:
            v = torch.tensor([0x7FC0DEAD], dtype=torch.int32, device="cuda")
            self.raw.view(torch.int32)[:PAD] = v
            self.raw.view(torch.int32)[-PAD:] = v
        else:
            self.raw[:PAD] = CANARY[dtype]
            self.raw[-PAD:] = CANARY[dtype]

    def intact(self):
        if self.dtype == torch.float32:
            b = self.raw.view(torch.int32)
            return bool((b[:PAD] == 0x7FC0DEAD).all() and (b[-PAD:] == 0x7FC0DEAD).all())
        return bool((self.raw[:PAD] == CANARY[self.dtype]).all()
                    and (self.raw[-PAD:] == CANARY[self.dtype]).all())


RAGGED = [9001, 3, 0, 4095, 8193, 1, 16384 + 2]


def _model(K, numels=RAGGED, seed=0):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    n = sum(numels)
    g = Guarded((n,), torch.float32, torch.randn(n, device="cuda", generator=gen) * 0.02)
    reps = [Guarded((n,), torch.float32,
                    g.t - torch.randn(n, device="cuda", generator=gen) * 1e-3) for _ in range(K)]
    m = Guarded((n,), torch.float32, torch.zeros(n, device="cuda"))
    return g, reps, m


def test_canaries_survive_every_entry_point(dl):
    K = 3
    F = dl.Fragment(RAGGED)
    n, T = F.n, F.T
    g, reps, m = _model(K)
    guards = [g, m] + reps
    stats = Guarded((K, T, 6), torch.int64)
    ws_s = Guarded((dl.stats_workspace_bytes(F, K),), torch.uint8, 0)
    codes = [Guarded((n,), torch.uint8) for _ in range(K)]
    cb = Guarded((K, T, 256), torch.float32)
    counts = Guarded((K, T, 256), torch.int32)
    ws_q = Guarded((dl.quantize_workspace_bytes(F, K),), torch.uint8, 0)
    db = Guarded((n,), torch.float32)
    guards += [stats, ws_s, cb, counts, ws_q, db] + codes
    R = [r.t for r in reps]
    dl.pseudograd_stats(g.t, R, F, 6.0, stats.t, ws_s.t)
    dl.quantize(g.t, R, F, stats.t, [c.t for c in codes], cb.t, counts.t, ws_q.t)
    dl.merge_outer_step(g.t, m.t, F, [c.t for c in codes], cb.t, delta_bar=db.t)
    dl.merge_outer_step(g.t, m.t, F, replicas=R, delta_bar=db.t)
    ws_r = Guarded((dl.rda_workspace_bytes(F, K),), torch.uint8, 0)
    dl.rda_merge_outer_step(g.t, m.t, F, [c.t for c in codes], cb.t, counts.t, delta_bar=db.t,
                            workspace=ws_r.t)
    ws_ring = Guarded((dl.ring_workspace_bytes(F),), torch.uint8, 0)
    dl.ring_outer_step(g.t, m.t, F, R, delta_bar=db.t, workspace=ws_ring.t)
    # values mode
    st1 = Guarded((1, T, 6), torch.int64)
    ws_s1 = Guarded((dl.stats_workspace_bytes(F, 1),), torch.uint8, 0)
    dl.pseudograd_stats(g.t, None, F, 6.0, st1.t, ws_s1.t)
    c1 = Guarded((n,), torch.uint8)
    cb1 = Guarded((1, T, 256), torch.float32)
    ws_q1 = Guarded((dl.quantize_workspace_bytes(F, 1),), torch.uint8, 0)
    dl.quantize(g.t, None, F, st1.t, [c1.t], cb1.t, None, ws_q1.t)
    guards += [ws_r, ws_ring, st1, ws_s1, c1, cb1, ws_q1]
    torch.cuda.synchronize()
    bad = [i for i, x in enumerate(guards) if not x.intact()]
    assert not bad, bad
    # the staged merge (K = 3) reports to the library's own word: clean
    assert dl.read_device_status(None) == 0


@pytest.mark.parametrize("mode", ["mean", "rda", "ring"])
def test_canaries_survive_outer_sync(dl, mode):
    K = 4
    flags = {"mean": 0, "rda": dl.DL_SYNC_RDA, "ring": dl.DL_SYNC_RING}[mode]
    layout = [[9001, 3, 0], [4095, 8193], [1], [16384 + 2, 77]]
    frags = [dl.Fragment(x) for x in layout]
    models = [_model(K, x, seed=i) for i, x in enumerate(layout)]
    ws = Guarded((dl.outer_sync_workspace_bytes(frags, K, flags),), torch.uint8, 0)
    dbs = [Guarded((F.n,), torch.float32) for F in frags]
    dl.outer_sync(frags, [mm[0].t for mm in models], [mm[2].t for mm in models],
                  [[r.t for r in mm[1]] for mm in models], K, workspace=ws.t,
                  delta_bar=[d.t for d in dbs], flags=flags)
    torch.cuda.synchronize()
    guards = [ws] + dbs + [x for mm in models for x in [mm[0], mm[2]] + mm[1]]
    assert all(x.intact() for x in guards)
    assert dl.read_device_status(ws.t) == 0
