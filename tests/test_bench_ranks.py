"""The benchmark's multi-rank harness on the CPU: two gloo ranks, as under
torchrun with --nproc-per-node 2. The outer step has no data exchange
(replicas only), so what N > 1 adds is the rank bookkeeping and the timing
rule: every rank times its own copy of the step and the job reports the
slowest."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.env_rank()
    # each rank's "timing" differs; every rank must see the maximum
    got = bench.max_over_ranks(10.0 + 7.5 * r, w, "cpu")
    out.put((r, w, local, got))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[:3] for x in res] == [(0, 2, 0), (1, 2, 1)]
    assert all(x[3] == 17.5 for x in res)


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.env_rank() == (0, 1, 0)
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_bench_fragments_and_oracle_sample():
    """The bench syncs the 10B set's median fragment (18 tensors, 415M
    elements) or its largest (the embedding alone, 525M); the oracle's
    bounded sample of the largest is the first values of that one tensor,
    the same values as the head of the whole tensor."""
    import numpy as np

    import bench
    import oracle
    import synthetic

    oracle.lib()
    wl = synthetic.WORKLOADS["decoder_10b"]()
    ts, f = bench.bench_fragment(wl, oracle.plan_fragments)
    assert (len(ts), sum(wl.numels[t] for t in ts)) == (18, 415260672)
    ts, f = bench.bench_fragment(wl, oracle.plan_fragments, "largest")
    assert (f, len(ts), wl.numels[ts[0]]) == (0, 1, 525336576)
    g, reps, off, tot, sel = bench.fragment_cpu_sample(wl, ts, 1 << 16)
    assert sel == ts and tot == 1 << 16 and list(off) == [0, 1 << 16]
    small = synthetic.WORKLOADS["decoder_1b"]()
    t = 5
    head = small.theta_global(t)[: 1 << 12]
    assert np.array_equal(small.theta_global(t, n=1 << 12), head)
