"""bench.py's multi-rank host logic on CPU (gloo, world size 2).

Each rank runs its own replica of the decode workload (requests are
independent, so the path shards by request with no exchange); the only
cross-rank steps are a barrier and the maximum of the per-rank times, and the
whole-job rate counts the units of every rank over the slowest rank's time."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        rate = bench.whole_job_rate(65_536, world, ms * 1e-3)
        q.put((rank, ms, rate))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(0.5, 0.75), (2.0, 1.25)])
def test_max_over_ranks_and_whole_job_rate_gloo(times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(times)
    for rank, ms, rate in got:
        assert ms == slowest, f"rank {rank} saw {ms}"
        assert rate == pytest.approx(2 * 65_536 / (slowest * 1e-3), rel=1e-12)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.whole_job_rate(10, 1, 2.0) == 5.0


def test_reference_arm_other_ranks_do_no_work(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus, impl = 1, 3, 2, "reference"

    assert bench.run_reference(Args, 1, 2) is None
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("n_layers", [1, 2, 5, 8, 9, 12, 23, 40, 78])
def test_e2e_copy_chunks_cover_every_layer_once(n_layers):
    """The end-to-end pass copies every layer's inputs and outputs exactly
    once per step, in chunks of at most six layers, and for the default 23
    layers starts and ends with one-layer chunks (the copies no decode hides)."""
    sys.path.insert(0, ROOT)
    import bench
    chunks = bench.e2e_chunks(n_layers)
    assert sum(chunks) == n_layers and min(chunks) >= 1
    assert max(chunks) <= max(6, n_layers if n_layers <= 6 else 6)
    if n_layers == 23:
        assert chunks[0] == 1 and chunks[-1] == 1
