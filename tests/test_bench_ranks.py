"""CPU: the multi-rank logic of bench.py on two gloo ranks — the timed region
is the slowest rank's, the value counts every rank's problem (weak scaling),
and the reference arm runs on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(times[rank], dist, "cpu")
    value = bench.weak_value(world, 1e12, ms)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, value))


def test_max_over_ranks_and_weak_value_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [12.5, 20.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == 20.0                        # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 1e12 / 20e-3 / 1e12)


def test_reference_arm_is_silent_on_other_ranks(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import synth
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(type("A", (), dict(steps=1, warmup=0, gpus=2))(), synth.CONFIGS["pr1"])
    assert buf.getvalue() == ""
