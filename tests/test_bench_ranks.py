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


def test_reference_arm_line_on_rank0_uses_the_oracle_pool(monkeypatch):
    """Rank 0 prints one JSON line whose CPU baseline ran one oracle process per
    head (the tiny workload has one head, so one core), extrapolated and marked so."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    import synth
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(type("A", (), dict(steps=1, warmup=0, gpus=1, iters=2))(),
                            synth.CONFIGS["pr1"])
    line = json.loads(buf.getvalue().strip())
    assert line["impl"] == "reference" and line["extrapolated"] is True
    assert line["cpu_baseline"]["cores"] == 1 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["value"] > 0 and line["sample_s_per_step"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_oracle_pool_runs_one_head_per_core():
    """Several heads at once: the extrapolation takes the slowest head's time,
    heads / cores rounds of it, and the row count scaled to every row."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    w = synth.CONFIGS["h8"]
    pool = bench.OraclePool(w.B * w.H)
    try:
        r = bench.cpu_oracle_sample(w, pool, rows_per_head=2, iters=1)
    finally:
        pool.close()
    assert 1 <= r["cores"] <= 8
    per_head = r["t_prep_head_s"] + r["t_rows_s"] * w.N / 2
    assert r["t_step_s"] <= -(-8 // r["cores"]) * per_head * (1 + 1e-9)
    assert r["value"] == pytest.approx(w.flops / r["t_step_s"] / 1e12)


def test_xu_roofline_counts_the_softmax_exponentials():
    sys.path.insert(0, ROOT)
    import bench
    import synth
    w = synth.CONFIGS["wan720p_fp4"]
    r = bench.xu_roofline(w, 64.7, 152, 2070.0)
    nb = (w.N + 127) // 128
    # one exponential per score, an ex2 and a lg2 per 16-score block scale, one
    # ex2 per row and key block
    assert r["ops_per_launch"] == pytest.approx(w.H * (w.N * w.N * 18 / 16 + w.N * nb))
    assert r["peak"] == pytest.approx(32 * 152 * 2070e6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert 0.3 < r["frac"] < 0.5
