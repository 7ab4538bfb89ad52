"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

The decode path shards by (batch row, kv head) with no exchange, so N GPUs run N
replicas; the only cross-rank steps are the barrier and the max-over-ranks timing.
"""

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        rate = bench.whole_job_rate(100.0, world, t)
        out.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, rate in res:
        assert t == 15.0  # every rank sees the slowest rank's time
        assert rate == pytest.approx(100.0 * world / 15.0)


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import synth

    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 1, 0, 2

    assert bench.run_reference(A(), synth.WORKLOADS["tiny-int8"]) == 0
    assert capsys.readouterr().out == ""


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(10, 1, 2.0) == 5.0


def test_reference_arm_line_on_rank_0(capsys, monkeypatch):
    """Rank 0 of the reference arm times the oracle and prints one JSON line with the
    contract's keys, the same workload config keys as the GPU arm, and its e2e block."""
    sys.path.insert(0, ROOT)
    import json

    import bench
    import synth

    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("KVQ_REF_SLICES", "1")

    class A:
        steps, warmup, gpus = 1, 1, 1

    w = synth.WORKLOADS["tiny-int8"]
    assert bench.run_reference(A(), w) == 0
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert {k: d["config"][k] for k in bench.workload_config(w, w.n_layers, w.seq)} == \
        bench.workload_config(w, w.n_layers, w.seq)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
