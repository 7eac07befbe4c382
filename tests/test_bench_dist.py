"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks, the slowest
rank's time taken for the whole job, throughput summed over the ranks."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    # rank r "took" 1 + r seconds for 100 steps
    t = bench.max_over_ranks(1.0 + r, w)
    value = bench.aggregate(100, t, w)
    q.put((r, w, lr, t, value))
    torch.distributed.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_sum_the_steps():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local_rank, t, value) in enumerate(got):
        assert (rank, world, local_rank) == (r, 2, r)
        assert t == 2.0                       # the slower rank's time
        assert value == pytest.approx(100 * 2 / 2.0)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate(10, 2.0, 1) == 5.0


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle, timed on the host cores) prints
    one JSON line with the contract's keys, the GPU arm's config and metric,
    and an e2e entry that moves no bytes."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "calls/s"
    for key in ("value", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD and "l2" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "calls/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
