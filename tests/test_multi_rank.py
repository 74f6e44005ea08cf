"""The multi-rank side of bench.py, on CPU: two gloo ranks (world size 2) on
127.0.0.1.  Every rank runs its own replica of the decode batch (independent
sequences, no data-path collective), so the timed step is the slowest rank's
and the whole-job rate counts the units of every rank; the reference arm runs
on rank 0 only and prints the contract's line there."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        # rank r measured (2 + 3 r) ms for its 4 queries
        ms, rate = bench.combine_over_ranks(2.0 + 3.0 * rank, 4, world, torch.device("cpu"))
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_slowest_ranks_and_rate_counts_all_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for _, ms, rate in got:
        assert ms == 5.0                        # the slower rank's step
        assert abs(rate - 8 / 5e-3) < 1e-6      # 2 ranks x 4 queries per 5 ms


def test_single_rank_keeps_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    ms, rate = bench.combine_over_ranks(4.0, 4, 1, torch.device("cpu"))
    assert ms == 4.0 and abs(rate - 1000.0) < 1e-9


def _bench(env_extra, *args):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_runs_on_rank_zero_only():
    r = _bench({"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"}, "--impl", "reference", "--gpus", "2",
               "--steps", "1", "--warmup", "0")
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""               # no work, no line on the other ranks


def test_reference_arm_line():
    r = _bench({"RANK": "0", "LOCAL_RANK": "0", "WORLD_SIZE": "1"}, "--impl", "reference", "--steps", "1",
               "--warmup", "0")
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["value"] > 0 and line["unit"] == "queries/s" and line["higher_is_better"] is True
    assert line["config"]["workload"] == "decode_1m"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "queries/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
