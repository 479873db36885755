"""The bench's multi-replica host logic on CPU ranks (gloo, world size 2).

The round does not shard: under torchrun each rank runs an independent
replica, and the whole job's figure is the rounds (and tokens) of all ranks
over the slowest rank's timed region.  These tests run that reduction on two
CPU processes, check that the reference arm prints from rank 0 only, and
that its one JSON line keeps the bench contract.
"""

import json
import time
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_ms = [12.5, 20.0][rank]
        rounds, tokens = [20, 20][rank], [33, 41][rank]
        t_max, sums = bench.reduce_over_ranks(world, "cpu", t_ms, rounds, tokens)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"t_max": t_max, "sums": sums}, f)
    finally:
        dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    mp.start_processes(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2,
                       start_method="spawn")
    for r in range(2):
        got = json.loads((tmp_path / f"r{r}.json").read_text())
        assert got["t_max"] == 20.0               # the slowest rank's timed region
        assert got["sums"] == [40.0, 74.0]        # rounds and tokens of both replicas


def test_reduce_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(1, "cpu", 7.25, 3, 9) == (7.25, [3, 9])


def test_reference_arm_other_ranks_exit_without_work():
    # rank 0 alone times the oracle and prints the line; rank 1 exits 0 silently
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_line_keeps_the_contract():
    # one step of the oracle arm on this host: the JSON line's keys, the
    # cpu_baseline describing this run and e2e equal to the line's own value
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    t0 = time.perf_counter()
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=900)
    wall = time.perf_counter() - t0
    assert p.returncode == 0, p.stderr
    lines = [l for l in p.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["higher_is_better"] is True and d["unit"] == "rounds/s"
    assert d["config"]["workload"].startswith("e2e_bf16")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # every step is real timed work: the timed region fits inside the run
    assert d["ms_per_step"] * d["steps"] / 1e3 <= wall
    assert abs(d["value"] - 1e3 / d["ms_per_step"]) <= 1e-3 * d["value"] + 1e-6
