"""The N > 1 host logic of bench.py on CPU (gloo, world size 2).  The round shards by sequence
with no exchange, so N GPUs run N independent replicas: each rank times its own, the job time is
the slowest rank's (all-reduce MAX), and the value counts every rank's rounds.  The reference arm
runs on rank 0 only; the other ranks exit without work."""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = bench.max_over_ranks(1.5 + rank, world, "cpu")  # rank 1 is the slow replica
    q.put((rank, ms, bench.job_rate(10, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_time_the_slowest_and_count_both():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2.5 for g in got)                      # both ranks see the slowest time
    assert all(abs(g[2] - 2 * 10 / 2.5e-3) < 1e-9 for g in got)  # 20 rounds in 2.5 ms


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0
    assert bench.job_rate(5, 1, 2.0) == 2500.0


def _reference(rank: int):
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                           "tiny_f32", "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True,
                          timeout=300, cwd=ROOT)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _reference(1)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _reference(0)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_side_call_cpu_baselines_cover_every_side_call():
    """The benchmark's oracle timings beside its separately timed calls (tiny workload, CPU)."""
    sys.path.insert(0, ROOT)
    import bench
    import datagen

    res = bench.side_cpu_baselines(datagen.WORKLOADS["tiny_f32"], 1)
    assert set(res) == {"kv_commit", "draft_attention", "static_tree", "sampled_build"}
    for v in res.values():
        assert v["kind"] == "oracle" and v["us"] > 0 and v["cores"] >= 1 and v["sample"]
    rl = bench._side_roofline(1e6, 10.0, "x")
    assert rl["bound"] == "hbm" and abs(rl["achieved"] - 100.0) < 1e-9 and rl["frac"] == rl["achieved"] / rl["peak"]
