"""The multi-GPU path of bench.py (replicas, no collective in the block):
its barrier and max-over-ranks run on any torch.distributed backend, so a
world_size-2 gloo group on the CPU checks that every rank sees the slowest
rank's step time and that the whole-job value counts every rank's tokens."""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        barrier, max_all = bench.collectives(dist, torch.device("cpu"))
        barrier()
        ms = max_all(1.0 + rank)  # rank 1 is the slower one
        q.put((rank, ms, bench.whole_job_tokens_per_s(world, 32, ms)))
        barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_time_the_slowest_rank_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in procs)
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2.0 for g in got)              # the slowest rank's 2 ms
    assert all(abs(g[2] - 2 * 32 / 2e-3) < 1e-6 for g in got)  # 2 ranks x 32 tokens


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    barrier, max_all = bench.collectives(None, None)
    barrier()
    assert max_all(3.5) == 3.5
    assert abs(bench.whole_job_tokens_per_s(1, 1, 0.025) - 40000.0) < 1e-6


def test_candidates_reference_arm_times_the_oracle():
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "candidates", "--cand-T", "2", "--cpu-budget", "1",
                          "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == "candidate_rows_per_s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "candidates_T2_N151936_k16"
