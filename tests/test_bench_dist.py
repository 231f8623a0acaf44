"""The benchmark's multi-process plumbing on CPU (gloo, world size 2): the max-over-ranks
timing, failure of a rank that never joins (a short process-group timeout ends the wait
with an error, no hang), and the reference arm under torchrun (rank 0 alone prints)."""
import json
import os
import socket
import subprocess
import sys
import time

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist = bench.dist_init(world, False, timeout_s=30)
    bench.barrier(dist)
    q.put((rank, bench.max_over_ranks(dist, 1.5 + rank)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2.5), (1, 2.5)]


def _lonely_rank(port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK="0", WORLD_SIZE="2")
    import bench
    t0 = time.time()
    try:
        bench.dist_init(2, False, timeout_s=3)
        q.put(("joined", time.time() - t0))
    except Exception as e:  # the missing rank is detected on the host
        q.put((type(e).__name__, time.time() - t0))


def test_missing_rank_is_detected_by_timeout():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_lonely_rank, args=(free_port(), q))
    p.start()
    what, took = q.get(timeout=120)
    p.join(timeout=60)
    assert what != "joined" and took < 60


def test_step_stats_single_process():
    import bench
    assert bench.step_stats([3.0, 1.0, 2.0, 10.0], None, None) == {"median": 2.5, "min": 1.0}


def test_reference_arm_under_torchrun_prints_one_line():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload", "tiny", "--cpu-procs", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["n_gpus"] == 2
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
    # two oracle processes, one per core asked for, timed over the same windows
    assert rec["cpu_baseline"]["cores"] == 2 and rec["cpu_baseline"]["value"] == rec["value"]
