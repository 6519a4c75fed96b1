"""The multi-rank logic of bench.py on CPU, with world size 2 over gloo.

The decode path shards by sequence with no data-path exchange, so N ranks
run N replicas; what must hold across ranks is the timing contract: every
rank meets at the barriers, the step time is the slowest rank's, and the
reported bandwidth counts the bytes of all ranks.  The reference arm runs on
rank 0 alone and the other ranks exit 0 without work."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    # rank r took 1 + r seconds for its steps: the job's time is the slowest
    t = bench.reduce_max(1.0 + r, w, "cpu")
    v = bench.aggregate(2e9, 10, w, t)
    bench.barrier(w)
    out.put((r, w, t, v))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_every_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    for r, (rank, world, t, v) in enumerate(res):
        assert (rank, world) == (r, 2)
        assert t == 2.0  # the slower rank's time on both ranks
        # 2 ranks x 10 steps x 2 GB over 2 s = 20 GB/s
        assert v == pytest.approx(20.0)


def test_reference_arm_prints_one_line_from_rank_zero_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", "bench.py", "--impl",
           "reference", "--workload", "tiny-f16-L200", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
