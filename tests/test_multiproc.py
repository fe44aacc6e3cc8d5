"""The N > 1 path of bench.py, on CPU with two gloo ranks.

The path partitions into independent matrices, so every rank runs its own
replica (weak scaling) and the only cross-rank steps are the barriers around
the timed region and the max of the ranks' times; rank 0 alone prints.  The
test launches two ranks as separate processes on 127.0.0.1 and checks the
rank bookkeeping, the barrier, the max over ranks and the whole-job
throughput; a second test runs the reference arm under two ranks and checks
that only rank 0 does work and prints.
"""

import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(script: str, ws: int = 2, args=(), timeout: float = 120.0):
    port = _free_port()
    procs = []
    for rank in range(ws):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(ws),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", script, *args], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=timeout)
            outs.append((p.returncode, out, err))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    return outs


def test_two_gloo_ranks_barrier_max_and_job_value():
    script = textwrap.dedent(f"""
        import json, sys
        sys.path.insert(0, {ROOT!r})
        import torch.distributed as dist
        import bench
        ws, rank, local = bench.dist_env()
        dist.init_process_group("gloo")
        bench.barrier(ws)
        t_ms = bench.max_over_ranks(10.0 + 5.0 * rank, ws)   # rank 1 is the slow one
        value = bench.job_value(1.0e9, 4, ws, t_ms)           # 1 GB per step per rank, 4 steps
        bench.barrier(ws)
        print(json.dumps({{"rank": rank, "ws": ws, "local": local, "t_ms": t_ms, "value": value}}))
        dist.destroy_process_group()
    """)
    outs = _launch(script)
    recs = []
    for rc, out, err in outs:
        assert rc == 0, err
        recs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(r["rank"] for r in recs) == [0, 1]
    for r in recs:
        assert r["ws"] == 2 and r["local"] == r["rank"]
        assert r["t_ms"] == 15.0                                   # max over ranks
        assert r["value"] == pytest.approx(2 * 4 * 1.0e9 / 15e-3 / 1e9)  # all ranks' bytes / slowest time


def test_reference_arm_two_ranks_only_rank0_prints():
    script = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        import bench
        sys.argv = ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
        ws, rank, local = bench.dist_env()
        if rank != 0:
            bench.run_reference(bench.argparse.Namespace(gpus=2, steps=1, warmup=0), ws, rank)
            print("rank1-done")
        else:
            print("rank0-skipped")
    """)
    outs = _launch(script)
    assert all(rc == 0 for rc, _, _ in outs), [e for _, _, e in outs]
    texts = [o.strip() for _, o, _ in outs]
    assert texts[0] == "rank0-skipped"
    assert texts[1] == "rank1-done"   # run_reference returned at once on rank 1: no work, no line
