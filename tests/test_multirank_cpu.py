"""World-size-2 host-side tests of the multi-rank bench path on CPU (gloo).

The operator shards over (sequence, head) with no exchange, so `bench.py --gpus N`
runs N independent replicas: the only cross-rank steps are the barriers around
the timed region and the max over ranks of the elapsed time.  These tests run
those steps with two gloo ranks, and the whole `bench.py --impl reference` launch
under torchrun (rank 0 prints the one JSON line, the other rank exits 0).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    # rank r took (r + 1) * 10 ms: the job took the slowest rank's time
    out[rank] = bench.max_over_ranks(10.0 * (rank + 1), w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs)
        assert dict(out) == {0: 20.0, 1: 20.0}



@pytest.mark.skipif(torch.cuda.is_available(), reason="the CPU (gloo) launch path")
def test_bench_reference_arm_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
           "--workload", "tiny", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["scaling"] == "weak"
    assert d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
