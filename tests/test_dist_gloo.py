"""The multi-process side of bench.py on CPU (gloo, world size 2).

One GPU per rank runs independent replicas; the job's time is the maximum
over ranks and only rank 0 prints.  These tests run the same host logic over
gloo on CPU: the max-over-ranks reduction and barrier, and the reference arm
under torchrun (rank 0 prints one JSON line, the other rank exits 0).
"""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    out[rank] = d.max(1.5 + rank * 2.0)
    d.barrier()
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init()
    assert not d.pg and d.max(2.0) == 2.0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-rows", "16",
           "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
