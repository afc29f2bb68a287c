"""World-size-2 checks (gloo, CPU) of the multi-rank benchmark logic: every rank runs an
independent replica; the job's time is the max over ranks and its work the sum."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_info() == (world, rank, rank)
    elapsed = 1.0 + rank          # rank 1 is the slow one
    units = 100.0 * (rank + 1)    # different per-rank work
    bench.barrier()
    t, u = bench.reduce_timing(elapsed, units)
    out[rank] = (t, u)
    dist.destroy_process_group()


def test_reduce_timing_two_ranks():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0] == res[1] == (2.0, 300.0)


def test_reduce_timing_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_timing(1.5, 7.0) == (1.5, 7.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm (the CPU oracle) runs and prints on rank 0 alone; the
    other ranks exit 0 without work or output (no process group is needed for it)."""
    import json
    import subprocess
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    outs = {}
    for rank in (1, 0):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank))
        r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs[rank] = r.stdout
    assert outs[1].strip() == ""
    lines = [ln for ln in outs[0].splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
