"""The multi-rank host logic of bench.py on CPU with gloo (world size 2): the
decode shards by sequence with no data-path collective, so the only
collectives are the barrier and the max-over-ranks of the timed region."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier(world)
    got = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, free_port(), out), nprocs=2, start_method="spawn", join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--workload", "llama70b_b12"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["n_gpus"] == 2
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
    # the line carries the bench contract's keys, for the same metric and workload as the GPU arm
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in rec, key
    sys.path.insert(0, ROOT)
    import bench
    assert rec["metric"] == bench.METRIC and rec["unit"] == bench.UNIT and rec["higher_is_better"] is True
    assert rec["config"]["workload"] == "llama70b_b12"
    assert (rec["steps"], rec["warmup"]) == (1, 3)            # at least three warm-up steps, always
    cb = rec["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == rec["value"]
    assert rec["e2e"]["value"] == rec["value"] and rec["e2e"]["unit"] == rec["unit"]
