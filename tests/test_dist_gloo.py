"""The N > 1 host logic on CPU with gloo, world size 2: disjoint sequence
shards covering the batch, whole-job aggregation (summed tokens, slowest
rank's time), and the benchmark's reference arm printing from rank 0 only."""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from hybrid_ssm_decode_gb300.replicas import aggregate, shard_range

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_shard_range_partitions():
    for total in (0, 1, 7, 256, 513):
        for world in (1, 2, 3, 8):
            spans = [shard_range(total, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == total
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0 and a0 <= a1
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_range(10, 2, 2)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    start, stop = shard_range(512, rank, world)
    dist.barrier()
    units, t = aggregate(stop - start, 10.0 * (rank + 1), dist)
    gathered = [None] * world
    dist.all_gather_object(gathered, (start, stop))
    if rank == 0:
        out.put((units, t, gathered))
    dist.destroy_process_group()


def test_gloo_world2_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    units, t, spans = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert units == 512 and t == 20.0
    assert spans == [(0, 256), (256, 512)]


def test_aggregate_without_group_is_local():
    assert aggregate(5, 3.0) == (5.0, 3.0)


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT
    port = 30500 + os.getpid() % 1000
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node=2", "--master-addr=127.0.0.1", f"--master-port={port}",
                        os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
