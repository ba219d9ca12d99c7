"""The multi-process (replicas) path of the benchmark on CPU, with gloo.

The verify step shards by sequence with no data-path collective: each rank
verifies its own seeded batch, the ranks meet at barriers around the timed
region, and the time taken is the maximum over ranks.  These tests run two
ranks as CPU processes (gloo on 127.0.0.1): the helpers that do the
rendezvous, the max over ranks and the per-rank shards, and the reference
arm under torchrun, where rank 0 alone prints its line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    from draft_verify_acceptance_gb300 import workloads as W
    r, w, local = bench.dist_init(world)
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # the time of the slowest rank is the job's time
    t = bench.max_over_ranks(0.25 + rank, w)
    inp = W.workload("tiny_sample_f32_B4_K4_V1000", seed=bench.shard_seed(0, rank))
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": t, "seed": bench.shard_seed(0, rank),
                   "first_logit": float(inp.target[0, 0, 0]), "B": inp.B}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_ranks_take_the_max_time_and_their_own_shards(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert res[0]["max"] == res[1]["max"] == 1.25
    assert res[0]["seed"] != res[1]["seed"]
    assert res[0]["first_logit"] != res[1]["first_logit"]  # independent batches
    assert res[0]["B"] == res[1]["B"] == 4  # fixed work per rank: weak scaling


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2",
           "--impl", "reference", "--workload", "tiny_sample_f32_B4_K4_V1000", "--steps", "2",
           "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
