"""The benchmark's multi-process path on the CPU: two gloo ranks run the
helpers bench.py uses under torchrun (barrier, max over ranks, whole-job
value) and the reference arm runs on rank 0 only. Decode attention shards
into independent replicas, so there is no collective on the data path to
test beyond these."""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_setup(2, backend="gloo")
bench.barrier(world)
slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)   # per-rank timed ms
value = bench.whole_job_gbs(world, 1_000_000, 100, slowest)

class Args:
    workload = "llama-b2-2048"; steps = 1; warmup = 3; rope = False; gpus = 2
t0 = time.perf_counter()
ref = bench.run_reference(Args, world, rank) if rank == 1 else None
took = time.perf_counter() - t0
bench.barrier(world)
print(json.dumps({{"rank": rank, "world": world, "slowest": slowest, "value": value,
                  "ref": ref, "ref_s": took}}), flush=True)
import torch.distributed as dist
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=300)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads([l for l in out.splitlines() if l.startswith("{")][-1]))
    for o in outs:
        assert o["world"] == 2
        assert o["slowest"] == 15.0                    # the max over the two ranks
        # 2 ranks x 1 MB x 100 steps in 15 ms
        assert abs(o["value"] - 2 * 1e6 * 100 / 0.015 / 1e9) < 1e-9
    rank1 = [o for o in outs if o["rank"] == 1][0]
    assert rank1["ref"] is None and rank1["ref_s"] < 1.0   # non-zero ranks do no work
