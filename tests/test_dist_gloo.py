"""Host logic of the multi-GPU bench path on CPU (gloo, world size 2).

Sessions are independent, so N GPUs run N replicas with no collective on the
data path; the only cross-rank steps are the barriers around the timed region
and the max over ranks of the step time.  Rank 1 of the reference arm exits
without work or output.
"""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


WORKER = r"""
import os, sys, json
sys.path.insert(0, os.environ["DSB_ROOT"])
import torch.distributed as dist
import bench
world, rank, local = bench._dist_env()
d = bench._maybe_init_dist(world, "gloo")
bench._barrier(d)
m = bench._max_over_ranks(d, 1.5 + rank, "cpu")
print(json.dumps({"rank": rank, "world": world, "max": m}), flush=True)
dist.destroy_process_group()
"""


def _launch(code, world=2, extra_env=None):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(world), LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), DSB_ROOT=ROOT, CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e
        outs.append(o)
    return outs


def test_max_over_ranks_and_barrier():
    import json
    outs = _launch(WORKER)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    assert sorted(r["rank"] for r in res) == [0, 1]
    assert all(r["world"] == 2 and r["max"] == 2.5 for r in res)


def test_reference_arm_prints_only_on_rank_zero():
    code = r"""
import os, sys
sys.path.insert(0, os.environ["DSB_ROOT"])
import bench
world, rank, _ = bench._dist_env()
if rank != 0:
    bench.run_reference(bench.argparse.Namespace(workload="llama-68m", b=8, T=1, steps=1, warmup=3))
    print("rank%d-silent" % rank)
else:
    print("rank0-skipped")
"""
    outs = _launch(code)
    assert outs[1].strip() == "rank1-silent"
