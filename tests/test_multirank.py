"""Host logic of the multi-rank benchmark on CPU (gloo, world size 2).

Every rank runs an independent replica of the workload; the job's time is the
slowest rank's, and only rank 0 prints. No GPU involved.
"""

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = bench.reduce_max([10.0 * (rank + 1), 3.0 - rank], "cpu")
    out[rank] = vals
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == [20.0, 3.0] and out[1] == [20.0, 3.0]


def test_reference_arm_prints_on_rank_zero_only():
    # torchrun-style environment for a non-zero rank: no output, exit 0
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", "mha_s64_d64"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", "mha_s64_d64"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    import json
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
