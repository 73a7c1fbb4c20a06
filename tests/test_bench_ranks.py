"""Host logic of bench.py's multi-GPU path (replicas only), on CPU with two gloo ranks."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


WORKER = r"""
import os, sys, json
sys.path.insert(0, os.environ["ROOT"])
import torch, torch.distributed as dist
dist.init_process_group("gloo", init_method="env://")
rank, world = dist.get_rank(), dist.get_world_size()
import bench
ms, tok = bench.combine_ranks(10.0 + 5.0 * rank, 100 + rank, torch.device("cpu"), world)
runs = bench.reference_runs_here()
print(json.dumps({"rank": rank, "ms": ms, "tok": tok, "ref": runs}), flush=True)
dist.barrier()
dist.destroy_process_group()
"""


def test_two_gloo_ranks_combine_max_time_and_summed_tokens():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, ROOT=ROOT, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err[-2000:]
        outs.append(out.strip().splitlines()[-1])
    import json
    res = sorted((json.loads(o) for o in outs), key=lambda r: r["rank"])
    for r in res:
        assert r["ms"] == 15.0          # the slowest rank's time
        assert r["tok"] == 201.0        # every rank's accepted tokens
    assert [r["ref"] for r in res] == [True, False]


def test_single_rank_passes_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_ranks(3.5, 7, None, 1) == (3.5, 7.0)
