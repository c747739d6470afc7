"""The benchmark's multi-rank arithmetic on CPU: two gloo ranks on 127.0.0.1, no GPU.

With N GPUs every rank runs its own copy of the workload (no collective on the data path), the
job's time is the slowest rank's and its rate counts the tokens of all ranks ("weak" scaling).
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, os.environ["REPO_ROOT"])
import torch.distributed as dist
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
import bench
got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)], world)
rate = bench.aggregate_rate(world, 8192, got[0])
dist.barrier()
dist.destroy_process_group()
print(json.dumps({"rank": rank, "got": got, "rate": rate}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_report_the_slowest_rank_and_all_tokens():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), REPO_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["got"] == [2.0, 5.0, 0.5]   # element-wise max over the two ranks, on both
        assert o["rate"] == 2 * 8192 / 2e-3  # both ranks' tokens over the slower rank's 2 ms


def test_one_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5], 1) == [3.0, 4.5]
    assert bench.aggregate_rate(1, 8192, 0.25) == 8192 / 0.25e-3
