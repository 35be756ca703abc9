"""bench.py's multi-rank bookkeeping at world size 2 on the gloo backend (CPU, no GPU).

With N GPUs the bench runs one replica per rank (the forward does not shard: independent heads and
batches, no exchange step), times every rank and reports the whole job: the slowest rank's time
(max over ranks) and the queries of all ranks over it. The timed loop's repetition count must be
the same on every rank. These are the host-side steps of that path; here two processes on
127.0.0.1 run them through torch.distributed's gloo backend.
"""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, sys.argv[1])
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
res = {
    # per-rank times 1.5 and 2.5: every rank reports the slower one
    "max": bench.max_over_ranks(1.5 + rank, world),
    # rank 0 wants ceil(1000 / (10 * 5)) = 20 repetitions, rank 1 ceil(1000 / (20 * 5)) = 10
    "reps": bench.timed_repeats(10.0 * (rank + 1), 5, world, min_s=1.0),
    # 1000 queries per rank, per-rank seconds 0.5 and 1.5
    "rate": bench.job_rate(1000, world, bench.max_over_ranks(0.5 + rank, world)),
    "single": bench.max_over_ranks(3.0, 1),
}
dist.barrier()
dist.destroy_process_group()
with open(os.path.join(sys.argv[2], "r%d.json" % rank), "w") as f:
    json.dump(res, f)
"""


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_agree_on_time_repetitions_and_rate(tmp_path):
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT, ROOT, str(tmp_path)],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT))
    for p in procs:
        out, _ = p.communicate(timeout=120)
        assert p.returncode == 0, out.decode()[-2000:]
    r0 = json.load(open(tmp_path / "r0.json"))
    r1 = json.load(open(tmp_path / "r1.json"))
    assert r0 == r1
    assert r0["max"] == 2.5
    assert r0["reps"] == 20
    assert r0["rate"] == 1000 * 2 / 1.5
    assert r0["single"] == 3.0
