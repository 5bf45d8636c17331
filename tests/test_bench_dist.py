"""Two-rank (gloo, CPU) test of bench.py's multi-process host logic: rendezvous,
barrier, and the whole-job aggregation (every rank's bytes over the slowest
rank's time).  The data path has no collective: ranks are independent replicas."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
assert d.world == 2 and d.pg is not None
d.barrier()
# rank r moves (r + 1) GB per step and takes (r + 1) * 100 ms for 10 steps
value, ms_max = bench.aggregate(d, (d.rank + 1) * 1e9, (d.rank + 1) * 100.0, 10)
out = {{"rank": d.rank, "value": value, "ms_max": ms_max, "max": d.max(float(d.rank)), "sum": d.sum(1.0)}}
open(os.path.join({tmp!r}, "rank%d.json" % d.rank), "w").write(json.dumps(out))
d.close()
"""


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_gloo_ranks_aggregate(tmp_path):
    port = free_port()
    code = CHILD.format(root=ROOT, tmp=str(tmp_path))
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                   LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=env))
    for p in procs:
        assert p.wait(timeout=120) == 0
    res = [json.loads(open(tmp_path / f"rank{r}.json").read()) for r in range(2)]
    for r in res:
        # (1 + 2) GB x 10 steps over the slowest rank's 0.2 s
        assert abs(r["value"] - 150.0) < 1e-9
        assert r["ms_max"] == 200.0
        assert r["max"] == 1.0 and r["sum"] == 2.0
