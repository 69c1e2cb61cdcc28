"""bench.py --shard (strong scaling: the headline's (b, h) problems split
over the ranks) on two gloo ranks without a GPU: the argument handling and
the partition each rank would time, gathered to rank 0 and printed as one
JSON line."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(world, *extra):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={world}", "--master-addr", "127.0.0.1",
           "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--backend", "gloo", "--gpus", str(world), "--steps", "3", "--warmup", "3", *extra]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    return json.loads(lines[0])


def test_shard_plan_two_ranks():
    line = _launch(2, "--shard")
    assert line["plan"] == "shard" and line["scaling"] == "strong" and line["n_gpus"] == 2
    assert line["ranges"] == [[0, 16], [16, 32]]
    assert line["timed"] is False


def test_replica_plan_two_ranks():
    line = _launch(2)
    assert line["plan"] == "replicas" and line["scaling"] == "weak"
    assert line["ranges"] == [[0, 32], [0, 32]]
