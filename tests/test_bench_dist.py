"""Host logic of the multi-process benchmark on CPU (gloo, world size 2): the barrier, the
max-over-ranks timing reduction, and the reference arm's rank-0-only rule."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys
sys.path.insert(0, {root!r})
import bench
ws, rank, local = bench._init_dist()
assert ws == 2 and bench._PG is not None
bench._barrier()
m = bench._max_over_ranks(1.5 + rank)      # rank 0: 1.5, rank 1: 2.5
assert abs(m - 2.5) < 1e-12, m
print("rank", rank, "ok", flush=True)
"""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _spawn(code, port, rank):
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
               LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    return subprocess.Popen([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                            text=True)


def test_two_rank_barrier_and_max_reduction():
    port = _free_port()
    code = CHILD.format(root=ROOT)
    procs = [_spawn(code, port, r) for r in range(2)]
    outs = [p.communicate(timeout=180)[0] for p in procs]
    for r, (p, out) in enumerate(zip(procs, outs)):
        assert p.returncode == 0, out
        assert f"rank {r} ok" in out


def test_reference_arm_prints_only_on_rank_zero(tmp_path):
    port = _free_port()
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); sys.argv = ['bench.py', '--impl', 'reference', '--gpus', '2', "
            f"'--steps', '1', '--warmup', '0', '--workload', 'tiny-f32', '--ref-budget', '4']; import bench; sys.exit(bench.main())")
    procs = [_spawn(code, port, r) for r in range(2)]
    outs = [p.communicate(timeout=600)[0] for p in procs]
    assert all(p.returncode == 0 for p in procs), outs
    import json
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    lines1 = [l for l in outs[1].splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and not lines1
    j = json.loads(lines0[0])
    assert j["impl"] == "reference" and j["cpu_baseline"]["kind"] == "oracle" and j["value"] > 0
    assert j["e2e"]["h2d_bytes_per_step"] == 0
