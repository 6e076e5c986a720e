"""The multi-process plumbing of bench.py on the CPU: two gloo ranks agree on the max over ranks and
pass the barrier; ranks other than 0 of the reference arm return without work."""
import json
import os
import socket
import subprocess
import sys
import types

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CHILD = """
import json, os, sys
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
v = d.max(10.0 + 5.0 * d.rank)
d.barrier()
print(json.dumps({{"rank": d.rank, "world": d.world, "max": v, "backend": d.pg.get_backend()}}), flush=True)
d.close()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.skipif(torch.cuda.is_available(), reason="the CPU (gloo) form of the plumbing")
def test_two_gloo_ranks_take_the_max_and_meet_at_the_barrier():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=120)
            assert p.returncode == 0, err[-2000:]
            outs.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["world"] == 2 and o["max"] == 15.0 and o["backend"] == "gloo" for o in outs)


def test_reference_arm_runs_on_rank_0_only():
    args = types.SimpleNamespace(workload="c1", steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args, types.SimpleNamespace(rank=1, world=2)) is None


def test_single_process_plumbing_is_a_no_op():
    d = bench.Dist()
    assert d.world == 1 and d.pg is None
    d.barrier()
    assert d.max(3.5) == 3.5
    d.close()
