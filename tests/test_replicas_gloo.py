"""The multi-GPU path is replicas only: every rank verifies its own batch, and
the benchmark adds a barrier and a max over ranks of the timed region, with no
collective on the data path. These tests run that host logic as two gloo
ranks on the CPU (no GPU needed)."""
import json
import os
import socket
import subprocess
import sys

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_RANK_SCRIPT = r"""
import argparse, json, sys
sys.path.insert(0, {root!r})
import bench
world, rank, local, pg = bench.dist_setup(argparse.Namespace(impl="ours"))
bench.barrier(pg)
m = bench.max_over_ranks(pg, 10.0 + 5.0 * rank)
print(json.dumps({{"world": world, "rank": rank, "local": local, "max": m}}), flush=True)
pg.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    env = dict(os.environ)
    env.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(port), SPEC_DIST_BACKEND="gloo", CUDA_VISIBLE_DEVICES="")
    return env


def test_two_ranks_barrier_and_max_over_ranks():
    port = _free_port()
    code = _RANK_SCRIPT.format(root=ROOT)
    procs = [subprocess.Popen([sys.executable, "-c", code], env=_env(r, 2, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            pytest.fail("gloo ranks did not finish")
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    assert all(o["world"] == 2 for o in outs)
    # every rank sees the slowest rank's time
    assert all(o["max"] == 15.0 for o in outs)


def test_replica_throughput_counts_every_rank_at_the_slowest_time():
    assert bench.replica_throughput(1, 10, 256, 8, 2.0) == pytest.approx(10 * 256 * 8 / 2e-3)
    # two replicas in the same time verify twice the positions
    assert bench.replica_throughput(2, 10, 256, 8, 2.0) == pytest.approx(2 * 10 * 256 * 8 / 2e-3)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank_zero_only(rank):
    """Under torchrun the reference arm (the oracle on the host cores) runs
    and prints on rank 0; the other ranks exit 0 without work."""
    env = _env(rank, 2, _free_port())
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny_B4_K4_V1024_f32", "--steps", "2", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    if rank == 0:
        assert len(lines) == 1
        line = json.loads(lines[0])
        assert line["impl"] == "reference" and line["n_gpus"] == 2
        assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    else:
        assert lines == []
