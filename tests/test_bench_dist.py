"""bench.py's multi-process logic on CPU with gloo, world size 2 (no GPU).

Each rank runs its own batch (weak scaling, no collective on the data path);
the timing reductions are the only collectives: the step time is the max
over ranks and the value is the units every rank processed divided by it.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(backend="gloo")
    try:
        seconds = 1.0 + rank            # rank 1 is the slow one
        value, t = bench.aggregate(units_per_rank_step=100.0, steps=10, max_seconds=seconds, dist=d)
        out[rank] = (value, t, d.max(rank * 3.0), d.sum(1.0))
    finally:
        d.close()


def test_aggregate_is_whole_job_over_slowest_rank():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        value, t, mx, sm = res[rank]
        assert t == 2.0                       # max over ranks
        assert value == pytest.approx(2 * 100.0 * 10 / 2.0)
        assert mx == 3.0 and sm == 2.0


def test_reference_arm_prints_only_on_rank_zero():
    port = _free_port()
    env_base = dict(os.environ, WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                    OMP_NUM_THREADS="2")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--ref-step-seconds", "0.05", "--workload", "decode_bgmv"]
    procs = []
    for rank in (0, 1):
        env = dict(env_base, RANK=str(rank), LOCAL_RANK=str(rank))
        procs.append(subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                                      cwd=ROOT))
    outs = [p.communicate(timeout=600) for p in procs]
    assert [p.returncode for p in procs] == [0, 0], [o[1][-2000:] for o in outs]
    lines0 = [l for l in outs[0][0].splitlines() if l.startswith("{")]
    lines1 = [l for l in outs[1][0].splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and not lines1
    line = json.loads(lines0[0])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
