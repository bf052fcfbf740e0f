"""The N > 1 path of bench.py on CPU: two gloo ranks (spawned processes).

Each rank decodes its own replay (weak scaling, no data-path collective); the
job time is the maximum over ranks and the throughput counts every rank's
lookups.  Only rank 0 prints the reference arm's line.
"""
import importlib.util
import os
import socket
import sys
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parent.parent


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", ROOT / "bench.py")
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, str(ROOT))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench = _load_bench()
    r, w, loc = bench.dist_env()
    total, value = bench.aggregate(1.0 + rank, 100, w, dist, "cpu")
    from trellis_row_decode_gb300 import synth
    idx = synth.WORKLOADS["tiny"].indices(synth.SEED_INDEX + r)
    q.put((r, w, loc, total, value, int(idx[:64].sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, t0, v0, s0), (r1, w1, l1, t1, v1, s1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2 and (l0, l1) == (0, 1)
    assert t0 == t1 == 2.0                       # slowest rank decides
    assert v0 == v1 == pytest.approx(100 * 2 / 2.0)
    assert s0 != s1                              # each rank replays its own ids


def test_reference_arm_prints_on_rank0_only(capsys):
    bench = _load_bench()
    from trellis_row_decode_gb300 import synth

    class A:
        steps, warmup, cpu_seconds, gpus = 1, 0, 0.5, 2
    bench.reference_arm(A, synth.WORKLOADS["tiny"], rank=1)
    assert capsys.readouterr().out == ""


def test_single_rank_aggregate_without_dist():
    bench = _load_bench()
    total, value = bench.aggregate(0.5, 1000, 1, None, "cpu")
    assert total == 0.5 and value == 2000.0
    assert np.isfinite(value)
