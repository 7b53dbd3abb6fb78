"""The benchmark's multi-rank aggregation (replicas only: each rank verifies
its own batches, the job takes the slowest rank's time) on two gloo ranks on
the CPU, as under torchrun with two GPUs."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import importlib.util
    import sys

    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.argv = ["bench.py"]
    spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    # rank r took (r + 1) ms for 100 (r + 1) positions
    out = bench.aggregate(float(rank + 1), 100 * (rank + 1), world, "cpu")
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        total_ms, positions, value = got[r]
        assert total_ms == 2.0 and positions == 300.0  # slowest rank, all positions
        assert abs(value - 300.0 / 2e-3) < 1e-6


def test_single_rank_is_local():
    import importlib.util
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.aggregate(4.0, 1000, 1) == (4.0, 1000, 1000 / 4e-3)


def test_algorithmic_bytes():
    """The roofline's algorithmic bytes: target rows 0..a_b and draft rows
    0..min(a_b + 1, gamma_b) - 1 of each row, V logits each (the rows the
    method must read, given where each row stops); greedy reads no draft."""
    import importlib.util

    import numpy as np
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    acc, gam = np.array([0, 4, 2]), np.array([4, 4, 2])
    # row 0: 1 target + 1 draft; row 1: 5 + 4; row 2 (all accepted): 3 + 2
    assert bench.bytes_read(acc, gam, 4, 10, False) == (1 + 1 + 5 + 4 + 3 + 2) * 10 * 4
    assert bench.bytes_read(acc, gam, 2, 10, True) == (1 + 5 + 3) * 10 * 2
