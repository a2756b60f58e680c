"""The bench's multi-GPU path is independent replicas: every rank times its
own decode loop, and rank 0 reports the slowest rank's step time (barrier +
MAX all-reduce).  Checked here with two gloo ranks on the CPU."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    ms = [2.0, 2.5][rank]
    e2e = [480.0, 450.0][rank]
    out[rank] = bench.slowest_over_ranks(ms, e2e, "cpu")
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        ms, e2e = res[r]
        assert ms == pytest.approx(2.5) and e2e == pytest.approx(450.0)
