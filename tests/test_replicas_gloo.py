"""The multi-GPU path is replicas (independent sequences per rank, no
exchange); its only cross-rank step is the aggregation of the benchmark's
numbers.  Checked here with two gloo ranks on the CPU: every rank gets the
units of both ranks over the slower rank's time."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    from lossless_draft_verify_gb300 import replicas
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        units = [300.0, 500.0][rank]
        ms = [10.0, 12.5][rank]
        rate, ms_max = replicas.whole_job_rate(units, ms, pg=dist)
        out[rank] = (rate, ms_max, replicas.max_over_ranks(rank + 1.0, pg=dist),
                     replicas.sum_over_ranks(rank + 1.0, pg=dist))
    finally:
        dist.destroy_process_group()


def test_whole_job_rate_over_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        rate, ms_max, mx, sm = res[rank]
        assert ms_max == 12.5
        assert abs(rate - 800.0 / 0.0125) < 1e-6
        assert mx == 2.0 and sm == 3.0


def test_single_process_is_local():
    from lossless_draft_verify_gb300 import replicas
    rate, ms = replicas.whole_job_rate(100.0, 20.0)
    assert ms == 20.0 and abs(rate - 5000.0) < 1e-9
