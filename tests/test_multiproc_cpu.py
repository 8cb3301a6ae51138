"""The multi-GPU (replicas) host logic of the benchmark on CPU with gloo,
world_size 2: each rank times its own replica; the job reports the slowest
rank's time and the units of all ranks over it."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    r, w, local, d = bench._dist()
    assert (r, w, local) == (rank, ws, rank) and d is dist
    ms_local = 2.0 + rank          # rank 1 is the slow one
    ms = bench.max_over_ranks(ms_local, dist, "cpu")
    out[rank] = (ms, bench.whole_job_tflops(1.0e12, ms, w))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_aggregate_over_two_gloo_ranks():
    ws = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(ws, _free_port(), out), nprocs=ws, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, tflops = res[0]
    assert ms == 3.0
    assert tflops == pytest.approx(2 * 1.0e12 / 3.0e-3 / 1e12)


def test_single_process_is_identity():
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.whole_job_tflops(1e12, 1.0, 1) == pytest.approx(1000.0)
