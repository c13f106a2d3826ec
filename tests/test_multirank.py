"""The multi-rank host logic of bench.py on CPU: two gloo ranks (no GPU).

bench.py --gpus N runs one process per GPU, each on an independent chunk of the
same shape (weak scaling, no data exchanged), and reports the work of all ranks
over the slowest rank's time.  Here two ranks check that their chunks differ,
that the max-over-ranks reduction picks the slowest rank on every rank, and that
the job throughput counts both ranks' work.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from block_sparse_video_row_b300 import synth
    w = bench.rank_workload(synth.WORKLOADS["tiny"], rank)
    q, _, _ = synth.make_qkv(w)
    ms = 10.0 + 5.0 * rank                    # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, world)
    value = bench.job_throughput(synth.useful_flop(w), world, slowest)
    out[rank] = (w.seed, float(q.astype(np.float64).sum()), slowest, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_and_reduce():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    from block_sparse_video_row_b300 import synth
    flop = synth.useful_flop(synth.WORKLOADS["tiny"])
    (seed0, sum0, slow0, val0), (seed1, sum1, slow1, val1) = res[0], res[1]
    assert seed0 != seed1 and sum0 != sum1          # independent chunks
    assert slow0 == slow1 == 15.0                   # every rank sees the slowest time
    assert val0 == val1 == pytest.approx(flop * 2 / 15e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1e12, 1, 1000.0) == pytest.approx(1.0)
