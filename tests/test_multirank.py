"""The multi-GPU host logic (independent copies per rank, MAX-reduced timing,
whole-job throughput), run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from exact_attention_blackwell_gb300 import inputs, sharding


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = [12.5, 20.0][rank]
        t = sharding.max_over_ranks(my_ms, dist, "cpu")
        # each rank draws a different slice of the workload from its own seed
        w = inputs.tiny()
        x = inputs.make_inputs(inputs.Workload(w.name, w.B, w.H, w.Hkv, w.N, w.d, w.causal,
                                               sharding.rank_seed(w.seed, rank)), with_dO=False)
        q = x["q"].float()
        gathered = [torch.zeros_like(q) for _ in range(world)]
        dist.all_gather(gathered, q)
        out[rank] = (t, bool(torch.equal(gathered[0], gathered[1])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_with_max_and_draw_distinct_inputs():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of a multi-threaded process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 20.0
    assert res[0][1] is False  # the ranks' inputs differ


def test_whole_job_throughput_counts_every_rank():
    assert sharding.whole_job_tflops(2e12, 10, 1000.0, 4) == pytest.approx(80.0)
    assert sharding.max_over_ranks(3.0) == 3.0
