"""The multi-GPU host logic (independent copies per rank, MAX-reduced timing,
whole-job throughput), run as two gloo ranks on the CPU."""
import os
import socket

import numpy as np
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


def test_head_pieces_cover_every_group_once():
    for B, Hkv, world in [(4, 16, 8), (3, 5, 4), (1, 8, 3), (2, 1, 4), (5, 3, 7), (1, 1, 2)]:
        seen = []
        for rank in range(world):
            for b0, b1, kh0, kh1 in sharding.head_pieces(B, Hkv, world, rank):
                assert 0 <= b0 < b1 <= B and 0 <= kh0 < kh1 <= Hkv
                seen += [(b, kh) for b in range(b0, b1) for kh in range(kh0, kh1)]
        assert sorted(seen) == [(b, kh) for b in range(B) for kh in range(Hkv)], (B, Hkv, world)
        sizes = [sharding.group_block(B, Hkv, world, r) for r in range(world)]
        counts = [e - s for s, e in sizes]
        assert max(counts) - min(counts) <= 1


def _shard_worker(rank, world, port, out):
    # each rank solves its pieces of one GQA problem with the oracle; rank 0
    # reassembles them and compares with the oracle on the whole problem
    import oracle

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = inputs.Workload("split", 3, 4, 2, 24, 16, True, 77)
        g = w.H // w.Hkv
        x = inputs.make_inputs(w)
        mine = []
        for pc in sharding.head_pieces(w.B, w.Hkv, world, rank):
            q, dO = (sharding.slice_piece(x[n], pc, g) for n in ("q", "dO"))
            k, v = (sharding.slice_piece(x[n], pc) for n in ("k", "v"))
            o, lse = oracle.attention_fwd(q, k, v, w.sm_scale, w.causal)
            dq, dk, dv = oracle.attention_bwd(q, k, v, dO, w.sm_scale, w.causal)
            mine.append((pc, o, lse, dq, dk, dv))
        parts = [None] * world
        dist.all_gather_object(parts, mine)
        if rank == 0:
            o_ref, lse_ref = oracle.attention_fwd(x["q"], x["k"], x["v"], w.sm_scale, w.causal)
            g_ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["dO"], w.sm_scale, w.causal)
            full = {n: np.zeros_like(r) for n, r in zip(("o", "lse", "dq", "dk", "dv"), (o_ref, lse_ref) + tuple(g_ref))}
            for rank_parts in parts:
                for (b0, b1, kh0, kh1), o, lse, dq, dk, dv in rank_parts:
                    full["o"][b0:b1, :, kh0 * g:kh1 * g] = o
                    full["lse"][b0:b1, kh0 * g:kh1 * g] = lse
                    full["dq"][b0:b1, :, kh0 * g:kh1 * g] = dq
                    full["dk"][b0:b1, :, kh0:kh1] = dk
                    full["dv"][b0:b1, :, kh0:kh1] = dv
            errs = [float(np.abs(full[n] - r).max()) for n, r in
                    zip(("o", "lse", "dq", "dk", "dv"), (o_ref, lse_ref) + tuple(g_ref))]
            out[0] = errs
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_one_problem_and_reassemble_the_whole(oracle_mod):
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_shard_worker, args=(world, port, out), nprocs=world, join=True)
        errs = out[0]
    # the same fp64 arithmetic on the same rows: the pieces reproduce the whole problem exactly
    assert max(errs) == 0.0, errs
