"""The N > 1 path of bench.py on CPU: two ranks over the gloo backend.

The layer is data-parallel over tokens, so N GPUs run N replicas: each rank takes its own
seeded batch of the same workload (same expert weights), nothing on the data path is
exchanged, and only the step time is reduced, as the maximum over ranks; the whole-job
rate counts the tokens of every rank.  Here each rank's replica is the CPU oracle on the
tiny workload, so the test needs no GPU.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import moe_inputs as mi
import oracle


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica_output(wl_base, rank):
    """The oracle's layer output for rank `rank`'s batch (weights of the base workload)."""
    wl = bench.replica_workload(wl_base, rank)
    q13, s13 = oracle.quant_128x128_bf16(mi.bf16_bits(mi.w13_bf16(wl_base)))
    q2, s2 = oracle.quant_128x128_bf16(mi.bf16_bits(mi.w2_bf16(wl_base)))
    return oracle.moe_forward(mi.bf16_bits(mi.hidden(wl)), mi.router_logits(wl).numpy(), q13, s13, q2, s2,
                              wl.topk)["out"]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out = _replica_output(mi.WORKLOADS["tiny"], rank)
        # stand-in step times, different on each rank: the reduction must return the slowest
        ms = bench.max_over_ranks([1.0 + rank, 10.0 * (rank + 1)], dist, "cpu")
        np.save(os.path.join(out_dir, f"out{rank}.npy"), out)
        np.save(os.path.join(out_dir, f"ms{rank}.npy"), np.array(ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_over_gloo(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    wl = mi.WORKLOADS["tiny"]
    outs = [np.load(tmp_path / f"out{r}.npy") for r in range(world)]
    # each rank computed its own batch: different tokens, and exactly its replica's output
    assert not np.array_equal(outs[0], outs[1])
    for r in range(world):
        np.testing.assert_array_equal(outs[r], _replica_output(wl, r))
    # the step time is the maximum over ranks, on every rank
    for r in range(world):
        assert np.load(tmp_path / f"ms{r}.npy").tolist() == [2.0, 20.0]
    # the whole-job rate counts every rank's tokens in the slowest rank's time
    assert bench.whole_job_rate(world, wl.T, 2.0) == world * wl.T / 2e-3


def test_replica_inputs_differ_only_in_tokens():
    wl = mi.WORKLOADS["tiny"]
    w0, w1 = bench.replica_workload(wl, 0), bench.replica_workload(wl, 1)
    assert w0 == wl and (w1.T, w1.H, w1.I, w1.E, w1.topk) == (wl.T, wl.H, wl.I, wl.E, wl.topk)
    assert not torch.equal(mi.hidden(w0), mi.hidden(w1))
    assert bench.max_over_ranks([3.0, 4.0], None, "cpu") == [3.0, 4.0]
