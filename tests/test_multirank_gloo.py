"""The bench's multi-rank harness on CPU: two gloo ranks (no GPU, no data-path collective).

Each rank runs an independently seeded pack of the same workload shape (weak
scaling); ranks meet only at the barrier and at the max/sum reductions of the
timing and FLOP counts, exactly as bench.py does under torchrun.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    from variable_length_causal_gb300 import synth

    w_, r_, l_ = bench.dist_setup()
    assert (w_, r_, l_) == (world, rank, rank)
    bench.barrier(world)
    mx = bench.max_over_ranks(float(rank + 1), world, "cpu")
    sm = bench.sum_over_ranks(float(rank + 1), world, "cpu")
    w = synth.workload(0)
    q, k, v, g, tokens, cu, ign = bench.make_inputs(w, "cpu", rank)
    out[rank] = (mx, sm, float(q.float().sum()), int(cu[-1]))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_seed_independently():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 2.0          # max over ranks
    assert out[0][1] == out[1][1] == 3.0          # sum over ranks
    assert out[0][3] == out[1][3]                 # same pack shape on every rank
    assert out[0][2] != out[1][2]                 # independently seeded tensors


def test_pack_assignment_by_quadratic_cost_across_ranks():
    from variable_length_causal_gb300 import synth

    w = synth.workload(2)
    bins = [w.lengths[(w.cu[:-1] >= b * 4096) & (w.cu[:-1] < (b + 1) * 4096)] for b in range(32)]
    costs = [float((b.astype(float) ** 2).sum()) for b in bins]
    parts = synth.assign_packs(costs, 4)
    loads = [sum(costs[i] for i in p) for p in parts]
    assert sorted(sum(parts, [])) == list(range(32))
    assert max(loads) / min(loads) < 1.25
