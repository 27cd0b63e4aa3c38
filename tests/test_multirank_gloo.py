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


def _shard_worker(rank, world, port, out):
    # every rank packs the same seeded length draw and shards the windows on its own;
    # the only exchange is this test's check that the shares agree
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import numpy as np
    import torch.distributed as dist

    import variable_length_causal_gb300 as vlc

    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(2024)
    L = np.clip(np.round(rng.lognormal(np.log(400), 0.8, size=20000)), 32, 4095).astype(np.int32)
    p = vlc.pack(L, 4096, extra=1)
    rank_of, load = vlc.shard_packs(L, p, world)
    mine = np.nonzero(rank_of == rank)[0]
    sq = sum(int((L[p.order[p.bin_start[b]:p.bin_start[b + 1]]].astype(np.int64) ** 2).sum()) for b in mine)
    gathered = [None] * world
    dist.all_gather_object(gathered, (mine.tolist(), sq, load.tolist(), p.nbins))
    out[rank] = gathered
    dist.destroy_process_group()


def test_ranks_shard_packs_consistently_without_exchange():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_shard_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        g = out[r]
        nbins = g[0][3]
        owned = sorted(sum((x[0] for x in g), []))
        assert owned == list(range(nbins))                   # every window on exactly one rank
        assert all(x[2] == g[0][2] for x in g)               # every rank computed the same loads
        assert [x[1] for x in g] == g[0][2]                  # a rank's load is its windows' sum L^2
    assert out[0] == out[1]


def _cp_worker(rank, world, port, out):
    """One rank of a context-parallel ring over gloo, forward and backward: the product's host
    partition and block rule decide what is held and computed; the oracle stands in for the device
    attention; the key halves' dk / dv are summed over the ranks with all_reduce."""
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import numpy as np
    import torch.distributed as dist

    import oracle
    import variable_length_causal_gb300 as vlc
    from oracle import cp as ocp

    dist.init_process_group("gloo", rank=rank, world_size=world)
    lengths = [48, 16, 96]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T, H, d = int(cu[-1]), 2, 8
    g = np.random.default_rng(5)                      # every rank draws the same pack
    q, k, v = (g.standard_normal((T, H, d)) for _ in range(3))
    seg_all = np.repeat(np.arange(len(lengths)), lengths)
    rows, pos, cu_chunk = vlc.cp_partition(cu, world, rank)
    # the rank keeps only its own rows; the ring hands the key/value halves around
    kv_local = torch.from_numpy(np.concatenate([k[rows], v[rows]], axis=1))
    gathered = [torch.empty_like(kv_local) for _ in range(world)]
    dist.all_gather(gathered, kv_local)
    meta = torch.from_numpy(np.stack([rows, pos.astype(np.int64)]))
    metas = [torch.empty_like(meta) for _ in range(world)]
    dist.all_gather(metas, meta)
    half = len(rows) // 2
    outs = []
    for qh in (0, 1):
        qs = slice(qh * half, (qh + 1) * half)
        o_parts, l_parts = [], []
        for step in range(world):
            src = (rank - step) % world
            kv = gathered[src].numpy()
            k_rows, k_pos = metas[src][0].numpy(), metas[src][1].numpy()
            for kh in (0, 1):
                mode = vlc.cp_block_mode(world, rank, qh, src, kh)
                if mode == vlc.binding.CP_BLOCK_NONE:
                    continue
                ks = slice(kh * half, (kh + 1) * half)
                o_p, l_p = ocp.block_attention(q[rows[qs]], kv[ks, :H], kv[ks, H:], seg_all[rows[qs]], pos[qs],
                                               seg_all[k_rows[ks]], k_pos[ks], 1.0 / np.sqrt(d))
                o_parts.append(o_p)
                l_parts.append(l_p)
        outs.append(ocp.lse_merge(o_parts, l_parts))
    o_full, l_full = ocp.block_attention(q[rows], k, v, seg_all[rows], pos, seg_all, np.arange(T) - cu[seg_all],
                                         1.0 / np.sqrt(d))
    err_o = max(float(np.abs(outs[h][0] - o_full[h * half:(h + 1) * half]).max()) for h in (0, 1))
    err_l = max(float(np.abs(outs[h][1] - l_full[:, h * half:(h + 1) * half]).max()) for h in (0, 1))

    # backward: the same blocks with the merged O / LSE; dq stays with the queries, the
    # dk / dv of a key half go back to the rank that holds it (summed over every rank)
    dout = g.standard_normal((T, H, d))
    scale = 1.0 / np.sqrt(d)
    dq = np.zeros((len(rows), H, d))
    dkv = torch.zeros((world, len(rows), 2 * H, d), dtype=torch.float64)   # per owner rank
    for qh in (0, 1):
        qs = slice(qh * half, (qh + 1) * half)
        o_m, l_m = outs[qh]
        delta = np.einsum("nhd,nhd->hn", dout[rows[qs]], o_m)
        for step in range(world):
            src = (rank - step) % world
            kv = gathered[src].numpy()
            k_rows, k_pos = metas[src][0].numpy(), metas[src][1].numpy()
            for kh in (0, 1):
                if vlc.cp_block_mode(world, rank, qh, src, kh) == vlc.binding.CP_BLOCK_NONE:
                    continue
                ks = slice(kh * half, (kh + 1) * half)
                bq, bk, bv = ocp.block_attention_backward(q[rows[qs]], kv[ks, :H], kv[ks, H:], dout[rows[qs]],
                                                          seg_all[rows[qs]], pos[qs], seg_all[k_rows[ks]],
                                                          k_pos[ks], l_m, delta, scale)
                dq[qs] += bq
                dkv[src, ks, :H] += torch.from_numpy(bk)
                dkv[src, ks, H:] += torch.from_numpy(bv)
    dist.all_reduce(dkv)
    dk_own, dv_own = dkv[rank, :, :H].numpy(), dkv[rank, :, H:].numpy()
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd_f64(dout, q, k, v, cu, theta=0.0)
    err_g = max(float(np.abs(dq - dq_ref[rows]).max()), float(np.abs(dk_own - dk_ref[rows]).max()),
                float(np.abs(dv_own - dv_ref[rows]).max()))
    out[rank] = (err_o, err_l, rows.tolist(), err_g)
    dist.destroy_process_group()


def test_context_parallel_ring_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_cp_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        assert out[r][0] < 1e-12 and out[r][1] < 1e-12
        assert out[r][3] < 1e-10
    assert sorted(out[0][2] + out[1][2]) == list(range(160))
