"""Multi-rank partitioning of the packed-attention work, on CPU.

Head and segment ranges partition the work; two gloo ranks that each compute
their shard (heads, or a contiguous run of segments) with the oracle
reproduce the unsharded result exactly, because every (segment, head) pair
is independent -- the multi-GPU path needs no exchange of data, only the
max of the ranks' times, which is checked here too.  The same holds for the
E4M3 forward, whose descales are per (segment, head): ranks that quantise
their own shard reproduce the unsharded codes and results."""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch

import oracle
from packed_variable_length_varlen_gb300 import sharding as S
from packed_variable_length_varlen_gb300 import workloads as W


def test_head_range_partitions():
    for H in (1, 2, 7, 16, 56):
        for world in (1, 2, 3, 4, 8):
            ranges = [S.head_range(H, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == H
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [h1 - h0 for h0, h1 in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        S.head_range(4, 2, 2)


def test_segment_range_partitions():
    rng = np.random.default_rng(11)
    for trial in range(40):
        B = int(rng.integers(1, 25))
        lq = rng.integers(0, 900, size=B)
        lk = rng.integers(0, 900, size=B)
        cu_q = [0] + list(np.cumsum(lq))
        cu_k = [0] + list(np.cumsum(lk))
        cost = [S.segment_cost(a, b) for a, b in zip(lq, lk)]
        total = sum(cost)
        for world in (1, 2, 3, 5):
            shards = [S.segment_range(cu_q, cu_k, world, r) for r in range(world)]
            assert shards[0].b0 == 0 and shards[-1].b1 == B
            for a, b in zip(shards, shards[1:]):
                assert a.b1 == b.b0 and a.q1 == b.q0 and a.k1 == b.k0
            for sh in shards:
                assert sh.cu_q == [x - cu_q[sh.b0] for x in cu_q[sh.b0:sh.b1 + 1]]
                assert sh.cu_k == [x - cu_k[sh.b0] for x in cu_k[sh.b0:sh.b1 + 1]]
                assert (sh.q0, sh.q1, sh.k0, sh.k1) == (cu_q[sh.b0], cu_q[sh.b1], cu_k[sh.b0], cu_k[sh.b1])
                share = sum(cost[sh.b0:sh.b1])
                assert share <= total / world + max(cost) + 1e-9
    with pytest.raises(ValueError):
        S.segment_range([0, 5, 3], [0, 1, 2], 2, 0)


def test_empty_shards_are_reported():
    """More ranks than heads or segments, or one segment dominating the
    cost, leave some ranks without work: the ranges say so (h0 == h1,
    SegmentShard.empty) and the non-empty shards still cover everything."""
    ranges = [S.head_range(3, 5, r) for r in range(5)]
    assert [h1 - h0 for h0, h1 in ranges] == [1, 1, 1, 0, 0]
    assert ranges[-1][0] == ranges[-1][1] == 3
    cu_q, cu_k = [0, 7, 9], [0, 7, 9]
    shards = [S.segment_range(cu_q, cu_k, 4, r) for r in range(4)]
    assert sum(not sh.empty for sh in shards) <= 2
    assert [b for sh in shards if not sh.empty for b in range(sh.b0, sh.b1)] == [0, 1]
    for sh in shards:
        if sh.empty:
            assert sh.q0 == sh.q1 and sh.k0 == sh.k1 and len(sh.cu_q) == 1
    # one dominant segment: the ranks between the boundaries it spans get nothing
    dom = S.segment_range([0, 1, 10001, 10002], [0, 1, 10001, 10002], 3, 1)
    assert dom.b1 - dom.b0 <= 1
    shards = [S.segment_range([0, 1, 10001, 10002], [0, 1, 10001, 10002], 3, r) for r in range(3)]
    assert any(sh.empty for sh in shards)
    assert sorted(b for sh in shards for b in range(sh.b0, sh.b1)) == [0, 1, 2]


def test_max_over_ranks_without_group():
    assert S.max_over_ranks(3.5) == 3.5


# ---------------------------------------------------------------- two ranks

_CASE = ([130, 0, 77, 256, 5, 64], [129, 9, 0, 300, 40, 64], 4, 64)


def _shard_result(w, cpu, mode, world, rank, window=(-1, -1)):
    """The oracle forward and backward of this rank's shard, keyed by global
    (row, head) pairs.  Masks are per segment, so they shard unchanged."""
    if mode == "heads":
        h0, h1 = S.head_range(w.num_heads, world, rank)
        view = lambda t: t[:, h0:h1]
        pb = oracle.Problem(view(cpu.q), view(cpu.k), view(cpu.v), w.cu_q, w.cu_k, w.softmax_scale,
                            dout=view(cpu.dout), window=window)
        rows, heads = oracle.all_pairs(w.total_q, h1 - h0)
        krows, kheads = oracle.all_pairs(w.total_k, h1 - h0)
        grows, gheads, gkrows, gkheads = rows, heads + h0, krows, kheads + h0
    else:
        sh = S.segment_range(w.cu_q, w.cu_k, world, rank)
        pb = oracle.Problem(cpu.q[sh.q0:sh.q1], cpu.k[sh.k0:sh.k1], cpu.v[sh.k0:sh.k1], sh.cu_q, sh.cu_k,
                            w.softmax_scale, dout=cpu.dout[sh.q0:sh.q1], window=window)
        rows, heads = oracle.all_pairs(sh.q1 - sh.q0, w.num_heads)
        krows, kheads = oracle.all_pairs(sh.k1 - sh.k0, w.num_heads)
        grows, gheads, gkrows, gkheads = rows + sh.q0, heads, krows + sh.k0, kheads
    o, lse = pb.fwd(rows, heads)
    dq, _ = pb.bwd_q(rows, heads)
    dk, dv = pb.bwd_kv(krows, kheads)
    return grows, gheads, o, lse, dq, gkrows, gkheads, dk, dv


def _worker(rank, world, port, mode, out_path, window=(-1, -1)):
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method="tcp://127.0.0.1:%d" % port)
    try:
        w = W.custom("shard", *_CASE[:2], _CASE[2], _CASE[3])
        cpu = W.make_inputs(w, 0)
        res = _shard_result(w, cpu, mode, world, rank, window)
        gathered = [None] * world
        dist.all_gather_object(gathered, res)  # only to bring the shards to one process for checking
        t_max = S.max_over_ranks(float(rank + 1))
        if rank == 0:
            cat = [np.concatenate([g[i] for g in gathered]) for i in range(9)]
            np.savez(out_path, *cat, t_max=np.float64(t_max))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("mode,window", [("heads", (-1, -1)), ("segments", (-1, -1)), ("heads", (-1, 0)),
                                         ("segments", (40, 3))])
def test_two_rank_shards_match_unsharded(mode, window):
    oracle.build()
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    world = 2
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "res.npz")
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, world, port, mode, out, window)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=240)
        for p in procs:
            if p.is_alive():
                p.kill()
                p.join()
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        z = np.load(out)
        rows, heads, o, lse, dq, krows, kheads, dk, dv = (z["arr_%d" % i] for i in range(9))
        assert float(z["t_max"]) == float(world)  # max over ranks of (rank + 1)

    w = W.custom("shard", *_CASE[:2], _CASE[2], _CASE[3])
    cpu = W.make_inputs(w, 0)
    full = oracle.Problem(cpu.q, cpu.k, cpu.v, w.cu_q, w.cu_k, w.softmax_scale, dout=cpu.dout, window=window)
    # every (row, head) pair computed exactly once across the ranks
    assert sorted(zip(rows.tolist(), heads.tolist())) == sorted(zip(*[a.tolist() for a in oracle.all_pairs(w.total_q, w.num_heads)]))
    assert sorted(zip(krows.tolist(), kheads.tolist())) == sorted(zip(*[a.tolist() for a in oracle.all_pairs(w.total_k, w.num_heads)]))
    o_ref, lse_ref = full.fwd(rows, heads)
    dq_ref, _ = full.bwd_q(rows, heads)
    dk_ref, dv_ref = full.bwd_kv(krows, kheads)
    # identical fp64 arithmetic per pair: the shards reproduce the full result bit for bit
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(lse, lse_ref)
    np.testing.assert_array_equal(dq, dq_ref)
    np.testing.assert_array_equal(dk, dk_ref)
    np.testing.assert_array_equal(dv, dv_ref)


# ---------------------------------------------------------------- two ranks, E4M3 forward

def _fp8_shard_result(w, cpu, mode, world, rank, causal=False):
    """The oracle's E4M3 forward of this rank's shard, keyed by global (row,
    head) pairs.  The rank quantises its own (segment, head) blocks: their
    descales depend on nothing outside the block, so a shard's codes are the
    unsharded codes of its blocks."""
    if mode == "heads":
        h0, h1 = S.head_range(w.num_heads, world, rank)
        q, k, v = (t[:, h0:h1] for t in (cpu.q, cpu.k, cpu.v))
        cu_q, cu_k = list(w.cu_q), list(w.cu_k)
        rows, heads = oracle.all_pairs(w.total_q, h1 - h0)
        grows, gheads = rows, heads + h0
    else:
        sh = S.segment_range(w.cu_q, w.cu_k, world, rank)
        q, k, v = cpu.q[sh.q0:sh.q1], cpu.k[sh.k0:sh.k1], cpu.v[sh.k0:sh.k1]
        cu_q, cu_k = sh.cu_q, sh.cu_k
        rows, heads = oracle.all_pairs(sh.q1 - sh.q0, w.num_heads)
        grows, gheads = rows + sh.q0, heads
    quant = [oracle.quantize_e4m3(x, cu) for x, cu in ((q, cu_q), (k, cu_k), (v, cu_k))]
    codes, desc = [c for c, _ in quant], [d for _, d in quant]
    o, lse = oracle.Fp8Problem(*codes, cu_q, cu_k, w.softmax_scale, *desc, causal=causal).fwd(rows, heads)
    return grows, gheads, o, lse


def _fp8_worker(rank, world, port, mode, out_path, causal):
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method="tcp://127.0.0.1:%d" % port)
    try:
        w = W.custom("shard", *_CASE[:2], _CASE[2], _CASE[3])
        cpu = W.make_inputs(w, 0, with_dout=False)
        res = _fp8_shard_result(w, cpu, mode, world, rank, causal)
        gathered = [None] * world
        dist.all_gather_object(gathered, res)  # only to bring the shards to one process for checking
        if rank == 0:
            np.savez(out_path, *[np.concatenate([g[i] for g in gathered]) for i in range(4)])
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode,causal", [("heads", False), ("segments", False), ("heads", True),
                                         ("segments", True)])
def test_two_rank_fp8_shards_match_unsharded(mode, causal):
    """Two gloo ranks each quantise and run their shard of the E4M3 forward
    (the oracle's reading); together they reproduce the unsharded
    quantisation and forward bit for bit, with no exchange of data."""
    oracle.build()
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    world = 2
    with tempfile.TemporaryDirectory() as d:
        out = os.path.join(d, "res.npz")
        port = _free_port()
        procs = [ctx.Process(target=_fp8_worker, args=(r, world, port, mode, out, causal)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=240)
        for p in procs:
            if p.is_alive():
                p.kill()
                p.join()
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        z = np.load(out)
        rows, heads, o, lse = (z["arr_%d" % i] for i in range(4))

    w = W.custom("shard", *_CASE[:2], _CASE[2], _CASE[3])
    cpu = W.make_inputs(w, 0, with_dout=False)
    quant = [oracle.quantize_e4m3(x, cu) for x, cu in ((cpu.q, w.cu_q), (cpu.k, w.cu_k), (cpu.v, w.cu_k))]
    full = oracle.Fp8Problem(*[c for c, _ in quant], list(w.cu_q), list(w.cu_k), w.softmax_scale,
                             *[d for _, d in quant], causal=causal)
    assert sorted(zip(rows.tolist(), heads.tolist())) == sorted(zip(*[a.tolist() for a in oracle.all_pairs(w.total_q, w.num_heads)]))
    o_ref, lse_ref = full.fwd(rows, heads)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(lse, lse_ref)
