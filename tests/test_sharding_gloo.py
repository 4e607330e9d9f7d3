"""Sequence sharding across ranks (no exchange step inside the op), run as two gloo
ranks on CPU: each rank computes its shard with the oracle, an all-gather reassembles
the full outputs, which must equal the unsharded result exactly."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.jfa_oracle as orc
from jagged_attention_recsys_jfa_gb300.inputs import JaggedConfig, make_batch
from jagged_attention_recsys_jfa_gb300.sharding import (scatter_bias_blocks, scatter_sequences, select_bias_blocks,
                                                        select_sequences, shard_sequences, visited_pairs)


def test_visited_pairs_matches_mask_count():
    for lq in range(0, 9):
        for lk in range(0, 9):
            for causal in (False, True):
                n = int(orc.causal_visible(lq, lk).sum()) if causal else lq * lk
                assert visited_pairs(lq, lk, causal) == n


def test_shards_cover_every_sequence_once_and_balance():
    g = torch.Generator().manual_seed(3)
    lq = torch.randint(1, 2000, (97,), generator=g).tolist()
    for world in (1, 2, 3, 8):
        shards = shard_sequences(lq, lq, world, causal=True)
        assert sorted(i for s in shards for i in s) == list(range(97))
        loads = [sum(visited_pairs(lq[i], lq[i], True) for i in s) for s in shards]
        assert max(loads) - min(loads) <= max(visited_pairs(x, x, True) for x in lq)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


CFG = JaggedConfig("shard", 7, 2, 8, ("uniform", 1, 40), kv_lengths=("uniform", 1, 50), causal=True,
                   bias_buckets=64, bias_center=32)


def _worker(rank, world, port, result):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = make_batch(CFG)
        shards = shard_sequences(b.q_lengths.tolist(), b.kv_lengths.tolist(), world, CFG.causal)
        mine = shards[rank]
        q, qo = select_sequences(b.q, b.q_offsets, mine)
        k, ko = select_sequences(b.k, b.kv_offsets, mine)
        v, _ = select_sequences(b.v, b.kv_offsets, mine)
        out, lse = orc.jagged_forward(q, k, v, qo, ko, CFG.scale, CFG.causal, b.bias, CFG.bias_center)
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine, out, lse, qo))
        if rank == 0:
            full_out = torch.zeros(b.q.shape, dtype=torch.float64)
            full_lse = torch.zeros((CFG.heads, b.q.shape[0]), dtype=torch.float64)
            for idx, o, l, off in gathered:
                scatter_sequences(full_out, b.q_offsets, idx, torch.from_numpy(o), off)
                scatter_sequences(full_lse.T, b.q_offsets, idx, torch.from_numpy(l).T, off)
            ref_out, ref_lse = orc.jagged_forward(b.q, b.k, b.v, b.q_offsets, b.kv_offsets, CFG.scale, CFG.causal,
                                                  b.bias, CFG.bias_center)
            result["out_equal"] = bool(np.array_equal(full_out.numpy(), ref_out))
            result["lse_equal"] = bool(np.array_equal(full_lse.numpy(), ref_lse))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_sharding_reassembles_exactly():
    mgr = mp.get_context("spawn").Manager()  # no fork of this (threaded) process
    result = mgr.dict()
    mp.spawn(_worker, args=(2, _free_port(), result), nprocs=2, join=True)
    assert result.get("out_equal") and result.get("lse_equal"), dict(result)


CFG_JB = JaggedConfig("shard_jb", 6, 2, 8, ("uniform", 1, 30), kv_lengths=("uniform", 1, 40), causal=True,
                      general_bias=True)


def _worker_bias(rank, world, port, result):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # general jagged bias: the shard's blocks travel with its sequences
        b = make_batch(CFG_JB)
        shards = shard_sequences(b.q_lengths.tolist(), b.kv_lengths.tolist(), world, CFG_JB.causal)
        mine = shards[rank]
        q, qo = select_sequences(b.q, b.q_offsets, mine)
        k, ko = select_sequences(b.k, b.kv_offsets, mine)
        v, _ = select_sequences(b.v, b.kv_offsets, mine)
        jv, jo = select_bias_blocks(b.jbias, b.jbias_offsets, mine)
        out, _ = orc.jagged_forward(q, k, v, qo, ko, CFG_JB.scale, CFG_JB.causal, jagged_bias=(jv, jo))
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine, out, qo))
        # relative-position table gradient: partial sums per rank, one all-reduce
        c = make_batch(CFG)
        cs = shard_sequences(c.q_lengths.tolist(), c.kv_lengths.tolist(), world, CFG.causal)[rank]
        cq, cqo = select_sequences(c.q, c.q_offsets, cs)
        ck, cko = select_sequences(c.k, c.kv_offsets, cs)
        cv, _ = select_sequences(c.v, c.kv_offsets, cs)
        cdo, _ = select_sequences(c.dout, c.q_offsets, cs)
        g = torch.from_numpy(orc.jagged_bias_grad(cdo, cq, ck, cv, cqo, cko, CFG.scale, CFG.causal, c.bias,
                                                  CFG.bias_center))
        dist.all_reduce(g, op=dist.ReduceOp.SUM)
        if rank == 0:
            full_out = torch.zeros(b.q.shape, dtype=torch.float64)
            for idx, o, off in gathered:
                scatter_sequences(full_out, b.q_offsets, idx, torch.from_numpy(o), off)
            ref_out, _ = orc.jagged_forward(b.q, b.k, b.v, b.q_offsets, b.kv_offsets, CFG_JB.scale, CFG_JB.causal,
                                            jagged_bias=(b.jbias, b.jbias_offsets))
            result["jb_out_equal"] = bool(np.array_equal(full_out.numpy(), ref_out))
            ref_g = orc.jagged_bias_grad(c.dout, c.q, c.k, c.v, c.q_offsets, c.kv_offsets, CFG.scale, CFG.causal,
                                         c.bias, CFG.bias_center)
            result["dbias_err"] = float(np.abs(g.numpy() - ref_g).max() / max(np.abs(ref_g).max(), 1e-30))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_biases_shard():
    """A general bias sharded with its sequences reassembles the unsharded output exactly;
    the relative-position table's gradient, summed over the ranks by one all-reduce, equals
    the unsharded gradient up to the order of the float64 additions."""
    mgr = mp.get_context("spawn").Manager()  # no fork of this (threaded) process
    result = mgr.dict()
    mp.spawn(_worker_bias, args=(2, _free_port(), result), nprocs=2, join=True)
    assert result.get("jb_out_equal"), dict(result)
    assert result.get("dbias_err", 1.0) <= 1e-12, dict(result)


CFG_BWD = JaggedConfig("shard_bwd", 9, 2, 8, ("uniform", 0, 30), kv_lengths=("uniform", 0, 40), causal=True,
                       general_bias=True)


def _worker_backward(rank, world, port, result):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # the backward of a sharded batch: each rank differentiates its own sequences (dq
        # by query rows, dk / dv by key rows, the general bias's gradient by blocks); an
        # all-gather puts the gradients back together with no other exchange
        b = make_batch(CFG_BWD)
        mine = shard_sequences(b.q_lengths.tolist(), b.kv_lengths.tolist(), world, CFG_BWD.causal)[rank]
        q, qo = select_sequences(b.q, b.q_offsets, mine)
        do, _ = select_sequences(b.dout, b.q_offsets, mine)
        k, ko = select_sequences(b.k, b.kv_offsets, mine)
        v, _ = select_sequences(b.v, b.kv_offsets, mine)
        jv, jo = select_bias_blocks(b.jbias, b.jbias_offsets, mine)
        kw = dict(scale=CFG_BWD.scale, causal=CFG_BWD.causal, jagged_bias=(jv, jo))
        dq, dk, dv = orc.jagged_backward(do, q, k, v, qo, ko, **kw)
        dj = orc.jagged_general_bias_grad(do, q, k, v, qo, ko, CFG_BWD.scale, CFG_BWD.causal, (jv, jo))
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine, dq, dk, dv, dj, qo, ko, jo))
        if rank == 0:
            full = {n: torch.zeros(t.shape, dtype=torch.float64) for n, t in (("dq", b.q), ("dk", b.k), ("dv", b.v))}
            full_dj = torch.zeros(b.jbias.shape, dtype=torch.float64)
            for idx, gq, gk, gv, gj, off_q, off_k, off_j in gathered:
                scatter_sequences(full["dq"], b.q_offsets, idx, torch.from_numpy(gq), off_q)
                scatter_sequences(full["dk"], b.kv_offsets, idx, torch.from_numpy(gk), off_k)
                scatter_sequences(full["dv"], b.kv_offsets, idx, torch.from_numpy(gv), off_k)
                scatter_bias_blocks(full_dj, b.jbias_offsets, idx, torch.from_numpy(gj), off_j)
            jb = (b.jbias, b.jbias_offsets)
            ref = orc.jagged_backward(b.dout, b.q, b.k, b.v, b.q_offsets, b.kv_offsets, CFG_BWD.scale, CFG_BWD.causal,
                                      jagged_bias=jb)
            ref_dj = orc.jagged_general_bias_grad(b.dout, b.q, b.k, b.v, b.q_offsets, b.kv_offsets, CFG_BWD.scale,
                                                  CFG_BWD.causal, jb)
            for n, r in zip(("dq", "dk", "dv"), ref):
                result[n + "_equal"] = bool(np.array_equal(full[n].numpy(), r))
            result["dj_equal"] = bool(np.array_equal(full_dj.numpy(), ref_dj))
            result["shards"] = [len(g[0]) for g in gathered]
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_sharded_backward_reassembles_exactly():
    """dq, dk, dv and the general bias's gradient of a batch sharded over two gloo ranks
    (empty sequences included), gathered and scattered back, equal the unsharded backward
    bit for bit: the backward has no exchange step either."""
    mgr = mp.get_context("spawn").Manager()  # no fork of this (threaded) process
    result = mgr.dict()
    mp.spawn(_worker_backward, args=(2, _free_port(), result), nprocs=2, join=True)
    res = dict(result)
    assert all(res.get(n) for n in ("dq_equal", "dk_equal", "dv_equal", "dj_equal")), res
    assert all(n > 0 for n in res["shards"]), res
