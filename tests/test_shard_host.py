"""Host side of the query-sharded indexer ("Scaling Training to 1M Token
Context on GLM-5.3-Flash", section "Across GPUs: Sharding"): each rank
selects for its own contiguous block of queries against all earlier pools,
then the int32 selections are gathered.  The split itself is tested here,
and the whole scheme on two gloo ranks on the CPU, with the oracle standing
in for each rank's GPU call (one GPU per box here)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import long_context_sparse_gb300 as dsa
import oracle
from long_context_sparse_gb300 import synth
from tests.helpers import bits


@pytest.mark.parametrize("S", [1, 4, 7, 4096, 6001, 131072])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_query_shard_partitions_the_sequence(S, world):
    spans = [dsa.query_shard(S, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == S
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0                      # contiguous, in rank order
    for a0, a1 in spans:
        assert 0 <= a0 <= a1 <= S
        assert a0 % 4 == 0 or a0 == S        # starts on a pool boundary
    sizes = [a1 - a0 for a0, a1 in spans]
    assert max(sizes) - min(sizes) <= 7      # one pool plus the ragged tail


def test_query_shard_rejects_bad_rank():
    with pytest.raises(ValueError):
        dsa.query_shard(100, 2, 2)
    with pytest.raises(ValueError):
        dsa.query_shard(100, 0, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, S, K_p, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.scaled(synth.WORKLOADS["tiny_fwd_s1k"], S, K_p=K_p)
        q_idx, k_idx, w = synth.indexer_inputs(wl, 5, "cpu")
        t0, t1 = dsa.query_shard(S, world, rank)
        rows = np.arange(t0, t1, dtype=np.int64)
        mine, _ = oracle.index_topk(bits(q_idx), bits(k_idx), w.numpy(), K_p, rows)
        # gather variable-length int32 blocks: pad to the longest shard
        n_max = max(b - a for a, b in (dsa.query_shard(S, world, r)
                                       for r in range(world)))
        buf = torch.full((n_max, K_p), -2, dtype=torch.int32)
        buf[: t1 - t0] = torch.from_numpy(mine)
        parts = [torch.empty_like(buf) for _ in range(world)]
        dist.all_gather(parts, buf)
        if rank == 0:
            full = torch.cat([p[: b - a] for p, (a, b) in zip(
                parts, (dsa.query_shard(S, world, r) for r in range(world)))])
            np.save(out_path, full.numpy())
    finally:
        dist.destroy_process_group()


def test_sharded_selection_on_two_gloo_ranks_equals_unsharded(tmp_path):
    S, K_p, world = 301, 16, 2
    out = str(tmp_path / "gathered.npy")
    mp.spawn(_rank_main, args=(world, _free_port(), S, K_p, out), nprocs=world,
             join=True)
    gathered = np.load(out)
    wl = synth.scaled(synth.WORKLOADS["tiny_fwd_s1k"], S, K_p=K_p)
    q_idx, k_idx, w = synth.indexer_inputs(wl, 5, "cpu")
    ref, _ = oracle.index_topk(bits(q_idx), bits(k_idx), w.numpy(), K_p)
    np.testing.assert_array_equal(gathered, ref)


def _attn_rank_main(rank, world, port, S, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.scaled(synth.WORKLOADS["tiny_fwd_s1k"], S, K_p=8, n_loc=3)
        q, k, v, dO = synth.attention_inputs(wl, 7, "cpu")
        idx = synth.random_selection(wl, 7, "cpu").numpy()
        scale = 1.0 / np.sqrt(wl.d_qk)
        t0, t1 = dsa.query_shard(S, world, rank)
        rows = np.arange(t0, t1, dtype=np.int64)
        # this rank's queries: dq rows, and partial dK/dV over every key
        dq, dk, dv = oracle.attn_bwd(bits(q)[rows], bits(k), bits(v), bits(dO)[rows],
                                     idx, wl.K_p, wl.n_loc, scale, rows)
        part = torch.from_numpy(np.concatenate([dk, dv], axis=1))
        dist.all_reduce(part)                 # the exchange: a sum over ranks
        n_max = max(b - a for a, b in (dsa.query_shard(S, world, r)
                                       for r in range(world)))
        buf = torch.zeros((n_max,) + dq.shape[1:], dtype=torch.float64)
        buf[: t1 - t0] = torch.from_numpy(dq)
        parts = [torch.empty_like(buf) for _ in range(world)]
        dist.all_gather(parts, buf)
        if rank == 0:
            full_dq = torch.cat([p[: b - a] for p, (a, b) in zip(
                parts, (dsa.query_shard(S, world, r) for r in range(world)))])
            np.savez(out_path, dq=full_dq.numpy(), dkv=part.numpy())
    finally:
        dist.destroy_process_group()


def test_query_sharded_attention_backward_on_two_gloo_ranks(tmp_path):
    """Attention backward split by query (the form of
    dsa_sparse_attn_bwd_range): per-rank dq rows gathered and per-rank
    partial dK/dV summed over ranks equal the unsharded backward."""
    S, world = 203, 2
    out = str(tmp_path / "bwd.npz")
    mp.spawn(_attn_rank_main, args=(world, _free_port(), S, out), nprocs=world,
             join=True)
    got = np.load(out)
    wl = synth.scaled(synth.WORKLOADS["tiny_fwd_s1k"], S, K_p=8, n_loc=3)
    q, k, v, dO = synth.attention_inputs(wl, 7, "cpu")
    idx = synth.random_selection(wl, 7, "cpu").numpy()
    dq, dk, dv = oracle.attn_bwd(bits(q), bits(k), bits(v), bits(dO), idx, wl.K_p,
                                 wl.n_loc, 1.0 / np.sqrt(wl.d_qk))
    np.testing.assert_array_equal(got["dq"], dq)      # row-local: exact
    ref = np.concatenate([dk, dv], axis=1)
    assert np.allclose(got["dkv"], ref, rtol=1e-12, atol=1e-14 * np.abs(ref).max())
