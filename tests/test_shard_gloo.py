"""Multi-rank host logic on CPU with the gloo backend (world size 2).

The path shards over (batch, head) units with no exchange: each rank's slice,
computed alone, must equal the matching slice of the whole computation.  The
float64 oracle stands in for the per-rank compute here (no GPU), so what is
tested is the partition, the per-rank seeds, the max-over-ranks timing
reduction and the all-gather that reassembles O and LSE.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from transformer_head_scaled_gb300 import inputs, shard


def test_shard_range_partitions():
    for B in (0, 1, 5, 64, 65):
        for world in (1, 2, 3, 8):
            spans = [shard.shard_range(B, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard.shard_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        global_B = 5
        w = inputs.Workload("g", global_B, 2, 33, 40, 16, inputs.MASK_KEY_PADDING, "bf16")
        q, k, v, lens = inputs.make_inputs(w)          # same global inputs on every rank
        a, b = shard.shard_range(global_B, world, rank)
        o, lse = oracle.attn_fwd(q[a:b], k[a:b], v[a:b], w.scale, w.mask, lens[a:b])
        o_all = shard.gather_batch(torch.from_numpy(o), global_B)
        l_all = shard.gather_batch(torch.from_numpy(lse), global_B)
        t = shard.max_over_ranks(1.0 + rank)
        np.save(os.path.join(result_dir, f"o{rank}.npy"), o_all.numpy())
        np.save(os.path.join(result_dir, f"l{rank}.npy"), l_all.numpy())
        np.save(os.path.join(result_dir, f"t{rank}.npy"), np.array([t]))
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_reassemble_without_exchange(tmp_path, oracle_mod):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    w = inputs.Workload("g", 5, 2, 33, 40, 16, inputs.MASK_KEY_PADDING, "bf16")
    q, k, v, lens = inputs.make_inputs(w)
    o_ref, l_ref = oracle_mod.attn_fwd(q, k, v, w.scale, w.mask, lens)
    for r in range(world):
        np.testing.assert_array_equal(np.load(tmp_path / f"o{r}.npy"), o_ref)
        np.testing.assert_array_equal(np.load(tmp_path / f"l{r}.npy"), l_ref)
        assert np.load(tmp_path / f"t{r}.npy")[0] == 2.0   # max over ranks of 1 + rank


def test_rank_seeds_distinct():
    assert shard.rank_seeds(0) == (0, 1, 2, 3)
    assert len({shard.rank_seeds(r) for r in range(8)}) == 8
