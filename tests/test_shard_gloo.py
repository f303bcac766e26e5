"""Multi-GPU sharding of a decode batch, exercised on CPU with gloo ranks.

Decode attention of different sequences is independent, so a batch is split
by sequence across ranks with no exchange on the data path.  Two gloo ranks
each compute their shard (here with the CPU oracle, as no GPU is assumed);
the shards, gathered only to check them, must equal the single-process
result bit for bit.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import pkv_workloads as W


def test_shards_cover_the_batch_disjointly_and_evenly():
    for n in (0, 1, 7, 64, 257):
        for ws in (1, 2, 3, 8):
            ranges = [W.shard_sequences(n, r, ws) for r in range(ws)]
            seqs = [s for r in ranges for s in r]
            assert seqs == list(range(n))
            sizes = [len(r) for r in ranges]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        W.shard_sequences(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_path):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.make("c1_tiny")
    mine = W.shard_sequences(w.num_seqs, rank, world)
    sl = slice(mine.start, mine.stop)
    out = oracle.decode_fp16(w.query[sl], w.k_pool, w.v_pool, w.block_tables[sl],
                             w.context_lens[sl], num_kv_heads=w.num_kv_heads,
                             softmax_scale=w.softmax_scale, num_threads=1)
    part = torch.from_numpy(out).reshape(-1, w.num_heads * w.head_dim)
    sizes = [len(W.shard_sequences(w.num_seqs, r, world)) for r in range(world)]
    assert len(set(sizes)) == 1  # all_gather wants equal shards
    gathered = [torch.zeros((sz, w.num_heads * w.head_dim), dtype=torch.float64) for sz in sizes]
    dist.all_gather(gathered, part)
    if rank == 0:
        np.save(result_path, torch.cat(gathered).numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_single_process_batch(tmp_path):
    import oracle
    w = W.make("c1_tiny")
    full = oracle.decode_fp16(w.query, w.k_pool, w.v_pool, w.block_tables, w.context_lens,
                              num_kv_heads=w.num_kv_heads, softmax_scale=w.softmax_scale,
                              num_threads=1)
    path = str(tmp_path / "gathered.npy")
    mp.start_processes(_rank_main, args=(2, _free_port(), path), nprocs=2, join=True,
                       start_method="spawn")
    got = np.load(path).reshape(full.shape)
    assert np.array_equal(got, full)
