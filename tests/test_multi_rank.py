"""The multi-process host logic on CPU (gloo, world size 2): layer shards,
the barrier and the maximum of the ranks' times around the timed region, and
CommitKV Eq. 4's shared index set when a sequence's layers are split across
ranks (each rank sums its own units' scores, one all-reduce adds the partial
sums, every rank then selects the same index set)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle as o
from budgeted_kv_cache_gb300.sharding import all_reduce_shared, barrier, layer_shard, max_over_ranks

B, L, HKV, T, BUDGET = 2, 5, 3, 257, 40


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _scores():
    # every rank draws the same unit scores [B][L][H_kv][T] and keeps its layers
    return np.random.default_rng(7).random((B, L, HKV, T)).astype(np.float32)


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        scores = _scores()
        l0, l1 = layer_shard(L, world, rank)
        # this rank's partial per-sequence sums, fp32 like kvc_shared_scores
        partial = torch.from_numpy(scores[:, l0:l1].reshape(B, -1, T).sum(axis=1, dtype=np.float32))
        shared = all_reduce_shared(partial, world).numpy()
        kept = [o.select_tokens(shared[b], T, BUDGET, 4, 8)[0] for b in range(B)]
        t = max_over_ranks(1.5 + rank, world)
        barrier(world)
        results[rank] = (shared, kept, t, (l0, l1))
    finally:
        dist.destroy_process_group()


def test_layer_shards_partition_the_layers():
    for n_layers in (1, 5, 36):
        for world in (1, 2, 3, 8):
            ranges = [layer_shard(n_layers, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n_layers
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            sizes = [b - a for a, b in ranges]
            assert max(sizes) - min(sizes) <= 1


def test_two_ranks_share_one_index_set_and_the_slowest_time():
    world = 2
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    scores = _scores()
    full = np.stack([o.shared_scores(scores[b].reshape(-1, T)) for b in range(B)])
    ref_kept = [o.select_tokens(full[b], T, BUDGET, 4, 8)[0] for b in range(B)]
    assert res[0][3] == (0, 3) and res[1][3] == (3, 5)
    for rank in range(world):
        shared, kept, t, _ = res[rank]
        np.testing.assert_allclose(shared, full, rtol=1e-6)         # fp32 partial sums
        for b in range(B):
            np.testing.assert_array_equal(kept[b], ref_kept[b])
        assert t == 2.5                                             # the slower rank's time
    np.testing.assert_array_equal(res[0][0], res[1][0])             # one index set everywhere
