"""The vocabulary-parallel tail's host side on CPU: slice boundaries, row
ownership blocks, and the candidate exchanges (all-gather; all-to-all of
owned rows) between gloo ranks, each holding one vocabulary slice.

Each rank's candidates come from the fp64 oracle on its own slice (the GPU
kernels need a GPU); after the exchange, the top k of the union by
(value desc, global id asc) must be the oracle's top k of the whole row.
"""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from decode_sampling_tail_gb300.vocab_parallel import shard_bounds, gather_candidates  # noqa: E402


@pytest.mark.parametrize("V,n", [(201088, 8), (4096, 3), (160, 10), (2048, 1)])
def test_shard_bounds_cover_the_vocabulary_in_even_pair_aligned_slices(V, n):
    b = shard_bounds(V, n)
    assert b[0] == 0 and b[-1] == V and len(b) == n + 1
    w = np.diff(b)
    assert np.all(w > 0) and np.all(np.asarray(b) % 16 == 0)
    assert w.max() - w.min() <= 16


def test_shard_bounds_reject_impossible_splits():
    with pytest.raises(ValueError):
        shard_bounds(100, 2)  # not whole pairs
    with pytest.raises(ValueError):
        shard_bounds(32, 3)   # fewer pairs than slices


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import gen
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = gen.custom(3, 64, 2048, 40, hidden_dtype="bf16", seed=71, dup_cols=2)  # ties across the slices
        b = shard_bounds(w.V, world)
        lo, hi = b[rank], b[rank + 1]
        logits = oracle.logits(w.hidden, w.hidden_dtype, w.gamma, np.ascontiguousarray(w.w_t[:, lo:hi]), w.Hu, w.eps,
                               w.zero_pad)
        vals, ids = oracle.topk(logits, w.k)          # slice-local ids
        v_all, i_all = gather_candidates(torch.from_numpy(vals.astype(np.float32)),
                                         torch.from_numpy(ids.astype(np.int32)))
        out[rank] = (v_all.numpy(), i_all.numpy(), b)
    finally:
        dist.destroy_process_group()


def test_two_ranks_exchange_candidates_and_the_union_gives_the_global_topk():
    import gen
    import oracle
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
    v_all, i_all, b = res[0]
    w = gen.custom(3, 64, 2048, 40, hidden_dtype="bf16", seed=71, dup_cols=2)
    full = oracle.logits(w.hidden, w.hidden_dtype, w.gamma, w.w_t, w.Hu, w.eps, w.zero_pad)
    ov, oi = oracle.topk(full, w.k)
    for r in range(w.B):
        gid = np.concatenate([i_all[s, r] + b[s] for s in range(2)])
        val = np.concatenate([v_all[s, r] for s in range(2)]).astype(np.float64)
        order = np.lexsort((gid, -val))[: w.k]
        assert np.array_equal(gid[order], oi[r])


@pytest.mark.parametrize("vtp,gbs", [(4, 8), (3, 3), (1, 5)])
def test_owned_row_blocks_partition_the_batch(vtp, gbs):
    from decode_sampling_tail_gb300.vocab_parallel import owned_row_block
    blocks = [owned_row_block(r, vtp, gbs) for r in range(vtp)]
    assert blocks[0][0] == 0 and all(n == gbs // vtp for _, n in blocks)
    assert all(blocks[r][0] + blocks[r][1] == blocks[r + 1][0] for r in range(vtp - 1))
    assert blocks[-1][0] + blocks[-1][1] == gbs


def test_owned_row_block_rejects_uneven_batches():
    from decode_sampling_tail_gb300.vocab_parallel import owned_row_block
    with pytest.raises(ValueError):
        owned_row_block(0, 3, 8)
    with pytest.raises(ValueError):
        owned_row_block(2, 2, 8)


def _rank_owned(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import gen
    import oracle
    from decode_sampling_tail_gb300.vocab_parallel import exchange_candidates
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = gen.custom(6, 64, 2400, 24, hidden_dtype="bf16", seed=72, dup_cols=2)
        b = shard_bounds(w.V, world)
        lo, hi = b[rank], b[rank + 1]
        logits = oracle.logits(w.hidden, w.hidden_dtype, w.gamma, np.ascontiguousarray(w.w_t[:, lo:hi]), w.Hu, w.eps,
                               w.zero_pad)
        vals, ids = oracle.topk(logits, w.k)
        v_own, i_own = exchange_candidates(torch.from_numpy(vals.astype(np.float32)),
                                           torch.from_numpy(ids.astype(np.int32)))
        out[rank] = (v_own.numpy(), i_own.numpy(), b)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_all_to_all_hands_each_rank_its_rows_and_their_union_gives_the_global_topk(world):
    import gen
    import oracle
    from decode_sampling_tail_gb300.vocab_parallel import owned_row_block
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_owned, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    w = gen.custom(6, 64, 2400, 24, hidden_dtype="bf16", seed=72, dup_cols=2)
    full = oracle.logits(w.hidden, w.hidden_dtype, w.gamma, w.w_t, w.Hu, w.eps, w.zero_pad)
    ov, oi = oracle.topk(full, w.k)
    for q in range(world):
        v_own, i_own, b = res[q]
        r0, n = owned_row_block(q, world, w.B)
        assert v_own.shape == (world, n, w.k)
        for j in range(n):
            gid = np.concatenate([i_own[s, j] + b[s] for s in range(world)])
            val = np.concatenate([v_own[s, j] for s in range(world)]).astype(np.float64)
            order = np.lexsort((gid, -val))[: w.k]
            assert np.array_equal(gid[order], oi[r0 + j])
