"""Vocabulary-parallel decode tail: N ranks, each holding a contiguous slice of
the vocabulary ("GPT-OSS Tail Chunked Megakernel Kernel API Reference",
section "Background" and parameter `replica_groups`: the lm_head's V split over
ranks, a per-rank top-k, one exchange, one global top-k).

Per step, every rank
  1. runs the whole tail on its slice (`Tail.run` with its [H, V_s] weight
     columns and no sampler) and keeps its sorted top-k: k values and
     slice-local ids per row;
  2. all-gathers those candidates over the group (gbs * k * 8 bytes per rank,
     the only collective);
  3. merges them with `merge_shards` (top-k of the union by value, then global
     id) and draws the token -- every rank the same token, so the sampler is
     replicated rather than owned.

Row ownership (the page's `owned_row_block`, single hop): instead of the
all-gather, an all-to-all sends every rank only the candidates of the rows it
owns, a contiguous block of gbs / N rows; each rank merges and samples those
rows alone, with `sampling_params` holding only its own rows.  The exchange
then moves gbs * k * 8 bytes per rank in total rather than N times that.

On one GPU the same functions run the slices one after another ("simulated
shards"); the result equals the unsharded tail bit for bit, because the
lm_head's arithmetic for a column does not depend on how the vocabulary is
split.
"""
from __future__ import annotations

from . import Tail, merge_shards

COL_ALIGN = 16  # slice boundaries on 16-column pairs (the kernels' V granularity)


def shard_bounds(V: int, nshard: int) -> list[int]:
    """Boundaries b_0 = 0 < b_1 < ... < b_n = V of n contiguous slices, multiples of 16 columns,
    as even as that allows (widths differ by at most 16)."""
    if V % COL_ALIGN or nshard < 1 or V // COL_ALIGN < nshard:
        raise ValueError(f"cannot split V={V} into {nshard} slices of whole 16-column pairs")
    pairs = V // COL_ALIGN
    return [COL_ALIGN * (pairs * s // nshard) for s in range(nshard + 1)]


def owned_row_block(rank: int, vtp: int, gbs: int) -> tuple[int, int]:
    """(row_start, n_rows): the contiguous block of batch rows `rank` owns after the exchange
    (page function `owned_row_block`, one hop).  gbs must split evenly over the vtp ranks."""
    if vtp < 1 or not 0 <= rank < vtp or gbs % vtp:
        raise ValueError(f"gbs={gbs} rows do not split into {vtp} equal blocks (rank {rank})")
    n = gbs // vtp
    return rank * n, n


def exchange_candidates(vals, idx, group=None):
    """All-to-all of this rank's [gbs, k] candidates: rank q receives, from every rank in rank
    order, the rows of q's block.  Returns [nshard, gbs / nshard, k] tensors for this rank's rows."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    gbs, k = int(vals.shape[0]), int(vals.shape[1])
    owned_row_block(0, world, gbs)  # validates the split
    out_v = torch.empty_like(vals)
    out_i = torch.empty_like(idx)
    # row blocks are contiguous in [gbs, k]: block q goes to rank q; the receive is source-rank major
    dist.all_to_all_single(out_v, vals.contiguous(), group=group)
    dist.all_to_all_single(out_i, idx.contiguous(), group=group)
    return out_v.view(world, gbs // world, k), out_i.view(world, gbs // world, k)


def gather_candidates(vals, idx, group=None):
    """All-gathers this rank's [gbs, k] candidates into [nshard, gbs, k] tensors (rank order)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    gbs, k = int(vals.shape[0]), int(vals.shape[1])
    out_v = torch.empty((world * gbs, k), dtype=vals.dtype, device=vals.device)  # ranks concatenated on dim 0
    out_i = torch.empty((world * gbs, k), dtype=idx.dtype, device=idx.device)
    dist.all_gather_into_tensor(out_v, vals.contiguous(), group=group)
    dist.all_gather_into_tensor(out_i, idx.contiguous(), group=group)
    return out_v.view(world, gbs, k), out_i.view(world, gbs, k)


class ShardedTail:
    """One rank's part of the vocabulary-parallel tail (the weight slice [H, V_s] is this rank's)."""

    def __init__(self, H: int, V: int, k: int, gbs_max: int, rank: int, world: int, device: int = 0, **kw):
        self.bounds = shard_bounds(V, world)
        self.rank, self.world, self.k = rank, world, k
        self.lo, self.hi = self.bounds[rank], self.bounds[rank + 1]
        if self.hi - self.lo < k:
            raise ValueError(f"slice of {self.hi - self.lo} columns is narrower than k={k}")
        self.tail = Tail(H, self.hi - self.lo, k, gbs_max, device=device, **kw)

    def close(self):
        self.tail.close()

    def local_topk(self, hidden, gamma, w_slice, out_vals, out_idx, stream=None):
        """This rank's sorted top-k (slice-local ids); no sampler."""
        self.tail.run(hidden, gamma, w_slice, None, out_topk_vals=out_vals, out_topk_idx=out_idx, stream=stream)

    def merge(self, all_vals, all_idx, params, out_tokens, out_topk_vals=None, out_topk_idx=None, stream=None):
        """Global top-k and the draw from every rank's candidates ([nshard, gbs, k])."""
        return merge_shards(all_vals, all_idx, self.bounds[:-1], self.k, params=params, out_tokens=out_tokens,
                            out_topk_vals=out_topk_vals, out_topk_idx=out_topk_idx, stream=stream)

    def step(self, hidden, gamma, w_slice, params, out_tokens, group=None, stream=None, owned_rows=False):
        """One vocabulary-parallel step on this rank: local top-k, exchange, merge and draw.

        owned_rows=False: all-gather, every rank draws every row (params and out_tokens [gbs]).
        owned_rows=True: all-to-all, this rank draws only its `owned_row_block` (params and
        out_tokens hold those gbs / N rows)."""
        import contextlib

        import torch
        gbs = int(hidden.shape[0])
        # the collective orders itself after the current stream: make that the kernels' stream
        ctx = torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()
        with ctx:
            vals = torch.empty((gbs, self.k), dtype=torch.float32, device=hidden.device)
            idx = torch.empty((gbs, self.k), dtype=torch.int32, device=hidden.device)
            self.local_topk(hidden, gamma, w_slice, vals, idx, stream=stream)
            if owned_rows:
                all_v, all_i = exchange_candidates(vals, idx, group)
            else:
                all_v, all_i = gather_candidates(vals, idx, group)
            return self.merge(all_v, all_i, params, out_tokens, stream=stream)
