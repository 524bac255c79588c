"""Split-V draft head across ranks (tensor-parallel candidate table).

"少读一张大表，草稿路径才真正快起来" splits the 65,536-row draft head over two
GB10 ranks (32,768 rows each): every rank takes the argmax over its own rows,
then the ranks exchange the best score and its global token id and keep the
overall best.  On one GPU the library does this merge inside the kernel
(packed-key atomicMax).  This module is the multi-rank form: each rank runs
the draft head on its shard, the (score, id) pairs are all-gathered over a
torch.distributed group, and the merge keeps the largest score and, on equal
scores, the lowest global id -- the same rule as the kernel, so the result
equals the single-GPU result over the union of the shards.
"""
from __future__ import annotations

import torch


def merge_rank_argmax(maxlogits: torch.Tensor, ids: torch.Tensor):
    """maxlogits float32 [R, B], ids int32 [R, B] (one row per rank) ->
    (ids [B], maxlogit [B]): the largest score per column, lowest id on ties.
    NaN scores count as -inf; -0 equals +0."""
    if maxlogits.shape != ids.shape or maxlogits.dim() != 2:
        raise ValueError("expected matching [ranks, B] tensors")
    s = torch.nan_to_num(maxlogits.float(), nan=float("-inf")) + 0.0
    best = s.max(dim=0, keepdim=True).values
    cand = torch.where(s == best, ids.long(), torch.full_like(ids, torch.iinfo(torch.int32).max, dtype=torch.long))
    win = cand.min(dim=0).values
    return win.to(torch.int32), best.squeeze(0)


def split_v_draft_argmax(local_fn, group=None):
    """Run `local_fn()` -> (ids [B] int32, maxlogit [B] float32) for this
    rank's shard, all-gather the pairs over `group`, and return the merged
    (ids, maxlogit) on every rank.

    `local_fn` is normally a closure over mtp_draft_head_argmax with this
    rank's candidate rows and global ids; anything that returns the same pair
    works.  The exchange moves 8 bytes per hidden row per rank."""
    import torch.distributed as dist
    ids, ml = local_fn()
    world = dist.get_world_size(group)
    ml_all = [torch.empty_like(ml) for _ in range(world)]
    ids_all = [torch.empty_like(ids) for _ in range(world)]
    dist.all_gather(ml_all, ml.contiguous(), group=group)
    dist.all_gather(ids_all, ids.contiguous(), group=group)
    return merge_rank_argmax(torch.stack(ml_all), torch.stack(ids_all))


def shard_rows(n_rows: int, rank: int, world: int):
    """Contiguous row range [lo, hi) of `rank` when n_rows are split over `world` ranks."""
    lo = n_rows * rank // world
    hi = n_rows * (rank + 1) // world
    return lo, hi
