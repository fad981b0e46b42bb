"""Host side of a row-sharded table (Engram listing, __init__: the embedding is a
ParallelEngramEmbedding).

The pages name the sharded embedding but not its split. This module reads it as the usual
vocabulary-parallel layout: rank r of W holds the contiguous rows
[floor(n r / W), floor(n (r + 1) / W)) of the n-row table. Every rank hashes the same tokens (the
hash is replicated), gathers the rows it holds and writes bf16 -0.0 for the others
(engram_embed_rows_shard), and one all-reduce (sum) of the [n_ids, head_dim] rows completes the
gather: each id has exactly one owner and -0 is the identity of IEEE addition, so the sum is the
unsharded gather bit for bit. The projection and the gate then run on the full rows.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import api


def table_shard_range(num_rows: int, world_size: int, rank: int) -> tuple[int, int]:
    """(first row, row count) that `rank` holds; the ranges tile [0, num_rows) in rank order and
    differ in size by at most one row."""
    if world_size < 1 or not 0 <= rank < world_size or num_rows < 0:
        raise ValueError("need world_size >= 1, 0 <= rank < world_size, num_rows >= 0")
    begin = num_rows * rank // world_size
    end = num_rows * (rank + 1) // world_size
    return begin, end - begin


def row_owner(ids, num_rows: int, world_size: int) -> np.ndarray:
    """The rank holding each row id in [0, num_rows): the largest r with floor(n r / W) <= id,
    i.e. ceil(W (id + 1) / n) - 1."""
    ids = np.asarray(ids, dtype=np.int64)
    if ids.size and (ids.min() < 0 or ids.max() >= num_rows):
        raise ValueError("row ids must lie in [0, num_rows)")
    return (world_size * (ids + 1) - 1) // num_rows


def exchange_rows(out: torch.Tensor, group=None) -> torch.Tensor:
    """The exchange step: sum every rank's partial rows in place (one all-reduce). bf16 sums of
    one value and -0.0s are exact in any order, so no wider type is needed."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    return out


def embed_rows_sharded(desc, table_shard, scales_shard, row_begin: int, ids, out, group=None):
    """Stage 2 over a row-sharded table: this rank's rows by engram_embed_rows_shard on the current
    stream, then exchange_rows. `out` (bf16 [n_ids, head_dim], on this rank's GPU) ends up equal
    on every rank of `group` to engram_embed_rows over the whole table."""
    api.engram_embed_rows_shard(desc, table_shard, scales_shard, row_begin, ids, out,
                                stream=torch.cuda.current_stream())
    return exchange_rows(out, group)
