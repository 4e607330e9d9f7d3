"""Splitting a jagged batch across ranks.

Every (sequence, head) of jagged attention is independent, forward and backward, so
a batch shards with no exchange step: each rank runs the kernels on its own sequences
and, if a caller wants the full outputs everywhere, one all-gather puts them back.
Sequences are balanced by the work they cost (the (query, key) pairs attention
visits), longest first onto the least-loaded rank.

Biases follow their sequences: a general jagged bias's blocks are packed per shard like
the values (select_bias_blocks). A relative-position table is shared by every sequence,
so its gradient is the one exchange a sharded backward has: each rank's table holds the
sum over its own sequences, and one all-reduce (sum) over the ranks gives the batch's.
"""
from __future__ import annotations

from typing import List, Sequence

import torch


def visited_pairs(lq: int, lk: int, causal: bool) -> int:
    """(query, key) pairs one sequence visits per head (bottom-right causal when causal)."""
    if lq <= 0 or lk <= 0:
        return 0
    if not causal:
        return lq * lk
    first = max(0, lq - lk)          # earlier rows see no key
    n = lq - first
    s0 = first + (lk - lq) + 1       # keys seen by row `first`
    return n * s0 + n * (n - 1) // 2


def shard_sequences(q_lengths: Sequence[int], kv_lengths: Sequence[int], world: int,
                    causal: bool = False) -> List[List[int]]:
    """Assign sequence indices to `world` ranks, longest-processing-time first.
    Returns one sorted index list per rank; every index appears exactly once."""
    if world < 1:
        raise ValueError("world must be >= 1")
    costs = [(visited_pairs(int(a), int(b), causal), i) for i, (a, b) in enumerate(zip(q_lengths, kv_lengths))]
    costs.sort(key=lambda t: (-t[0], t[1]))
    load = [0] * world
    shards: List[List[int]] = [[] for _ in range(world)]
    for c, i in costs:
        r = min(range(world), key=lambda k: (load[k], k))
        shards[r].append(i)
        load[r] += c
    return [sorted(s) for s in shards]


def select_sequences(values: torch.Tensor, offsets: torch.Tensor, index: Sequence[int]):
    """Pack the chosen sequences of a jagged tensor (values [T, ...], offsets [B+1])
    into a new jagged tensor; returns (values, offsets)."""
    off = offsets.tolist()
    parts = [values[off[b]:off[b + 1]] for b in index]
    lens = [off[b + 1] - off[b] for b in index]
    new_off = torch.zeros(len(index) + 1, dtype=torch.int64)
    if lens:
        new_off[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)
    packed = torch.cat(parts, 0) if parts else values[:0]
    return packed, new_off.to(offsets.device)


def scatter_sequences(full: torch.Tensor, offsets: torch.Tensor, index: Sequence[int], part: torch.Tensor,
                      part_offsets: torch.Tensor) -> None:
    """Write a rank's packed results (part, part_offsets) back into the full jagged
    tensor at the rows of sequences `index` (inverse of select_sequences)."""
    off = offsets.tolist()
    poff = part_offsets.tolist()
    for k, b in enumerate(index):
        full[off[b]:off[b + 1]] = part[poff[k]:poff[k + 1]]


def select_bias_blocks(values: torch.Tensor, block_offsets: torch.Tensor, index: Sequence[int]):
    """Pack the general jagged bias blocks (values [H, plane], block offsets [B+1]) of the
    chosen sequences into the bias of a shard; returns (values, block offsets).  A block's
    layout depends only on its sequence's lengths, so blocks move unchanged."""
    off = block_offsets.tolist()
    parts = [values[:, off[b]:off[b + 1]] for b in index]
    sizes = [off[b + 1] - off[b] for b in index]
    new_off = torch.zeros(len(index) + 1, dtype=torch.int64)
    if sizes:
        new_off[1:] = torch.cumsum(torch.tensor(sizes, dtype=torch.int64), 0)
    packed = torch.cat(parts, 1).contiguous() if parts else values[:, :0]
    return packed, new_off.to(block_offsets.device)


def scatter_bias_blocks(full: torch.Tensor, block_offsets: torch.Tensor, index: Sequence[int], part: torch.Tensor,
                        part_offsets: torch.Tensor) -> None:
    """Write a shard's packed general-bias blocks (part [H, plane'], part_offsets) back into
    the full [H, plane] array at the blocks of sequences `index` (inverse of
    select_bias_blocks; used for the bias's gradient)."""
    off = block_offsets.tolist()
    poff = part_offsets.tolist()
    for k, b in enumerate(index):
        full[:, off[b]:off[b + 1]] = part[:, poff[k]:poff[k + 1]]
