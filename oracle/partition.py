"""Partition index oracle (pure Python loops over the definitions).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

TransformerEngine PR #3221, section "Why": the default DualChunkSwap
partition divides every sequence into 2*cp_size chunks; the NO_LOAD_BALANCE
partition cuts the complete physical buffer into cp_size contiguous chunks,
one per rank in rank-major order ("What changed"; the commit note "Rank-major
ownership needs no KV reorder"). The rank r -> chunks {r, 2*cp_size-1-r}
assignment is the head-tail split (torchtitan PR #2144, "Summary",
_HeadTailLoadBalancer) applied to each document.

Readings where the pages are silent:
* Within a rank, DualChunkSwap lists document 0..N-1 in pack order, and for
  each document chunk r before chunk 2*cp_size-1-r. The rank-local offset
  array is therefore cu_seqlens_padded / cp_size.
* DualChunkSwap requires every padded document length to be divisible by
  2*cp_size (the pages give divisibility as the reason NO_LOAD_BALANCE
  exists); NO_LOAD_BALANCE requires T % cp_size == 0 ("equal local Q/K/V
  physical lengths", section "Scope and constraints").
"""
from __future__ import annotations

from typing import List, Sequence

DUAL_CHUNK_SWAP = "dcs"
NO_LOAD_BALANCE = "nlb"
PACKED_MIRRORED = "mirrored"


class PartitionError(ValueError):
    pass


def local_tokens(strategy: str, T: int, cp_size: int) -> int:
    """Tokens each rank holds: T / cp_size under either strategy."""
    if cp_size < 1:
        raise PartitionError("cp_size must be >= 1")
    if T % cp_size != 0:
        raise PartitionError("T must be divisible by cp_size")
    return T // cp_size


def dual_chunk_swap_indices(cu_seqlens_padded: Sequence[int], cp_size: int, rank: int) -> List[int]:
    """Physical token indices owned by ``rank`` under DualChunkSwap."""
    cup = [int(x) for x in cu_seqlens_padded]
    if not (0 <= rank < cp_size):
        raise PartitionError("rank out of range")
    out: List[int] = []
    for j in range(len(cup) - 1):
        start, end = cup[j], cup[j + 1]
        P = end - start
        if P < 0:
            raise PartitionError("cu_seqlens_padded must be non-decreasing")
        if P % (2 * cp_size) != 0:
            raise PartitionError(f"document {j}: padded length {P} not divisible by 2*cp_size")
        chunk = P // (2 * cp_size)
        for c in (rank, 2 * cp_size - 1 - rank):
            for t in range(chunk):
                out.append(start + c * chunk + t)
    return out


def no_load_balance_indices(T: int, cp_size: int, rank: int) -> List[int]:
    """Physical token indices owned by ``rank`` under NO_LOAD_BALANCE."""
    if not (0 <= rank < cp_size):
        raise PartitionError("rank out of range")
    n = local_tokens(NO_LOAD_BALANCE, T, cp_size)
    out: List[int] = []
    for t in range(n):
        out.append(rank * n + t)
    return out


def packed_mirrored_indices(T: int, cp_size: int, rank: int) -> List[int]:
    """The PR's interim packed super-sequence partition (commit notes: the
    complete physical token buffer represented as one partitioning sequence,
    mirrored chunks): DualChunkSwap of the single sequence [0, T)."""
    if T % (2 * cp_size) != 0:
        raise PartitionError("T must be divisible by 2*cp_size")
    return dual_chunk_swap_indices([0, T], cp_size, rank)


def partition_index(strategy: str, cu_seqlens_padded: Sequence[int], cp_size: int, rank: int) -> List[int]:
    T = int(cu_seqlens_padded[-1])
    if strategy == DUAL_CHUNK_SWAP:
        return dual_chunk_swap_indices(cu_seqlens_padded, cp_size, rank)
    if strategy == NO_LOAD_BALANCE:
        return no_load_balance_indices(T, cp_size, rank)
    if strategy == PACKED_MIRRORED:
        return packed_mirrored_indices(T, cp_size, rank)
    raise PartitionError(f"unknown strategy {strategy!r}")


def restore_index(strategy: str, cu_seqlens_padded: Sequence[int], cp_size: int) -> List[int]:
    """K/V restoration after an all-gather (TE PR, Greptile summary: "stable
    K/V restoration"): the gathered buffer is the rank-major concatenation of
    the ranks' index lists; restore[p] is the position of physical slot p in
    that concatenation, so gathered[restore] is back in token order."""
    T = int(cu_seqlens_padded[-1])
    concat: List[int] = []
    for r in range(cp_size):
        concat += partition_index(strategy, cu_seqlens_padded, cp_size, r)
    restore = [-1] * T
    for pos, p in enumerate(concat):
        restore[p] = pos
    return restore


def local_cu_seqlens_padded(cu_seqlens_padded: Sequence[int], cp_size: int) -> List[int]:
    """Rank-local physical offsets under DualChunkSwap: each document keeps
    1/cp_size of its padded length on every rank."""
    return [int(x) // cp_size for x in cu_seqlens_padded]
