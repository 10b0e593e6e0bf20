"""Host-side request sharding across ranks (one process per GPU).

Requests of the verification step are independent (attention reads only its own request's
cache and layout, acceptance only its own logits), so a global batch splits across GPUs
with no exchange step. `shard_requests` balances the attention work, which grows with the
prompt length, by longest-processing-time-first assignment.
"""
from __future__ import annotations

import heapq
from typing import List, Sequence


def shard_requests(prompt_len: Sequence[int], world_size: int) -> List[List[int]]:
    """Request indices per rank. Work of a request is taken as P + 1 (prompt keys plus its
    response tile); requests are placed longest first on the least-loaded rank (ties: lower
    rank). Each rank's list is sorted by request index."""
    if world_size < 1:
        raise ValueError("world_size must be >= 1")
    order = sorted(range(len(prompt_len)), key=lambda r: (-(max(int(prompt_len[r]), 0) + 1), r))
    heap = [(0, rank) for rank in range(world_size)]
    shards: List[List[int]] = [[] for _ in range(world_size)]
    for r in order:
        load, rank = heapq.heappop(heap)
        shards[rank].append(r)
        heapq.heappush(heap, (load + max(int(prompt_len[r]), 0) + 1, rank))
    return [sorted(s) for s in shards]
