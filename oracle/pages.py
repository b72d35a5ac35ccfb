"""Page-allocator model — test infrastructure only.

The paged KV arena is the "true goal" KV layout of the mlx-bun parallel-slots
design ("KV memory: dynamic allocation, not static partition", rung 3: fixed
size blocks in a shared pool plus a block manager). The pages fix no
allocation order, so the reading taken is: a step visits its lanes in input
order; a lane whose length is a multiple of the page size takes the LOWEST
free page index; resetting a lane returns all of its pages. A step that needs
more pages than are free changes nothing (the call is atomic).

Lane lengths and the per-call validation follow the primitive's contract in
"Fat-station continuous batching" ("The capture": each lane advances by one
token; positions are per lane and advanced by the call).
"""
from __future__ import annotations

import heapq

OK, ERR_ARG, ERR_LANE, ERR_DUP_LANE, ERR_POSITION, ERR_TOKEN, ERR_KV_FULL = (
    0, -1, -2, -3, -4, -5, -6)


class PageModel:
    def __init__(self, n_pages: int, page_size: int, max_lanes: int,
                 max_pages_per_lane: int):
        self.page_size = page_size
        self.max_lanes = max_lanes
        self.max_pages_per_lane = max_pages_per_lane
        self.free = list(range(n_pages))
        heapq.heapify(self.free)
        self.tables = [[] for _ in range(max_lanes)]
        self.length = [0] * max_lanes

    def reset(self, lane: int) -> int:
        if not 0 <= lane < self.max_lanes:
            return ERR_LANE
        for p in self.tables[lane]:
            heapq.heappush(self.free, p)
        self.tables[lane] = []
        self.length[lane] = 0
        return OK

    def step(self, lanes, positions, tokens, vocab: int) -> int:
        """Validate one decode step and allocate its pages; atomic."""
        n = len(lanes)
        if n < 0 or len(positions) != n or len(tokens) != n:
            return ERR_ARG
        seen = set()
        need = 0
        for i in range(n):
            k = int(lanes[i])
            if not 0 <= k < self.max_lanes:
                return ERR_LANE
            if k in seen:
                return ERR_DUP_LANE
            seen.add(k)
            if int(positions[i]) != self.length[k]:
                return ERR_POSITION
            if not 0 <= int(tokens[i]) < vocab:
                return ERR_TOKEN
            if self.length[k] % self.page_size == 0:
                if self.length[k] // self.page_size >= self.max_pages_per_lane:
                    return ERR_KV_FULL
                need += 1
        if need > len(self.free):
            return ERR_KV_FULL
        for i in range(n):
            k = int(lanes[i])
            if self.length[k] % self.page_size == 0:
                self.tables[k].append(heapq.heappop(self.free))
            self.length[k] += 1
        return OK

    def table(self, lane: int):
        return list(self.tables[lane])
