"""Page-allocator model — test infrastructure only.

The paged KV arena is the "true goal" KV layout of the mlx-bun parallel-slots
design ("KV memory: dynamic allocation, not static partition", rung 3: fixed
size blocks in a shared pool plus a block manager). The pages fix no
allocation order, so the reading taken is: a step visits its lanes in input
order; a lane whose length is a multiple of the page size takes the LOWEST
free page index; resetting a lane returns all of its pages. A step that needs
more pages than are free changes nothing (the call is atomic).

Clone and Evict ("MODEL-BATCHING-RESULTS", "Why in-kernel batching, not
vLLM": per-user prefix reuse and quarantine of a span, kept under batching)
act on pages as follows, the reading taken for sharing. A page carries the
count of lanes that hold it and is free when that count is 0. Clone gives an
empty lane the source lane's full pages (count + 1) and, when the source's
length is not a multiple of the page size, one fresh page (lowest free) for
the copy of its partial last page. Evict of [start, end) keeps the first
ceil(new_length / page_size) pages of the table; among them the pages from
index start // page_size on are written, and each such page that another
lane holds is replaced, in ascending index order, by the lowest free page
(the old page loses one holder); then the pages past the new end lose one
holder each. Both are atomic (no free page for a copy: nothing changes).

Lane lengths and the per-call validation follow the primitive's contract in
"Fat-station continuous batching" ("The capture": each lane advances by one
token; positions are per lane and advanced by the call).
"""
from __future__ import annotations

import heapq

OK, ERR_ARG, ERR_LANE, ERR_DUP_LANE, ERR_POSITION, ERR_TOKEN, ERR_KV_FULL = (
    0, -1, -2, -3, -4, -5, -6)
ERR_STATE = -9


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
        self.ref = [0] * n_pages

    def _take(self) -> int:
        p = heapq.heappop(self.free)
        self.ref[p] = 1
        return p

    def _release(self, p: int) -> None:
        self.ref[p] -= 1
        if self.ref[p] == 0:
            heapq.heappush(self.free, p)

    def reset(self, lane: int) -> int:
        if not 0 <= lane < self.max_lanes:
            return ERR_LANE
        for p in self.tables[lane]:
            self._release(p)
        self.tables[lane] = []
        self.length[lane] = 0
        return OK

    def clone(self, src: int, dst: int) -> int:
        if not (0 <= src < self.max_lanes and 0 <= dst < self.max_lanes):
            return ERR_LANE
        if src == dst:
            return ERR_ARG
        if self.length[dst] or self.tables[dst]:
            return ERR_STATE
        n, ps = self.length[src], self.page_size
        full = n // ps
        if n % ps and not self.free:
            return ERR_KV_FULL
        t = self.tables[src][:full]
        for p in t:
            self.ref[p] += 1
        if n % ps:
            t.append(self._take())
        self.tables[dst] = t
        self.length[dst] = n
        return OK

    def evict(self, lane: int, start: int, end: int) -> int:
        if not 0 <= lane < self.max_lanes:
            return ERR_LANE
        n, ps = self.length[lane], self.page_size
        if not 0 <= start <= end <= n:
            return ERR_ARG
        if start == end:
            return OK
        nl = n - (end - start)
        keep = -(-nl // ps)
        old = self.tables[lane]
        written = range(start // ps, keep)
        if sum(self.ref[old[x]] > 1 for x in written) > len(self.free):
            return ERR_KV_FULL
        t = old[:keep]
        for x in written:
            if self.ref[old[x]] > 1:
                self.ref[old[x]] -= 1
                t[x] = self._take()
        for p in old[keep:]:
            self._release(p)
        self.tables[lane] = t
        self.length[lane] = nl
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
                self.tables[k].append(self._take())
            self.length[k] += 1
        return OK

    def table(self, lane: int):
        return list(self.tables[lane])
