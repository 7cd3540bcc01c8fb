"""The tile hand-out protocol of the standalone amax pass (TileQueue in
csrc/nvfp4_tiles.cuh), model-checked on the CPU over many random orders of
the CTAs' atomic requests: every tile is processed exactly once, every CTA
makes exactly one request that finds the tiles exhausted, exactly one request
sees the counter's final value, and that one leaves the counter at zero for
the next call.  The model follows the device code step for step: the first
`stages` loads of CTA b are the static tiles b + k*G, one request is made
after them, and each later refill takes the pending ticket and (if it was a
tile) requests the next one."""
import random

import pytest

NO_TILE = None


class Queue:
    """One CTA's thread-0 state (the device struct's fields)."""

    def __init__(self, cta, grid, ntiles, stages, counter):
        self.cta, self.grid, self.ntiles, self.counter = cta, grid, ntiles, counter
        self.first_dyn = stages * grid
        self.final_v = max(ntiles - self.first_dyn, 0) + grid - 1
        self.pending = None
        self.done = False
        self.saw_final = False

    def static_tile(self, k):
        t = self.cta + k * self.grid
        return t if t < self.ntiles else NO_TILE

    def request(self):
        self.pending = self.counter[0]  # atomicAdd returns the old value
        self.counter[0] += 1

    def start(self, complete):
        self.request()
        if not complete:
            self.finish()

    def next(self):
        if self.done:
            return NO_TILE
        t = self.first_dyn + self.pending
        if t < self.ntiles:
            self.request()
            return t
        self.finish()
        return NO_TILE

    def finish(self):
        self.done = True
        if self.pending == self.final_v:
            self.saw_final = True
            self.counter[0] = 0


def run(grid, ntiles, stages, rng):
    counter = [0]
    qs = [Queue(b, grid, ntiles, stages, counter) for b in range(grid)]
    processed = []
    # per CTA: the tiles currently in its stages (in load order)
    inflight = {b: [] for b in range(grid)}
    waiting = list(range(grid))  # CTAs not started yet: they start in any order, between others' refills
    live = []
    while waiting or live:
        if waiting and (not live or rng.random() < 0.5):
            b = waiting.pop(rng.randrange(len(waiting)))
            q = qs[b]
            complete = True
            for k in range(stages):
                t = q.static_tile(k)
                inflight[b].append(t)
                complete = t is not NO_TILE
                if not complete:
                    break
            q.start(complete)
            live.append(b)
            continue
        b = rng.choice(live)  # the next CTA to finish a load and refill its stage
        q = inflight[b]
        t = q.pop(0)
        if t is NO_TILE:  # the end marker: this CTA leaves its loop
            live.remove(b)
            continue
        processed.append(t)
        if not qs[b].done:
            q.append(qs[b].next())
    return processed, qs, counter[0]


@pytest.mark.parametrize("grid,ntiles,stages", [
    (456, 4096, 3),   # 8192x4096 bf16 on 152 SMs x 3 CTAs: 1368 static tiles, 2728 from the counter
    (456, 1368, 3),   # exactly the static tiles
    (456, 1000, 3),   # fewer tiles than static slots
    (7, 100, 3), (5, 5, 3), (3, 4, 1), (1, 9, 3), (64, 3000, 2),
])
def test_every_tile_once_and_one_reset(grid, ntiles, stages):
    rng = random.Random(grid * 1000 + ntiles)
    for _ in range(20):
        processed, qs, counter = run(grid, ntiles, stages, rng)
        assert sorted(processed) == list(range(ntiles))
        assert all(q.done for q in qs)
        assert sum(q.saw_final for q in qs) == 1
        assert counter == 0
