"""Oracle of the bounded expert slot pool -- TEST INFRASTRUCTURE ONLY.

The pages keep the routed experts in storage and cache the frequently used
ones in a pool of bounded size, evicting by least frequent use combined with
recency (Swiftlet README on the wpnews page, section "How it works", and the
same README's list of what it borrowed; creativeainews, "How Expert Streaming
Works").  They give no formula.
Readings, plainest first:

* one step is one forward call; the experts it needs are the distinct
  experts of its T*k (token, expert) pairs;
* an expert's frequency is the number of pairs routed to it since it entered
  the pool (its count restarts when it is evicted and fetched again);
  recency is the step of its last use;
* a needed expert already in the pool is a hit: frequency += its pairs,
  last use = this step;
* the misses are filled in ascending expert id; each takes an empty slot if
  there is one (lowest slot first), else evicts, among the slots whose expert
  this step does not need, the one with the lowest frequency, then the least
  recent last use, then the lowest slot id;
* a miss with no slot left to take (the step needs more distinct experts
  than the pool holds) stays unmapped and is counted as an overflow.

Frequencies saturate at 2^23 - 1 and steps at 2^24 - 1 (the device packs
both into one 64-bit key).
"""
from __future__ import annotations

FREQ_MAX = (1 << 23) - 1
STEP_MAX = (1 << 24) - 1


class SlotPool:
    def __init__(self, n_experts: int, n_slots: int):
        self.E, self.S = n_experts, n_slots
        self.table = [-1] * n_experts       # expert -> slot
        self.owner = [-1] * n_slots         # slot -> expert
        self.freq = [0] * n_slots
        self.last = [0] * n_slots
        self.step_no = 0
        self.hits = self.misses = self.evictions = self.overflows = 0

    def step(self, topk_idx) -> list:
        """Apply one forward's routing (any iterable of expert ids, one per
        pair).  Returns the fills of this step as (expert, slot) pairs."""
        self.step_no = min(self.step_no + 1, STEP_MAX)
        count = {}
        for e in topk_idx:
            count[int(e)] = count.get(int(e), 0) + 1
        needed = sorted(count)
        for e in needed:
            s = self.table[e]
            if s >= 0:
                self.hits += 1
                self.freq[s] = min(self.freq[s] + count[e], FREQ_MAX)
                self.last[s] = self.step_no
        fills = []
        for e in needed:
            if self.table[e] >= 0:  # a hit (evictions only touch unneeded experts)
                continue
            best = None
            for s in range(self.S):
                o = self.owner[s]
                if o >= 0 and o in count:
                    continue  # needed by this step
                key = (0, 0, 0, s) if o < 0 else (1, self.freq[s], self.last[s], s)
                if best is None or key < best[0]:
                    best = (key, s)
            if best is None:
                self.overflows += 1
                continue
            s = best[1]
            if self.owner[s] >= 0:
                self.table[self.owner[s]] = -1
                self.evictions += 1
            self.owner[s] = e
            self.table[e] = s
            self.freq[s] = min(count[e], FREQ_MAX)
            self.last[s] = self.step_no
            self.misses += 1
            fills.append((e, s))
        return fills
