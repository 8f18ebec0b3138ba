"""Pins of the slot-pool policy oracle (oracle/pool_policy.py).  CPU only.

The policy is integer bookkeeping, so the pins are a hand-worked trace, closed
forms for special pool sizes, and invariants on random traces.
"""
import random

from oracle.pool_policy import SlotPool


def test_hand_worked_trace():
    """S = 3 slots, 8 experts.
    step 1 [1, 2]: both miss, empty slots 0, 1; freq 1, 1.
    step 2 [1, 3]: 1 hits (freq 2, last 2); 3 misses into empty slot 2.
    step 3 [4, 4]: 4 misses; slots 0 (e1: freq 2, last 2), 1 (e2: 1, 1),
      2 (e3: 1, 2); lowest frequency 1 ties between slots 1 and 2, the least
      recent is slot 1 -> e2 evicted, e4 in slot 1 with freq 2 (two pairs).
    step 4 [2, 5]: both miss; e1 (2, 2), e4 (2, 3), e3 (1, 2): e3 goes for e2
      (slot 2); then e1 (2, 2) against e4 (2, 3): e1 is less recent -> e5 in
      slot 0.
    """
    p = SlotPool(8, 3)
    assert p.step([1, 2]) == [(1, 0), (2, 1)]
    assert p.step([1, 3]) == [(3, 2)]
    assert p.step([4, 4]) == [(4, 1)]
    assert p.owner == [1, 4, 3] and p.freq == [2, 2, 1] and p.last == [2, 3, 2]
    assert p.step([2, 5]) == [(2, 2), (5, 0)]
    assert p.owner == [5, 4, 2]
    assert (p.hits, p.misses, p.evictions, p.overflows) == (1, 6, 3, 0)


def test_frequency_beats_recency():
    """A twice-used expert outlives a once-used one that was used later."""
    p = SlotPool(4, 2)
    p.step([0])
    p.step([0])      # e0: freq 2
    p.step([1])      # e1: freq 1, more recent
    p.step([2])      # must evict e1 (lower frequency), not e0
    assert sorted(p.owner) == [0, 2]


def test_pool_as_large_as_the_working_set_only_misses_once():
    """S >= number of distinct experts ever used: compulsory misses only."""
    rng = random.Random(3)
    p = SlotPool(64, 20)
    used = set()
    for _ in range(200):
        step = [rng.randrange(20) for _ in range(6)]
        used.update(step)
        p.step(step)
    assert p.misses == len(used) and p.evictions == 0 and p.overflows == 0


def test_one_slot_alternating_experts_always_miss():
    p = SlotPool(4, 1)
    for i in range(10):
        p.step([i % 2])
    assert p.misses == 10 and p.hits == 0 and p.evictions == 9


def test_overflow_when_a_step_needs_more_than_the_pool():
    p = SlotPool(16, 3)
    fills = p.step([0, 1, 2, 3, 4])
    assert fills == [(0, 0), (1, 1), (2, 2)] and p.overflows == 2
    assert p.table[3] == -1 and p.table[4] == -1


def test_invariants_on_random_traces():
    rng = random.Random(7)
    for trial in range(20):
        E, S = rng.randint(4, 40), 0
        S = rng.randint(1, E - 1)
        p = SlotPool(E, S)
        distinct_total = 0
        for _ in range(60):
            k = rng.randint(1, min(S, 6))
            step = [rng.randrange(E) for _ in range(k)]
            before = {e: p.table[e] for e in set(step)}
            p.step(step)
            distinct_total += len(set(step))
            # the table and the owners are inverse maps
            for e in range(E):
                if p.table[e] >= 0:
                    assert p.owner[p.table[e]] == e
            for s in range(S):
                if p.owner[s] >= 0:
                    assert p.table[p.owner[s]] == s
            # every expert of the step is resident after it (no overflow: k <= S)
            assert all(p.table[e] >= 0 for e in step)
            # hits keep their slot
            for e, s in before.items():
                if s >= 0:
                    assert p.table[e] == s
        assert p.hits + p.misses == distinct_total
        assert p.overflows == 0
