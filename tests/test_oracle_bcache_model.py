"""The block-cache residency model (oracle/bcache_model.py) pinned to CLOCK
worked by hand: three slots, the textbook second-chance sweep, a call that
never evicts what it reads, and an overflow once every slot is in use."""
from oracle.bcache_model import ClockCache


def test_clock_worked_example():
    c = ClockCache(n_pages=8, n_slots=3)
    # cold: three misses fill slots 0, 1, 2 in order; the hand ends at 0
    assert c.resolve([0, 1, 2]) == [0, 1, 2]
    assert c.hand == 0
    # page 0 hits (slot 0, used by this call); page 3 misses: the sweep skips
    # slot 0, clears the bits of slots 1 and 2, skips slot 0 again and takes
    # slot 1 (page 1 evicted); the hand stops at 2
    assert c.resolve([0, 3]) == [0, 1]
    assert c.table[1] == -1 and c.table[3] == 1 and c.hand == 2
    # page 2 hits (slot 2); pages 4, 5, 6 miss: slot 0 loses its bit, slot 1
    # (page 3, placed last call) too, then slot 0 is taken for 4 and slot 1
    # for 5; every slot is now used by this call, so 6 overflows (id 3 + 0)
    assert c.resolve([4, 5, 6, 2]) == [0, 1, 3, 2]
    assert c.table[6] == -1 and c.table[0] == -1 and c.table[3] == -1
    assert (c.calls, c.lookups, c.hits, c.misses, c.overflow) == (3, 9, 2, 7, 1)


def test_clock_claims_once_and_skips_invalid():
    c = ClockCache(n_pages=4, n_slots=2)
    # page 1 named three times is one miss; -1 lookups are skipped
    assert c.resolve([1, -1, 1, 2, 1]) == [0, -1, 0, 1, 0]
    assert (c.lookups, c.misses) == (4, 2)
    c.reset()
    assert c.table == [-1] * 4 and c.hand == 0 and c.calls == 0


def test_clock_demand_above_capacity_is_stable():
    # the same selection twice: the resident pages stay, the rest overflow
    c = ClockCache(n_pages=10, n_slots=3)
    sel = [5, 6, 7, 8, 9]
    first = c.resolve(sel)
    assert first == [0, 1, 2, 3, 4]
    second = c.resolve(sel)
    assert second[:3] == [0, 1, 2] and second[3:] == [3, 4]
    assert c.hits == 3 and c.overflow == 4
