"""Block-cache residency restated as a plain sequential model (test
infrastructure: only tests/ import it).

Follows the resolve rules of the "Strata compare" page, KV streaming section
(the resolve steps of its design notes): a resident page named by the call
gets the call's mark and its CLOCK reference bit; a missing page is claimed
once, however many lookups name it; each claimed miss then takes one victim
slot by a CLOCK (second-chance) sweep that never takes a slot this call uses,
and the table is re-pointed (old page -> absent, new page -> slot).

Readings this library adds, stated where the page is silent:
  * the unit is one (block, KV head) page, because selections are per KV head;
  * misses are claimed in the order of their first lookup (sequence, KV head,
    selection order);
  * a miss that finds no slot (every slot is used by this call or already
    taken) is read into the call's overflow area instead: its page id is
    n_slots + (its index among the overflowed misses), and it stays absent.

The sweep is the textbook loop, one slot at a time: skip a slot this call
uses; take a free slot or one whose reference bit is clear; otherwise clear
the bit and move on.  Slots taken by this call count as used.
"""


class ClockCache:
    def __init__(self, n_pages: int, n_slots: int):
        self.table = [-1] * n_pages          # page -> slot, or -1
        self.slot_page = [-1] * n_slots      # slot -> page, or -1
        self.ref = [0] * n_slots
        self.hand = 0
        self.calls = self.lookups = self.hits = self.misses = self.overflow = 0

    def reset(self):
        self.__init__(len(self.table), len(self.slot_page))

    def resolve(self, pages):
        """pages: page id of every lookup in lookup order (-1: invalid, skipped).
        Returns the pool page id of every lookup (-1 for invalid lookups)."""
        n = len(self.slot_page)
        used = set()
        n_look = n_hit = 0
        for p in pages:
            if p < 0:
                continue
            n_look += 1
            s = self.table[p]
            if s >= 0:
                used.add(s)
                self.ref[s] = 1
                n_hit += 1
        misses, seen = [], set()
        for p in pages:
            if p >= 0 and self.table[p] < 0 and p not in seen:
                seen.add(p)
                misses.append(p)
        where = {}
        n_over = 0
        for p in misses:
            victim = None
            for _ in range(2 * n):               # two revolutions clear every bit on the way
                j = self.hand
                if j not in used and (self.slot_page[j] < 0 or self.ref[j] == 0):
                    victim = j
                    self.hand = (j + 1) % n
                    break
                if j not in used:
                    self.ref[j] = 0              # second chance used up
                self.hand = (j + 1) % n
            if victim is None:
                where[p] = n + n_over
                n_over += 1
                continue
            old = self.slot_page[victim]
            if old >= 0:
                self.table[old] = -1
            self.slot_page[victim] = p
            self.table[p] = victim
            self.ref[victim] = 1
            used.add(victim)
            where[p] = victim
        self.calls += 1
        self.lookups += n_look
        self.hits += n_hit
        self.misses += len(misses)
        self.overflow += n_over
        out = []
        for p in pages:
            if p < 0:
                out.append(-1)
            elif p in where:
                out.append(where[p])
            else:
                out.append(self.table[p])
        return out
