"""The decode schedules' partition arithmetic, checked on the CPU.

The balanced schedule lays the pages of all (sequence, head group) units end
to end (TP pages) and gives CTA c the pages [c*TP/G, (c+1)*TP/G) with
G = min(grid, TP); the CTA holding a unit's first page records the unit's
last owner as floor(((x + 1) * G - 1) / TP) for the unit's last page x, and
the combine merges the partials of every CTA from the first to the last
owner.  The split schedule cuts a sequence into chunks of
C = ceil(ceil(hint / bs) / S) pages with the last split taking the rest
(reading R11).  These tests restate those formulas and check the invariants
the kernels rely on: every page covered exactly once, the recorded owners
are the true ones, and every CTA between them holds part of the unit.
"""

import random


def _balanced(P, grid):
    tp = sum(P)
    G = min(grid, tp if tp > 0 else 1)
    owners = {}
    covered = [0] * tp
    for c in range(grid):
        lo, hi = (c * tp // G, (c + 1) * tp // G) if c < G else (tp, tp)
        for x in range(lo, hi):
            covered[x] += 1
            owners.setdefault(x, c)
    return tp, G, covered, owners


def test_balanced_partition_covers_every_page_once_and_owners_are_consistent():
    rng = random.Random(11)
    for _ in range(2000):
        U = rng.choice([1, 2, 5, 64, 300])
        P = [rng.choice([0, 0, 1, 3, 16, 100, 1024]) for _ in range(U)]
        grid = rng.choice([1, 2, 7, 148, 152])
        tp, G, covered, owners = _balanced(P, grid)
        assert all(n == 1 for n in covered)
        start = 0
        for p in P:
            if p == 0:
                continue
            first, last = start, start + p - 1
            c_first = owners[first]
            c_last = ((last + 1) * G - 1) // tp          # the kernel's formula
            assert c_last == owners[last]
            assert c_first == ((first + 1) * G - 1) // tp
            # every CTA from the first to the last owner holds part of the unit
            held = {owners[x] for x in range(first, last + 1)}
            assert held == set(range(c_first, c_last + 1))
            start += p


def test_split_partition_covers_every_key_once_for_any_hint():
    rng = random.Random(12)
    for _ in range(1500):
        bs = rng.choice([16, 32, 256])
        L = rng.randint(0, 6000)
        S = rng.randint(1, 256)
        hint = rng.choice([L, L // 2, 1, 6000, max(L, 1) * 3])
        hint_pages = (max(hint, 1) + bs - 1) // bs
        C = max(1, (hint_pages + S - 1) // S)        # pages per split
        P = (L + bs - 1) // bs
        seen = [0] * L
        for j in range(S):
            p0 = min(j * C, P)
            p1 = P if j == S - 1 else min((j + 1) * C, P)   # the last split takes the rest
            for k in range(p0 * bs, min(p1 * bs, L)):
                seen[k] += 1
        assert all(n == 1 for n in seen)
