"""Invariants of the split-KV partition plan (CPU).

These pin the plan's restatement in oracle/mla_sched.py without relying on
it: whatever the plan is, every 64-key tile of every request must be covered
exactly once, split counts must add up, split slots must be dense, and no
part may exceed its budget except the last (which absorbs the remainder).
"""

import numpy as np
import pytest

from oracle import mla_sched as sp


def cost_of(ranges, F):
    return sum(t1 - t0 + F for (_, t0, t1, _) in ranges)


@pytest.mark.parametrize("num_parts", [1, 2, 3, 7, 38, 76, 152])
@pytest.mark.parametrize("F", [0, 1, 4])
def test_plan_covers_every_tile_once(num_parts, F):
    rng = np.random.default_rng(num_parts * 10 + F)
    for trial in range(25):
        B = int(rng.integers(1, 70))
        L = rng.integers(0, 5000, size=B)
        L[rng.random(B) < 0.1] = 0
        sched, off = sp.plan(L.tolist(), num_parts, F)
        assert len(sched) == num_parts and len(off) == B + 1
        nt = [-(-int(x) // 64) for x in L]
        seen = {b: np.zeros(nt[b], int) for b in range(B)}
        splits = {b: [] for b in range(B)}
        total = sum(n + F for n in nt if n > 0)
        cap = -(-total // num_parts) + F if total else 0
        for p, e in enumerate(sched):
            rs = sp.part_ranges(e, L.tolist())
            for (b, t0, t1, s) in rs:
                assert 0 <= t0 < t1 <= nt[b]
                seen[b][t0:t1] += 1
                splits[b].append(s)
            if p < num_parts - 1:
                assert cost_of(rs, F) <= cap
            else:
                assert cost_of(rs, F) <= 2 * cap + F
        for b in range(B):
            assert (seen[b] == 1).all()
            n = off[b + 1] - off[b]
            assert n == len(splits[b])
            assert splits[b] == list(range(n))        # split slots 0..n-1 in part order
            assert (n == 0) == (nt[b] == 0)


def _forced(L, num_parts, F, cap):
    """The plan's walk with a given cap (the oracle's own walk, cap fixed)."""
    saved = sp.choose_cap
    sp.choose_cap = lambda nt, P, F_: cap
    try:
        return sp.plan(L, num_parts, F)
    finally:
        sp.choose_cap = saved


@pytest.mark.parametrize("num_parts", [2, 7, 38, 76])
def test_plan_cap_never_worse_than_the_plain_cap(num_parts):
    """The chosen cap's plan has a largest part no costlier than the plan with
    cap = c0 + F, and when a smaller cap is chosen the last part fits in it."""
    rng = np.random.default_rng(num_parts + 300)
    F = 4
    for trial in range(30):
        B = int(rng.integers(1, 70))
        L = rng.integers(0, 5000, size=B).tolist()
        nt = [-(-int(x) // 64) for x in L]
        total = sum(n + F for n in nt if n > 0)
        if total == 0:
            continue
        c0 = -(-total // num_parts)
        cap = sp.choose_cap(nt, num_parts, F)
        assert c0 <= cap <= c0 + F

        def part_costs(sched):
            return [cost_of(sp.part_ranges(e, L), F) for e in sched]
        chosen = part_costs(sp.plan(L, num_parts, F)[0])
        plain = part_costs(_forced(L, num_parts, F, c0 + F)[0])
        assert max(chosen) <= max(plain)
        if cap < c0 + F:
            assert chosen[-1] <= cap
            # and no smaller cap in the range would do: its last part overflows
            for c in range(c0, cap):
                assert part_costs(_forced(L, num_parts, F, c)[0])[-1] > c


def test_plan_cap_by_hand():
    """Requests of 2, 1, 1, 1 tiles, 4 parts, F = 4: costs 6, 5, 5, 5, total 21,
    c0 = ceil(21 / 4) = 6.  Cap 6: part 0 takes request 0 (6, then 1 + 4 > 0
    left), parts 1 and 2 one request each, the last part request 3 (5 <= 6):
    cap 6 is chosen.  The plain cap c0 + F = 10 puts requests 1 and 2 in part 1
    (5 + 5) and leaves the last part empty."""
    L = [128, 64, 64, 64]
    assert sp.choose_cap([2, 1, 1, 1], 4, 4) == 6
    sched, off = sp.plan(L, 4, 4)
    assert sched == [(0, 0, 1, 0, 0, 0, 0, 0), (1, 0, 2, 0, 0, 0, 0, 0), (2, 0, 3, 0, 0, 0, 0, 0),
                     (3, 0, 4, 0, 0, 0, 0, 0)]
    assert off == [0, 1, 2, 3, 4]
    plain = _forced(L, 4, 4, 10)[0]
    assert [cost_of(sp.part_ranges(e, L), 4) for e in plain] == [6, 10, 5, 0]


def test_plan_single_request_long_context():
    sched, off = sp.plan([65536], 76, 4)
    rs = [sp.part_ranges(e, [65536]) for e in sched]
    sizes = [r[0][2] - r[0][1] for r in rs if r]
    assert sum(sizes) == 1024 and off[1] == len(sizes)
    assert max(sizes) - min(sizes[:-1]) <= 1 + 4


def test_plan_all_empty():
    sched, off = sp.plan([0, 0, 0], 5, 4)
    assert off == [0, 0, 0, 0]
    assert all(sp.part_ranges(e, [0, 0, 0]) == [] for e in sched)


# ---------------------------------------------------------------- request-local plan

@pytest.mark.parametrize("num_parts", [1, 5, 16, 38, 76, 152])
def test_request_local_plan_invariants(num_parts):
    rng = np.random.default_rng(num_parts + 7)
    for trial in range(40):
        B = int(rng.integers(1, 40))
        L = rng.integers(0, 5000, size=B)
        L[rng.random(B) < 0.15] = 0
        sched, off = sp.plan_request_local(L.tolist(), num_parts, 4)
        nt = [-(-int(x) // 64) for x in L]
        active = sum(1 for n in nt if n > 0)
        assert len(sched) == num_parts and len(off) == B + 1
        if active == 0 or active > num_parts:
            assert (sched, off) == sp.plan(L.tolist(), num_parts, 4)
            continue
        seen = {b: np.zeros(nt[b], int) for b in range(B)}
        per_unit = {b: [] for b in range(B)}
        for e in sched:
            rs = sp.part_ranges(e, L.tolist())
            assert len(rs) <= 1                      # no part spans two units
            for (b, t0, t1, s) in rs:
                seen[b][t0:t1] += 1
                per_unit[b].append((s, t1 - t0))
        for b in range(B):
            assert (seen[b] == 1).all()
            n = off[b + 1] - off[b]
            assert [s for s, _ in per_unit[b]] == list(range(n))
            if nt[b]:
                sizes = [z for _, z in per_unit[b]]
                assert 1 <= n <= nt[b] and max(sizes) - min(sizes) <= 1
            else:
                assert n == 0
        # every part is used unless a unit ran out of tiles to give
        used = off[-1]
        assert used == num_parts or any(off[b + 1] - off[b] == nt[b] for b in range(B) if nt[b])


def test_request_local_plan_by_hand():
    # 3 units with 10, 30, 0 and 20 tiles (64 keys each), 10 parts: 3 active, 7 spare;
    # quotas 10*7/60 = 1 r 10, 30*7/60 = 3 r 30, 20*7/60 = 2 r 20 -> 6 given, one more to the
    # largest remainder (unit 1): seats 2, 5, 0, 3.
    L = [640, 1920, 0, 1280]
    sched, off = sp.plan_request_local(L, 10, 4)
    assert off == [0, 2, 7, 7, 10]
    assert sched[:2] == [(0, 0, 0, 5, 0, 0, 0, 0), (0, 5, 1, 0, 1, 0, 0, 0)]
    assert [e[1] for e in sched[2:7]] == [0, 6, 12, 18, 24] and sched[6][2:4] == (2, 0)
    assert sched[7:] == [(3, 0, 3, 6, 0, 0, 0, 0), (3, 6, 3, 13, 1, 0, 0, 0), (3, 13, 4, 0, 2, 0, 0, 0)]
