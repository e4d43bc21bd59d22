"""CPU restatement of the split-KV partition plan (test infrastructure only).

FlashMLA PR #183 (*Add SM80 (Ampere/A100) dense MLA decode kernel*, section
*How the occupancy work went*) describes the scheduler this follows: the KV
work of the whole batch is cut into ``num_parts`` contiguous partitions, the
part count follows from how many CTAs (here: CTA pairs) actually fit on the
GPU, and every extra partition carries a fixed cost (Q reload, prologue and
epilogue, one more combine row).  The page gives no formula, so the plan
below is this library's own; it is written out plainly here so the GPU
metadata can be compared with it integer for integer.  It is additionally
pinned by invariants that do not depend on this code (every tile of every
request is covered exactly once; the split counts add up; no part exceeds
its budget except the last), see tests/test_sched.py.

Plan
----
Work unit = one request b with n_b = ceil(L_b / 64) tiles of 64 keys.
cost(b) = n_b + F for n_b > 0 (F = fixed cost of a split, in tiles).
Parts p = 0..P-1 take consecutive ranges of (request, tile) in order.  With
budget ``cap``, a part completes whole requests while remaining + F fits in
its budget, then takes ``budget - F`` tiles of the next request if that is
positive, and stops.  The last part takes everything left.  Requests with
n_b = 0 are skipped (they get 0 splits).
cap: with c0 = ceil(sum_b cost(b) / P), the smallest cap in c0 .. c0 + F
whose walk over parts 0..P-2 leaves the last part a cost (remaining tiles +
F per request touched) of at most cap; c0 + F if none does.  The search is
the library's only where it is cheap: at most SEARCH_MAX_UNITS requests, at
most SEARCH_MAX_PARTS parts, F <= SEARCH_MAX_F and c0 + F < 2^30; otherwise
cap = c0 + F.  (With c0 + F alone the walk often
finishes early and leaves the last parts empty: 2 of 76 parts idle for 64
requests of 2048-4096 keys.)

Metadata (int32):
  sched[p] = (begin_b, begin_t, end_b, end_t, begin_split, 0, 0, 0)
    part p covers tiles [begin_t, ...) of begin_b, whole requests in
    between, and tiles [0, end_t) of end_b (nothing of end_b if end_t = 0);
    begin_split = how many earlier parts touched begin_b.
  split_offset[B + 1]: prefix sum of per-request split counts.
"""

from __future__ import annotations

TILE = 64
SEARCH_MAX_UNITS = 4096
SEARCH_MAX_PARTS = 128
SEARCH_MAX_F = 4


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def leftover(nt, num_parts: int, fixed_cost: int, cap: int) -> int:
    """Cost left for the last part after parts 0..P-2 walk with budget cap."""
    B = len(nt)
    b, t = 0, 0
    for _ in range(num_parts - 1):
        budget = cap
        while b < B:
            if nt[b] == 0:
                b, t = b + 1, 0
                continue
            rem = nt[b] - t
            if rem + fixed_cost <= budget:
                budget -= rem + fixed_cost
                b, t = b + 1, 0
            else:
                take = budget - fixed_cost
                if take > 0:
                    t += take
                break
    return sum(nt[bb] - (t if bb == b else 0) + fixed_cost for bb in range(b, B) if nt[bb] > 0)


def choose_cap(nt, num_parts: int, fixed_cost: int) -> int:
    total = sum(n + fixed_cost for n in nt if n > 0)
    if total == 0:
        return 0
    c0 = ceil_div(total, num_parts)
    if (len(nt) <= SEARCH_MAX_UNITS and num_parts <= SEARCH_MAX_PARTS and fixed_cost <= SEARCH_MAX_F
            and c0 + fixed_cost < 2 ** 30):
        for cap in range(c0, c0 + fixed_cost + 1):
            if leftover(nt, num_parts, fixed_cost, cap) <= cap:
                return cap
    return c0 + fixed_cost


def plan(seqlens, num_parts: int, fixed_cost: int, tile: int = TILE):
    B = len(seqlens)
    nt = [ceil_div(max(int(L), 0), tile) for L in seqlens]
    cap = choose_cap(nt, num_parts, fixed_cost)
    touched = [0] * B
    sched = []
    b, t = 0, 0
    for p in range(num_parts):
        while b < B and nt[b] == 0:
            b, t = b + 1, 0
        begin = (b, t)
        begin_split = touched[b] if b < B else 0
        if p == num_parts - 1:
            b, t = B, 0
        else:
            budget = cap
            while b < B:
                if nt[b] == 0:
                    b, t = b + 1, 0
                    continue
                rem = nt[b] - t
                if rem + fixed_cost <= budget:
                    budget -= rem + fixed_cost
                    b, t = b + 1, 0
                else:
                    take = budget - fixed_cost
                    if take > 0:
                        t += take
                    break
        end = (b, t)
        # requests this part touches
        if begin != end:
            last = end[0] if end[1] > 0 else end[0] - 1
            for bb in range(begin[0], min(last, B - 1) + 1):
                if nt[bb] > 0:
                    touched[bb] += 1
        sched.append((begin[0], begin[1], end[0], end[1], begin_split, 0, 0, 0))
    split_offset = [0]
    for bb in range(B):
        split_offset.append(split_offset[-1] + touched[bb])
    return sched, split_offset


def part_ranges(entry, seqlens, tile: int = TILE):
    """Expand one sched entry into [(b, t0, t1, split_local), ...]."""
    b0, t0, b1, t1, s0 = entry[:5]
    nt = [ceil_div(max(int(L), 0), tile) for L in seqlens]
    out = []
    b = b0
    while b < len(seqlens) and (b < b1 or (b == b1 and t1 > 0)):
        lo = t0 if b == b0 else 0
        hi = t1 if b == b1 else nt[b]
        if hi > lo:
            out.append((b, lo, hi, s0 if b == b0 else 0))
        b += 1
    return out


def plan_request_local(seqlens, num_parts: int, fixed_cost: int, tile: int = TILE):
    """Request-local plan: no part spans two work units.

    FlashMLA PR #200 (*[SM90] Add packed selected-KV sparse decode*, section
    *Scheduler policy*) names a "compact request-local scheduler" for its
    H=64 path and says the native scheduler is kept where it measured faster;
    the page does not define it.  Reading taken here: every part works on the
    tiles of a single unit (query token), and the parts are shared out over
    the units in proportion to their tile counts:
      * units with n_b > 0 tiles: A of them; if A > P, or there are no tiles,
        the native plan above is used instead;
      * each active unit gets one part, and the other R = P - A parts go by
        largest remainder: q_b, r_b = divmod(n_b * R, sum n), one more part to
        the (R - sum q) units with the largest r_b (ties: lower b first);
      * a unit never gets more parts than tiles;
      * unit b's k-th of s_b parts covers tiles [k*n_b//s_b, (k+1)*n_b//s_b).
    Parts are numbered in unit order; unused parts are empty (B, 0, B, 0).
    Same metadata format as ``plan``.
    """
    B = len(seqlens)
    nt = [ceil_div(max(int(L), 0), tile) for L in seqlens]
    active = [b for b in range(B) if nt[b] > 0]
    if not active or len(active) > num_parts:
        return plan(seqlens, num_parts, fixed_cost, tile)
    total = sum(nt)
    spare = num_parts - len(active)
    seats = [0] * B
    remainders = []
    given = 0
    for b in active:
        q, r = divmod(nt[b] * spare, total)
        seats[b] = 1 + q
        given += q
        remainders.append((-r, b))
    for _, b in sorted(remainders)[:spare - given]:
        seats[b] += 1
    sched = []
    split_offset = [0]
    for b in range(B):
        s = min(seats[b], nt[b])
        for k in range(s):
            lo, hi = k * nt[b] // s, (k + 1) * nt[b] // s
            end_b, end_t = (b, hi) if hi < nt[b] else (b + 1, 0)
            sched.append((b, lo, end_b, end_t, k, 0, 0, 0))
        split_offset.append(split_offset[-1] + s)
    while len(sched) < num_parts:
        sched.append((B, 0, B, 0, 0, 0, 0, 0))
    return sched, split_offset
