"""Integer split planner: per-request split counts and the plan buffer.

Test infrastructure only (see the package docstring). The device planner
kernel must reproduce these outputs bit for bit.

What the pages fix (balanced-MLA page, module overview and ``BalancedMla``):
a small device kernel turns each request's KV length into a split count and a
work list, once per decode step, reused by every layer; the list buffer is
pre-filled with -1; "balanced" plans per request from the lengths, while the
uniform (tokenspeed) schedule gives every request the same number of chunks,
fixed by the batch shape. The drafter-attention page's ``_plan_kernel`` ranks
requests longest first, ties to the lower row. The pages do not give the
formula; the one below is this project's reading:

* pages p_i = ceil(len_i / 64); T = sum p_i; Rn = number of non-empty requests.
* A request's M = k*H query rows are processed in row blocks of NR rows
  (NR = 32 when M <= 32, else 64), nb = ceil(M / NR) jobs per item. The plan
  targets U = max(1, num_ctas // nb) concurrent work items (units).
* balanced: c0 = max(minp, ceil(T / U)) pages per split, minp =
  ceil(min_split_tokens / 64). If every non-empty request fits in one wave
  (Rn <= U) the chunk c is the smallest c >= c0 whose item count
  sum_i min(ceil(p_i / c), max_splits) is at most U (one wave, the smallest
  largest item); otherwise c = c0. n_i = min(ceil(p_i / c), max_splits);
  split s of request i covers pages [floor(s p_i / n_i), floor((s+1) p_i / n_i)).
* balanced, packed: when items have several row blocks (nb >= 2: long,
  tensor-bound jobs, for which a piece's own overhead is small) and there are
  at most U requests (empty ones included: the decode launch then knows from
  the shape that the plan may be packed), with big = max_i ceil(p_i / n_i)
  (that plan's largest item, in pages) and each piece charged J = JOB_PAGES
  pages of overhead (its query load and epilogue), if
  8 (c0 + 2 J) <= 7 (big + J) (a unit holding the end of one request and the
  start of the next costs c0 + 2 J) and U <= MAX_PACKED_UNITS, the requests'
  pages are laid end to end in rank order and cut into segments of c0 pages;
  unit u processes the pieces of segment u in order. n_i = number of segments
  request i overlaps; an empty request is one empty piece, given to unit (its
  index among the empty requests) mod (number of segments). The packed plan is
  used if its costliest unit, max_u (pages of segment u + J * pieces of u),
  is at most 7/8 of big + J, every n_i <= max_splits and no unit holds more
  than UNIT_SLOTS pieces; otherwise the per-request plan stands.
* uniform: S = clamp(ceil(U / R), 1, max_splits) for every request,
  n_i = min(S, p_i), equal splits as above.
* an empty request gets one (empty) split in every mode.

The plan buffer (int32, ``list_len`` entries):

* entries [0, E): requests with two or more pieces first, then the others,
  each group in rank order (length descending, ties to the lower index), each
  request's pieces in ascending s; entry (i << 12) | s, with bit 30 set in
  every entry of a packed plan; the rest -1. A multi-piece entry's partial
  slot is its index. (In the per-request plans n_i never decreases with the
  length, so this is plain rank order.)
* [E, E + 2): two words the decode uses as job counters, -1.
* ranges [E + 2, 3E + 2), packed plans: entry e's first and end page within
  its request, at E + 2 + 2e and E + 3 + 2e; -1 past the entries.
* units [3E + 2, 3E + 2 + UNIT_SLOTS * U), packed plans: unit u's pieces
  (entry indices) in order, slot-major: its j-th at j * U + u, -1 padded.
* When the plan is not packed its pieces are the equal splits above and the
  ranges and the unit table are not used: the device planner leaves them as
  they were, this planner writes -1 there.

E = U + R for balanced, R * S for uniform.
"""
from __future__ import annotations

import numpy as np

PAGE = 64
BALANCED, UNIFORM = 0, 1
SPLIT_BITS = 12
MAX_SPLITS_LIMIT = 1 << SPLIT_BITS
PACKED_BIT = 1 << 30     # set in every entry of a packed plan
SCHED_WORDS = 2          # the decode's job counters after the entries
UNIT_SLOTS = 8           # pieces a unit of a packed plan may hold
MAX_PACKED_UNITS = 1024  # the device planner's per-unit tables
JOB_PAGES = 4            # overhead charged per piece of a packed plan, in pages


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


def row_block(M: int) -> int:
    return 32 if M <= 32 else 64


def row_blocks(M: int) -> int:
    """Jobs a work item is processed as: blocks of the request's M query rows."""
    return cdiv(M, row_block(M))


def units(M: int, num_ctas: int) -> int:
    return max(1, num_ctas // row_blocks(M))


def uniform_splits(R: int, M: int, num_ctas: int, max_splits: int) -> int:
    return min(max(1, cdiv(units(M, num_ctas), max(R, 1))), max_splits)


def items_len(R: int, M: int, num_ctas: int, policy: int, max_splits: int) -> int:
    """Entry capacity E that every length vector of R requests fits in."""
    if policy == BALANCED:
        return units(M, num_ctas) + R
    return R * uniform_splits(R, M, num_ctas, max_splits)


def list_len(R: int, M: int, num_ctas: int, policy: int, max_splits: int) -> int:
    """Length of the whole plan buffer (entries, counters, ranges, units)."""
    E = items_len(R, M, num_ctas, policy, max_splits)
    return 3 * E + SCHED_WORDS + UNIT_SLOTS * units(M, num_ctas)


def regions(R: int, M: int, num_ctas: int, policy: int, max_splits: int):
    """(E, offset of the ranges, offset of the unit table) in the buffer."""
    E = items_len(R, M, num_ctas, policy, max_splits)
    return E, E + SCHED_WORDS, 3 * E + SCHED_WORDS


def partial_slots(R: int, M: int, num_ctas: int, policy: int, max_splits: int) -> int:
    """Upper bound on multi-piece entries (the only ones that write partials).
    Per-request plans: a multi-split request has more than c0 pages, so fewer
    than U of them, and sum ceil(p_i / c) <= U + their count. Packed: a
    request with b_i >= 1 segment cuts inside has b_i + 1 <= 2 b_i pieces,
    and there are at most U - 1 cuts."""
    if policy == BALANCED:
        return min(items_len(R, M, num_ctas, policy, max_splits), 2 * units(M, num_ctas))
    s = uniform_splits(R, M, num_ctas, max_splits)
    return R * s if s >= 2 else 0


def rank_order(seq_lens) -> list[int]:
    """Request indices, longest first, ties to the lower index."""
    lens = [int(x) for x in np.asarray(seq_lens).ravel()]
    return sorted(range(len(lens)), key=lambda i: (-lens[i], i))


def _per_request_counts(p, R, M, num_ctas, minp, max_splits, policy):
    """n_i of the balanced (one-wave or not) or the uniform plan."""
    U = units(M, num_ctas)
    if policy == UNIFORM:
        S = uniform_splits(R, M, num_ctas, max_splits)
        return [1 if pi == 0 else min(S, pi) for pi in p]
    T = sum(p)
    Rn = sum(1 for pi in p if pi > 0)
    c = max(minp, cdiv(T, U))

    def count(cc: int) -> int:
        return sum(min(cdiv(pi, cc), max_splits) for pi in p if pi > 0)

    if Rn <= U and count(c) > U:
        lo, hi = c + 1, max(p)              # count(hi) = Rn <= U
        while lo < hi:
            mid = (lo + hi) // 2
            if count(mid) <= U:
                hi = mid
            else:
                lo = mid + 1
        c = lo
    return [1 if pi == 0 else min(cdiv(pi, c), max_splits) for pi in p]


def _packed(p, order, U, c0, max_splits, big):
    """Pieces of the packed plan: per request a list of (unit, first, end)
    pages within the request, or None when it does not apply or gains too
    little over the per-request plan's largest item ``big``."""
    T = sum(p)
    nseg = cdiv(T, c0)
    pieces = {}
    per_unit = [0] * U
    P = 0
    n_empty = 0
    for i in order:
        if p[i] == 0:
            u = n_empty % nseg
            n_empty += 1
            pieces[i] = [(u, 0, 0)]
            per_unit[u] += 1
            continue
        u0, u1 = P // c0, (P + p[i] - 1) // c0
        lst = []
        for u in range(u0, u1 + 1):
            a = max(P, u * c0) - P
            b = min(P + p[i], (u + 1) * c0) - P
            lst.append((u, a, b))
            per_unit[u] += 1
        pieces[i] = lst
        P += p[i]
    if max(len(v) for v in pieces.values()) > max_splits or max(per_unit) > UNIT_SLOTS:
        return None
    cost = max(min(c0, T - u * c0) + JOB_PAGES * per_unit[u] for u in range(nseg))
    if 8 * cost > 7 * (big + JOB_PAGES):
        return None
    return pieces


def plan_pieces(seq_lens, M: int, num_ctas: int, min_split_tokens: int, max_splits: int,
                policy: int):
    """-> (pieces per request: list of (unit or -1, first page, end page),
    packed flag). The decision rule of the module docstring."""
    lens = [max(0, int(x)) for x in np.asarray(seq_lens).ravel()]
    R = len(lens)
    p = [cdiv(L, PAGE) for L in lens]
    U = units(M, num_ctas)
    minp = max(1, cdiv(min_split_tokens, PAGE))
    n = _per_request_counts(p, R, M, num_ctas, minp, max_splits, policy)
    order = rank_order(lens)
    if policy == BALANCED:
        T = sum(p)
        Rn = sum(1 for pi in p if pi > 0)
        c0 = max(minp, cdiv(T, U))
        big = max([cdiv(pi, ni) for pi, ni in zip(p, n) if pi > 0], default=0)
        if T > 0 and row_blocks(M) >= 2 and R <= U <= MAX_PACKED_UNITS and \
                8 * (c0 + 2 * JOB_PAGES) <= 7 * (big + JOB_PAGES):
            packed = _packed(p, order, U, c0, max_splits, big)
            if packed is not None:
                return [packed[i] for i in range(R)], True
    out = []
    for i in range(R):
        out.append([(-1, (s * p[i]) // n[i], ((s + 1) * p[i]) // n[i]) for s in range(n[i])])
    return out, False


def plan(seq_lens, M: int, num_ctas: int, min_split_tokens: int, max_splits: int,
         policy: int, capacity: int | None = None):
    """-> (counts [R] int32, plan buffer [capacity] int32)."""
    lens = [max(0, int(x)) for x in np.asarray(seq_lens).ravel()]
    R = len(lens)
    E, off_rng, off_unit = regions(R, M, num_ctas, policy, max_splits)
    need = list_len(R, M, num_ctas, policy, max_splits)
    if capacity is None:
        capacity = need
    if capacity < need:
        raise ValueError("plan buffer shorter than the plan needs")
    pieces, packed = plan_pieces(lens, M, num_ctas, min_split_tokens, max_splits, policy)
    counts = np.array([len(v) for v in pieces], dtype=np.int32)
    order = rank_order(lens)
    listed = [i for i in order if counts[i] >= 2] + [i for i in order if counts[i] < 2]
    buf = np.full(capacity, -1, dtype=np.int64)
    e = 0
    unit_fill = [0] * units(M, num_ctas)
    where = {}
    for i in listed:
        for s, (u, a, b) in enumerate(pieces[i]):
            if e >= E:
                raise ValueError("more entries than the entry capacity")
            buf[e] = (PACKED_BIT if packed else 0) | (i << SPLIT_BITS) | s
            buf[off_rng + 2 * e] = a
            buf[off_rng + 2 * e + 1] = b
            where[(i, s)] = e
            e += 1
    if not packed:
        buf[off_rng:] = -1                   # only the entries and counters are defined
    else:
        # Each unit's pieces in segment order: the requests in rank order
        # (every empty request after the non-empty ones).
        for i in order:
            for s, (u, _, _) in enumerate(pieces[i]):
                buf[off_unit + unit_fill[u] * units(M, num_ctas) + u] = where[(i, s)]
                unit_fill[u] += 1
    return counts, buf.astype(np.int32)


def entry_request(w: int) -> int:
    return (int(w) & ~PACKED_BIT) >> SPLIT_BITS


def entry_split(w: int) -> int:
    return int(w) & (MAX_SPLITS_LIMIT - 1)


def entry_keys(buf, counts, e: int, length: int, R: int, M: int, num_ctas: int,
               policy: int, max_splits: int) -> tuple[int, int]:
    """Keys [j0, j1) of entry e of a plan buffer for a request of ``length``
    keys: from the ranges in a packed plan, else the equal split."""
    _, off_rng, _ = regions(R, M, num_ctas, policy, max_splits)
    if int(buf[e]) & PACKED_BIT:
        a, b = int(buf[off_rng + 2 * e]), int(buf[off_rng + 2 * e + 1])
        return PAGE * a, min(int(length), PAGE * b)
    return split_range(int(length), int(counts[entry_request(buf[e])]), entry_split(buf[e]))


def fold_factor(k: int, heads: int, max_heads: int = 128) -> int:
    """Query tokens folded into one decode row when a row may hold at most
    `max_heads` heads: the largest divisor of k whose heads fit
    (drafter-attention page, `fold_plan`, the LSE-returning route; 1 if even a
    single token's heads do not fit)."""
    fits = [d for d in range(1, k + 1) if k % d == 0 and d * heads <= max_heads]
    return max(fits) if fits else 1


def split_range(length: int, n: int, s: int) -> tuple[int, int]:
    """Keys [j0, j1) of split s of n equal splits of a request of ``length``
    keys (the per-request plans)."""
    p = cdiv(length, PAGE)
    p0 = (s * p) // n
    p1 = ((s + 1) * p) // n
    return PAGE * p0, min(length, PAGE * p1)
