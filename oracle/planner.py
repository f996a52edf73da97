"""Integer split planner: per-request split counts and the work list.

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
  targets U = max(1, num_ctas // nb) concurrent work items.
* balanced: c0 = max(minp, ceil(T / U)) pages per split, minp =
  ceil(min_split_tokens / 64). If every non-empty request fits in one wave
  (Rn <= U) the chunk c is the smallest c >= c0 whose item count
  sum_i min(ceil(p_i / c), max_splits) is at most U (one wave, the smallest
  largest item); otherwise c = c0. n_i = min(ceil(p_i / c), max_splits).
* uniform: S = clamp(ceil(U / R), 1, max_splits) for every request,
  n_i = min(S, p_i).
* an empty request gets one (empty) split in both policies.
* split s of request i covers pages [floor(s p_i / n_i), floor((s+1) p_i / n_i)),
  i.e. keys [64 p0, min(len_i, 64 p1)).
* work list: requests in rank order (length descending, ties to the lower
  index), each request's splits in ascending s, entry (i << 12) | s, the rest
  -1. Because n_i never decreases with the length, every multi-split item sits
  before every single-split item; a multi-split item's partial slot is its
  list index.
"""
from __future__ import annotations

import numpy as np

PAGE = 64
BALANCED, UNIFORM = 0, 1
SPLIT_BITS = 12
MAX_SPLITS_LIMIT = 1 << SPLIT_BITS


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


def list_len(R: int, M: int, num_ctas: int, policy: int, max_splits: int) -> int:
    """Work-list capacity that every length vector of R requests fits in."""
    if policy == BALANCED:
        return units(M, num_ctas) + R
    return R * uniform_splits(R, M, num_ctas, max_splits)


def partial_slots(R: int, M: int, num_ctas: int, policy: int, max_splits: int) -> int:
    """Upper bound on multi-split items (the only ones that write partials)."""
    if policy == BALANCED:
        return min(list_len(R, M, num_ctas, policy, max_splits), 2 * units(M, num_ctas))
    s = uniform_splits(R, M, num_ctas, max_splits)
    return R * s if s >= 2 else 0


def split_counts(seq_lens, M: int, num_ctas: int, min_split_tokens: int, max_splits: int,
                 policy: int) -> np.ndarray:
    lens = [int(x) for x in np.asarray(seq_lens).ravel()]
    R = len(lens)
    p = [cdiv(L, PAGE) for L in lens]
    U = units(M, num_ctas)
    if policy == UNIFORM:
        S = uniform_splits(R, M, num_ctas, max_splits)
        return np.array([1 if L == 0 else min(S, pi) for L, pi in zip(lens, p)], dtype=np.int32)
    T = sum(p)
    Rn = sum(1 for L in lens if L > 0)
    minp = max(1, cdiv(min_split_tokens, PAGE))
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
    return np.array([1 if pi == 0 else min(cdiv(pi, c), max_splits) for pi in p], dtype=np.int32)


def rank_order(seq_lens) -> list[int]:
    """Request indices, longest first, ties to the lower index."""
    lens = [int(x) for x in np.asarray(seq_lens).ravel()]
    return sorted(range(len(lens)), key=lambda i: (-lens[i], i))


def plan(seq_lens, M: int, num_ctas: int, min_split_tokens: int, max_splits: int,
         policy: int, capacity: int | None = None):
    """-> (counts [R] int32, work [capacity] int32)."""
    lens = np.asarray(seq_lens).ravel()
    R = lens.size
    if capacity is None:
        capacity = list_len(R, M, num_ctas, policy, max_splits)
    counts = split_counts(lens, M, num_ctas, min_split_tokens, max_splits, policy)
    work = []
    for i in rank_order(lens):
        for s in range(int(counts[i])):
            work.append((i << SPLIT_BITS) | s)
    if len(work) > capacity:
        raise ValueError("work list longer than its capacity")
    out = np.full(capacity, -1, dtype=np.int32)
    out[: len(work)] = np.array(work, dtype=np.int64).astype(np.int32)
    return counts, out


def fold_factor(k: int, heads: int, max_heads: int = 128) -> int:
    """Query tokens folded into one decode row when a row may hold at most
    `max_heads` heads: the largest divisor of k whose heads fit
    (drafter-attention page, `fold_plan`, the LSE-returning route; 1 if even a
    single token's heads do not fit)."""
    fits = [d for d in range(1, k + 1) if k % d == 0 and d * heads <= max_heads]
    return max(fits) if fits else 1


def split_range(length: int, n: int, s: int) -> tuple[int, int]:
    """Keys [j0, j1) of split s of n of a request of ``length`` keys."""
    p = cdiv(length, PAGE)
    p0 = (s * p) // n
    p1 = ((s + 1) * p) // n
    return PAGE * p0, min(length, PAGE * p1)
