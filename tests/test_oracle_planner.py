"""The integer split planner against its worked example, brute force and
properties (no GPU)."""
import os

import numpy as np
import pytest

from oracle import planner as pl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        vals[key] = rest
    return vals


def _golden_words(vals):
    out = []
    for tok in vals:
        if "x" in tok:                       # "-1 x64": the value, repeated
            continue
        out.append(int(tok))
    if vals and "x" in vals[-1]:
        out += [out[-1]] * (int(vals[-1][1:]) - 1)
    return out


@pytest.mark.parametrize("name", ["plan_worked_example.txt", "plan_packed_example.txt"])
def test_worked_examples(name):
    g = _read_golden(name)
    lens = [int(x) for x in g["seq_lens"]]
    M, G = int(g["M"][0]), int(g["num_ctas"][0])
    mst, ms = int(g["min_split_tokens"][0]), int(g["max_splits"][0])
    policy = {"balanced": pl.BALANCED, "uniform": pl.UNIFORM}[g["policy"][0]]
    counts, buf = pl.plan(lens, M, G, mst, ms, policy)
    want = sum((_golden_words(g[k]) for k in ("entries", "counters", "ranges", "units")), [])
    assert counts.tolist() == [int(x) for x in g["counts"]]
    assert buf.tolist() == want


def _count(p, c, max_splits):
    return sum(min(-(-x // c), max_splits) for x in p if x > 0)


def _chunk_brute(lens, M, G, minp_tokens, max_splits):
    """Linear scan for the balanced chunk: the plain statement of the rule."""
    p = [-(-L // 64) for L in lens]
    U = pl.units(M, G)
    minp = max(1, -(-minp_tokens // 64))
    c0 = max(minp, -(-sum(p) // U))
    Rn = sum(1 for L in lens if L > 0)
    if Rn <= U and _count(p, c0, max_splits) > U:
        c = c0
        while _count(p, c, max_splits) > U:
            c += 1
        return c
    return c0


def _random_lengths(rng, R):
    kind = rng.integers(0, 4)
    if kind == 0:
        return rng.integers(0, 9000, size=R)
    if kind == 1:
        return np.clip(np.round(np.exp(rng.normal(np.log(2048), 1.0, size=R))), 0, 40000).astype(int)
    if kind == 2:
        lens = rng.integers(1, 600, size=R)
        lens[rng.integers(0, R)] = rng.integers(10000, 140000)
        return lens
    return rng.integers(0, 3, size=R) * rng.integers(0, 70, size=R)


def _unpack(buf, R, M, G, policy, ms):
    E, off_rng, off_unit = pl.regions(R, M, G, policy, ms)
    U = pl.units(M, G)
    entries = buf[:E]
    rng = buf[off_rng:off_rng + 2 * E].reshape(E, 2)
    table = buf[off_unit:off_unit + pl.UNIT_SLOTS * U].reshape(pl.UNIT_SLOTS, U).T   # [unit, slot]
    return E, entries, rng, table


@pytest.mark.parametrize("seed", range(60))
def test_plan_properties(seed):
    rng_ = np.random.default_rng(seed)
    R = int(rng_.integers(1, 160))
    lens = _random_lengths(rng_, R)
    M = int(rng_.choice([1, 8, 32, 56, 64, 65, 256, 448]))
    G = int(rng_.choice([1, 7, 16, 148, 152, 304]))
    mst = int(rng_.choice([64, 256, 1000]))
    ms = int(rng_.choice([1, 3, 64, 4096]))
    p = -(-lens // 64)
    U = pl.units(M, G)
    for policy in (pl.BALANCED, pl.UNIFORM):
        counts, buf = pl.plan(lens, M, G, mst, ms, policy)
        assert buf.size == pl.list_len(R, M, G, policy, ms)
        E, entries, rng, table = _unpack(buf, R, M, G, policy, ms)
        assert np.all(buf[E:E + pl.SCHED_WORDS] == -1)
        n = counts.astype(int)
        assert np.all(n >= 1) and np.all(n <= ms)
        items = entries[entries >= 0]
        k = items.size
        assert k == n.sum() <= E
        assert np.all(entries[k:] == -1)                # -1 tail, no holes
        assert np.all(rng[k:] == -1)
        # multi-piece requests first, then the rest, each in rank order;
        # pieces ascending; multi-piece entries fit the partial slots
        packed = bool(table[0, 0] >= 0)
        assert np.all((items & pl.PACKED_BIT) == (pl.PACKED_BIT if packed else 0))
        reqs = (items & ~pl.PACKED_BIT) >> pl.SPLIT_BITS
        order = pl.rank_order(lens)
        listed = [i for i in order if n[i] >= 2] + [i for i in order if n[i] < 2]
        assert reqs.tolist() == [i for i in listed for _ in range(n[i])]
        assert (items & (pl.MAX_SPLITS_LIMIT - 1)).tolist() == [s for i in listed
                                                                 for s in range(n[i])]
        nmulti = int(sum(n[i] for i in range(R) if n[i] >= 2))
        assert nmulti <= pl.partial_slots(R, M, G, policy, ms)
        # each request's pieces tile its pages exactly
        first = {}
        for e in range(k):
            first.setdefault(int(reqs[e]), e)
        for i in range(R):
            e0 = first[i]
            prev = 0
            for s in range(n[i]):
                j0, j1 = pl.entry_keys(buf, counts, e0 + s, int(lens[i]), R, M, G, policy, ms)
                assert j0 == min(prev, int(lens[i])) and j1 >= j0 and j0 % 64 == 0
                prev = j1 if j1 < lens[i] else 64 * p[i]
                if packed:
                    assert tuple(rng[e0 + s]) == (j0 // 64, -(-j1 // 64))
            assert prev == 64 * p[i]
        if policy == pl.UNIFORM:
            S = pl.uniform_splits(R, M, G, ms)
            assert not packed
            assert np.all(n[lens > 0] == np.minimum(S, p[lens > 0]))
            continue
        c = _chunk_brute(lens, M, G, mst, ms)
        n_req = np.where(p > 0, np.minimum(-(-p // c), ms), 1)
        minp = max(1, -(-mst // 64))
        c0 = max(minp, -(-int(p.sum()) // U))
        Rn = int(np.count_nonzero(lens))
        big = max([-(-int(pi) // int(ni)) for pi, ni in zip(p, n_req) if pi > 0], default=0)
        J = pl.JOB_PAGES
        wants = (p.sum() > 0 and pl.row_blocks(M) >= 2 and R <= U <= pl.MAX_PACKED_UNITS
                 and 8 * (c0 + 2 * J) <= 7 * (big + J))
        if not wants:
            assert not packed                            # the cost test comes on top
        if not packed:
            # the per-request plan: equal page-aligned splits
            assert np.all(n == n_req)
            for i in range(R):
                for s in range(n[i]):
                    j0, _ = pl.entry_keys(buf, counts, first[i] + s, int(lens[i]), R, M, G,
                                          policy, ms)
                    assert j0 == min(64 * ((s * p[i]) // n[i]), int(lens[i]))
            if Rn <= U:
                assert n[lens > 0].sum() <= U            # one wave
            continue
        # packed: every unit's pieces, in its table, cover its c0-page segment
        # of the rank-ordered pages, in order; empty requests add empty pieces
        assert wants
        where = np.zeros(E, dtype=int) - 1
        for u in range(U):
            row = table[u]
            got = row[row >= 0]
            assert np.all(row[got.size:] == -1) and got.size <= pl.UNIT_SLOTS
            where[got] = u
            pages = int(sum(rng[e][1] - rng[e][0] for e in got))
            assert pages == max(0, min(c0, int(p.sum()) - u * c0))
        assert np.all(where[:k] >= 0)                     # every entry has a unit
        pos = 0
        for i in order:
            for s in range(n[i]):
                e = first[i] + s
                a, b = rng[e]
                if p[i] > 0:
                    assert where[e] == (pos + a) // c0 and (pos + b - 1) // c0 == where[e]
            pos += int(p[i])


@pytest.mark.parametrize("seed", range(30))
def test_packed_plans_balance_one_wave_batches(seed):
    """Batches of at most U requests: the plan is packed exactly when items
    have several row blocks and
    c0 + 2 JOB_PAGES and the packing's costliest unit (its pages plus
    JOB_PAGES per piece) both come to at most 7/8 of the per-request plan's
    largest item plus JOB_PAGES (and the packing fits its limits); then every
    unit holds the pages of its segment, at most c0. Brute force over the
    rank-ordered pages, against the per-request chunk found by linear scan."""
    rng_ = np.random.default_rng(1000 + seed)
    G = int(rng_.choice([16, 64, 152]))
    M = int(rng_.choice([32, 56, 256, 448]))
    U = pl.units(M, G)
    R = int(rng_.integers(1, U + 1))
    lens = rng_.integers(256, 70000, size=R)
    counts, buf = pl.plan(lens, M, G, 64, 64, pl.BALANCED)
    E, entries, rng, table = _unpack(buf, R, M, G, pl.BALANCED, 64)
    p = -(-lens // 64)
    T = int(p.sum())
    c0 = max(1, -(-T // U))
    c = _chunk_brute(lens, M, G, 64, 64)
    largest = int(max(-(-pi // min(-(-pi // c), 64)) for pi in p))
    starts = np.concatenate([[0], np.cumsum(p[pl.rank_order(lens)])])
    nseg = -(-T // c0)
    per_req = [(s1 - 1) // c0 - s0 // c0 + 1 for s0, s1 in zip(starts[:-1], starts[1:])]
    per_unit = [sum(1 for s0, s1 in zip(starts[:-1], starts[1:])
                    if s0 < (u + 1) * c0 and s1 > u * c0) for u in range(nseg)]
    cost = max(min(c0, T - u * c0) + pl.JOB_PAGES * per_unit[u] for u in range(nseg))
    J = pl.JOB_PAGES
    wants = (pl.row_blocks(M) >= 2 and 8 * (c0 + 2 * J) <= 7 * (largest + J) and max(per_req) <= 64
             and max(per_unit) <= pl.UNIT_SLOTS and 8 * cost <= 7 * (largest + J))
    assert bool(np.any(table >= 0)) == wants
    if wants:
        loads = [int(sum(rng[e][1] - rng[e][0] for e in row[row >= 0])) for row in table]
        assert loads == [max(0, min(c0, T - u * c0)) for u in range(U)]
        assert [int((row >= 0).sum()) for row in table[:nseg]] == per_unit


def test_packed_plan_places_empty_requests():
    """A packed plan gives the k-th empty request (in rank order, that is by
    index) one empty piece in unit k mod (number of segments), after that
    unit's non-empty pieces."""
    lens = [0, 13474, 4345, 6990, 0, 0, 3742, 4383]
    M, G = 256, 44                              # four 64-row blocks, U = 11
    counts, buf = pl.plan(lens, M, G, 64, 64, pl.BALANCED)
    E, entries, rng, table = _unpack(buf, len(lens), M, G, pl.BALANCED, 64)
    assert int(entries[0]) & pl.PACKED_BIT
    p = [-(-L // 64) for L in lens]
    c0 = -(-sum(p) // pl.units(M, G))
    nseg = -(-sum(p) // c0)
    empties = [0, 4, 5]
    for k, i in enumerate(empties):
        e = [j for j in range(E) if entries[j] >= 0 and pl.entry_request(entries[j]) == i]
        assert len(e) == 1 and tuple(rng[e[0]]) == (0, 0)
        row = [x for x in table[k % nseg] if x >= 0]
        slot = row.index(e[0])
        assert all(pl.entry_request(entries[x]) not in empties for x in row[:slot])
        assert all(pl.entry_request(entries[x]) in empties for x in row[slot:])


def test_packing_cost_keeps_the_per_request_plan():
    """The unit cost decides: nine requests of 1021 .. 5808 keys, M = 128 (two
    row blocks), 29 CTAs: U = 14, pages 16 28 48 91 89 12 63 76 46 (T = 469),
    c0 = 34; the per-request plan's largest item is 46 pages, so
    8 (c0 + 2 J) = 336 <= 7 (46 + J) = 350 lets packing be tried, but segment
    12 ([408, 442), full) would hold three pieces: cost >= 34 + 3 J = 46 and
    8 * 46 = 368 > 350, so the per-request plan stands."""
    lens = [1021, 1786, 3049, 5808, 5645, 717, 3996, 4808, 2938]
    assert pl.JOB_PAGES == 4
    _, packed = pl.plan_pieces(lens, 128, 29, 64, 64, pl.BALANCED)
    assert not packed
    counts, buf = pl.plan(lens, 128, 29, 64, 64, pl.BALANCED)
    assert not int(buf[0]) & pl.PACKED_BIT


def test_empty_and_degenerate():
    counts, work = pl.plan([0, 0, 0], 32, 152, 256, 64, pl.BALANCED)
    assert counts.tolist() == [1, 1, 1]
    assert work[:3].tolist() == [0, 1 << 12, 2 << 12]
    counts, work = pl.plan([1], 1, 1, 64, 64, pl.BALANCED)
    # E = 2 entries, 2 counters, 4 range words, 8 unit-table words (not packed)
    assert counts.tolist() == [1] and work.tolist() == [0] + [-1] * 15
    # max_splits = 1 never splits
    counts, _ = pl.plan([100000, 5], 32, 152, 64, 1, pl.BALANCED)
    assert counts.tolist() == [1, 1]


def test_skewed_batch_balances_better_than_uniform():
    """A 128k request among short ones: balanced splits it, uniform cannot."""
    lens = [131072] + [32768] * 7 + [2000] * 120
    cb, _ = pl.plan(lens, 448, 152, 256, 64, pl.BALANCED)
    cu, _ = pl.plan(lens, 448, 152, 256, 64, pl.UNIFORM)
    p = -(-np.array(lens) // 64)
    largest_b = max(-(-p // cb))
    largest_u = max(-(-p // cu))
    assert largest_u >= 1.5 * largest_b


def test_fold_factor_worked_example():
    """The pages' example: k = 4 at 64 heads with a 128-head cap folds pairs."""
    for line in open(os.path.join(GOLDEN, "fold_plan_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, H, cap, want = (int(x) for x in line.split())
        assert pl.fold_factor(k, H, cap) == want


@pytest.mark.parametrize("k", range(1, 13))
@pytest.mark.parametrize("H", [1, 8, 16, 64, 96, 128, 200])
def test_fold_factor_properties(k, H):
    f = pl.fold_factor(k, H, 128)
    assert k % f == 0
    assert f == 1 or f * H <= 128
    assert all(not (k % d == 0 and d * H <= 128) for d in range(f + 1, k + 1))
