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


def test_worked_example():
    g = _read_golden("plan_worked_example.txt")
    lens = [int(x) for x in g["seq_lens"]]
    policy = {"balanced": pl.BALANCED, "uniform": pl.UNIFORM}[g["policy"][0]]
    counts, work = pl.plan(lens, int(g["M"][0]), int(g["num_ctas"][0]),
                           int(g["min_split_tokens"][0]), int(g["max_splits"][0]), policy)
    assert counts.tolist() == [int(x) for x in g["counts"]]
    assert work.tolist() == [int(x) for x in g["work"]]


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


@pytest.mark.parametrize("seed", range(40))
def test_plan_properties(seed):
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 160))
    lens = _random_lengths(rng, R)
    M = int(rng.choice([1, 8, 32, 56, 64, 65, 256, 448]))
    G = int(rng.choice([1, 7, 148, 152, 304]))
    mst = int(rng.choice([64, 256, 1000]))
    ms = int(rng.choice([1, 3, 64, 4096]))
    for policy in (pl.BALANCED, pl.UNIFORM):
        counts, work = pl.plan(lens, M, G, mst, ms, policy)
        cap = pl.list_len(R, M, G, policy, ms)
        assert work.size == cap
        n = counts.astype(int)
        assert np.all(n >= 1) and np.all(n <= ms)
        items = work[work >= 0]
        assert items.size == n.sum() <= cap
        assert np.all(work[items.size:] == -1)          # -1 tail, no holes
        # rank order: longest first, ties to the lower index; splits ascending
        reqs = items >> pl.SPLIT_BITS
        order = pl.rank_order(lens)
        expect = [i for i in order for _ in range(n[i])]
        assert reqs.tolist() == expect
        assert (items & (pl.MAX_SPLITS_LIMIT - 1)).tolist() == [s for i in order for s in range(n[i])]
        # the splits of each request tile its keys exactly, page aligned
        for i, L in enumerate(lens):
            prev = 0
            for s in range(n[i]):
                j0, j1 = pl.split_range(int(L), int(n[i]), s)
                assert j0 == prev and j0 % 64 == 0 and j1 >= j0
                prev = j1
            assert prev == L
        # multi-split items come first and fit the partial slots
        multi = np.nonzero(n[reqs] >= 2)[0]
        if multi.size:
            assert multi.max() + 1 == multi.size
            assert multi.size <= pl.partial_slots(R, M, G, policy, ms)
        if policy == pl.UNIFORM:
            S = pl.uniform_splits(R, M, G, ms)
            p = -(-lens // 64)
            assert np.all(n[lens > 0] == np.minimum(S, p[lens > 0]))
        else:
            c = _chunk_brute(lens, M, G, mst, ms)
            p = -(-lens // 64)
            assert np.all(n[lens > 0] == np.minimum(-(-p[lens > 0] // c), ms))
            U = pl.units(M, G)
            if np.count_nonzero(lens) <= U:
                assert n[lens > 0].sum() <= U            # one wave


def test_empty_and_degenerate():
    counts, work = pl.plan([0, 0, 0], 32, 152, 256, 64, pl.BALANCED)
    assert counts.tolist() == [1, 1, 1]
    assert work[:3].tolist() == [0, 1 << 12, 2 << 12]
    counts, work = pl.plan([1], 1, 1, 64, 64, pl.BALANCED)
    assert counts.tolist() == [1] and work.tolist() == [0, -1]
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
