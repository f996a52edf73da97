"""The tiered launch's host rules (drafter-attention page, `balanced_tiers`,
`_balanced_tables`, `_plan_kernel`) against a worked example, the pages'
stated cut-offs and properties; the binding's host copy of `balanced_tiers`
against the oracle's. No GPU."""
import os

import numpy as np
import pytest

import mla_decode_attention_folded_gb300 as mla
from oracle import tiers as ot

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tier_worked_example.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        key, *rest = line.split()
        vals[key] = [int(x) for x in rest]
    return vals


def test_worked_example():
    g = _golden()
    rest, rows, lens = ot.tier_tables(g["seq_lens"], g["split_rows"][0], g["pairs"][0],
                                      tuple(g["move"]))
    assert rest == g["rest_lens"] and rows == g["tier_rows"] and lens == g["tier_lens"]


def test_balanced_tiers_cutoffs():
    # the pages: no tiers while rows * 4 <= SMs; at least half the rows unsplit
    assert ot.balanced_tiers(38, 152) == ()
    assert ot.balanced_tiers(39, 152) == (8,)          # 39 // 2 = 19: 8 fits, 8 + 16 not
    assert ot.balanced_tiers(32, 100) == (8,)          # 32 // 2 = 16: 8 + 16 > 16
    assert ot.balanced_tiers(48, 100) == (8, 16)       # 8 + 16 = 24 <= 24
    assert ot.balanced_tiers(64, 152) == (8, 16)
    assert ot.balanced_tiers(128, 152) == (8, 16, 32)
    assert ot.balanced_tiers(1024, 152) == (8, 16, 32)
    for rows in range(1, 300):
        t = ot.balanced_tiers(rows, 152)
        assert sum(t) <= rows // 2
        if rows * 4 <= 152:
            assert t == ()


def test_binding_rule_matches_oracle():
    for sms in (8, 32, 148, 152):
        for rows in range(1, 400):
            assert mla.balanced_tiers(rows, sms) == ot.balanced_tiers(rows, sms), (rows, sms)
    assert mla.TIERS == ot.TIERS and mla.MOVE == ot.MOVE


@pytest.mark.parametrize("seed", range(20))
def test_tier_tables_properties(seed):
    rng = np.random.default_rng(seed)
    rows = int(rng.integers(1, 200))
    lens = rng.integers(0, 5000, size=rows)
    lens[rng.random(rows) < 0.2] = 777                   # ties
    split_rows = int(rng.integers(0, rows + 1))
    pairs = int(rng.integers(1, 100))
    rest, trows, tlens = ot.tier_tables(lens, split_rows, pairs)
    total = int(lens.sum())
    moved = [r for r in trows if r < rows]
    assert len(set(moved)) == len(moved)
    for i in range(rows):                                 # every key once
        assert rest[i] + (lens[i] if i in moved else 0) == lens[i]
        assert (rest[i] == 0) or (i not in moved)
    for r, (i, L) in enumerate(zip(trows, tlens)):
        if i < rows:
            assert L == lens[i] and L * pairs > total     # moved: longer than a pair's share
            longer = int((lens > L).sum()) + int((lens[:i] == L).sum())
            assert longer == r                            # its rank, ties to the lower row
        else:
            assert L == 0
    # a candidate that stays is never longer than one that moves
    stay = [lens[i] for i in np.argsort(-lens, kind="stable")[:split_rows] if i not in moved]
    if moved and stay:
        assert max(stay) <= min(lens[i] for i in moved)
