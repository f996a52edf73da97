"""Split tiers of the tiered launch: which rows leave the unsplit launch.

Test infrastructure only (see the package docstring). The device tier planner
must reproduce ``tier_tables`` bit for bit.

What the pages fix (drafter-attention page, ``balanced_tiers``,
``_balanced_tables`` and ``_plan_kernel``; ``balanced_decode`` runs the
result):

* ``balanced_tiers``: no tiers when rows * 4 <= SMs (the single launch then
  splits every row already); otherwise the tier sizes of ``TIERS``, in order,
  while their running sum stays at most rows // 2 (at least half the rows stay
  in the unsplit launch).
* the tier rows are chosen among the ``split_rows`` = sum(tiers) longest rows,
  ranked by length, longest first, ties to the lower row; a ranked row moves
  into its tier when its length exceeds ``MOVE`` of a pair's share of the
  batch's keys: len * MOVE_DEN * pairs > MOVE_NUM * total, pairs = SMs // 2.
* outputs: every row's length in the unsplit launch (0 for a moved row);
  per rank r < split_rows the batch row it takes (``rows`` when that rank's
  row stays in the unsplit launch) and its length in the tier (0 when not
  moved).

``TIERS`` and ``MOVE`` have no values on the pages; the ones below are this
project's.
"""
from __future__ import annotations

TIERS = (8, 16, 32)        # rows per tier, longest rows first
MOVE = (1, 1)              # MOVE_NUM / MOVE_DEN: longer than one pair's share


def balanced_tiers(rows: int, sms: int, tiers=TIERS) -> tuple:
    if rows * 4 <= sms:
        return ()
    out: list[int] = []
    for size in tiers:
        if sum(out) + size > rows // 2:
            break
        out.append(size)
    return tuple(out)


def tier_tables(seq_lens, split_rows: int, pairs: int, move=MOVE):
    """-> (rest [rows], tier_rows [split_rows], tier_lens [split_rows]) as int
    lists. Negative lengths are read as 0."""
    lens = [max(0, int(x)) for x in seq_lens]
    rows = len(lens)
    assert 0 <= split_rows <= rows
    total = sum(lens)
    ranked = sorted(range(rows), key=lambda i: (-lens[i], i))
    rest = list(lens)
    tier_rows = [rows] * split_rows
    tier_lens = [0] * split_rows
    for r, i in enumerate(ranked[:split_rows]):
        if lens[i] * move[1] * pairs > move[0] * total:
            rest[i] = 0
            tier_rows[r] = i
            tier_lens[r] = lens[i]
    return rest, tier_rows, tier_lens
