"""Plant plausible mistakes in the packed plan of the CPU planner and check
that the planner's pins (its worked examples, the property and balance tests,
the empty-request pin) catch every one: the same check as for the attention
oracle, for the split planner's newest part. No GPU."""
import inspect
import textwrap

import numpy as np
import pytest

from oracle import planner as pl
from tests import test_oracle_planner as tp

# (function, source text, its replacement): one plausible mistake each.
MUTANTS = {
    "segment_off_by_one": ("_packed", "u0, u1 = P // c0, (P + p[i] - 1) // c0",
                           "u0, u1 = (P + 1) // c0, (P + p[i]) // c0"),
    "ranges_not_relative": ("_packed", "a = max(P, u * c0) - P", "a = max(P, u * c0)"),
    "empty_always_unit_0": ("_packed", "u = n_empty % nseg", "u = 0"),
    "no_piece_cost": ("_packed",
                      "cost = max(min(c0, T - u * c0) + JOB_PAGES * per_unit[u] for u in range(nseg))",
                      "cost = max(min(c0, T - u * c0) for u in range(nseg))"),
    "cost_of_last_unit_only": ("_packed",
                               "cost = max(min(c0, T - u * c0) + JOB_PAGES * per_unit[u] for u in range(nseg))",
                               "cost = min(c0, T - (nseg - 1) * c0) + JOB_PAGES * per_unit[nseg - 1]"),
    "entries_in_rank_order": ("plan",
                              "listed = [i for i in order if counts[i] >= 2] + [i for i in order if counts[i] < 2]",
                              "listed = list(order)"),
    "unit_table_unit_major": ("plan",
                              "buf[off_unit + unit_fill[u] * units(M, num_ctas) + u] = where[(i, s)]",
                              "buf[off_unit + u * UNIT_SLOTS + unit_fill[u]] = where[(i, s)]"),
    "no_packed_bit": ("plan", "buf[e] = (PACKED_BIT if packed else 0) | (i << SPLIT_BITS) | s",
                      "buf[e] = (i << SPLIT_BITS) | s"),
    "single_block_items_pack": ("plan_pieces", "row_blocks(M) >= 2", "row_blocks(M) >= 1"),
}


def _mutated(name):
    fn_name, old, new = MUTANTS[name]
    src = textwrap.dedent(inspect.getsource(getattr(pl, fn_name)))
    assert src.count(old) == 1, (name, old)
    ns = dict(vars(pl))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    return fn_name, ns[fn_name]


def _pins():
    """Every planner pin that concerns packed plans; raises on a mismatch."""
    for golden in ("plan_worked_example.txt", "plan_packed_example.txt"):
        tp.test_worked_examples(golden)
    for seed in range(60):
        tp.test_plan_properties(seed)
    for seed in range(30):
        tp.test_packed_plans_balance_one_wave_batches(seed)
    tp.test_packed_plan_places_empty_requests()
    tp.test_packing_cost_keeps_the_per_request_plan()


def test_pins_pass_on_the_real_planner():
    _pins()


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    fn_name, fn = _mutated(name)
    monkeypatch.setattr(pl, fn_name, fn)
    with pytest.raises(Exception):
        _pins()
