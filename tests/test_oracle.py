"""The CPU oracle against its pins (no GPU)."""
import math

import numpy as np
import pytest
import torch

import oracle.e4m3 as e4m3
import oracle.merge as merge
from tests import oracle_pins as pins


def test_e4m3_table_matches_torch_cast():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(np.isnan(e4m3.TABLE), nan)
    assert np.array_equal(e4m3.TABLE[~nan], ref[~nan])


def test_e4m3_known_points():
    t = e4m3.TABLE
    assert t[0x00] == 0.0 and t[0x80] == 0.0 and math.copysign(1, t[0x80]) < 0
    assert t[0x01] == 2.0 ** -9            # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert t[0x08] == 2.0 ** -6            # smallest normal
    assert t[0x38] == 1.0 and t[0xB8] == -1.0
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)        # codes order like their values
    with pytest.raises(ValueError):
        e4m3.decode(np.array([0x7F], dtype=np.uint8))


def test_oracle_matches_brute_force():
    assert pins.check_brute_force() == []


def test_oracle_closed_forms():
    assert pins.check_closed_forms() == []


def test_oracle_matches_torch_softmax_on_one_page():
    assert pins.check_library_softmax() == []


def test_fold_equals_unfold():
    assert pins.check_fold_equals_unfold() == []


def test_split_merge_invariance():
    assert pins.check_split_merge() == []


def test_convexity():
    assert pins.check_convexity() == []


def test_row_sampler_matches_brute_force_and_whole_batch():
    assert pins.check_row_sampler() == []


def test_merge_empty_and_single():
    o = np.random.default_rng(0).standard_normal((3, 4, 8))
    l = np.full((3, 4), -np.inf)
    mo, ml = merge.combine(o, l)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))
    l[1] = 2.5                                   # one live split: passes through
    mo, ml = merge.combine(o, l)
    assert np.allclose(mo, o[1], rtol=0, atol=1e-15) and np.all(ml == 2.5)
    l[:] = 1.0                                   # equal LSE: plain mean, +log2(3)
    mo, ml = merge.combine(o, l)
    assert np.allclose(mo, o.mean(axis=0), atol=1e-15)
    assert np.allclose(ml, 1.0 + math.log2(3), atol=1e-15)
