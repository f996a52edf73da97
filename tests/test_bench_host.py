"""Host-side pieces of bench.py that need no GPU: the oracle sampler's row
accounting and the algorithmic-byte count the roofline divides by."""
import numpy as np
import pytest

import bench
from workloads import make_batch_from_lengths


def test_sampler_counts_whole_requests_after_one_cycle():
    # lengths that end mid-chunk and one empty request
    lens = [300, 0, 256, 513]
    b = make_batch_from_lengths(lens, 2, 3, seed=5)
    s = bench.OracleSampler(b)
    chunks_needed = sum(-(-L // s.CHUNK) for L in lens)
    rows = 0.0
    for _ in range(chunks_needed):
        _, r, _, n = s.run(0.0)           # exactly one chunk per call
        assert n == 1
        rows += r
    assert rows == pytest.approx(sum(1 for L in lens if L > 0) * b.k, rel=1e-12)
    assert (s.r, s.j) == (0, 0)           # back at the first request


def test_sampler_refuses_all_empty_batch():
    b = make_batch_from_lengths([0, 0], 1, 2, seed=6)
    with pytest.raises(ValueError):
        bench.OracleSampler(b)


def test_algorithmic_bytes_formula():
    lens = np.array([100, 37])
    M, pages = 32, int(sum(-(-L // 64) for L in lens))
    got = bench.algorithmic_bytes(lens, M)
    want = 576 * lens.sum() + len(lens) * M * (576 + 1028) + 4 * pages
    assert got == want
