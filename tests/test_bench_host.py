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


def test_roofline_picks_binding_bound():
    hbm, _ = bench.measured_hbm_peak()
    fp8, _ = bench.fp8_tensor_peak()
    ridge = fp8 * 1e12 / (hbm * 1e9)
    lo = bench.roofline(10**9, int(0.5 * ridge * 10**9), 1e-3)
    hi = bench.roofline(10**9, int(2.0 * ridge * 10**9), 1e-3)
    assert lo["bound"] == "hbm" and lo["unit"] == "GB/s"
    assert lo["achieved"] == pytest.approx(1000.0) and lo["frac"] == pytest.approx(1000.0 / hbm)
    assert hi["bound"] == "tensor" and hi["unit"] == "TFLOP/s"
    assert hi["frac"] == pytest.approx(hi["achieved"] / fp8)
    assert bench.algorithmic_flops([100, 28], 3) == 2 * 3 * 1088 * 128


def test_source_hash_ignores_comments_only():
    code = "int f(int a) {\n  return a + 1;  // one more\n}\n"
    commented = "/* a note\n   over lines */\nint f(int a) {\n  // first\n  return a + 1;\n}\n"
    changed = "int f(int a) {\n  return a + 2;  // one more\n}\n"
    assert bench.strip_comments(code) == bench.strip_comments(commented)
    assert bench.strip_comments(code) != bench.strip_comments(changed)
    assert len(bench.source_hash()) == 16
