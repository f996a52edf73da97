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


def test_one_thread_oracle_runs_in_its_own_interpreter():
    r = bench.one_thread_oracle("R2_k4_H8_len100+37", 0.2)
    assert "error" not in r, r
    assert r["cores"] == 1 and r["kind"] == "oracle" and r["value"] > 0


def test_workload_summary_gains():
    b = make_batch_from_lengths([640, 64], 2, 4, seed=7)
    s = bench.workload_summary("none", b, 0.02, 0.015,
                               {"folded_uniform": 0.03, "unfolded_balanced": 0.05})
    assert s["step_us"] == pytest.approx(20.0) and s["decode_us"] == pytest.approx(15.0)
    assert s["balanced_over_uniform"] == pytest.approx(1.5)
    assert s["folded_over_unfolded"] == pytest.approx(2.5)
    assert s["rows_per_s"] == pytest.approx(b.R * b.k / 0.02e-3)
    assert s["traffic"] is None            # no capture of a workload called "none"
    assert s["variants_step_us"]["folded_balanced"] == pytest.approx(20.0)
