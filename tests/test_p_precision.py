"""Why P enters the PV product as two E4M3 terms: a model of the kernels'
softmax arithmetic (tests/kernel_numerics.py) against the oracle, on short
requests of each workload's recipe (few keys per row: the hardest case for a
rounded P). The balanced-MLA page stores P as E4M3, unscaled (module
overview); the tolerance |out - ref| <= 2e-2 + 2e-2 |ref| is the one every
GPU test uses. No GPU."""
import pytest

from tests import kernel_numerics as kn
from workloads import WORKLOADS, make_batch_from_lengths

# (workload, short lengths from its recipe) -- the tiny workload as stated.
SAMPLES = [
    ("R2_k4_H8_len100+37", (100, 37)),
    ("R32_k4_H8_len1k-8k", (1024, 1100)),
    ("R64_k7_H8_lognormal2k", (256, 300)),
    ("R16_k4_H64_len16k-64k", (16384,)),
    ("R128_k7_H64_skewed128k", (512, 560)),
]


def _batch(name, lens):
    w = WORKLOADS[name]
    return make_batch_from_lengths(lens, w.k, w.H, seed=w.seed, value_std=w.value_std,
                                   scaling=w.scaling)


def _worst(name, lens, mode):
    b = _batch(name, lens)
    errs = [kn.request_error(b, r, mode) for r in range(b.R)]
    return max(e[0] for e in errs), max(e[1] for e in errs)


@pytest.mark.parametrize("name,lens", SAMPLES)
def test_two_term_p_meets_the_bound_with_margin(name, lens):
    excess, lse = _worst(name, lens, "two_term")
    assert excess <= -5e-3, f"{name}: two-term P within {-excess:.4f} of the bound"
    assert lse <= 1e-4


@pytest.mark.parametrize("mode", ["one_term", "one_term_rounded_sum"])
@pytest.mark.parametrize("name,lens", [SAMPLES[0], SAMPLES[4]])
def test_single_term_p_misses_the_bound(name, lens, mode):
    """One E4M3 term, whether normalised by the FP32 sum of P or by the sum of
    the rounded values the MMA used, exceeds the bound on the tiny workload
    and on the skewed workload's short requests: hence the second term."""
    excess, lse = _worst(name, lens, mode)
    assert excess > 0, f"{name} {mode}: inside the bound by {-excess:.4f}"
    assert lse <= 1e-4                       # the LSE comes from the FP32 sum either way
