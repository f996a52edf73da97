"""Parity of the CUDA path (through the C ABI) with the CPU oracle."""
import numpy as np
import pytest
import torch

import mla_decode_attention_folded_gb300 as mla
import oracle.attention as att
from oracle import planner as pl
from tests.gpu_util import assert_close, oracle_full, run_decode, to_device, bmm_scales
from workloads import WORKLOADS, make_batch, make_batch_from_lengths

pytestmark = pytest.mark.gpu

TINY = "R2_k4_H8_len100+37"
FULL = [n for n in WORKLOADS if n != TINY]


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


# ---------------------------------------------------------------- planner
def _gpu_plan(lens, M, G, mst, ms, policy):
    R = len(lens)
    s = mla.make_shape(R, 1, M, 1, 1, G, mst, ms, policy)
    n = mla.plan_list_len(s)
    d = torch.tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    counts = torch.zeros(R, dtype=torch.int32, device="cuda")
    work = torch.full((n,), 7, dtype=torch.int32, device="cuda")   # not pre-filled with -1
    mla.plan_splits(s, d, counts, work)
    return counts.cpu().numpy(), work.cpu().numpy()


def _same_plan(c, wk, c2, wk2, R, M, G, policy, ms):
    """Device plan == CPU plan: counts, entries and counters always; ranges
    and unit table when the plan is packed (the device planner leaves them
    unwritten otherwise)."""
    E, off_rng, off_unit = pl.regions(R, M, G, policy, ms)
    if not (np.array_equal(c, c2) and np.array_equal(wk[:off_rng], wk2[:off_rng])):
        return False
    if int(wk2[0]) >= 0 and int(wk2[0]) & pl.PACKED_BIT:
        return np.array_equal(wk[off_rng:], wk2[off_rng:])
    return True


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("policy", [pl.BALANCED, pl.UNIFORM])
def test_planner_bit_exact_on_workloads(name, policy):
    w = WORKLOADS[name]
    b = make_batch(name) if name == TINY else None
    from workloads import draw_lengths
    gen = torch.Generator().manual_seed(w.seed)
    lens = draw_lengths(w.lengths, w.R, gen) if b is None else b.seq_lens.numpy()
    for G in (8, _sms()):
        c, wk = _gpu_plan(lens, w.M, G, 256, 64, policy)
        c2, wk2 = pl.plan(lens, w.M, G, 256, 64, policy, capacity=len(wk))
        assert _same_plan(c, wk, c2, wk2, len(lens), w.M, G, policy, 64)


@pytest.mark.parametrize("lens,M,G", [
    ([6390, 5100, 3800], 256, 16),                                  # packed worked example
    ([0, 13474, 4345, 6990, 0, 0, 3742, 4383], 256, 44),            # packed, empty requests
    ([1021, 1786, 3049, 5808, 5645, 717, 3996, 4808, 2938], 128, 29),   # kept by the cost
    ([16384, 40000, 65536, 30000] * 4, 256, 152),                   # packed, 16 requests
])
def test_planner_bit_exact_on_packing_pins(lens, M, G):
    """The device planner takes the packing decision and lays out a packed
    plan exactly as the CPU planner's pinned cases do."""
    c, wk = _gpu_plan(lens, M, G, 64, 64, pl.BALANCED)
    c2, wk2 = pl.plan(lens, M, G, 64, 64, pl.BALANCED, capacity=len(wk))
    assert _same_plan(c, wk, c2, wk2, len(lens), M, G, pl.BALANCED, 64)
    assert bool(int(wk[0]) & pl.PACKED_BIT) == bool(int(wk2[0]) & pl.PACKED_BIT)


def test_planner_bit_exact_random():
    rng = np.random.default_rng(123)
    for trial in range(2000):
        R = int(rng.integers(1, 1025)) if trial % 50 == 0 else int(rng.integers(1, 200))
        kind = trial % 4
        if kind == 0:
            lens = rng.integers(0, 9000, size=R)
        elif kind == 1:
            lens = np.clip(np.round(np.exp(rng.normal(7.6, 1.2, size=R))), 0, 200000).astype(int)
        elif kind == 2:
            lens = rng.integers(0, 3, size=R) * rng.integers(0, 200, size=R)
        else:
            lens = rng.integers(1, 600, size=R)
            lens[0] = int(rng.integers(50000, 500000))
        M = int(rng.choice([1, 8, 32, 33, 56, 64, 256, 448, 4096]))
        G = int(rng.choice([1, 3, 148, 152, 304, 2048]))
        mst = int(rng.choice([1, 64, 256, 5000]))
        ms = int(rng.choice([1, 2, 64, 4096]))
        policy = int(rng.integers(0, 2))
        c, wk = _gpu_plan(lens, M, G, mst, ms, policy)
        c2, wk2 = pl.plan(lens, M, G, mst, ms, policy, capacity=len(wk))
        assert _same_plan(c, wk, c2, wk2, R, M, G, policy, ms), (trial, R, M, G)


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("policy", [pl.BALANCED, pl.UNIFORM])
@pytest.mark.parametrize("num_ctas", [1, 8, None])
def test_tiny_workload_matches_oracle(policy, num_ctas):
    b = make_batch(TINY)
    ref_o, ref_l = oracle_full(b)
    out, lse, status, _ = run_decode(b, policy=policy, num_ctas=num_ctas, min_split_tokens=64)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"tiny policy={policy} ctas={num_ctas}")


CASES = [
    # lengths, k, H: ragged tails, page boundaries, empty and one-key requests
    ((1, 63, 64, 65, 127, 128, 129), 2, 4),
    ((0, 5, 0), 3, 2),
    ((700, 1500, 3), 1, 1),
    ((1000, 257, 4096), 4, 8),
    ((333, 2000), 7, 8),
    ((2100, 640), 3, 11),
    ((1500,), 1, 64),
    ((900, 130), 2, 40),
    ((2500, 64), 4, 64),
    ((2100, 640), 7, 64),
    ((500, 70), 2, 65),
    ((1300, 90), 6, 64),
    ((800, 200), 15, 32),
]


@pytest.mark.parametrize("lens,k,H", CASES)
@pytest.mark.parametrize("policy", [pl.BALANCED, pl.UNIFORM])
def test_small_cases_match_oracle(lens, k, H, policy):
    b = make_batch_from_lengths(lens, k, H, seed=sum(lens) + 17 * k + H, value_std=1.0,
                                scaling="amax", fill=-5, extra_pages=3)
    ref_o, ref_l = oracle_full(b)
    for G in (2, 13, None):
        out, lse, status, _ = run_decode(b, policy=policy, num_ctas=G, min_split_tokens=64)
        assert status == 0
        assert_close(out, lse, ref_o, ref_l, f"{lens} k={k} H={H} G={G}")
    if max(lens) > 0:
        empty = [i for i, L in enumerate(lens) if L == 0]
        for i in empty:
            assert torch.all(out[i] == 0) and torch.all(torch.isneginf(lse[i]))


def test_planner_bit_exact_with_row_groups():
    rng = np.random.default_rng(7)
    for trial in range(300):
        R = int(rng.integers(1, 120))
        k = int(rng.choice([2, 4, 6, 7, 8]))
        groups = int(rng.choice([d for d in range(1, k + 1) if k % d == 0]))
        if R * groups > 1024:
            continue
        H = int(rng.choice([8, 16, 64]))
        lens = rng.integers(0, 20000, size=R)
        G = int(rng.choice([8, 152]))
        policy = int(rng.integers(0, 2))
        s = mla.make_shape(R, k, H, 1, 1, G, 256, 64, policy, groups)
        n = mla.plan_list_len(s)
        counts = torch.zeros(R * groups, dtype=torch.int32, device="cuda")
        work = torch.full((n,), 7, dtype=torch.int32, device="cuda")
        mla.plan_splits(s, torch.tensor(lens.astype(np.int32), device="cuda"), counts, work)
        c2, w2 = pl.plan(np.repeat(lens, groups), (k // groups) * H, G, 256, 64, policy,
                         capacity=n)
        assert _same_plan(counts.cpu().numpy(), work.cpu().numpy(), c2, w2, R * groups,
                          (k // groups) * H, G, policy, 64), trial


@pytest.mark.parametrize("lens,k,H", [((900, 77, 2000), 4, 64), ((1500, 300), 7, 8),
                                      ((700, 0, 64), 6, 16)])
def test_row_groups_match_oracle(lens, k, H):
    """Unfolded (groups = k), the pages' partial fold and every divisor in
    between give the same attention as the oracle."""
    b = make_batch_from_lengths(lens, k, H, seed=sum(lens) + k, scaling="amax", fill=-5)
    ref_o, ref_l = oracle_full(b)
    divisors = [g for g in range(1, k + 1) if k % g == 0]
    assert k // mla.fold_factor(k, H) in divisors
    for groups in divisors:
        for policy in (pl.BALANCED, pl.UNIFORM):
            out, lse, status, _ = run_decode(b, policy=policy, groups=groups, min_split_tokens=64)
            assert status == 0
            assert_close(out, lse, ref_o, ref_l, f"groups={groups} policy={policy}")


@pytest.mark.parametrize("policy", [pl.BALANCED, pl.UNIFORM])
def test_page_and_tile_boundaries(policy):
    """Lengths on every page / tile boundary and the degenerate ones: empty, one
    key, one key short of and past a page (64) and a tile (128)."""
    lens = (0, 1, 63, 64, 65, 127, 128, 129, 191, 192, 255, 256, 257)
    b = make_batch_from_lengths(lens, 3, 4, seed=17, scaling="amax", fill=-5)
    ref_o, ref_l = oracle_full(b)
    for mst in (64, 256):
        out, lse, status, _ = run_decode(b, policy=policy, min_split_tokens=mst)
        assert status == 0
        assert_close(out, lse, ref_o, ref_l, f"boundaries mst={mst}")


def test_one_row_per_request():
    """k = 1, H = 1: a single query row per request (31 padding rows of the
    32-row block)."""
    b = make_batch_from_lengths((900, 3, 2000, 64), 1, 1, seed=19, scaling="amax")
    ref_o, ref_l = oracle_full(b)
    out, lse, status, _ = run_decode(b, min_split_tokens=64)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, "M=1")


def test_maximum_row_groups():
    """R * groups = 1024 row groups, the most the planner takes."""
    rng = np.random.default_rng(21)
    lens = rng.integers(0, 400, size=512)
    b = make_batch_from_lengths(lens, 2, 4, seed=23, scaling="amax")
    ref_o, ref_l = oracle_full(b)
    for groups in (1, 2):
        out, lse, status, _ = run_decode(b, groups=groups, min_split_tokens=64)
        assert status == 0
        assert_close(out, lse, ref_o, ref_l, f"1024 row groups, groups={groups}")


def test_maximum_rows_per_request():
    """M = k * H = 4096 query rows per request (the largest M): 64 row blocks
    of 64 rows per work item."""
    b = make_batch_from_lengths((700, 130), 16, 256, seed=29, scaling="amax")
    ref_o, ref_l = oracle_full(b)
    out, lse, status, _ = run_decode(b, min_split_tokens=64)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, "M=4096")


def test_folded_equals_unfolded():
    b = make_batch_from_lengths((900, 77, 2000), 4, 8, seed=5, scaling="amax")
    ref_o, ref_l = oracle_full(b)
    for policy in (pl.BALANCED, pl.UNIFORM):
        fo, fl, s1, _ = run_decode(b, policy=policy)
        uo, ul, s2, _ = run_decode(b, policy=policy, folded=False)
        assert s1 == 0 and s2 == 0
        assert_close(fo, fl, ref_o, ref_l, "folded")
        assert_close(uo, ul, ref_o, ref_l, "unfolded")


def test_many_splits_of_one_request():
    b = make_batch_from_lengths((20000,), 2, 16, seed=9, scaling="amax")
    ref_o, ref_l = oracle_full(b)
    out, lse, status, (counts, _) = run_decode(b, min_split_tokens=64, max_splits=4096)
    assert status == 0 and int(counts[0]) > 100
    assert_close(out, lse, ref_o, ref_l, "many splits")


def _random_cases(n, seed):
    """Seeded random shapes: R, k, H, row groups, lengths (page and tile
    edges, empty and one-key requests mixed in), policy, CTA count and split
    limits; each case's oracle work (rows x keys) kept to a few million."""
    rng = np.random.default_rng(seed)
    edges = [0, 1, 63, 64, 65, 95, 96, 97, 127, 128, 129, 191, 192, 193]
    out = []
    while len(out) < n:
        R = int(rng.integers(1, 10))
        k = int(rng.integers(1, 9))
        H = int(rng.choice([1, 2, 3, 5, 8, 16, 33, 64]))
        lens = [int(rng.choice(edges)) if rng.random() < 0.4 else int(rng.integers(1, 3000))
                for _ in range(R)]
        if k * H * sum(lens) > 3_000_000 or max(lens) == 0:
            continue
        divisors = [d for d in range(1, k + 1) if k % d == 0]
        groups = int(rng.choice(divisors))
        policy = int(rng.choice([pl.BALANCED, pl.UNIFORM]))
        num_ctas = int(rng.choice([1, 3, 16, 57, 152]))
        mst = int(rng.choice([64, 256]))
        ms = int(rng.choice([3, 64]))
        out.append((tuple(lens), k, H, groups, policy, num_ctas, mst, ms))
    return out


@pytest.mark.parametrize("lens,k,H,groups,policy,G,mst,ms", _random_cases(40, 2026))
def test_random_shapes_match_oracle(lens, k, H, groups, policy, G, mst, ms):
    """Seeded random shapes against the oracle, element by element."""
    b = make_batch_from_lengths(lens, k, H, seed=len(lens) * 1009 + k * 31 + H, value_std=1.0,
                                scaling="amax", fill=-5, extra_pages=2)
    ref_o, ref_l = oracle_full(b)
    out, lse, status, _ = run_decode(b, policy=policy, num_ctas=G, min_split_tokens=mst,
                                     max_splits=ms, groups=groups)
    assert status == 0
    assert_close(out, lse, ref_o, ref_l, f"{lens} k={k} H={H} groups={groups} G={G}")
    for i, L in enumerate(lens):
        if L == 0:
            assert torch.all(out[i] == 0) and torch.all(torch.isneginf(lse[i]))


@pytest.mark.parametrize("lens,k,H,G,groups,policy", [
    ((6000,) + (300,) * 30 + (0, 90), 4, 8, 5, 1, pl.BALANCED),   # 32-row kernel, an empty request
    ((4000, 2500) + (700,) * 12, 7, 8, 7, 1, pl.BALANCED),       # 64-row kernel
    ((3000, 1500, 400, 64), 2, 64, 3, 1, pl.BALANCED),           # M = 128: two 64-row blocks
    ((5000, 900, 60) + (400,) * 9, 4, 16, 6, 2, pl.BALANCED),    # row groups, 32-row blocks
    ((2500, 1800, 0, 700), 2, 64, 4, 2, pl.BALANCED),            # row groups, 64-row blocks
    ((3000, 100) + (500,) * 6, 4, 8, 3, 1, pl.UNIFORM),          # uniform splits
])
def test_claimed_jobs_and_repeated_decodes_of_one_plan(lens, k, H, G, groups, policy):
    """Far more jobs than CTAs: after its first job a CTA claims the next ones
    in list order from the counters after the items. Three decodes of one plan
    agree bit for bit and with the oracle, and each leaves the work list as the
    plan wrote it (both counters back at -1)."""
    b = make_batch_from_lengths(lens, k, H, seed=sum(lens) + G, scaling="amax")
    d = to_device(b)
    eng = mla.FoldedMla(b.R, b.k, b.H, d["bt"].shape[1], d["kv"].shape[0], "cuda", num_ctas=G,
                        min_split_tokens=64, policy=policy, groups=groups)
    bmm1, bmm2 = bmm_scales(b)
    eng.plan(d["lens"])
    torch.cuda.synchronize()
    planned = eng.work.cpu().clone()
    E = pl.items_len(b.R * groups, (k // groups) * H, G, policy, 64)
    assert torch.all(planned[E:E + 2] == -1)                # the job counters
    runs = []
    for _ in range(3):
        out, lse = eng.decode(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2)
        torch.cuda.synchronize()
        assert torch.equal(eng.work.cpu(), planned)
        runs.append((out.clone(), lse.clone()))
    assert int(eng.status.item()) == 0
    for o, l in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1])
    ref_o, ref_l = oracle_full(b)
    assert_close(runs[0][0].float().cpu(), runs[0][1].cpu(), ref_o, ref_l,
                 f"lens={len(lens)} requests k={k} H={H} G={G} groups={groups} policy={policy}")


@pytest.mark.parametrize("lens,k,H,G,groups", [
    ((2625, 797, 6485, 1686), 2, 64, 10, 1),                # two 64-row blocks per item
    ((5400, 0, 4962, 1294, 6586), 2, 64, 11, 1),            # two blocks, an empty request
    ((3000, 2500, 2000, 1500), 4, 64, 16, 1),               # four blocks
    ((9000, 4000, 0, 0, 2000, 64, 1), 7, 64, 56, 1),        # seven blocks, empty requests
    ((258, 4369, 1331, 3613), 4, 64, 25, 2),                # row groups of two blocks
    ((0, 5322, 7175, 1472), 4, 64, 22, 2),                  # row groups, an empty request
])
def test_packed_plans(lens, k, H, G, groups):
    """Batches of at most one request per unit whose per-request plan leaves
    one large item, with several row blocks per item: the plan packs the
    rank-ordered pages into equal segments and each unit's CTAs walk their own
    entries. The device plan equals the oracle's bit for bit, three
    decodes of it agree bit for bit and with the oracle, and the buffer is left
    as planned."""
    b = make_batch_from_lengths(lens, k, H, seed=sum(lens) + G + 5, scaling="amax")
    rows = np.repeat(np.asarray(lens), groups)
    M = (k // groups) * H
    want_counts, want_buf = pl.plan(rows, M, G, 64, 64, pl.BALANCED)
    assert int(want_buf[0]) & pl.PACKED_BIT, "the case must give a packed plan"
    d = to_device(b)
    eng = mla.FoldedMla(b.R, b.k, b.H, d["bt"].shape[1], d["kv"].shape[0], "cuda", num_ctas=G,
                        min_split_tokens=64, groups=groups)
    bmm1, bmm2 = bmm_scales(b)
    eng.plan(d["lens"])
    torch.cuda.synchronize()
    planned = eng.work.cpu().clone()
    assert _same_plan(eng.counts.cpu().numpy(), planned.numpy(), want_counts, want_buf,
                      len(rows), M, G, pl.BALANCED, 64)
    runs = []
    for _ in range(3):
        out, lse = eng.decode(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2)
        torch.cuda.synchronize()
        assert torch.equal(eng.work.cpu(), planned)
        runs.append((out.clone(), lse.clone()))
    assert int(eng.status.item()) == 0
    for o, l in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(l, runs[0][1])
    ref_o, ref_l = oracle_full(b)
    assert_close(runs[0][0].float().reshape(b.R, b.M, 512).cpu(), runs[0][1].reshape(b.R, b.M).cpu(),
                 ref_o, ref_l, f"packed {lens} k={k} H={H} G={G} groups={groups}")


def test_out_of_range_page_sets_status_without_fault():
    b = make_batch_from_lengths((300, 100), 2, 8, seed=3, scaling="amax")
    b.block_table[0, 2] = b.kv.shape[0] + 1000          # inside request 0's pages
    _, _, status, _ = run_decode(b)
    assert status & mla.FAULT_PAGE_RANGE
    b.block_table[0, 2] = -3
    _, _, status, _ = run_decode(b)
    assert status & mla.FAULT_PAGE_RANGE


def test_wait_that_runs_out_stops_one_cta_and_the_plan_stays_reusable():
    """Failure detection without a fault: CTA 0's first KV copy is withheld and
    the pipeline waits are bounded at 20 ms, so a wait runs out. The call
    returns with MLA_FAULT_WAIT_TIMEOUT set, and a regular decode of the same
    plan and work list afterwards matches the oracle (the job counters were put
    back). 32-row kernel, 64-row kernel with one and with two row blocks."""
    for lens, k, H in (((3000, 700, 64), 4, 8), ((2100, 640), 7, 8), ((1300, 90), 2, 64)):
        b = make_batch_from_lengths(lens, k, H, seed=43, scaling="amax")
        d = to_device(b)
        eng = mla.FoldedMla(b.R, b.k, b.H, d["bt"].shape[1], d["kv"].shape[0], "cuda",
                            num_ctas=_sms(), min_split_tokens=64)
        bmm1, bmm2 = bmm_scales(b)
        eng.plan(d["lens"])
        out = torch.empty((b.R, b.M, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((b.R, b.M), dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        mla.folded_decode_wait_test(eng.shape, d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2,
                                    eng.counts, eng.work, eng.workspace, out, lse, status,
                                    20_000_000)
        mla.split_combine(eng.shape, eng.counts, eng.work, eng.workspace, bmm2, out, lse)
        torch.cuda.synchronize()
        assert int(status.item()) & mla.FAULT_WAIT_TIMEOUT, (lens, k, H)
        eng.status.zero_()
        o, l = eng.decode(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2)
        torch.cuda.synchronize()
        assert int(eng.status.item()) == 0
        ref_o, ref_l = oracle_full(b)
        assert_close(o.float().reshape(b.R, b.M, 512).cpu(), l.cpu(), ref_o, ref_l,
                     f"after a timed-out decode {lens}")


def test_wait_test_entry_refuses_limits_out_of_range():
    # Device inputs are NULL: a working range check answers MLA_ERR_SHAPE
    # first; without it the call would stop at MLA_ERR_NULL, launching nothing.
    import ctypes
    from mla_decode_attention_folded_gb300 import _lib
    s = mla.make_shape(2, 2, 8, 8, 16, _sms())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = _lib.load()
    for limit in (0, 999_999, 3_000_000_000):
        rc = lib.mla_folded_decode_wait_test(ctypes.byref(s), None, None, None, None, 0.1, 1.0,
                                             None, None, mla.plan_list_len(s), None, 0, None,
                                             None, status.data_ptr(), limit, None)
        assert rc == -2, limit                                  # MLA_ERR_SHAPE


def test_no_lse_route_matches_lse_route():
    """lse = NULL (the route without an LSE): the same out, bit for bit, on
    single- and multi-split requests and on the 32-row and 64-row kernels, with
    one and two 64-row blocks."""
    for lens, k, H in (((3000, 700, 64, 0), 4, 8), ((2100, 640), 7, 8), ((1300, 90), 2, 64)):
        b = make_batch_from_lengths(lens, k, H, seed=41, scaling="amax")
        d = to_device(b)
        G = _sms()
        eng = mla.FoldedMla(b.R, b.k, b.H, d["bt"].shape[1], d["kv"].shape[0], "cuda",
                            num_ctas=G, min_split_tokens=64)
        bmm1, bmm2 = bmm_scales(b)
        eng.plan(d["lens"])
        out1, lse1 = eng.decode(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2)
        out2, lse2 = eng.decode(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2,
                                return_lse=False)
        torch.cuda.synchronize()
        assert lse2 is None and int(eng.status.item()) == 0
        assert torch.equal(out1.view(torch.int16), out2.view(torch.int16)), (lens, k, H)
        assert int((eng.counts >= 2).sum()) > 0
        ref_o, ref_l = oracle_full(b)
        assert_close(out2.float().reshape(b.R, b.M, 512).cpu(), lse1.cpu(), ref_o, ref_l,
                     f"no-lse {lens}")


def test_no_lse_route_writes_nothing_outside_its_buffers():
    """Without an LSE output, one-split rows have nowhere to put theirs: the
    decode must not write it anywhere (a one-split plan needs no workspace at
    all). Canary bytes around the workspace stay untouched; 32-row, 64-row and
    one and two 64-row blocks, one-split and mixed plans."""
    for lens, k, H, max_splits in (((3000, 700, 0, 64), 4, 8, 1), ((2100, 640, 0), 7, 8, 1),
                                   ((1300, 90, 0), 2, 64, 1), ((3000, 700, 0, 64), 4, 8, 64)):
        b = make_batch_from_lengths(lens, k, H, seed=45, scaling="amax")
        d = to_device(b)
        s = mla.make_shape(b.R, b.k, b.H, d["bt"].shape[1], d["kv"].shape[0], _sms(), 64,
                           max_splits, pl.UNIFORM if max_splits == 1 else pl.BALANCED)
        ws = mla.workspace_bytes(s)
        canary = torch.full(((ws + 255) // 256 * 256 + (1 << 20),), 0x5A, dtype=torch.uint8,
                            device="cuda")
        workspace = canary[:max(ws, 256)]          # never NULL: a stray write lands here
        counts = torch.zeros(b.R, dtype=torch.int32, device="cuda")
        work = torch.full((mla.plan_list_len(s),), -1, dtype=torch.int32, device="cuda")
        out = torch.empty((b.R, b.M, 512), dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        mla.plan_splits(s, d["lens"], counts, work)
        mla.folded_decode(s, d["q"], d["kv"], d["bt"], d["lens"], *bmm_scales(b), counts, work,
                          workspace, out, None, status)
        mla.split_combine(s, counts, work, workspace, bmm_scales(b)[1], out, None)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert bool((canary[ws:] == 0x5A).all()), (lens, k, H, max_splits)
        ref_o, ref_l = oracle_full(b)
        assert_close(out.float().cpu(), ref_l, ref_o, ref_l, f"no-lse {lens} {max_splits}")


def test_lse_merge_without_lse_output():
    S, rows = 3, 70
    g = torch.Generator().manual_seed(8)
    parts = (torch.randn(S, rows, 512, generator=g)).to(torch.bfloat16).cuda()
    plse = (torch.randn(S, rows, generator=g) * 4).float().cuda()
    o1 = torch.empty(rows, 512, dtype=torch.bfloat16, device="cuda")
    l1 = torch.empty(rows, dtype=torch.float32, device="cuda")
    o2 = torch.empty_like(o1)
    mla.lse_merge(parts, plse, o1, l1)
    mla.lse_merge(parts, plse, o2, None)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


# ---------------------------------------------------------------- combine alone
def test_combine_on_oracle_partials():
    """mla_split_combine on partials the oracle made over the planned splits."""
    b = make_batch_from_lengths((3000, 700, 64, 0), 2, 8, seed=77, scaling="amax")
    G = 16
    s = mla.make_shape(b.R, b.k, b.H, b.block_table.shape[1], b.kv.shape[0], G, 64, 64)
    counts, work = pl.plan(b.seq_lens.numpy(), b.M, G, 64, 64, pl.BALANCED,
                           capacity=mla.plan_list_len(s))
    slots = pl.partial_slots(b.R, b.M, G, pl.BALANCED, 64)
    ws = torch.zeros(mla.workspace_bytes(s), dtype=torch.uint8)
    po_bytes = (slots * b.M * 512 * 4 + 255) // 256 * 256
    po = ws[:po_bytes].view(torch.float32)[: slots * b.M * 512].view(slots, b.M, 512)
    plse = ws[po_bytes:].view(torch.float32)[: slots * b.M].view(slots, b.M)
    lens = b.seq_lens.numpy()
    for idx, e in enumerate(work):
        if e < 0:
            break
        r = pl.entry_request(e)
        if counts[r] < 2:
            continue
        kr = np.zeros((b.R, 2), dtype=np.int64)
        kr[r] = pl.entry_keys(work, counts, idx, int(lens[r]), b.R, b.M, G, pl.BALANCED, 64)
        o, l = att.mla_decode(b.q.numpy(), b.kv.numpy(), b.block_table.numpy(), lens, b.k,
                              b.sm_scale, b.q_scale, b.kv_scale, key_range=kr, requests=[r])
        po[idx] = torch.from_numpy(o.reshape(b.R, b.M, 512)[r] / b.kv_scale).float()
        plse[idx] = torch.from_numpy(l.reshape(b.R, b.M)[r]).float()
    out = torch.zeros((b.R, b.M, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((b.R, b.M), dtype=torch.float32, device="cuda")
    mla.split_combine(s, torch.from_numpy(counts).cuda(), torch.from_numpy(work).cuda(),
                      ws.cuda(), b.kv_scale, out, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle_full(b)
    multi = [r for r in range(b.R) if counts[r] >= 2]
    assert multi
    assert_close(out.float().cpu()[multi], lse.cpu()[multi], ref_o[multi], ref_l[multi],
                 "combine")


# ---------------------------------------------------------------- full sizes, sampled
def _picks(b, counts, n=40, seed=0):
    rng = np.random.default_rng(seed)
    lens = b.seq_lens.numpy()
    reqs = [int(np.argmax(lens)), int(np.argmin(lens))]
    reqs += [int(r) for r in np.nonzero(counts.numpy() >= 2)[0][:3]]
    reqs += [int(r) for r in rng.integers(0, b.R, size=4)]
    picks = []
    for r in dict.fromkeys(reqs):
        for m in sorted(set([0, b.M - 1] + rng.integers(0, b.M, size=3).tolist())):
            picks.append((r, m))
    return picks[:n]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled(name):
    b = make_batch(name)
    out, lse, status, (counts, _) = run_decode(b)
    assert status == 0
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    picks = _picks(b, counts)
    ref_o, ref_l = att.mla_decode_rows(b.q.numpy(), b.kv.numpy(), b.block_table.numpy(),
                                       b.seq_lens.numpy(), b.k, b.sm_scale, b.q_scale,
                                       b.kv_scale, picks)
    got_o = np.stack([out[r, m].numpy() for r, m in picks])
    got_l = np.array([float(lse[r, m]) for r, m in picks])
    assert_close(got_o, got_l, ref_o, ref_l, name)
