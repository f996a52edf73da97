"""The tiered launch on the GPU (drafter-attention page, `balanced_decode`):
the device tier planner bit for bit against the CPU rule, the row
gather/scatter byte for byte, and the whole tiered decode against the oracle."""
import numpy as np
import pytest
import torch

import mla_decode_attention_folded_gb300 as mla
from oracle import tiers as ot
from tests.gpu_util import assert_close, bmm_scales, oracle_full, to_device
from workloads import make_batch_from_lengths

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(12))
def test_tier_plan_bit_exact(seed):
    rng = np.random.default_rng(seed)
    rows = int(rng.choice([1, 2, 37, 128, 640, 1024]))
    lens = rng.integers(-5, 200000, size=rows).astype(np.int32)
    lens[rng.random(rows) < 0.25] = 4096                 # ties
    lens[rng.random(rows) < 0.1] = 0
    split_rows = int(rng.integers(0, rows + 1))
    pairs = int(rng.integers(1, 200))
    move = (int(rng.integers(1, 5)), int(rng.integers(1, 5)))
    dev_lens = torch.from_numpy(lens).cuda()
    rest = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    n = max(split_rows, 1)
    trows = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    tlens = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    mla.tier_plan(rows, split_rows, pairs, move, dev_lens, rest, trows, tlens)
    torch.cuda.synchronize()
    want = ot.tier_tables(lens, split_rows, pairs, move)
    assert rest.cpu().tolist() == want[0]
    assert trows.cpu().tolist()[:split_rows] == want[1]
    assert tlens.cpu().tolist()[:split_rows] == want[2]


@pytest.mark.parametrize("row_bytes", [4, 36, 2304, 65536 + 48])
def test_row_copy_gather_and_scatter(row_bytes):
    g = torch.Generator().manual_seed(row_bytes)
    bound, targets = 50, 23
    src = torch.randint(0, 256, (bound, row_bytes), dtype=torch.uint8, generator=g)
    index = torch.randint(-3, bound + 5, (targets,), dtype=torch.int32, generator=g)
    dst = torch.randint(0, 256, (targets, row_bytes), dtype=torch.uint8, generator=g)
    want = dst.clone()
    for i, t in enumerate(index.tolist()):
        if 0 <= t < bound:
            want[i] = src[t]
    d = dst.cuda()
    mla.row_copy(src.cuda(), d, index.cuda(), targets, bound, True)
    torch.cuda.synchronize()
    assert torch.equal(d.cpu(), want)
    # scatter back into a fresh buffer (distinct targets only)
    perm = torch.randperm(bound + 5, generator=g)[:targets].to(torch.int32) - 2
    back = torch.zeros((bound, row_bytes), dtype=torch.uint8)
    want = back.clone()
    for i, t in enumerate(perm.tolist()):
        if 0 <= t < bound:
            want[t] = dst[i]
    b = back.cuda()
    mla.row_copy(dst.cuda(), b, perm.cuda(), targets, bound, False)
    torch.cuda.synchronize()
    assert torch.equal(b.cpu(), want)


@pytest.mark.parametrize("k,H,sms,lens", [
    (4, 8, 32, [10000, 100, 64, 0] * 12),                    # 48 rows: tiers (8, 16), 12 move
    (7, 64, 16, [2200, 300, 90, 1800, 513, 64, 5, 1000] * 2),  # 16 rows, M = 448: tier (8,)
])
def test_tiered_decode_matches_oracle(k, H, sms, lens):
    b = make_batch_from_lengths(tuple(lens), k, H, seed=len(lens) + k, scaling="amax")
    d = to_device(b)
    eng = mla.TieredMla(b.R, b.k, b.H, d["bt"].shape[1], d["kv"].shape[0], "cuda", sms=sms)
    assert eng.split_rows > 0
    bmm1, bmm2 = bmm_scales(b)
    out, lse = eng.decode(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2)
    torch.cuda.synchronize()
    assert int((eng.tier_rows < b.R).sum()) > 0              # some rows really moved
    assert int(eng.unsplit.status.item()) == 0
    assert all(int(e.status.item()) == 0 for e in eng.engines)
    ref_o, ref_l = oracle_full(b)
    assert_close(out.float().cpu(), lse.cpu(), ref_o, ref_l, f"tiered k={k} H={H}")
    out2, lse2 = eng.decode(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2, return_lse=False)
    torch.cuda.synchronize()
    assert lse2 is None
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
