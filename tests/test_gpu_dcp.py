"""Decode-context-parallel merge on one GPU: every request's pages are
interleaved over D shards, each shard is decoded on its own by the regular
path, and mla_lse_merge combines the shards' BF16 rows and log2 LSEs; the
result must match the oracle on the whole request (drafter-attention page,
`DraftDcp`: the same attention as the unsharded decode)."""
import numpy as np
import pytest
import torch

import mla_decode_attention_folded_gb300 as mla
from tests.gpu_util import assert_close, oracle_full, run_decode
from workloads import make_batch_from_lengths, shard_pages

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shards", [2, 3, 4])
@pytest.mark.parametrize("lens,k,H", [((3000, 100, 64, 37), 4, 8), ((1900, 700), 7, 8),
                                      ((2600, 130), 4, 64)])
def test_sharded_decode_merged_matches_oracle(shards, lens, k, H):
    b = make_batch_from_lengths(lens, k, H, seed=shards * 1000 + sum(lens), scaling="amax")
    ref_o, ref_l = oracle_full(b)
    outs, lses = [], []
    for d in range(shards):
        part = shard_pages(b, shards, d)
        o, l, status, _ = run_decode(part, min_split_tokens=64)
        assert status == 0
        outs.append(o)                       # float32 copies of the BF16 rows
        lses.append(l)
    parts_out = torch.stack(outs).to(torch.bfloat16).cuda().contiguous()
    parts_lse = torch.stack(lses).cuda().contiguous()
    out = torch.empty((b.R, b.M, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((b.R, b.M), dtype=torch.float32, device="cuda")
    mla.lse_merge(parts_out, parts_lse, out, lse)
    torch.cuda.synchronize()
    assert_close(out.float().cpu(), lse.cpu(), ref_o, ref_l, f"{shards} shards")


def test_merge_of_empty_sources():
    S, rows = 3, 5
    parts_out = torch.randn(S, rows, 512).to(torch.bfloat16).cuda()
    parts_lse = torch.full((S, rows), float("-inf"), device="cuda")
    parts_lse[1, 2] = 3.0                    # row 2 has one live source
    out = torch.empty((rows, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(rows, device="cuda")
    mla.lse_merge(parts_out, parts_lse, out, lse)
    torch.cuda.synchronize()
    o, l = out.float().cpu(), lse.cpu()
    for r in range(rows):
        if r == 2:
            assert torch.equal(o[r], parts_out[1, 2].float().cpu()) and float(l[r]) == 3.0
        else:
            assert torch.all(o[r] == 0) and torch.isneginf(l[r])
