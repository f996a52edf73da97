"""The seeded input recipe (workloads/): shapes, length distributions, page
layout, quantisation and determinism of the five workloads and of the batches
the tests build. No GPU."""
import math

import numpy as np
import torch

from workloads import (E4M3_MAX, PAGE, WORKLOADS, draw_lengths, make_batch,
                       make_batch_from_lengths, make_w_uv, quantize)

# name -> (R, k, H): the five workloads of the pages' draft-block decode.
SHAPES = {
    "R2_k4_H8_len100+37": (2, 4, 8),
    "R32_k4_H8_len1k-8k": (32, 4, 8),
    "R64_k7_H8_lognormal2k": (64, 7, 8),
    "R16_k4_H64_len16k-64k": (16, 4, 64),
    "R128_k7_H64_skewed128k": (128, 7, 64),
}


def _lengths(name):
    w = WORKLOADS[name]
    return draw_lengths(w.lengths, w.R, torch.Generator().manual_seed(w.seed))


def test_workload_shapes_and_seeds():
    assert list(WORKLOADS) == list(SHAPES)
    for i, (name, (R, k, H)) in enumerate(SHAPES.items()):
        w = WORKLOADS[name]
        assert (w.R, w.k, w.H, w.M) == (R, k, H, k * H)
        assert w.seed == 1000 + i


def test_lengths_follow_the_recipe():
    assert _lengths("R2_k4_H8_len100+37").tolist() == [100, 37]
    c2 = _lengths("R32_k4_H8_len1k-8k")
    assert c2.size == 32 and c2.min() >= 1024 and c2.max() <= 8192
    c3 = _lengths("R64_k7_H8_lognormal2k")
    assert c3.size == 64 and c3.min() >= 256 and c3.max() <= 32768
    # log-lengths centred on ln 2048 with unit spread (64 draws: loose bounds)
    logs = np.log(c3.astype(np.float64))
    assert abs(np.median(logs) - math.log(2048)) < 0.5
    assert 0.6 < np.std(logs) < 1.4
    c4 = _lengths("R16_k4_H64_len16k-64k")
    assert c4.size == 16 and c4.min() >= 16384 and c4.max() <= 65536
    c5 = _lengths("R128_k7_H64_skewed128k")
    assert c5.size == 128
    assert int(np.sum(c5 == 131072)) == 1 and int(np.sum(c5 == 32768)) == 7
    rest = c5[(c5 != 131072) & (c5 != 32768)]
    assert rest.size == 120 and rest.min() >= 512 and rest.max() <= 4096
    assert not np.all(np.diff(c5) <= 0)          # the rows are shuffled, not sorted


def test_lengths_are_seeded():
    for name in SHAPES:
        assert np.array_equal(_lengths(name), _lengths(name))
    w = WORKLOADS["R32_k4_H8_len1k-8k"]
    other = draw_lengths(w.lengths, w.R, torch.Generator().manual_seed(w.seed + 1))
    assert not np.array_equal(_lengths(w.name), other)


def test_block_tables_partition_the_pages():
    lens = (100, 37, 0, 64, 65, 1)
    b = make_batch_from_lengths(lens, 2, 3, seed=5, fill=-9, extra_pages=4)
    pages = [(L + PAGE - 1) // PAGE for L in lens]
    bt = b.block_table.numpy()
    assert bt.shape == (len(lens), max(pages)) and b.kv.shape == (sum(pages) + 4, PAGE, 576)
    used = []
    for r, p in enumerate(pages):
        used += bt[r, :p].tolist()
        assert np.all(bt[r, p:] == -9)           # past the request's pages: the fill
    assert sorted(used) == sorted(set(used))      # no page shared between requests
    assert set(used) <= set(range(b.kv.shape[0]))
    assert b.seq_lens.tolist() == list(lens)
    assert b.q.shape == (len(lens) * 2, 3, 576)


def test_batches_are_deterministic():
    a = make_batch_from_lengths((300, 70), 3, 4, seed=11, scaling="amax")
    b = make_batch_from_lengths((300, 70), 3, 4, seed=11, scaling="amax")
    c = make_batch_from_lengths((300, 70), 3, 4, seed=12, scaling="amax")
    for x, y in ((a.q, b.q), (a.kv, b.kv), (a.block_table, b.block_table)):
        assert torch.equal(x, y)
    assert a.q_scale == b.q_scale and a.kv_scale == b.kv_scale
    assert not torch.equal(a.kv, c.kv)
    t1, t2 = make_batch("R2_k4_H8_len100+37"), make_batch("R2_k4_H8_len100+37")
    assert torch.equal(t1.kv, t2.kv) and t1.seq_lens.tolist() == [100, 37]


def _decode(codes):
    return codes.view(torch.float8_e4m3fn).float()


def test_quantisation():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(4096, generator=g) * 7.0
    codes, scale = quantize(x.clone(), "amax")
    assert codes.dtype == torch.uint8
    assert scale == float(np.float32(float(x.abs().max()) / E4M3_MAX))
    assert float(_decode(codes).abs().max()) == E4M3_MAX   # amax lands on 448 exactly
    assert not torch.any((codes & 0x7F) == 0x7F)            # no E4M3 NaN codes
    # the stored codes are the round-to-nearest E4M3 of x / scale
    assert torch.equal(codes, (x / scale).clamp(-E4M3_MAX, E4M3_MAX)
                       .to(torch.float8_e4m3fn).view(torch.uint8))
    big = torch.tensor([1000.0, -1000.0, 3.0])
    ucodes, uscale = quantize(big.clone(), "unit")
    assert uscale == 1.0 and _decode(ucodes).tolist() == [448.0, -448.0, 3.0]   # clipped


def test_w_uv_is_seeded_bf16_with_unit_output_scale():
    w = make_w_uv(4, seed=9)
    assert w.dtype == torch.bfloat16 and w.shape == (4, 512, 128)
    assert torch.equal(w, make_w_uv(4, seed=9)) and not torch.equal(w, make_w_uv(4, seed=10))
    # N(0, 1) / sqrt(512) per element: each column has unit norm on average
    col = w.float().pow(2).sum(dim=1)
    assert abs(float(col.mean()) - 1.0) < 0.05
