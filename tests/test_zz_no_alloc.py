"""The allocation-free decode entry point against the regular one.

mla_folded_decode_noalloc serves callers that may not allocate device memory
(for example a host application whose own allocator owns the GPU, or code that
runs while a memory pool is being sized): it keeps the split-KV partials in a
fixed device array inside the library rather than in a caller workspace. On
the same plan it runs the same kernels as mla_folded_decode followed by
mla_split_combine, so its results must be bit-identical to theirs. This file
runs last so that a failure here never hides the other tests; it also passes
alone in a fresh process.
"""
import ctypes

import pytest
import torch

import mla_decode_attention_folded_gb300 as mla
from mla_decode_attention_folded_gb300 import _lib
from tests.gpu_util import assert_close, bmm_scales, oracle_full, to_device
from workloads import make_batch_from_lengths

pytestmark = pytest.mark.gpu


def _decode_both(b):
    """(regular out, lse), (no-alloc out, lse) for one batch, same plan."""
    d = to_device(b)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    eng = mla.FoldedMla(b.R, b.k, b.H, d["bt"].shape[1], d["kv"].shape[0], "cuda", num_ctas=G,
                        min_split_tokens=64)
    bmm1, bmm2 = bmm_scales(b)
    eng.plan(d["lens"])
    ref_o, ref_l = eng.decode(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2)
    out = torch.full((b.R, b.M, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((b.R, b.M), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.folded_decode_noalloc(eng.shape, d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2,
                              eng.counts, eng.work, out, lse, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(eng.status.item()) == 0
    assert int(eng.counts.max()) >= 2          # the scratch really held partials
    return (ref_o.cpu(), ref_l.cpu()), (out.cpu(), lse.cpu())


def test_noalloc_matches_regular_entry_point_twice_in_a_row():
    first = make_batch_from_lengths((3000, 700, 64, 0, 1900), 4, 8, seed=101, scaling="amax")
    second = make_batch_from_lengths((5000, 130, 2600), 7, 8, seed=202, scaling="amax")
    for b in (first, second):
        (ro, rl), (o, l) = _decode_both(b)
        assert torch.equal(o.view(torch.int16), ro.view(torch.int16)), "out differs"
        assert torch.equal(l, rl), "lse differs"
        ref_o, ref_l = oracle_full(b)
        assert_close(o.float().numpy(), l.numpy(), ref_o, ref_l, "no-alloc vs oracle")


def test_noalloc_on_a_packed_plan():
    """Eleven requests of 256 rows (four row blocks) on every SM: the plan packs
    the requests' pages into equal per-unit segments; the allocation-free call
    and the regular one agree bit for bit and with the oracle."""
    from oracle import planner as pl
    lens = (13435, 22970, 14236, 18445, 2082, 8967, 5989, 10509, 4787, 11033, 22350)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    _, packed = pl.plan_pieces(lens, 256, G, 64, 64, pl.BALANCED)
    if not packed:
        pytest.skip("this device's SM count does not pack the batch")
    b = make_batch_from_lengths(lens, 4, 64, seed=303, scaling="amax")
    (ro, rl), (o, l) = _decode_both(b)
    assert torch.equal(o.view(torch.int16), ro.view(torch.int16)), "out differs"
    assert torch.equal(l, rl), "lse differs"
    ref_o, ref_l = oracle_full(b)
    assert_close(o.float().numpy(), l.numpy(), ref_o, ref_l, "no-alloc, packed plan")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # Every device pointer is NULL: a working size check returns
    # MLA_ERR_SCRATCH_LIMIT first; were it missing, the null checks of the
    # decode would refuse the call before any launch.
    lib = _lib.load()
    s = mla.make_shape(1024, 64, 64, 4096, 1 << 20, 2048)      # M = 4096 rows per request
    assert mla.workspace_bytes(s) > _lib.NOALLOC_SCRATCH_BYTES
    rc = lib.mla_folded_decode_noalloc(ctypes.byref(s), None, None, None, None, 1.0, 1.0, None, None,
                                       mla.plan_list_len(s), None, None, None, None)
    assert rc == -8                                             # MLA_ERR_SCRATCH_LIMIT
