"""Helpers for the GPU tests: move a host batch to the device, run the folded
decode through the C ABI, compare with the oracle at the stated tolerance."""
from __future__ import annotations

import math

import numpy as np
import torch

import mla_decode_attention_folded_gb300 as mla
import oracle.attention as att

# Tolerances of the decode: |out - ref| <= ATOL + RTOL |ref|, |lse2 - ref| <= LSE_TOL.
ATOL, RTOL, LSE_TOL = 2e-2, 2e-2, 1e-3


def bmm_scales(b):
    bmm1 = float(np.float32(b.sm_scale) * np.float32(b.q_scale) * np.float32(b.kv_scale))
    return bmm1, float(b.kv_scale)


def to_device(b, dev="cuda"):
    return dict(q=b.q.to(dev), kv=b.kv.to(dev), bt=b.block_table.to(dev),
                lens=b.seq_lens.to(dev))


def unfold(b):
    """The stock flattened layout: R*k single-token rows, replicated tables."""
    rep = torch.arange(b.R).repeat_interleave(b.k)
    return dict(R=b.R * b.k, k=1, H=b.H, bt=b.block_table[rep].contiguous(),
                lens=b.seq_lens[rep].contiguous())


def run_decode(b, policy=mla.POLICY_BALANCED, num_ctas=None, folded=True,
               min_split_tokens=256, max_splits=64, dev="cuda", d=None, groups=1):
    """-> (out [R, k*H, 512] float32 CPU, lse [R, k*H] CPU, status int, plan).
    folded=False runs the stock flattened layout with replicated tables;
    groups > 1 runs row groups of k/groups tokens on the request's own KV."""
    d = d or to_device(b, dev)
    if folded:
        R, k, H, bt, lens = b.R, b.k, b.H, d["bt"], d["lens"]
    else:
        u = unfold(b)
        R, k, H, bt, lens = u["R"], u["k"], u["H"], u["bt"].to(dev), u["lens"].to(dev)
    if num_ctas is None:
        num_ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    eng = mla.FoldedMla(R, k, H, bt.shape[1], d["kv"].shape[0], dev, num_ctas=num_ctas,
                        min_split_tokens=min_split_tokens, max_splits=max_splits, policy=policy,
                        groups=groups if folded else 1)
    bmm1, bmm2 = bmm_scales(b)
    eng.plan(lens)
    out, lse = eng.decode(d["q"], d["kv"], bt, lens, bmm1, bmm2)
    torch.cuda.synchronize()
    out = out.float().reshape(b.R, b.M, 512).cpu()
    lse = lse.reshape(b.R, b.M).cpu()
    return out, lse, int(eng.status.item()), (eng.counts.cpu(), eng.work.cpu())


def oracle_full(b):
    o, l = att.mla_decode(b.q.numpy(), b.kv.numpy(), b.block_table.numpy(), b.seq_lens.numpy(),
                          b.k, b.sm_scale, b.q_scale, b.kv_scale)
    return o.reshape(b.R, b.M, 512), l.reshape(b.R, b.M)


def assert_close(out, lse, ref_o, ref_l, what=""):
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite out"
    err = np.abs(out - ref_o) - (ATOL + RTOL * np.abs(ref_o))
    assert err.max() <= 0, f"{what}: out exceeds tolerance by {err.max():.3e} " \
                           f"(max abs err {np.abs(out - ref_o).max():.3e})"
    both_inf = np.isneginf(lse) & np.isneginf(ref_l)
    with np.errstate(invalid="ignore"):
        lerr = np.where(both_inf, 0.0, np.abs(lse - ref_l))
    assert np.all(np.isfinite(lerr)) and lerr.max() <= LSE_TOL, \
        f"{what}: lse error {np.nanmax(lerr):.3e}"
