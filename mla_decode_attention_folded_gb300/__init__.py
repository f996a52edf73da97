"""Folded, KV-balanced FP8 MLA decode for GB300 (sm_103a).

A thin Python binding over the C ABI of ``include/mlafold.h``: it marshals
PyTorch device tensors into pointers and calls the library; every step of the
decode runs in the library's CUDA kernels. PyTorch only owns the memory and
the stream.

The API follows the pages (drafter-attention page, ``folded_decode``;
balanced-MLA page, ``BalancedMla.require`` / ``plan`` / ``decode``):

* ``FoldedMla(R, k, H, max_pages, num_pages, device)`` allocates the plan
  buffers (``counts`` zeros, ``work`` -1) and the split-KV workspace up front,
  so nothing is allocated later (and a CUDA graph can capture the calls);
* ``.plan(seq_lens)`` plans the step's splits on the device, once per step;
* ``.decode(q, kv, block_table, seq_lens, bmm1_scale, bmm2_scale)`` runs the
  split-KV decode and the LSE reduction: BF16 ``out [R, k*H, 512]`` and the
  base-2 ``lse [R, k*H]``, in the stock token-major-then-head order.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (FAULT_PAGE_RANGE, FAULT_WAIT_TIMEOUT, FAULT_WORK_ITEM, MlaError, MlaShape,
                   POLICY_BALANCED, POLICY_UNIFORM)

__all__ = ["MlaShape", "MlaError", "POLICY_BALANCED", "POLICY_UNIFORM", "make_shape",
           "plan_list_len", "workspace_bytes", "plan_splits", "folded_decode",
           "split_combine", "uv_combine", "lse_merge", "folded_decode_noalloc",
           "folded_decode_wait_test", "tier_plan", "row_copy", "balanced_tiers", "TIERS", "MOVE",
           "FoldedMla", "TieredMla", "fold_factor", "FAULT_WAIT_TIMEOUT", "FAULT_PAGE_RANGE",
           "FAULT_WORK_ITEM", "library_path"]

PAGE = 64


def library_path() -> str:
    return _lib.LIB_PATH


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def make_shape(R: int, k: int, H: int, max_pages: int, num_pages: int, num_ctas: int,
               min_split_tokens: int = 256, max_splits: int = 64,
               policy: int = POLICY_BALANCED, groups: int = 1) -> MlaShape:
    return MlaShape(R, k, H, PAGE, max_pages, num_pages, num_ctas, min_split_tokens,
                    max_splits, policy, groups)


def fold_factor(k: int, H: int, max_heads: int = 128) -> int:
    """Tokens folded into one decode row when a row may hold at most
    `max_heads` heads: the largest divisor f of k with f * H <= max_heads
    (1 when even one token's heads exceed it). The drafter-attention page's
    `fold_plan` rule for the LSE-returning kernel (its example: k = 4 at 64
    heads folds pairs). Use groups = k // f row groups per request."""
    best = 1
    for f in range(1, k + 1):
        if k % f == 0 and f * H <= max_heads:
            best = f
    return best


def plan_list_len(shape: MlaShape) -> int:
    return _lib.check("mla_plan_list_len", _lib.load().mla_plan_list_len(ctypes.byref(shape)))


def workspace_bytes(shape: MlaShape) -> int:
    out = ctypes.c_size_t(0)
    _lib.check("mla_workspace_bytes", _lib.load().mla_workspace_bytes(ctypes.byref(shape),
                                                                      ctypes.byref(out)))
    return out.value


def plan_splits(shape: MlaShape, seq_lens, counts, work, stream=None) -> None:
    _lib.check("mla_plan_splits", _lib.load().mla_plan_splits(
        ctypes.byref(shape), _ptr(seq_lens), _ptr(counts), _ptr(work), work.numel(),
        _stream(stream)))


def folded_decode(shape: MlaShape, q, kv, block_table, seq_lens, bmm1_scale: float,
                  bmm2_scale: float, counts, work, workspace, out, lse, status=None,
                  stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.check("mla_folded_decode", _lib.load().mla_folded_decode(
        ctypes.byref(shape), _ptr(q), _ptr(kv), _ptr(block_table), _ptr(seq_lens),
        float(bmm1_scale), float(bmm2_scale), _ptr(counts), _ptr(work), work.numel(),
        _ptr(workspace), ws_bytes, _ptr(out), _ptr(lse), _ptr(status), _stream(stream)))


def folded_decode_wait_test(shape: MlaShape, q, kv, block_table, seq_lens, bmm1_scale: float,
                            bmm2_scale: float, counts, work, workspace, out, lse, status,
                            wait_limit_ns: int, stream=None) -> None:
    """Failure-detection test hook: the decode with every pipeline wait bounded
    by wait_limit_ns and CTA 0's first KV copy withheld, so that a wait runs
    out and MLA_FAULT_WAIT_TIMEOUT is set in `status` (see include/mlafold.h)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.check("mla_folded_decode_wait_test", _lib.load().mla_folded_decode_wait_test(
        ctypes.byref(shape), _ptr(q), _ptr(kv), _ptr(block_table), _ptr(seq_lens),
        float(bmm1_scale), float(bmm2_scale), _ptr(counts), _ptr(work), work.numel(),
        _ptr(workspace), ws_bytes, _ptr(out), _ptr(lse), _ptr(status), int(wait_limit_ns),
        _stream(stream)))


def split_combine(shape: MlaShape, counts, work, workspace, bmm2_scale: float, out, lse,
                  stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.check("mla_split_combine", _lib.load().mla_split_combine(
        ctypes.byref(shape), _ptr(counts), _ptr(work), work.numel(), _ptr(workspace), ws_bytes,
        float(bmm2_scale), _ptr(out), _ptr(lse), _stream(stream)))


def uv_combine(shape: MlaShape, counts, work, workspace, bmm2_scale: float, out, w_uv, y,
               status=None, stream=None) -> None:
    """The split reduction fused with the W_UV up-projection: y [R*k, H, 128]
    BF16 from the decode's workspace partials and one-split rows `out`, with
    w_uv [H, 128, 512] BF16 (W_UV[h] transposed, latent-contiguous)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _lib.check("mla_uv_combine", _lib.load().mla_uv_combine(
        ctypes.byref(shape), _ptr(counts), _ptr(work), work.numel(), _ptr(workspace), ws_bytes,
        float(bmm2_scale), _ptr(out), _ptr(w_uv), _ptr(y), _ptr(status), _stream(stream)))


def lse_merge(parts_out, parts_lse, out, lse, stream=None) -> None:
    """Merge S partial results over disjoint key sets: parts_out [S, rows, 512]
    BF16 and parts_lse [S, rows] FP32 log2 -> out [rows, 512], lse [rows]
    (the decode-context-parallel combine; see include/mlafold.h)."""
    S, rows = parts_lse.shape[0], parts_lse.numel() // parts_lse.shape[0]
    _lib.check("mla_lse_merge", _lib.load().mla_lse_merge(
        S, rows, _ptr(parts_out), _ptr(parts_lse), _ptr(out), _ptr(lse), _stream(stream)))


def folded_decode_noalloc(shape: MlaShape, q, kv, block_table, seq_lens, bmm1_scale: float,
                          bmm2_scale: float, counts, work, out, lse, status=None,
                          stream=None) -> None:
    """Decode plus LSE reduction with the library's own fixed device scratch
    (no workspace argument, no allocation): for callers that may not allocate
    device memory. Shapes whose workspace exceeds the library's 64 MiB scratch
    raise MlaError(MLA_ERR_SCRATCH_LIMIT). Calls that overlap on the GPU share
    that scratch and race."""
    _lib.check("mla_folded_decode_noalloc", _lib.load().mla_folded_decode_noalloc(
        ctypes.byref(shape), _ptr(q), _ptr(kv), _ptr(block_table), _ptr(seq_lens),
        float(bmm1_scale), float(bmm2_scale), _ptr(counts), _ptr(work), work.numel(), _ptr(out),
        _ptr(lse), _ptr(status), _stream(stream)))


# The tiered launch's constants. The pages name TIERS and MOVE without values
# (drafter-attention page, `balanced_tiers`, `_balanced_tables`); these are
# this library's: tiers of 8, 16 and 32 rows, and a row moves when it is longer
# than one pair's share of the batch's keys.
TIERS = (8, 16, 32)
MOVE = (1, 1)


def balanced_tiers(rows: int, sms: int, tiers=TIERS) -> tuple:
    """Tier sizes for `rows` decode rows on `sms` SMs (drafter-attention page,
    `balanced_tiers`): none when rows * 4 <= sms, else the sizes of `tiers` in
    order while their sum stays at most rows // 2."""
    if rows * 4 <= sms:
        return ()
    out: list = []
    for size in tiers:
        if sum(out) + size > rows // 2:
            break
        out.append(size)
    return tuple(out)


def tier_plan(rows: int, split_rows: int, pairs: int, move, seq_lens, rest_lens, tier_rows,
              tier_lens, stream=None) -> None:
    """Which rows move into the tiers (see mla_tier_plan in include/mlafold.h)."""
    _lib.check("mla_tier_plan", _lib.load().mla_tier_plan(
        rows, split_rows, pairs, int(move[0]), int(move[1]), _ptr(seq_lens), _ptr(rest_lens),
        _ptr(tier_rows), _ptr(tier_lens), _stream(stream)))


def row_copy(src, dst, index, targets: int, bound: int, gather: bool, stream=None) -> None:
    """Whole-row gather (dst[i] = src[index[i]]) or scatter (dst[index[i]] =
    src[i]) of the rows whose index lies in [0, bound); rows are the leading
    dimension of src and dst (see mla_row_copy in include/mlafold.h)."""
    row_bytes = src[0].numel() * src.element_size()
    if dst[0].numel() * dst.element_size() != row_bytes:
        raise ValueError("src and dst rows differ in size")
    _lib.check("mla_row_copy", _lib.load().mla_row_copy(
        _ptr(src), _ptr(dst), _ptr(index), int(targets), int(bound), int(row_bytes),
        1 if gather else 0, _stream(stream)))


class FoldedMla:
    """Plan buffers and split-KV workspace of one decode shape. `groups` row
    groups per request (a divisor of k): 1 folds all k tokens into one decode
    row, k is the stock unfolded layout, `k // fold_factor(k, H)` the partial
    fold of the pages' `fold_plan`; out and lse keep the same layout.

    Everything is allocated here, before any capture; ``plan`` and ``decode``
    only launch kernels (balanced-MLA page, ``BalancedMla.require``: prepared
    before capture, one shared scratch)."""

    def __init__(self, R: int, k: int, H: int, max_pages: int, num_pages: int,
                 device=None, num_ctas: int | None = None, min_split_tokens: int = 256,
                 max_splits: int = 64, policy: int = POLICY_BALANCED, groups: int = 1):
        self.device = torch.device(device if device is not None else "cuda")
        if num_ctas is None:
            num_ctas = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.shape = make_shape(R, k, H, max_pages, num_pages, num_ctas, min_split_tokens,
                                max_splits, policy, groups)
        self.R, self.k, self.H, self.M = R, k, H, k * H
        self.groups = groups
        i32 = dict(dtype=torch.int32, device=self.device)
        self.counts = torch.zeros(R * groups, **i32)
        self.work = torch.full((plan_list_len(self.shape),), -1, **i32)
        self.workspace = torch.empty(max(workspace_bytes(self.shape), 256), dtype=torch.uint8,
                                     device=self.device)
        self.status = torch.zeros(1, **i32)

    def plan(self, seq_lens, stream=None) -> None:
        plan_splits(self.shape, seq_lens, self.counts, self.work, stream)

    def decode(self, q, kv, block_table, seq_lens, bmm1_scale: float, bmm2_scale: float,
               out=None, lse=None, stream=None, return_lse: bool = True):
        """out [R, M, 512] BF16 and, with return_lse, the base-2 lse [R, M]
        (else None: the no-LSE route, nothing written for it)."""
        if out is None:
            out = torch.empty((self.R, self.M, 512), dtype=torch.bfloat16, device=self.device)
        if lse is None and return_lse:
            lse = torch.empty((self.R, self.M), dtype=torch.float32, device=self.device)
        if not return_lse:
            lse = None
        folded_decode(self.shape, q, kv, block_table, seq_lens, bmm1_scale, bmm2_scale,
                      self.counts, self.work, self.workspace, out, lse, self.status, stream)
        split_combine(self.shape, self.counts, self.work, self.workspace, bmm2_scale, out, lse,
                      stream)
        return out, lse

    def decode_uv(self, q, kv, block_table, seq_lens, bmm1_scale: float, bmm2_scale: float,
                  w_uv, y=None, out=None, stream=None):
        """The decode followed by the split reduction fused with W_UV:
        y [R*k, H, 128] BF16 (w_uv [H, 128, 512] BF16, latent-contiguous).
        `out` receives the one-split requests' rows only; no LSE is written."""
        if out is None:
            out = torch.empty((self.R, self.M, 512), dtype=torch.bfloat16, device=self.device)
        if y is None:
            y = torch.empty((self.R * self.k, self.H, 128), dtype=torch.bfloat16,
                            device=self.device)
        folded_decode(self.shape, q, kv, block_table, seq_lens, bmm1_scale, bmm2_scale,
                      self.counts, self.work, self.workspace, out, None, self.status, stream)
        uv_combine(self.shape, self.counts, self.work, self.workspace, bmm2_scale, out, w_uv, y,
                   self.status, stream)
        return y


class TieredMla:
    """The pages' tiered launch (drafter-attention page, `balanced_decode`),
    built from this library's kernels for comparison with the single
    persistent decode of `FoldedMla`: the longest decode rows move out of one
    unsplit launch into tiers of TIERS rows, each tier a decode launch of its
    own with split rows, on streams of decreasing priority (the unsplit launch
    on the highest, then the tiers from the coarsest split to the finest).

    One folded decode row per request (groups = 1). Split counts: the unsplit
    launch gives every row one split; a tier of m rows gets this library's
    uniform split count for m rows (the pages' stock kernel gives sms // (2m)
    splits: CTA pairs per row split; here the plan's concurrent items per row).
    Every buffer is allocated here, before any capture."""

    def __init__(self, R: int, k: int, H: int, max_pages: int, num_pages: int, device=None,
                 sms: int | None = None, tiers=None, move=MOVE):
        self.device = torch.device(device if device is not None else "cuda")
        if sms is None:
            sms = torch.cuda.get_device_properties(self.device).multi_processor_count
        self.R, self.k, self.H, self.M, self.max_pages = R, k, H, k * H, max_pages
        self.tiers = balanced_tiers(R, sms) if tiers is None else tuple(tiers)
        self.split_rows = sum(self.tiers)
        if self.split_rows > R:
            raise ValueError("the tiers hold more rows than the batch")
        self.pairs = max(1, sms // 2)
        self.move = tuple(move)
        self.unsplit = FoldedMla(R, k, H, max_pages, num_pages, self.device, num_ctas=sms,
                                 max_splits=1, policy=POLICY_UNIFORM)
        self.engines = [FoldedMla(m, k, H, max_pages, num_pages, self.device, num_ctas=sms,
                                  policy=POLICY_UNIFORM) for m in self.tiers]
        n = max(self.split_rows, 1)
        i32 = dict(dtype=torch.int32, device=self.device)
        self.rest = torch.zeros(R, **i32)
        self.tier_rows = torch.full((n,), R, **i32)
        self.tier_lens = torch.zeros(n, **i32)
        self.q_s = torch.empty((n * k, H, 576), dtype=torch.uint8, device=self.device)
        self.bt_s = torch.zeros((n, max_pages), **i32)
        self.out_s = torch.empty((n, self.M, 512), dtype=torch.bfloat16, device=self.device)
        self.lse_s = torch.empty((n, self.M), dtype=torch.float32, device=self.device)
        low, high = torch.cuda.Stream.priority_range()
        self.streams = [torch.cuda.Stream(self.device, priority=min(low, high + i))
                        for i in range(len(self.tiers) + 1)]

    def decode(self, q, kv, block_table, seq_lens, bmm1_scale: float, bmm2_scale: float,
               out=None, lse=None, return_lse: bool = True):
        """out [R, M, 512] BF16 and the base-2 lse [R, M] (None without
        return_lse), as FoldedMla.decode returns them."""
        if out is None:
            out = torch.empty((self.R, self.M, 512), dtype=torch.bfloat16, device=self.device)
        if lse is None and return_lse:
            lse = torch.empty((self.R, self.M), dtype=torch.float32, device=self.device)
        if not return_lse:
            lse = None
        main = torch.cuda.current_stream(self.device)
        R, k, n = self.R, self.k, self.split_rows
        tier_plan(R, n, self.pairs, self.move, seq_lens, self.rest, self.tier_rows,
                  self.tier_lens, main)
        first = self.streams[0]
        first.wait_stream(main)
        self.unsplit.plan(self.rest, first)
        self.unsplit.decode(q, kv, block_table, self.rest, bmm1_scale, bmm2_scale, out=out,
                            lse=lse, stream=first, return_lse=return_lse)
        if n:
            row_copy(q.view(R, -1), self.q_s.view(n, -1), self.tier_rows, n, R, True, main)
            row_copy(block_table, self.bt_s, self.tier_rows, n, R, True, main)
            launches, start = [], 0
            for m, eng in zip(self.tiers, self.engines):
                launches.append((start, m, eng))
                start += m
            for stream, (b, m, eng) in zip(self.streams[1:], reversed(launches)):
                stream.wait_stream(main)
                lens = self.tier_lens[b:b + m]
                eng.plan(lens, stream)
                eng.decode(self.q_s[b * k:(b + m) * k], kv, self.bt_s[b:b + m], lens, bmm1_scale,
                           bmm2_scale, out=self.out_s[b:b + m],
                           lse=self.lse_s[b:b + m] if return_lse else None, stream=stream,
                           return_lse=return_lse)
        for stream in self.streams:
            main.wait_stream(stream)
        if n:
            row_copy(self.out_s, out, self.tier_rows, n, R, False, main)
            if lse is not None:
                row_copy(self.lse_s, lse, self.tier_rows, n, R, False, main)
        return out, lse
