"""Exact absorbed-MLA decode over a paged FP8 latent cache, in float64.

Test infrastructure only (see the package docstring).

Definition followed (drafter-attention page, module overview and
``folded_decode``; balanced-MLA page, module overview and ``BalancedMla.decode``):

* The cache holds one latent row of 576 dims per key: dims 0..511 are the
  latent (also the value, ``kv_lora_rank`` = 512) and 512..575 the rope part.
  Key j of request r lives in page ``block_table[r][j // 64]``, slot j % 64.
* Absorbed MLA decode is MQA: every query row (token t, head h) of request r
  attends, with its own softmax, over the same keys j < seq_lens[r]. A draft
  block is non-causal, so there is no mask beyond the length.
* Scores are ``sm_scale * (q_scale * Q) . (kv_scale * K)``, the stock bmm1
  scale applied to raw FP8 dot products (drafter-attention page, ``_scales``).
* The output is the softmax-weighted sum of the 512 value dims; the returned
  LSE is base 2 over the scaled scores (balanced-MLA page: log2 LSE).

The fold changes no result (drafter-attention page, module overview: the same
attention, exactly), so this oracle has no fold: it computes each (token, head)
row of the stock layout ``[R*k, H, ...]``. The folded ``[R, k*H, ...]`` output
has the same memory order.

Readings where the pages are silent (listed again in the design notes):

* an empty request (length 0) yields out = 0 and lse = -inf;
* ``key_range`` restricts request r to keys [j0, j1): the split partial of the
  split-KV decode, normalised by its own sum, with its own LSE.
"""
from __future__ import annotations

import math

import numpy as np

from . import e4m3

PAGE = 64
D_QK = 576
D_V = 512
LN2 = math.log(2.0)


def request_keys(kv_codes, block_table_row, j0: int, j1: int, kv_scale: float) -> np.ndarray:
    """Dequantised key rows j0..j1-1 of one request: [j1-j0, 576] float64."""
    j = np.arange(j0, j1, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[j // PAGE]
    slots = j % PAGE
    kv = np.asarray(kv_codes)
    return e4m3.decode(kv[pages, slots, :]) * float(kv_scale)


def attend(qd: np.ndarray, kd: np.ndarray, sm_scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Softmax attention of dequantised query rows over dequantised key rows.

    qd: [n, 576], kd: [L, 576]. Returns out [n, 512] and the base-2 LSE [n]
    of the scaled scores. L = 0 gives out = 0, lse = -inf.
    """
    n = qd.shape[0]
    if kd.shape[0] == 0:
        return np.zeros((n, D_V)), np.full(n, -np.inf)
    s = sm_scale * (qd @ kd.T)                          # [n, L] scores
    mx = s.max(axis=1, keepdims=True)
    e = np.exp(s - mx)
    z = e.sum(axis=1, keepdims=True)
    out = (e / z) @ kd[:, :D_V]                         # value = latent slice
    lse_natural = mx[:, 0] + np.log(z[:, 0])
    return out, lse_natural / LN2


def mla_decode(q_codes, kv_codes, block_table, seq_lens, tokens_per_request: int,
               sm_scale: float, q_scale: float, kv_scale: float,
               key_range=None, requests=None):
    """Stock-layout decode of R requests x k tokens.

    q_codes: [R*k, H, 576] uint8 E4M3; kv_codes: [pages, 64, 576] uint8;
    block_table: [R, max_pages]; seq_lens: [R].
    key_range: optional [R, 2] array of per-request key ranges [j0, j1).
    requests: optional subset of request indices to compute (others stay NaN).
    Returns out [R*k, H, 512] and lse2 [R*k, H] in float64.
    """
    q = np.asarray(q_codes)
    rows, H, dim = q.shape
    assert dim == D_QK
    k = int(tokens_per_request)
    lens = np.asarray(seq_lens, dtype=np.int64)
    R = lens.size
    assert rows == R * k
    out = np.full((rows, H, D_V), np.nan)
    lse = np.full((rows, H), np.nan)
    for r in (range(R) if requests is None else requests):
        j0, j1 = (0, int(lens[r])) if key_range is None else (int(key_range[r][0]), int(key_range[r][1]))
        kd = request_keys(kv_codes, np.asarray(block_table)[r], j0, j1, kv_scale)
        qd = e4m3.decode(q[r * k:(r + 1) * k].reshape(k * H, D_QK)) * float(q_scale)
        o, l2 = attend(qd, kd, sm_scale)
        out[r * k:(r + 1) * k] = o.reshape(k, H, D_V)
        lse[r * k:(r + 1) * k] = l2.reshape(k, H)
    return out, lse


def mla_decode_rows(q_codes, kv_codes, block_table, seq_lens, tokens_per_request: int,
                    sm_scale: float, q_scale: float, kv_scale: float, picks):
    """Selected (request, folded row m = t*H + h) outputs only: for sampled
    parity checks on workloads too large to decode whole on the CPU.
    Returns out [len(picks), 512] and lse2 [len(picks)]."""
    q = np.asarray(q_codes)
    _, H, _ = q.shape
    k = int(tokens_per_request)
    lens = np.asarray(seq_lens, dtype=np.int64)
    outs, lses = [], []
    for r, m in picks:
        t, h = divmod(int(m), H)
        kd = request_keys(kv_codes, np.asarray(block_table)[r], 0, int(lens[r]), kv_scale)
        qd = e4m3.decode(q[r * k + t, h][None, :]) * float(q_scale)
        o, l2 = attend(qd, kd, sm_scale)
        outs.append(o[0])
        lses.append(l2[0])
    return np.stack(outs), np.array(lses)
