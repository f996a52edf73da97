"""LSE merge of split-KV partials, in float64.

Test infrastructure only (see the package docstring).

Follows the combine the pages describe for partial rows over disjoint key sets
(drafter-attention page, ``DraftDcp``: each partial weighted by
exp2(lse - max) over the sum of the weights; balanced-MLA page, module
overview: FP32 split partials with a log2 LSE, reduced per row). Each partial
is its key set's normalised output with that set's base-2 LSE; the merged LSE
is max + log2(sum of weights).

A partial over an empty key set has lse = -inf and weight 0. If every partial
is empty the row is empty: out = 0, lse = -inf.
"""
from __future__ import annotations

import numpy as np


def combine(parts_out, parts_lse):
    """parts_out: [S, n, D], parts_lse: [S, n] -> out [n, D], lse [n]."""
    o = np.asarray(parts_out, dtype=np.float64)
    l = np.asarray(parts_lse, dtype=np.float64)
    mx = l.max(axis=0)                                   # [n]
    empty = np.isneginf(mx)
    safe = np.where(empty, 0.0, mx)
    w = np.where(np.isneginf(l), 0.0, np.exp2(l - safe[None, :]))   # [S, n]
    z = w.sum(axis=0)
    zsafe = np.where(empty, 1.0, z)
    out = (w[:, :, None] * o).sum(axis=0) / zsafe[:, None]
    out[empty] = 0.0
    lse = np.where(empty, -np.inf, safe + np.log2(zsafe))
    return out, lse
