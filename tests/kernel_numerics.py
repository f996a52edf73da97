"""A float64/float32 model of the decode kernels' softmax arithmetic, for
deciding how P enters the PV product (test infrastructure, like the oracle;
nothing on the product path imports it).

The balanced-MLA page (module overview) fixes the precision contract: FP32
split partials, a row max kept while it grows by at most 2^8, and P stored as
E4M3, unscaled. It does not say how the softmax normaliser relates to the
rounded P. This model follows the kernels' steps tile by tile (128 keys):
scores in FP32 times bmm1 * log2(e); the lazy max (moved to 2 below the tile's
maximum when a score exceeds it by more than 8); P = 2^(x - m) in FP32; the PV
product accumulated in FP32; then one of three ways of feeding P:

* ``"two_term"`` -- the kernels' choice: P rounded to FP16, hi = e4m3(P16),
  lo = e4m3(P16 - hi), the MMA sees hi + lo; normaliser = FP32 sum of P;
* ``"one_term"`` -- one E4M3 term, normaliser = FP32 sum of P;
* ``"one_term_rounded_sum"`` -- one E4M3 term, normaliser = the sum of the
  E4M3 values the MMA used (out stays a convex combination of value rows);
  the LSE still from the FP32 sum.

E4M3 and FP16 roundings use PyTorch's casts (round to nearest even).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.attention as att

MODES = ("two_term", "one_term", "one_term_rounded_sum")
TILE = 128
LOG2E = 1.4426950408889634


def _e4m3(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).to(torch.float32).numpy()


def _bf16(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def simulate_rows(qd: np.ndarray, kd: np.ndarray, bmm1: float, bmm2: float, mode: str,
                  lead: float = 2.0):
    """One request decoded as one split. qd [n, 576] raw dequantised query
    codes (no scale), kd [L, 576] raw dequantised key codes; bmm1 and bmm2 as
    the kernels take them. Returns out [n, 512] (BF16-rounded, as float64) and
    the base-2 LSE [n]."""
    n, L = qd.shape[0], kd.shape[0]
    scale = np.float32(np.float64(bmm1) * LOG2E)
    s = (qd @ kd.T).astype(np.float32)                 # FP8 products, FP32 accumulation
    m = np.full(n, -np.inf, dtype=np.float32)
    l = np.zeros(n, dtype=np.float32)
    le = np.zeros(n, dtype=np.float32)
    o = np.zeros((n, 512), dtype=np.float32)
    v = kd[:, :512].astype(np.float32)
    for t0 in range(0, L, TILE):
        x = s[:, t0:t0 + TILE] * scale
        tm = x.max(axis=1)
        move = tm > m + np.float32(8.0)
        mn = np.where(move, tm - np.float32(lead), m).astype(np.float32)
        alpha = np.where(np.isneginf(m), np.float32(0.0),
                         np.exp2(np.minimum(m - mn, 0.0))).astype(np.float32)
        o *= alpha[:, None]
        l *= alpha
        le *= alpha
        m = mn
        p = np.exp2(x - m[:, None]).astype(np.float32)
        l += p.sum(axis=1, dtype=np.float32)
        if mode == "two_term":
            p16 = p.astype(np.float16)
            hi = _e4m3(p16.astype(np.float32))
            lo = _e4m3((p16 - hi.astype(np.float16)).astype(np.float32))
            w = hi + lo
        else:
            w = _e4m3(p)
            le += w.sum(axis=1, dtype=np.float32)
        o += w @ v[t0:t0 + TILE]
    norm = le if mode == "one_term_rounded_sum" else l
    out = _bf16((o / norm[:, None]) * np.float32(bmm2)).astype(np.float64)
    lse = m.astype(np.float64) + np.log2(l.astype(np.float64))
    return out, lse


def request_error(batch, r: int, mode: str):
    """(worst out excess over |err| <= 2e-2 + 2e-2 |ref| (negative = inside
    the bound), worst |lse err|) of request r of `batch`, against the oracle."""
    b = batch
    k, H = b.k, b.H
    L = int(b.seq_lens[r])
    codes = b.q.numpy()[r * k:(r + 1) * k].reshape(k * H, 576)
    qd = att.e4m3.decode(codes)
    kd = att.request_keys(b.kv.numpy(), b.block_table.numpy()[r], 0, L, 1.0)
    bmm1 = float(np.float32(b.sm_scale) * np.float32(b.q_scale) * np.float32(b.kv_scale))
    out, lse = simulate_rows(qd, kd, bmm1, float(b.kv_scale), mode)
    ref_o, ref_l = att.attend(qd * float(b.q_scale), kd * float(b.kv_scale), b.sm_scale)
    excess = np.abs(out - ref_o) - (2e-2 + 2e-2 * np.abs(ref_o))
    return float(excess.max()), float(np.abs(lse - ref_l).max())
