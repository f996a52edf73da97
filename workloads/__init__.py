"""Seeded synthetic inputs for the folded FP8 MLA decode.

This module is shared by the CPU oracle (``oracle/``), the tests and the
benchmark. It holds no arithmetic of the method itself: it only draws random
values, quantises them to FP8 E4M3 codes with PyTorch's own cast (the stored
inputs), lays out the paged cache and its block tables, and names the
workloads.

Workloads follow the shapes the pages describe for the Kimi-K3 draft block
(drafter-attention page, module overview: R requests x k draft tokens x H
heads, 576-dim FP8 latent rows of 512 latent + 64 rope, page size 64). No
public dataset exists for this path; every workload is synthetic.

Recipe (stated once, used everywhere):

* lengths: ``fixed`` list, ``uniform`` integers in [lo, hi] inclusive,
  ``lognormal`` round(exp(N(ln median, sigma))) clipped to [lo, hi], or
  ``skewed`` (a head of fixed long requests, the rest uniform in [lo, hi]),
  shuffled with the seed;
* values: Q and KV drawn N(0, 1) * ``value_std`` in float32;
* quantisation: ``unit`` clips to +-448 and casts with scale 1.0; ``amax``
  uses scale = amax / 448 (float32) and stores e4m3(clip(x / scale, +-448));
  PyTorch's cast rounds to nearest even and does not saturate, hence the clip;
* pages: one random permutation of [0, total pages) handed out to the
  requests in order; block-table entries past a request's pages hold
  ``fill`` (0 for timing runs, an out-of-range sentinel in bounds tests);
* softmax scale 1/sqrt(192) (qk_nope 128 + rope 64) for every workload;
* W_UV (the up-projection after the merge): N(0, 1) / sqrt(512) per element,
  rounded to BF16, seeded per use (``make_w_uv``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Sequence

import numpy as np
import torch

PAGE = 64          # tokens per cache page
D_QK = 576         # latent 512 + rope 64
D_V = 512          # kv_lora_rank: the value is the latent slice of the key row
E4M3_MAX = 448.0
SM_SCALE = 1.0 / math.sqrt(192.0)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int
    k: int
    H: int
    lengths: tuple
    value_std: float
    scaling: str            # "unit" or "amax"
    seed: int

    @property
    def M(self) -> int:
        return self.k * self.H


# The five workloads, named by what they are and their sizes.
WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in (
        Workload("R2_k4_H8_len100+37", 2, 4, 8, ("fixed", (100, 37)), 1.0, "unit", 1000),
        Workload("R32_k4_H8_len1k-8k", 32, 4, 8, ("uniform", 1024, 8192), 0.5, "amax", 1001),
        Workload("R64_k7_H8_lognormal2k", 64, 7, 8, ("lognormal", 2048, 1.0, 256, 32768), 1.0, "amax", 1002),
        Workload("R16_k4_H64_len16k-64k", 16, 4, 64, ("uniform", 16384, 65536), 1.0, "amax", 1003),
        Workload("R128_k7_H64_skewed128k", 128, 7, 64,
                 ("skewed", (131072,) + (32768,) * 7, 512, 4096), 1.0, "amax", 1004),
    )
}
ORDER = list(WORKLOADS)      # tiny first, then the four full-size workloads


@dataclasses.dataclass
class Batch:
    """One decode batch on the host. FP8 tensors hold raw E4M3 codes (uint8)."""
    q: torch.Tensor            # [R*k, H, 576] uint8, token-major per request
    kv: torch.Tensor           # [num_pages, 64, 576] uint8
    block_table: torch.Tensor  # [R, max_pages] int32
    seq_lens: torch.Tensor     # [R] int32
    k: int
    H: int
    q_scale: float
    kv_scale: float
    sm_scale: float = SM_SCALE

    @property
    def R(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def M(self) -> int:
        return self.k * self.H


def draw_lengths(spec: tuple, R: int, gen: torch.Generator) -> np.ndarray:
    kind = spec[0]
    if kind == "fixed":
        out = np.asarray(spec[1], dtype=np.int64)
        assert out.size == R
        return out
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return torch.randint(lo, hi + 1, (R,), generator=gen).numpy().astype(np.int64)
    if kind == "lognormal":
        median, sigma, lo, hi = spec[1:]
        z = torch.randn(R, generator=gen, dtype=torch.float64).numpy()
        return np.clip(np.round(np.exp(np.log(median) + sigma * z)), lo, hi).astype(np.int64)
    if kind == "skewed":
        head, lo, hi = spec[1], spec[2], spec[3]
        rest = torch.randint(lo, hi + 1, (R - len(head),), generator=gen).numpy()
        out = np.concatenate([np.asarray(head, dtype=np.int64), rest.astype(np.int64)])
        perm = torch.randperm(R, generator=gen).numpy()
        return out[perm]
    raise ValueError(f"unknown length recipe {kind!r}")


def quantize(x: torch.Tensor, scaling: str) -> tuple[torch.Tensor, float]:
    """float32 values -> (E4M3 codes as uint8, per-tensor scale)."""
    if scaling == "unit":
        scale = 1.0
        y = x
    elif scaling == "amax":
        amax = float(x.abs().max())
        scale = float(np.float32(amax / E4M3_MAX)) if amax > 0 else 1.0
        y = x / scale
    else:
        raise ValueError(scaling)
    codes = y.clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def make_batch_from_lengths(lengths: Sequence[int], k: int, H: int, *, seed: int,
                            value_std: float = 1.0, scaling: str = "unit",
                            fill: int = 0, extra_pages: int = 0,
                            max_pages: int | None = None) -> Batch:
    """A batch with the given per-request KV lengths (any R, k, H)."""
    gen = torch.Generator().manual_seed(seed)
    lens = np.asarray(lengths, dtype=np.int64)
    R = lens.size
    pages = (lens + PAGE - 1) // PAGE
    total = int(pages.sum())
    num_pages = max(1, total + extra_pages)
    width = max(1, int(pages.max()) if R else 1)
    if max_pages is not None:
        assert max_pages >= width
        width = max_pages
    perm = torch.randperm(num_pages, generator=gen).numpy().astype(np.int64)
    bt = np.full((R, width), fill, dtype=np.int64)
    off = 0
    for i in range(R):
        bt[i, : pages[i]] = perm[off: off + pages[i]]
        off += pages[i]
    qf = torch.randn((R * k, H, D_QK), generator=gen, dtype=torch.float32) * value_std
    q, q_scale = quantize(qf, scaling)
    del qf
    kvf = torch.randn((num_pages, PAGE, D_QK), generator=gen, dtype=torch.float32) * value_std
    kv, kv_scale = quantize(kvf, scaling)
    del kvf
    return Batch(q=q.contiguous(), kv=kv.contiguous(),
                 block_table=torch.from_numpy(bt.astype(np.int32)),
                 seq_lens=torch.from_numpy(lens.astype(np.int32)),
                 k=k, H=H, q_scale=q_scale, kv_scale=kv_scale)


def make_batch(name: str, *, fill: int = 0) -> Batch:
    """The named workload's batch, seeded by its seed (1000 + its index)."""
    w = WORKLOADS[name]
    gen = torch.Generator().manual_seed(w.seed)
    lens = draw_lengths(w.lengths, w.R, gen)
    return make_batch_from_lengths(lens, w.k, w.H, seed=w.seed + 7919, value_std=w.value_std,
                                   scaling=w.scaling, fill=fill)



def shard_pages(batch: Batch, shards: int, shard: int) -> Batch:
    """The part of `batch` that shard `shard` of `shards` holds when each
    request's KV pages are interleaved over the shards page by page (page p of
    a request lives on shard p % shards), as a decode-context-parallel cache
    is laid out. Queries and the cache buffer are shared; the block table and
    lengths are the shard's local ones (its pages in order; only a request's
    last page can be partial, and it is also the last page of its shard)."""
    lens = batch.seq_lens.numpy().astype(np.int64)
    bt = batch.block_table.numpy()
    R = lens.size
    local_pages = [list(range(shard, int((L + PAGE - 1) // PAGE), shards)) for L in lens]
    width = max(1, max(len(p) for p in local_pages))
    lbt = np.zeros((R, width), dtype=np.int32)
    llen = np.zeros(R, dtype=np.int32)
    for r, pages in enumerate(local_pages):
        for j, p in enumerate(pages):
            lbt[r, j] = bt[r, p]
            llen[r] += min(PAGE, int(lens[r]) - PAGE * p)
    return Batch(q=batch.q, kv=batch.kv, block_table=torch.from_numpy(lbt),
                 seq_lens=torch.from_numpy(llen), k=batch.k, H=batch.H,
                 q_scale=batch.q_scale, kv_scale=batch.kv_scale, sm_scale=batch.sm_scale)


def make_w_uv(H: int, seed: int) -> torch.Tensor:
    """Synthetic per-head W_UV [H, 512, 128] as BF16 (no trained weights exist
    here): N(0, 1) / sqrt(512) drawn in float32, rounded to BF16 by PyTorch's
    cast, so each output has about unit variance for unit-variance inputs."""
    gen = torch.Generator().manual_seed(seed)
    w = torch.randn((H, D_V, 128), generator=gen, dtype=torch.float32) / math.sqrt(D_V)
    return w.to(torch.bfloat16)
