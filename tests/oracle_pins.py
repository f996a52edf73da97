"""Checks that pin the CPU oracle to things other than itself.

Each check returns a list of failure strings (empty = pass). They call the
oracle through its module attributes, so a test can plant a mistake in the
oracle (monkeypatching one of its functions) and confirm that some check
catches it.

Pins used (none re-types the oracle's own expression):
* brute force: pure-Python loops with math.exp / math.fsum, E4M3 decoded by
  PyTorch's float8_e4m3fn cast, pages looked up one key at a time;
* closed forms: one key; zero query (uniform weights); identical keys;
  one dominant key;
* library special case: float64 torch.softmax(S) @ V on one contiguous page;
* invariants: fold == unfold row by row, split-merge invariance, convexity;
* the per-row sampler against the brute force and the whole-batch oracle.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle.attention as att
import oracle.merge as merge
from workloads import make_batch_from_lengths

LOG2E = 1.0 / math.log(2.0)


def torch_decode(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def brute_force(batch):
    """Pure-Python per-(token, head) attention. Returns (out, lse2) stock layout."""
    q = torch_decode(batch.q.numpy()) * batch.q_scale
    kv = batch.kv.numpy()
    bt = batch.block_table.numpy()
    lens = batch.seq_lens.numpy()
    R, k, H = batch.R, batch.k, batch.H
    out = np.zeros((R * k, H, 512))
    lse = np.zeros((R * k, H))
    for r in range(R):
        L = int(lens[r])
        keys = []
        for j in range(L):
            page = int(bt[r][j // 64])
            keys.append(torch_decode(kv[page, j % 64]) * batch.kv_scale)
        for t in range(k):
            for h in range(H):
                qrow = q[r * k + t, h]
                if L == 0:
                    lse[r * k + t, h] = -math.inf
                    continue
                s = [batch.sm_scale * math.fsum(float(a) * float(b) for a, b in zip(qrow, key))
                     for key in keys]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                z = math.fsum(e)
                for d in range(512):
                    out[r * k + t, h, d] = math.fsum(e[j] * keys[j][d] for j in range(L)) / z
                lse[r * k + t, h] = (mx + math.log(z)) * LOG2E
    return out, lse


def run_oracle(batch, **kw):
    return att.mla_decode(batch.q.numpy(), batch.kv.numpy(), batch.block_table.numpy(),
                          batch.seq_lens.numpy(), batch.k, batch.sm_scale, batch.q_scale,
                          batch.kv_scale, **kw)


def _cmp(name, got, want, tol, fails):
    got = np.asarray(got)
    want = np.asarray(want)
    same_inf = np.isinf(got) & np.isinf(want) & (np.sign(got) == np.sign(want))
    with np.errstate(invalid="ignore"):
        diff = np.where(same_inf, 0.0, np.abs(got - want))
    if not np.all(np.isfinite(diff)) or diff.max(initial=0.0) > tol:
        fails.append(f"{name}: max diff {np.nanmax(diff) if diff.size else 0} > {tol}")


# Tiny cases for the brute force: (lengths, k, H, seed, value_std, scaling).
TINY_CASES = [
    ((100, 37), 4, 2, 11, 1.0, "unit"),
    ((1, 64, 65), 2, 3, 12, 1.0, "unit"),
    ((130,), 3, 1, 13, 0.5, "amax"),
    ((0, 7), 1, 4, 14, 1.0, "unit"),
]


_BF_CACHE: dict = {}


def _tiny(case):
    lens, k, H, seed, std, scaling = case
    b = make_batch_from_lengths(lens, k, H, seed=seed, value_std=std, scaling=scaling,
                                extra_pages=2)
    if case not in _BF_CACHE:          # the brute force never depends on the oracle
        _BF_CACHE[case] = brute_force(b)
    return b, _BF_CACHE[case]


def check_brute_force(cases=TINY_CASES):
    fails = []
    for case in cases:
        lens = case[0]
        b, (o_ref, l_ref) = _tiny(case)
        o, l = run_oracle(b)
        _cmp(f"bf out {lens}", o, o_ref, 1e-12, fails)
        _cmp(f"bf lse {lens}", l, l_ref, 1e-12, fails)
    return fails


def check_closed_forms():
    fails = []
    # (1) one key: out = V_0 exactly, lse2 = s_0 * log2(e).
    b = make_batch_from_lengths((1,), 2, 3, seed=21, extra_pages=3)
    o, l = run_oracle(b)
    page = int(b.block_table[0, 0])
    key = torch_decode(b.kv[page, 0].numpy()) * b.kv_scale
    q = torch_decode(b.q.numpy()) * b.q_scale
    for t in range(2):
        for h in range(3):
            _cmp("one key out", o[t, h], key[:512], 1e-12, fails)
            s0 = b.sm_scale * float(np.dot(q[t, h], key))
            _cmp("one key lse", l[t, h], s0 * LOG2E, 1e-12, fails)
    # (2) zero query: every weight equal; lse2 = log2(L), out = mean of V.
    b = make_batch_from_lengths((77, 3), 2, 2, seed=22, extra_pages=1)
    b.q.zero_()
    o, l = run_oracle(b)
    for r, L in enumerate((77, 3)):
        keys = np.stack([torch_decode(b.kv[int(b.block_table[r, j // 64]), j % 64].numpy())
                         for j in range(L)]) * b.kv_scale
        mean = keys[:, :512].mean(axis=0)
        for t in range(2):
            for h in range(2):
                _cmp("zero q out", o[r * 2 + t, h], mean, 1e-12, fails)
                _cmp("zero q lse", l[r * 2 + t, h], math.log2(L), 1e-12, fails)
    # (3) identical keys: out = V, lse2 = s + log2(L).
    b = make_batch_from_lengths((90,), 1, 2, seed=23)
    row = b.kv[0, 0].clone()
    b.kv[:] = row
    o, l = run_oracle(b)
    key = torch_decode(row.numpy()) * b.kv_scale
    q = torch_decode(b.q.numpy()) * b.q_scale
    for h in range(2):
        _cmp("same keys out", o[0, h], key[:512], 1e-12, fails)
        s = b.sm_scale * float(np.dot(q[0, h], key))
        _cmp("same keys lse", l[0, h], s * LOG2E + math.log2(90), 1e-12, fails)
    # (4) one dominant key: out -> V of that key.
    b = make_batch_from_lengths((50,), 1, 1, seed=24)
    b.kv.zero_()
    b.q.zero_()
    one = torch.tensor([1.0]).to(torch.float8_e4m3fn).view(torch.uint8)
    big = torch.tensor([448.0]).to(torch.float8_e4m3fn).view(torch.uint8)
    b.q[0, 0, 520] = big[0]                       # a rope dim: scores need all 576 dims
    dom = 17
    pg, sl = int(b.block_table[0, dom // 64]), dom % 64
    b.kv[pg, sl, 520] = big[0]
    b.kv[pg, sl, 5] = one[0]                      # V of the dominant key: e_5
    o, l = run_oracle(b)
    want = np.zeros(512)
    want[5] = 1.0
    _cmp("dominant out", o[0, 0], want, 1e-9, fails)
    s_dom = b.sm_scale * 448.0 * 448.0
    _cmp("dominant lse", l[0, 0], s_dom * LOG2E, 1e-9, fails)
    return fails


def check_library_softmax():
    """float64 torch.softmax over one contiguous page equals the oracle."""
    fails = []
    b = make_batch_from_lengths((64,), 3, 4, seed=31, value_std=1.0)
    o, l = run_oracle(b)
    page = int(b.block_table[0, 0])
    K = torch.from_numpy(torch_decode(b.kv[page].numpy()) * b.kv_scale)
    Q = torch.from_numpy(torch_decode(b.q.numpy()) * b.q_scale).reshape(12, 576)
    S = b.sm_scale * (Q @ K.T)
    ref = torch.softmax(S, dim=-1) @ K[:, :512]
    lse = torch.logsumexp(S, dim=-1) / math.log(2.0)
    _cmp("lib out", o.reshape(12, 512), ref.numpy(), 1e-12, fails)
    _cmp("lib lse", l.reshape(12), lse.numpy(), 1e-12, fails)
    return fails


def check_fold_equals_unfold():
    """Folded (R, k, H) equals R*k single-token requests with replicated tables."""
    fails = []
    b = make_batch_from_lengths((150, 64, 9), 3, 2, seed=41, extra_pages=1)
    o, l = run_oracle(b)
    R, k = b.R, b.k
    rep = np.repeat(np.arange(R), k)
    o2, l2 = att.mla_decode(b.q.numpy(), b.kv.numpy(), b.block_table.numpy()[rep],
                            b.seq_lens.numpy()[rep], 1, b.sm_scale, b.q_scale, b.kv_scale)
    _cmp("fold out", o, o2, 1e-12, fails)
    _cmp("fold lse", l, l2, 1e-12, fails)
    return fails


def check_split_merge(seed=51):
    """Any partition of each request's keys, merged by LSE, equals no split."""
    fails = []
    b = make_batch_from_lengths((300, 129, 5), 2, 3, seed=seed)
    o, l = run_oracle(b)
    rng = np.random.default_rng(seed)
    lens = b.seq_lens.numpy()
    for S in (2, 3, 5):
        cuts = []
        for L in lens:
            inner = np.sort(rng.integers(0, L + 1, size=S - 1)) if L > 0 else np.zeros(S - 1, int)
            cuts.append(np.concatenate([[0], inner, [L]]))
        parts_o, parts_l = [], []
        for s in range(S):
            kr = np.array([[c[s], c[s + 1]] for c in cuts])
            po, pl = run_oracle(b, key_range=kr)
            parts_o.append(po.reshape(-1, 512))
            parts_l.append(pl.reshape(-1))
        mo, ml = merge.combine(np.stack(parts_o), np.stack(parts_l))
        _cmp(f"split{S} out", mo, o.reshape(-1, 512), 1e-12, fails)
        _cmp(f"split{S} lse", ml, l.reshape(-1), 1e-12, fails)
    return fails


def check_convexity():
    """out lies in the per-dim hull of the request's value rows."""
    fails = []
    b = make_batch_from_lengths((200, 33), 2, 2, seed=61)
    o, _ = run_oracle(b)
    for r, L in enumerate(b.seq_lens.numpy()):
        keys = np.stack([torch_decode(b.kv[int(b.block_table[r, j // 64]), j % 64].numpy())
                         for j in range(int(L))]) * b.kv_scale
        lo, hi = keys[:, :512].min(axis=0), keys[:, :512].max(axis=0)
        rows = o[r * 2:(r + 1) * 2].reshape(-1, 512)
        if np.any(rows < lo - 1e-12) or np.any(rows > hi + 1e-12):
            fails.append(f"convexity violated in request {r}")
    return fails


def _row_picks(R, M, n, rng):
    """(request, folded row) picks: the first and last row of every request
    plus n random ones."""
    picks = [(r, 0) for r in range(R)] + [(r, M - 1) for r in range(R)]
    picks += [(int(rng.integers(R)), int(rng.integers(M))) for _ in range(n)]
    return picks


def check_row_sampler(cases=TINY_CASES, seed=71):
    """The per-row sampler the full-size GPU checks use as ground truth: every
    pick (request r, folded row m = t*H + h) equals the brute force's row for
    token r*k + t, head h (drafter-attention page, module overview: rows run
    token-major, then head), and the whole-batch oracle's row on a batch with
    k and H both above one."""
    fails = []
    rng = np.random.default_rng(seed)
    for case in cases:
        b, (o_ref, l_ref) = _tiny(case)
        M = b.k * b.H
        picks = _row_picks(b.R, M, 12, rng)
        o, l = att.mla_decode_rows(b.q.numpy(), b.kv.numpy(), b.block_table.numpy(),
                                   b.seq_lens.numpy(), b.k, b.sm_scale, b.q_scale, b.kv_scale,
                                   picks)
        for i, (r, m) in enumerate(picks):
            t, h = r * b.k + m // b.H, m % b.H
            _cmp(f"rows bf out {case[0]} pick {(r, m)}", o[i], o_ref[t, h], 1e-12, fails)
            _cmp(f"rows bf lse {case[0]} pick {(r, m)}", l[i], l_ref[t, h], 1e-12, fails)
    b = make_batch_from_lengths((200, 70, 1), 3, 5, seed=seed, extra_pages=1)
    o_all, l_all = run_oracle(b)
    M = b.k * b.H
    picks = _row_picks(b.R, M, 20, rng)
    o, l = att.mla_decode_rows(b.q.numpy(), b.kv.numpy(), b.block_table.numpy(),
                               b.seq_lens.numpy(), b.k, b.sm_scale, b.q_scale, b.kv_scale, picks)
    for i, (r, m) in enumerate(picks):
        t, h = r * b.k + m // b.H, m % b.H
        _cmp(f"rows out pick {(r, m)}", o[i], o_all[t, h], 1e-12, fails)
        _cmp(f"rows lse pick {(r, m)}", l[i], l_all[t, h], 1e-12, fails)
    return fails


ALL_CHECKS = (check_brute_force, check_closed_forms, check_library_softmax,
              check_fold_equals_unfold, check_split_merge, check_convexity, check_row_sampler)


def all_failures():
    fails = []
    for c in ALL_CHECKS:
        fails += c()
    return fails
