"""The split reduction fused with the W_UV up-projection (mla_uv_combine)
against the oracle's exact product (drafter-attention page, `DraftDcp`).

Tolerance, derived from the arithmetic: the kernel rounds each merged latent
row o to BF16 (relative error <= 2^-9, taken as 2^-8), multiplies by the BF16
W_UV with FP32 accumulation (relative error well below 2^-16 over 512 terms)
and rounds y to BF16 (2^-8 again). Against the exact y = o_exact . W:
    |y - y_ref| <= sum_c |W[c, j]| * e_c + 2^-8 |y_ref| + 1e-4,
where e_c bounds |o_c - o_exact_c| per element: 2^-8 |o_exact_c| + 1e-6 when the
partials are the oracle's own (the merge is then exact up to FP32), and the
decode's tolerance ATOL + RTOL |o_exact_c| (plus 2^-8 |o_exact_c|) end to end.
"""
import numpy as np
import pytest
import torch

import mla_decode_attention_folded_gb300 as mla
import oracle.attention as att
import oracle.uv as ouv
from oracle import planner as pl
from tests.gpu_util import ATOL, RTOL, bmm_scales, oracle_full, to_device
from workloads import make_batch, make_batch_from_lengths, make_w_uv

pytestmark = pytest.mark.gpu

EPS = 2.0 ** -8


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _w_views(H, seed):
    w = make_w_uv(H, seed)                                 # [H, 512, 128] BF16
    dev = w.transpose(1, 2).contiguous().cuda()            # [H, 128, 512], latent-contiguous
    return w.float().double().numpy(), dev


def _check(y, ref_y, o_ref, w, elem_err, what):
    """y [T, H, 128] vs ref_y with the bound of the module docstring."""
    y = np.asarray(y, dtype=np.float64)
    e = elem_err(np.abs(o_ref))                            # [T, H, 512]
    bound = np.einsum("thc,hcj->thj", e, np.abs(w)) + EPS * np.abs(ref_y) + 1e-4
    assert np.all(np.isfinite(y)), f"{what}: non-finite y"
    excess = np.abs(y - ref_y) - bound
    assert excess.max() <= 0, f"{what}: y exceeds its bound by {excess.max():.3e}"


def _decode_uv(b, w_dev, groups=1, policy=mla.POLICY_BALANCED, min_split_tokens=64):
    d = to_device(b)
    eng = mla.FoldedMla(b.R, b.k, b.H, d["bt"].shape[1], d["kv"].shape[0], "cuda",
                        num_ctas=_sms(), min_split_tokens=min_split_tokens, policy=policy,
                        groups=groups)
    bmm1, bmm2 = bmm_scales(b)
    eng.plan(d["lens"])
    y = eng.decode_uv(d["q"], d["kv"], d["bt"], d["lens"], bmm1, bmm2, w_dev)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), int(eng.status.item()), eng.counts.cpu().numpy()


@pytest.mark.parametrize("lens,k,H,groups", [
    ((3000, 700, 64, 0), 4, 8, 1),        # multi-split, single-split and an empty request
    ((2100, 640, 90), 7, 8, 1),           # 21 tokens: one ragged 32-token block
    ((1300, 90), 4, 64, 1),               # M = 256: four 64-row blocks; 64 heads
    ((1300, 900), 4, 64, 2),              # row groups (the pages' partial fold)
    ((500,) * 9, 4, 2, 1),                # 36 tokens: two blocks, the second ragged
])
def test_decode_uv_matches_oracle(lens, k, H, groups):
    b = make_batch_from_lengths(lens, k, H, seed=61, scaling="amax")
    w, w_dev = _w_views(H, seed=7)
    y, status, counts = _decode_uv(b, w_dev, groups=groups)
    assert status == 0
    assert (counts >= 2).any()
    ref_o, _ = oracle_full(b)                              # [R, M, 512]
    o_ref = ref_o.reshape(b.R * b.k, b.H, 512)
    ref_y = ouv.uv_project(o_ref, w)
    _check(y, ref_y, o_ref, w, lambda a: ATOL + (RTOL + EPS) * a, f"lens={lens} k={k} H={H}")


def _random_uv_cases(n, seed):
    """Seeded random shapes for the fused reducer: tokens per row block
    (k / groups), heads, lengths at page and tile edges, empty requests."""
    rng = np.random.default_rng(seed)
    edges = [0, 1, 63, 64, 65, 127, 128, 129]
    out = []
    while len(out) < n:
        R = int(rng.integers(1, 8))
        k = int(rng.integers(1, 9))
        H = int(rng.choice([1, 2, 4, 8, 16, 64]))
        lens = [int(rng.choice(edges)) if rng.random() < 0.3 else int(rng.integers(1, 3500))
                for _ in range(R)]
        if k * H * sum(lens) > 2_000_000 or max(lens) == 0:
            continue
        groups = int(rng.choice([d for d in range(1, k + 1) if k % d == 0]))
        out.append((tuple(lens), k, H, groups))
    return out


@pytest.mark.parametrize("lens,k,H,groups", _random_uv_cases(12, 2027))
def test_random_shapes_uv_match_oracle(lens, k, H, groups):
    """Decode + fused W_UV reduction on seeded random shapes against the
    oracle's exact product, with the end-to-end bound of the module docstring."""
    b = make_batch_from_lengths(lens, k, H, seed=len(lens) * 101 + k * 7 + H, scaling="amax")
    w, w_dev = _w_views(H, seed=k + H)
    y, status, _ = _decode_uv(b, w_dev, groups=groups, min_split_tokens=64)
    assert status == 0
    ref_o, _ = oracle_full(b)
    o_ref = ref_o.reshape(b.R * b.k, b.H, 512)
    ref_y = ouv.uv_project(o_ref, w)
    _check(y, ref_y, o_ref, w, lambda a: ATOL + (RTOL + EPS) * a,
           f"lens={lens} k={k} H={H} groups={groups}")


def test_uv_on_oracle_partials():
    """The fused reducer alone, on split partials and one-split rows the oracle
    made over the planned splits."""
    b = make_batch_from_lengths((3000, 700, 64, 0, 2500), 2, 8, seed=77, scaling="amax")
    G = 16
    s = mla.make_shape(b.R, b.k, b.H, b.block_table.shape[1], b.kv.shape[0], G, 64, 64)
    counts, work = pl.plan(b.seq_lens.numpy(), b.M, G, 64, 64, pl.BALANCED,
                           capacity=mla.plan_list_len(s))
    slots = pl.partial_slots(b.R, b.M, G, pl.BALANCED, 64)
    ws = torch.zeros(mla.workspace_bytes(s), dtype=torch.uint8)
    po_bytes = (slots * b.M * 512 * 4 + 255) // 256 * 256
    po = ws[:po_bytes].view(torch.float32)[: slots * b.M * 512].view(slots, b.M, 512)
    plse = ws[po_bytes:].view(torch.float32)[: slots * b.M].view(slots, b.M)
    lens = b.seq_lens.numpy()
    ref_o, _ = oracle_full(b)
    out = torch.zeros((b.R, b.M, 512), dtype=torch.bfloat16)
    for r in range(b.R):
        if counts[r] < 2:
            out[r] = torch.from_numpy(ref_o[r]).to(torch.bfloat16)
    for idx, e in enumerate(work):
        if e < 0:
            break
        r = pl.entry_request(e)
        if counts[r] < 2:
            continue
        kr = np.zeros((b.R, 2), dtype=np.int64)
        kr[r] = pl.entry_keys(work, counts, idx, int(lens[r]), b.R, b.M, G, pl.BALANCED, 64)
        o, l = att.mla_decode(b.q.numpy(), b.kv.numpy(), b.block_table.numpy(), lens, b.k,
                              b.sm_scale, b.q_scale, b.kv_scale, key_range=kr, requests=[r])
        po[idx] = torch.from_numpy(o.reshape(b.R, b.M, 512)[r] / b.kv_scale).float()
        plse[idx] = torch.from_numpy(l.reshape(b.R, b.M)[r]).float()
    w, w_dev = _w_views(b.H, seed=3)
    y = torch.empty((b.R * b.k, b.H, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.uv_combine(s, torch.from_numpy(counts).cuda(), torch.from_numpy(work).cuda(), ws.cuda(),
                   b.kv_scale, out.cuda(), w_dev, y, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert (counts >= 2).sum() >= 2
    o_ref = ref_o.reshape(b.R * b.k, b.H, 512)
    ref_y = ouv.uv_project(o_ref, w)
    _check(y.float().cpu().numpy(), ref_y, o_ref, w, lambda a: EPS * a + 1e-6, "oracle partials")


def test_bench_workload_sampled():
    """The bench workload at full size through decode + fused reducer, checked
    on sampled (token, head) rows the oracle computes one by one."""
    b = make_batch("R32_k4_H8_len1k-8k")
    w, w_dev = _w_views(b.H, seed=11)
    y, status, counts = _decode_uv(b, w_dev, min_split_tokens=256)
    assert status == 0
    rng = np.random.default_rng(4)
    picks = [(int(r), int(m)) for r, m in zip(rng.integers(0, b.R, 24), rng.integers(0, b.M, 24))]
    picks += [(int(np.argmax(counts)), 0), (int(np.argmin(counts)), b.M - 1)]
    o, _ = att.mla_decode_rows(b.q.numpy(), b.kv.numpy(), b.block_table.numpy(),
                               b.seq_lens.numpy(), b.k, b.sm_scale, b.q_scale, b.kv_scale, picks)
    for (r, m), orow in zip(picks, o):
        t, h = divmod(m, b.H)
        ref = orow @ w[h]
        bound = (ATOL + (RTOL + EPS) * np.abs(orow)) @ np.abs(w[h]) + EPS * np.abs(ref) + 1e-4
        got = y[r * b.k + t, h]
        assert np.all(np.abs(got - ref) <= bound), (r, m)


def test_uv_rejects_bad_arguments():
    b = make_batch_from_lengths((300,), 2, 8, seed=1)
    s = mla.make_shape(b.R, b.k, b.H, 8, 16, 8, 64, 64)
    n = mla.plan_list_len(s)
    i32 = dict(dtype=torch.int32, device="cuda")
    counts, work = torch.ones(1, **i32), torch.full((n,), -1, **i32)
    ws = torch.zeros(max(mla.workspace_bytes(s), 256), dtype=torch.uint8, device="cuda")
    out = torch.zeros((1, b.M, 512), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((b.H, 128, 512), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((2, b.H, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mla.MlaError):
        mla.uv_combine(s, counts, work, ws, 1.0, out, None, y)
    with pytest.raises(mla.MlaError):
        mla.uv_combine(s, counts, work[:1], ws, 1.0, out, w, y)
    with pytest.raises(mla.MlaError):            # y not 16-byte aligned
        mla.uv_combine(s, counts, work, ws, 1.0, out, w, y.view(-1)[1:].view(torch.int16))
