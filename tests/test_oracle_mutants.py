"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch every one of them: a pin set that a dropped term, a wrong sign or index,
or a transposed operand slips through would not pin anything."""
import numpy as np
import pytest

import oracle.attention as att
import oracle.merge as merge
from tests import oracle_pins as pins

_attend = att.attend
_request_keys = att.request_keys
_mla_decode = att.mla_decode
_combine = merge.combine


def _attend_variant(score_dims=slice(0, 576), value=slice(0, 512), scale=True, axis=1,
                    subtract_max=True):
    def attend(qd, kd, sm_scale):
        n = qd.shape[0]
        if kd.shape[0] == 0:
            return np.zeros((n, 512)), np.full(n, -np.inf)
        s = (sm_scale if scale else 1.0) * (qd[:, score_dims] @ kd[:, score_dims].T)
        mx = s.max(axis=axis, keepdims=True) if subtract_max else np.zeros_like(s[:, :1])
        with np.errstate(over="ignore", invalid="ignore"):
            e = np.exp(s - mx)
            z = e.sum(axis=axis, keepdims=True)
            w = e / z
            if axis == 0:
                z = e.sum(axis=1, keepdims=True)
            out = w @ kd[:, value]
            lse = (mx if mx.shape[0] == n else mx.T)[:, 0] + np.log(z[:, 0])
        return out, lse / att.LN2
    return attend


def _keys_variant(page_shift=0, slot_shift=0, scale=True, extra=0):
    def request_keys(kv_codes, row, j0, j1, kv_scale):
        j = np.arange(j0, j1 + extra, dtype=np.int64)
        row = np.asarray(row, dtype=np.int64)
        pages = row[(j // 64 + page_shift) % row.size]
        slots = (j + slot_shift) % 64
        return att.e4m3.decode(np.asarray(kv_codes)[pages, slots, :]) * (kv_scale if scale else 1.0)
    return request_keys


def _head_major_decode(*a, **kw):
    out, lse = _mla_decode(*a, **kw)
    k = a[4]
    rows, H = lse.shape
    R = rows // k
    o = out.reshape(R, k, H, 512).transpose(0, 2, 1, 3).reshape(R, k * H, 512)
    l = lse.reshape(R, k, H).transpose(0, 2, 1).reshape(R, k * H)
    return o.reshape(rows, H, 512), l.reshape(rows, H)


def _rows_variant(split_by_k=False, no_request_offset=False):
    """mla_decode_rows with one index mistake."""
    def mla_decode_rows(q_codes, kv_codes, block_table, seq_lens, tokens_per_request,
                        sm_scale, q_scale, kv_scale, picks):
        q = np.asarray(q_codes)
        _, H, _ = q.shape
        k = int(tokens_per_request)
        outs, lses = [], []
        for r, m in picks:
            t, h = divmod(int(m), k if split_by_k else H)
            t, h = min(t, k - 1), min(h, H - 1)
            row = t if no_request_offset else r * k + t
            kd = att.request_keys(kv_codes, np.asarray(block_table)[r], 0,
                                  int(np.asarray(seq_lens)[r]), kv_scale)
            qd = att.e4m3.decode(q[row, h][None, :]) * float(q_scale)
            o, l2 = att.attend(qd, kd, sm_scale)
            outs.append(o[0])
            lses.append(l2[0])
        return np.stack(outs), np.array(lses)
    return mla_decode_rows


def _combine_natural(o, l):
    o = np.asarray(o); l = np.asarray(l)
    mx = l.max(axis=0)
    w = np.exp(l - mx)
    return (w[:, :, None] * o).sum(0) / w.sum(0)[:, None], mx + np.log(w.sum(0))


MUTANTS = {
    "scores drop the rope dims": ("attend", _attend_variant(score_dims=slice(0, 512))),
    "value taken from the wrong slice": ("attend", _attend_variant(value=slice(64, 576))),
    "softmax scale dropped": ("attend", _attend_variant(scale=False)),
    "no max subtraction": ("attend", _attend_variant(subtract_max=False)),
    "natural-log LSE": ("LN2", 1.0),
    "next page instead of this one": ("request_keys", _keys_variant(page_shift=1)),
    "slot off by one": ("request_keys", _keys_variant(slot_shift=1)),
    "kv scale not applied": ("request_keys", _keys_variant(scale=False)),
    "one key past the length": ("request_keys", _keys_variant(extra=1)),
    "head-major row order": ("mla_decode", _head_major_decode),
    "merge weights in base e": ("combine", _combine_natural),
    "row sampler splits rows by k": ("mla_decode_rows", _rows_variant(split_by_k=True)),
    "row sampler drops the request offset": ("mla_decode_rows",
                                             _rows_variant(no_request_offset=True)),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, value = MUTANTS[name]
    module = merge if attr == "combine" else att
    monkeypatch.setattr(module, attr, value)
    assert pins.all_failures(), f"no pin caught: {name}"


def test_pins_pass_on_the_real_oracle():
    assert pins.all_failures() == []
