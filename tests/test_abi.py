"""The C-ABI library loads, exports every symbol include/mlafold.h declares,
and its host-only sizing and validation agree with the oracle planner.
No GPU: nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

import mla_decode_attention_folded_gb300 as mla
from mla_decode_attention_folded_gb300 import _lib
from oracle import planner as pl

HEADER = os.path.join(os.path.dirname(__file__), "..", "include", "mlafold.h")
def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTS)
    for name in names:
        assert hasattr(lib, name), name


def test_noalloc_limit_matches_header():
    """The allocation-free entry point's scratch size as the header defines it
    (the library derives its array from the same macro) is the binding's."""
    text = open(HEADER).read()
    m = re.search(r"#define\s+MLA_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "MLA_NOALLOC_SCRATCH_BYTES not found in the header"
    assert int(m.group(1)) << int(m.group(2)) == _lib.NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("R,k,H,G,policy,ms", [
    (2, 4, 8, 8, pl.BALANCED, 64), (32, 4, 8, 152, pl.BALANCED, 64),
    (64, 7, 8, 152, pl.UNIFORM, 64), (16, 4, 64, 152, pl.BALANCED, 64),
    (128, 7, 64, 152, pl.UNIFORM, 64), (1000, 1, 1, 2048, pl.BALANCED, 4096),
    (5, 3, 3, 1, pl.UNIFORM, 1)])
def test_sizes_match_oracle_planner(R, k, H, G, policy, ms):
    s = mla.make_shape(R, k, H, 10, 100, G, 256, ms, policy)
    M = k * H
    assert mla.plan_list_len(s) == pl.list_len(R, M, G, policy, ms)
    slots = pl.partial_slots(R, M, G, policy, ms)
    align = lambda x: (x + 255) // 256 * 256
    want = 0 if slots == 0 else align(slots * M * 512 * 4) + align(slots * M * 4)
    assert mla.workspace_bytes(s) == want


@pytest.mark.parametrize("field,value,code", [
    ("page_size", 32, -5), ("R", 0, -2), ("R", 1025, -2), ("k", 0, -2), ("H", 0, -2),
    ("H", 5000, -2), ("num_ctas", 0, -2), ("max_splits", 4097, -2), ("policy", 7, -2),
    ("min_split_tokens", 0, -2), ("num_pages", 0, -2), ("max_pages", 0, -2),
    ("max_pages", 1 << 25, -2)])
def test_bad_shape_rejected_on_host(field, value, code):
    s = mla.make_shape(4, 2, 8, 10, 100, 152)
    setattr(s, field, value)
    assert _lib.load().mla_plan_list_len(ctypes.byref(s)) == code
    with pytest.raises(mla.MlaError):
        mla.workspace_bytes(s)


def test_null_pointers_rejected_before_any_launch():
    lib = _lib.load()
    s = mla.make_shape(4, 2, 8, 10, 100, 152)
    assert lib.mla_plan_splits(ctypes.byref(s), None, None, None, 100, None) == -1
    assert lib.mla_folded_decode(ctypes.byref(s), None, None, None, None, 1.0, 1.0, None, None,
                                 100, None, 0, None, None, None, None) == -1
    assert lib.mla_split_combine(ctypes.byref(s), None, None, 100, None, 0, 1.0, None, None,
                                 None) == -1
    assert lib.mla_workspace_bytes(ctypes.byref(s), None) == -1
    assert lib.mla_plan_list_len(None) == -1


def test_short_list_and_workspace_rejected_before_any_launch():
    lib = _lib.load()
    s = mla.make_shape(32, 4, 8, 10, 100, 152)
    n = mla.plan_list_len(s)
    fake = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced
    assert lib.mla_plan_splits(ctypes.byref(s), fake, fake, fake, n - 1, None) == -4
    args = [ctypes.byref(s), fake, fake, fake, fake, 1.0, 1.0, fake, fake]
    assert lib.mla_folded_decode(*args, n, fake, 0, fake, fake, None, None) == -3
    assert lib.mla_folded_decode(*args, n - 1, fake, 1 << 30, fake, fake, None, None) == -4
    odd = ctypes.c_void_p((1 << 20) + 8)     # not 16-byte aligned
    args2 = [ctypes.byref(s), odd, fake, fake, fake, 1.0, 1.0, fake, fake]
    assert lib.mla_folded_decode(*args2, n, fake, 1 << 30, fake, fake, None, None) == -7


def test_binding_fold_factor_matches_oracle():
    for k in range(1, 13):
        for H in (1, 8, 16, 64, 96, 128, 200):
            assert mla.fold_factor(k, H, 128) == pl.fold_factor(k, H, 128)


@pytest.mark.parametrize("R,k,H,groups", [(16, 4, 64, 2), (128, 7, 8, 7), (100, 6, 8, 3)])
def test_row_group_sizes_match_oracle(R, k, H, groups):
    for policy in (pl.BALANCED, pl.UNIFORM):
        s = mla.make_shape(R, k, H, 10, 100, 152, 256, 64, policy, groups)
        Rg, Mg = R * groups, (k // groups) * H
        assert mla.plan_list_len(s) == pl.list_len(Rg, Mg, 152, policy, 64)
        slots = pl.partial_slots(Rg, Mg, 152, policy, 64)
        align = lambda x: (x + 255) // 256 * 256
        want = 0 if slots == 0 else align(slots * Mg * 512 * 4) + align(slots * Mg * 4)
        assert mla.workspace_bytes(s) == want


@pytest.mark.parametrize("R,k,groups", [(4, 4, 3), (4, 6, 4), (600, 2, 2), (4, 2, -1)])
def test_bad_row_groups_rejected(R, k, groups):
    s = mla.make_shape(R, k, 8, 10, 100, 152, 256, 64, 0, groups)
    assert _lib.load().mla_plan_list_len(ctypes.byref(s)) == -2


def test_zero_groups_reads_as_one():
    s0 = mla.make_shape(32, 4, 8, 10, 100, 152, 256, 64, 0, 0)
    s1 = mla.make_shape(32, 4, 8, 10, 100, 152, 256, 64, 0, 1)
    assert mla.plan_list_len(s0) == mla.plan_list_len(s1)
    assert mla.workspace_bytes(s0) == mla.workspace_bytes(s1)
