"""ctypes view of libmlafold.so (the C ABI of include/mlafold.h).

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmlafold.so")

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", -1: "MLA_ERR_NULL", -2: "MLA_ERR_SHAPE", -3: "MLA_ERR_WORKSPACE",
                -4: "MLA_ERR_LIST", -5: "MLA_ERR_UNSUPPORTED", -6: "MLA_ERR_CUDA",
                -7: "MLA_ERR_ALIGN", -8: "MLA_ERR_SCRATCH_LIMIT"}
POLICY_BALANCED, POLICY_UNIFORM = 0, 1
FAULT_WAIT_TIMEOUT, FAULT_PAGE_RANGE, FAULT_WORK_ITEM = 0x1, 0x2, 0x4

# Every symbol include/mlafold.h declares.
EXPORTS = ("mla_plan_list_len", "mla_workspace_bytes", "mla_plan_splits",
           "mla_folded_decode", "mla_split_combine", "mla_lse_merge",
           "mla_folded_decode_noalloc", "mla_uv_combine", "mla_folded_decode_wait_test",
           "mla_tier_plan", "mla_row_copy")
NOALLOC_SCRATCH_BYTES = 64 << 20


class MlaShape(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("k", ctypes.c_int32), ("H", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("min_split_tokens", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("policy", ctypes.c_int32), ("groups", ctypes.c_int32)]


class MlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}")
        self.code = code


_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m mla_decode_attention_folded_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    SP = ctypes.POINTER(MlaShape)
    lib.mla_plan_list_len.argtypes = [SP]
    lib.mla_plan_list_len.restype = I32
    lib.mla_workspace_bytes.argtypes = [SP, ctypes.POINTER(SZ)]
    lib.mla_workspace_bytes.restype = I32
    lib.mla_plan_splits.argtypes = [SP, P, P, P, I32, P]
    lib.mla_plan_splits.restype = I32
    lib.mla_folded_decode.argtypes = [SP, P, P, P, P, F, F, P, P, I32, P, SZ, P, P, P, P]
    lib.mla_folded_decode.restype = I32
    lib.mla_folded_decode_wait_test.argtypes = [SP, P, P, P, P, F, F, P, P, I32, P, SZ, P, P, P,
                                                ctypes.c_uint64, P]
    lib.mla_folded_decode_wait_test.restype = I32
    lib.mla_tier_plan.argtypes = [I32, I32, I32, I32, I32, P, P, P, P, P]
    lib.mla_tier_plan.restype = I32
    lib.mla_row_copy.argtypes = [P, P, P, I32, I32, ctypes.c_int64, I32, P]
    lib.mla_row_copy.restype = I32
    lib.mla_split_combine.argtypes = [SP, P, P, I32, P, SZ, F, P, P, P]
    lib.mla_split_combine.restype = I32
    lib.mla_lse_merge.argtypes = [I32, I32, P, P, P, P, P]
    lib.mla_lse_merge.restype = I32
    lib.mla_folded_decode_noalloc.argtypes = [SP, P, P, P, P, F, F, P, P, I32, P, P, P, P]
    lib.mla_folded_decode_noalloc.restype = I32
    lib.mla_uv_combine.argtypes = [SP, P, P, I32, P, SZ, F, P, P, P, P, P]
    lib.mla_uv_combine.restype = I32
    _lib = lib
    return lib


def check(fn: str, code: int) -> int:
    if code < 0:
        raise MlaError(fn, code)
    return code
