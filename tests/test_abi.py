"""The C ABI library loads, exports every declared entry point, and rejects
bad arguments on the host without launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from sparse_mla_decode_04_gb300 import smla as S

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "smla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(smla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["smla_plan_num_splits", "smla_workspace_bytes", "smla_decode", "smla_read_device_error",
              "smla_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(smla_lib):
    for n in declared_functions():
        assert hasattr(smla_lib, n), n
        assert ctypes.cast(getattr(smla_lib, n), ctypes.c_void_p).value


def test_status_strings(smla_lib):
    for st in range(7):
        assert S.smla_status_string(st)
    assert S.smla_status_string(99) == "unknown status"


def test_workspace_bytes(smla_lib):
    a = S.smla_workspace_bytes(32, 128, 8)
    b = S.smla_workspace_bytes(32, 128, 10)
    assert 0 < a < b
    assert b - a == 32 * 2 * 128 * (512 * 4 + 2 * 8)
    # at least rows + 95 partial slots, whatever the split budget
    unit = 128 * (512 * 4 + 2 * 8)
    assert S.smla_workspace_bytes(32, 128, 1) == S.smla_workspace_bytes(32, 128, 3)
    assert S.smla_workspace_bytes(32, 128, 4) - S.smla_workspace_bytes(32, 128, 1) == (128 - 127) * unit
    assert S.smla_workspace_bytes(0, 128, 1) == 0
    assert S.smla_workspace_bytes(1, 129, 1) == 0
    assert S.smla_workspace_bytes(1, 128, 33) == 0
    assert S.smla_workspace_bytes(1025, 128, 1) == 0


def _fake_args(**kw):
    """Arguments that look well formed; pointers are fake host integers, so
    every case below must fail a host check before any launch."""
    a = S.smla_decode_args()
    base = 1 << 20
    for i, f in enumerate(["q_nope", "q_rope", "kv_pool", "kv_scales", "main_idx", "swa_start", "swa_len",
                           "cmp_pool", "cmp_scales", "cmp_start", "cmp_len", "sink", "out", "lse"]):
        setattr(a, f, base + i * 4096)
    a.n_main, a.n_cmp, a.topk, a.sm_scale = 1024, 192, 128, 0.044
    a.num_rows, a.num_heads, a.num_splits = 2, 16, 1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


WS = 1 << 30  # fake, 256-aligned workspace address


@pytest.mark.parametrize("field,value,status", [
    ("num_rows", 0, S.SMLA_ERR_BAD_SHAPE), ("num_rows", 1025, S.SMLA_ERR_BAD_SHAPE),
    ("num_heads", 0, S.SMLA_ERR_BAD_SHAPE), ("num_heads", 129, S.SMLA_ERR_BAD_SHAPE),
    ("num_splits", 0, S.SMLA_ERR_BAD_SHAPE), ("num_splits", 33, S.SMLA_ERR_BAD_SHAPE),
    ("topk", -1, S.SMLA_ERR_BAD_SHAPE), ("n_main", -5, S.SMLA_ERR_BAD_SHAPE),
    ("sm_scale", float("nan"), S.SMLA_ERR_BAD_SHAPE),
    ("q_nope", None, S.SMLA_ERR_NULL_POINTER), ("out", None, S.SMLA_ERR_NULL_POINTER),
    ("main_idx", None, S.SMLA_ERR_NULL_POINTER), ("kv_pool", None, S.SMLA_ERR_NULL_POINTER),
    ("swa_start", None, S.SMLA_ERR_NULL_POINTER), ("cmp_pool", None, S.SMLA_ERR_NULL_POINTER),
    ("q_nope", (1 << 20) + 8, S.SMLA_ERR_MISALIGNED), ("kv_scales", (1 << 20) + 3 * 4096 + 4, S.SMLA_ERR_MISALIGNED),
    ("lse", (1 << 20) + 13 * 4096 + 2, S.SMLA_ERR_MISALIGNED),
])
def test_decode_rejects_bad_arguments(smla_lib, field, value, status):
    a = _fake_args(**{field: value})
    assert S.smla_decode(a, WS, 1 << 40) == status


def test_decode_rejects_small_workspace(smla_lib):
    need = S.smla_workspace_bytes(2, 16, 1)
    assert S.smla_decode(_fake_args(), WS, need - 1) == S.SMLA_ERR_WORKSPACE_TOO_SMALL
    assert S.smla_decode(_fake_args(), WS + 16, 1 << 40) == S.SMLA_ERR_MISALIGNED


def test_decode_null_struct_and_workspace(smla_lib):
    lib = smla_lib
    assert lib.smla_decode(None, ctypes.c_void_p(WS), 1 << 40, None) == S.SMLA_ERR_NULL_POINTER
    a = _fake_args()
    assert lib.smla_decode(ctypes.byref(a), None, 1 << 40, None) == S.SMLA_ERR_NULL_POINTER


def test_read_device_error_null(smla_lib):
    assert smla_lib.smla_read_device_error(None, None, None) == S.SMLA_ERR_NULL_POINTER
