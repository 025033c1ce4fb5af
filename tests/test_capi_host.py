"""The C-ABI library loads, exports every symbol include/moe_fp4.h declares,
and rejects bad arguments on the host before touching a GPU.

These tests run without a GPU: every call below fails its argument checks,
which come before any CUDA runtime call, so no pointer is dereferenced (the
"device pointers" here are plain integers that are never used).
"""
import ctypes as C
import os
import re

import pytest

from block_scaled_fp4_moe_gb300 import _build, moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return moe.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "moe_fp4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(L):
    declared = header_functions()
    assert "moe_layer_forward" in declared and "moe_route_topk" in declared
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(moe.exported_symbols()) == declared


def test_status_strings(L):
    for code in range(9):
        s = moe.moe_status_string(code)
        assert s and s != "unknown status"
    assert moe.moe_status_string(99) == "unknown status"


def test_workspace_size(L):
    a = moe.moe_workspace_size(1, 5120, 1536, 160, 8, 1)
    b = moe.moe_workspace_size(4, 5120, 1536, 160, 8, 1)
    assert 0 < a < b
    assert a % 256 == 0
    assert moe.moe_workspace_size(1, 5120, 1536, 160, 0, 1) == 0
    assert moe.moe_workspace_size(-1, 5120, 1536, 160, 8, 1) == 0


FAKE = 1 << 40          # 16-byte aligned integer that is never dereferenced


def bank(w13=FAKE, s13=FAKE, w2=FAKE, s2=FAKE, packed=FAKE, E=160, S=1, H=5120, I=1536):
    return moe._Bank(w13, s13, w2, s2, packed, E, S, H, I)


def forward(L, b, T=1, k=8, x=FAKE, wr=FAKE, y=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return L.moe_layer_forward(C.c_void_p(x), C.c_void_p(wr), None, T, k, C.byref(b), 1.0, C.c_void_p(y), None,
                               None, C.c_void_p(ws), ws_bytes, None)


def test_layer_forward_argument_checks(L):
    assert forward(L, bank(packed=0)) == moe.MOE_ERR_INVALID_ARG
    assert forward(L, bank(), x=0) == moe.MOE_ERR_INVALID_ARG
    assert forward(L, bank(), T=-1) == moe.MOE_ERR_INVALID_ARG
    assert forward(L, bank(S=2)) == moe.MOE_ERR_INVALID_ARG
    assert forward(L, bank(), k=0) == moe.MOE_ERR_INVALID_ARG
    assert forward(L, bank(), k=161) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert forward(L, bank(H=5000)) == moe.MOE_ERR_UNSUPPORTED_SHAPE       # not a multiple of 64
    assert forward(L, bank(I=16448)) == moe.MOE_ERR_UNSUPPORTED_SHAPE      # I > 16384
    assert forward(L, bank(E=2000)) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert forward(L, bank(), T=5000) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert forward(L, bank(packed=FAKE + 8)) == moe.MOE_ERR_MISALIGNED
    assert forward(L, bank(), x=FAKE + 2) == moe.MOE_ERR_MISALIGNED
    assert forward(L, bank(), ws=FAKE + 16) == moe.MOE_ERR_MISALIGNED
    need = moe.moe_workspace_size(1, 5120, 1536, 160, 8, 1)
    assert forward(L, bank(), ws_bytes=need - 1) == moe.MOE_ERR_WORKSPACE_TOO_SMALL


def test_pack_argument_checks(L):
    p = C.c_void_p(FAKE)
    assert moe.moe_packed_bank_size(5120, 1536, 160, 1) == moe.moe_packed_bank_size(5120, 1536, 160, 1)
    n = moe.moe_packed_bank_size(5120, 1536, 160, 1)
    # the canonical bytes (a permutation) and one exponent base per weight row
    # (2I gate/up rows and H down rows per expert), up to section alignment
    canon = 161 * (2 * 1536 * 5120 // 2 + 2 * 1536 * 5120 // 32 + 5120 * 1536 // 2 + 5120 * 1536 // 32)
    rowexp = 161 * (2 * 1536 + 5120)
    assert canon + rowexp <= n < canon + rowexp + 1024
    assert moe.moe_packed_bank_size(5000, 1536, 160, 1) == 0
    assert L.moe_pack_bank(C.byref(bank(w13=0)), p, n, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pack_bank(C.byref(bank()), None, n, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pack_bank(C.byref(bank(s2=FAKE + 4)), p, n, None) == moe.MOE_ERR_MISALIGNED
    assert L.moe_pack_bank(C.byref(bank()), C.c_void_p(FAKE + 16), n, None) == moe.MOE_ERR_MISALIGNED
    assert L.moe_pack_bank(C.byref(bank()), p, n - 1, None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL


def forward_mx(L, b, T=1, k=8, pmx=FAKE, x=FAKE, y=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return L.moe_layer_forward_mxfp8(C.c_void_p(x), C.c_void_p(FAKE), None, T, k, C.byref(b), C.c_void_p(pmx), 1.0,
                                     C.c_void_p(y), None, None, C.c_void_p(ws), ws_bytes, None)


def test_mxfp8_argument_checks(L):
    # the canonical arrays, 256-byte aligned sections (no padding at these sizes)
    n = moe.lib().moe_packed_mx_bank_size(5120, 1536, 160, 1)
    assert n == 161 * 3 * 1536 * 5120 * 17 // 32
    assert moe.lib().moe_packed_mx_bank_size(5120 + 64, 1536, 160, 1) == 0      # H % 128
    assert moe.lib().moe_packed_mx_bank_size(5120, 1536 + 64, 160, 1) == 0      # I % 128
    p = C.c_void_p(FAKE)
    assert L.moe_pack_bank_mx(C.byref(bank(w2=0)), p, n, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pack_bank_mx(C.byref(bank()), C.c_void_p(FAKE + 16), n, None) == moe.MOE_ERR_MISALIGNED
    assert L.moe_pack_bank_mx(C.byref(bank()), p, n - 1, None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_pack_bank_mx(C.byref(bank(H=5120 + 64)), p, n, None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert forward_mx(L, bank(), pmx=0) == moe.MOE_ERR_INVALID_ARG
    assert forward_mx(L, bank(), pmx=FAKE + 16) == moe.MOE_ERR_MISALIGNED
    assert forward_mx(L, bank(H=5120 + 64)) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert forward_mx(L, bank(), x=0) == moe.MOE_ERR_INVALID_ARG
    assert forward_mx(L, bank(), k=161) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    need = moe.moe_workspace_size(1, 5120, 1536, 160, 8, 1)
    assert forward_mx(L, bank(), ws_bytes=need - 1) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    ev = (C.c_void_p * 5)()
    assert L.moe_layer_forward_mxfp8_profiled(C.c_void_p(FAKE), C.c_void_p(FAKE), None, 1, 8, C.byref(bank()), p,
                                              1.0, C.c_void_p(FAKE), C.c_void_p(FAKE), 1 << 40, ev, 4,
                                              None) == moe.MOE_ERR_INVALID_ARG      # fewer than 5 events


def test_other_entry_points_argument_checks(L):
    p = C.c_void_p(FAKE)
    assert L.moe_route_topk(p, p, None, 1, 5120, 160, 9, 1, 1.0, None, p, p, 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_route_topk(p, p, None, 1, 5120, 8, 9, 1, 1.0, p, p, p, 1 << 30, None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_route_topk(p, p, None, 1, 5120, 160, 8, 1, 1.0, p, p, p, 16, None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_group_tokens(p, 1, 9, 161, p, p, p, p, None, p, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_group_tokens(p, 1, 40, 161, p, p, p, p, p, p, 1 << 20, None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    b = bank()
    assert L.moe_expert_ffn_mxfp4(p, p, None, 1, 8, C.byref(b), p, p, 1 << 40, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_check_device_status(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_init(None, 1024, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_init(C.c_void_p(FAKE + 16), 1024, None) == moe.MOE_ERR_MISALIGNED
    assert L.moe_workspace_init(p, 64, None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_layer_forward_profiled(p, p, None, 1, 8, C.byref(b), 1.0, p, p, 1 << 40, None, 5, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_decode_e2m1(None, p, 4, None) == moe.MOE_ERR_INVALID_ARG


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(moe, "_libs", {})
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_build, "DEBUG_LIB_PATH", str(tmp_path / "missing_debug.so"))
    with pytest.raises(RuntimeError, match="missing"):
        moe.lib()
    with pytest.raises(RuntimeError, match="missing"):
        with moe.debug_bounds():
            pass


def test_debug_build_exports_the_same_symbols():
    """libmoe_fp4_debug.so (range checks on) has the same C ABI."""
    _build.build(debug=True)
    with moe.debug_bounds() as L:
        assert moe.library_path() == _build.DEBUG_LIB_PATH
        for name in moe.exported_symbols():
            assert hasattr(L, name), name
        assert L.moe_status_string(moe.MOE_ERR_DEVICE_ASSERT) == b"device-side input check failed"
    assert moe.library_path() == _build.LIB_PATH
