"""The C-ABI library builds, loads and exports every function include/mok.h
declares; host-only calls (size queries, argument checks) behave as
documented.  No device work: these run without a GPU."""
import ctypes
import os
import re

import pytest

from routing_dispatch_grouped_router_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "mok.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mok_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_lib.exported_names())


def _desc(**kw):
    base = dict(T=256, d=128, E=8, I=256, k=2)
    base.update(kw)
    return _lib.MoeDesc(T=base["T"], d=base["d"], E=base["E"], I=base["I"], k=base["k"],
                        dtype=base.get("dtype", 0), mb_tokens=0, ring_slots=0, flags=0, reserved=0)


def _sizes(lib, desc):
    f, s, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    code = lib.mok_moe_workspace_size(ctypes.byref(desc), ctypes.byref(f), ctypes.byref(s),
                                      ctypes.byref(b))
    return code, f.value, s.value, b.value


def test_workspace_sizes_cover_the_layout(lib):
    d = _desc()
    code, f, s, b = _sizes(lib, d)
    assert code == 0 and f > 0 and s > 0 and b > 0
    L = _lib.SavedLayout()
    assert lib.mok_moe_saved_layout(ctypes.byref(d), ctypes.byref(L)) == 0
    assert L.total == s
    R = 256 * 2
    assert L.rows_max == (R + 127 * 8 + 127) // 128 * 128
    offs = [L.status, L.topk_idx, L.topk_w, L.counts, L.offsets, L.pos, L.token_of_row,
            L.padded_offsets, L.padded_pos, L.padded_token, L.row_weight, L.x_perm, L.gate_up]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.gate_up + L.rows_max * 2 * 256 * 2 <= L.total


@pytest.mark.parametrize("kw,expect", [
    (dict(k=9, E=16), 2), (dict(k=3, E=2), 2), (dict(E=513), 2), (dict(d=96), 2),
    (dict(I=200), 2), (dict(dtype=1), 2), (dict(T=-1), 1), (dict(k=0), 1), (dict(d=0), 1),
])
def test_invalid_shapes_are_rejected(lib, kw, expect):
    code, *_ = _sizes(lib, _desc(**kw))
    assert code == expect


def test_zero_tokens_is_valid(lib):
    code, f, s, b = _sizes(lib, _desc(T=0))
    assert code == 0


def test_null_pointers_rejected_before_any_device_call(lib):
    d = _desc()
    code = lib.mok_moe_forward(ctypes.byref(d), None, None, None, None, None, None, None, 0,
                               None, 0, None)
    assert code == 1
    code = lib.mok_gemm_bf16(128, 128, 100, None, 0, None, 0, None, None, 0, None)
    assert code == 1
    code = lib.mok_gemm_bf16(128, 128, 100, ctypes.c_void_p(16), 0, ctypes.c_void_p(16), 0,
                             ctypes.c_void_p(16), ctypes.c_void_p(16), 256, None)
    assert code == 2


def test_status_strings(lib):
    for c in (0, 1, 2, 3, 4, 5, 16, 17, 18):
        assert lib.mok_status_string(c).decode()
    assert lib.mok_status_string(999) == b"unknown status"
