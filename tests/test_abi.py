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
                        dtype=base.get("dtype", 0), mb_tokens=base.get("mb", 0),
                        ring_slots=base.get("ring", 0), flags=base.get("flags", 0), reserved=0)


def _sizes(lib, desc):
    f, s, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    code = lib.mok_moe_workspace_size(ctypes.byref(desc), ctypes.byref(f), ctypes.byref(s),
                                      ctypes.byref(b))
    return code, f.value, s.value, b.value


def _regions(L, T, k, E, I, d, mb=None):
    """(offset, bytes) of every field of one micro-batch, plus ring slot 0."""
    Tk = (mb or T) * k
    rows = L.rows_max
    return [(L.status, 4), (L.topk_idx, Tk * 4), (L.topk_w, Tk * 4), (L.counts, E * 4),
            (L.offsets, (E + 1) * 4), (L.pos, Tk * 4), (L.token_of_row, Tk * 4),
            (L.padded_offsets, (E + 1) * 4), (L.padded_pos, Tk * 4), (L.padded_token, rows * 4),
            (L.row_weight, rows * 4), (L.gate_up, rows * 2 * I * 4), (L.x_perm, rows * d * 2)]


def _no_overlap(regions, total):
    regions = sorted(regions)
    for (o1, n1), (o2, _) in zip(regions, regions[1:]):
        assert o1 + n1 <= o2
    assert regions[-1][0] + regions[-1][1] <= total
    assert all(o % 256 == 0 for o, _ in regions)


def test_workspace_sizes_cover_the_layout(lib):
    d = _desc()
    code, f, s, b = _sizes(lib, d)
    assert code == 0 and f > 0 and s > 0 and b > 0
    L = _lib.SavedLayout()
    assert lib.mok_moe_saved_layout(ctypes.byref(d), ctypes.byref(L)) == 0
    assert L.total == s and L.mb_count == 1 and L.ring_slots == 1
    R = 256 * 2
    assert L.rows_max == (R + 127 * 8 + 127) // 128 * 128
    _no_overlap(_regions(L, 256, 2, 8, 256, 128), L.total)


def test_mxfp8_keeps_no_dispatched_rows(lib):
    """MXFP8 quantises the dispatched x rows straight from the token rows, so
    `saved` has no ring of bf16 rows: x_perm is not kept.  It keeps the
    weights in the backward's orientations instead (W_gate_up along 2I as
    codes and scales, W_down along d as bf16 values)."""
    bf = _desc(T=1024, mb=256, ring=2)
    mx = _desc(T=1024, mb=256, ring=2)
    mx.dtype = 1
    Lb, Lm = _lib.SavedLayout(), _lib.SavedLayout()
    assert lib.mok_moe_saved_layout(ctypes.byref(bf), ctypes.byref(Lb)) == 0
    assert lib.mok_moe_saved_layout(ctypes.byref(mx), ctypes.byref(Lm)) == 0
    assert Lm.x_perm == (1 << 64) - 1 and Lm.ring_slot_bytes == 0  # MOK_NOT_KEPT
    # ... and keeps the weights' backward forms instead (after everything else)
    n = mx.E * 2 * mx.I * mx.d
    wt = (n + n // 32 + 255) // 256 * 256
    wd = (mx.E * mx.d * mx.I * 2 + 255) // 256 * 256
    assert Lm.w_gate_up_t + wt == Lm.w_down_col and Lm.w_down_col + wd == Lm.total
    assert Lb.total - (Lm.total - wt - wd) == 2 * Lb.ring_slot_bytes
    assert Lb.w_gate_up_t == Lb.w_down_col == (1 << 64) - 1
    _no_overlap(_regions(Lm, 1024, 2, 8, 256, 128, mb=256)[:-1], Lm.total)


def test_nvfp4_weight_scales_sit_in_the_status_block(lib):
    """NVFP4 keeps the weights' two fp32 tensor scales for the backward inside
    the 256-byte status block (after the status word), and W_gate_up along 2I
    after everything else; the other dtypes keep neither."""
    bf = _desc(T=1024, mb=256, ring=2)
    nv = _desc(T=1024, mb=256, ring=2)
    nv.dtype, nv.d, nv.I = 2, 256, 256
    Lb, Ln = _lib.SavedLayout(), _lib.SavedLayout()
    assert lib.mok_moe_saved_layout(ctypes.byref(bf), ctypes.byref(Lb)) == 0
    assert lib.mok_moe_saved_layout(ctypes.byref(nv), ctypes.byref(Ln)) == 0
    assert Lb.nv_weight_scales == (1 << 64) - 1 and Lb.w_gate_up_t == (1 << 64) - 1
    # W_gate_up along 2I after everything else: codes and scales of E*2I*d values
    n = nv.E * 2 * nv.I * nv.d
    assert Ln.w_gate_up_t % 256 == 0 and Ln.w_gate_up_t + n // 2 + n // 16 <= Ln.total
    assert Ln.w_gate_up_t >= 256 + Ln.mb_count * Ln.mb_stride  # after the micro-batch blocks
    assert Ln.status + 4 <= Ln.nv_weight_scales and Ln.nv_weight_scales + 8 <= Ln.topk_idx
    assert Ln.nv_weight_scales % 4 == 0 and Ln.topk_idx == 256


def test_micro_batch_layout(lib):
    d = _desc(T=1024, mb=256, ring=2)
    L = _lib.SavedLayout()
    assert lib.mok_moe_saved_layout(ctypes.byref(d), ctypes.byref(L)) == 0
    assert L.mb_count == 4 and L.ring_slots == 2
    assert L.rows_max == (512 + 127 * 8 + 127) // 128 * 128  # per micro-batch
    regs = []
    for i in range(4):
        for o, n in _regions(L, 1024, 2, 8, 256, 128, mb=256)[:-1]:
            regs.append((o + i * L.mb_stride if o else o, n) if o else (o, n))
    regs = [r for r in regs if r[0] != 0] + [(0, 4)]
    for j in range(2):
        regs.append((L.x_perm + j * L.ring_slot_bytes, L.rows_max * 128 * 2))
    _no_overlap(list(set(regs)), L.total)
    # micro-batching needs a divisor of T, a ring no larger than the batches,
    # and fp32 weight gradients
    assert _sizes(lib, _desc(T=1000, mb=256))[0] == 2
    assert _sizes(lib, _desc(T=1024, mb=256, ring=5))[0] == 2
    assert _sizes(lib, _desc(T=1024, mb=256, flags=2))[0] == 2


def test_recompute_flag_drops_gate_up_from_saved(lib):
    base, rec = _desc(T=1024, mb=256, ring=2), _desc(T=1024, mb=256, ring=2, flags=8)
    Lb, Lr = _lib.SavedLayout(), _lib.SavedLayout()
    assert lib.mok_moe_saved_layout(ctypes.byref(base), ctypes.byref(Lb)) == 0
    assert lib.mok_moe_saved_layout(ctypes.byref(rec), ctypes.byref(Lr)) == 0
    assert Lr.gate_up == (1 << 64) - 1
    per_mb = Lb.rows_max * 2 * 256 * 4
    assert Lb.total - Lr.total == 4 * per_mb
    _, _, sb, bb = _sizes(lib, base)
    _, _, sr, br = _sizes(lib, rec)
    assert sr == Lr.total and br - bb == per_mb  # one micro-batch of g, u in the scratch


def test_recompute_dispatch_flag_drops_the_dispatched_rows_from_saved(lib):
    """MOK_FLAG_RECOMPUTE_DISPATCH: no ring of dispatched x rows in `saved`;
    one slot moves to the forward scratch and, without micro-batches, one to
    the backward scratch (with them the backward already dispatches each
    micro-batch into its own weight-gradient slot)."""
    for mb, ring in ((0, 0), (256, 2)):
        T = 1024
        base, rec = _desc(T=T, mb=mb, ring=ring), _desc(T=T, mb=mb, ring=ring, flags=0x20)
        Lb, Lr = _lib.SavedLayout(), _lib.SavedLayout()
        assert lib.mok_moe_saved_layout(ctypes.byref(base), ctypes.byref(Lb)) == 0
        assert lib.mok_moe_saved_layout(ctypes.byref(rec), ctypes.byref(Lr)) == 0
        assert Lr.x_perm == (1 << 64) - 1 and Lr.ring_slot_bytes == 0
        slot = Lb.rows_max * 128 * 2
        assert Lb.total - Lr.total == Lb.ring_slots * slot
        _, fb, _, bb = _sizes(lib, base)
        _, fr, sr, br = _sizes(lib, rec)
        assert sr == Lr.total and fr - fb == slot
        assert br - bb == (slot if mb == 0 else 0)
    # accepted with MXFP8, which keeps no dispatched rows anyway
    mx, mxr = _desc(dtype=1), _desc(dtype=1, flags=0x20)
    assert _sizes(lib, mx)[1:] == _sizes(lib, mxr)[1:]


def test_backward_rejects_a_missing_x(lib):
    """Every backward with tokens reads x (the router-weight gradient), so a
    NULL x is rejected before any device call, whatever the ring."""
    d = _desc(T=1024, mb=256)
    p = ctypes.c_void_p(256)
    code = lib.mok_moe_backward(ctypes.byref(d), p, None, p, None, p, p, p, 1 << 40, p, p, p,
                                p, p, 1 << 40, None)
    assert code == 1


@pytest.mark.parametrize("kw,expect", [
    (dict(k=9, E=16), 2), (dict(k=3, E=2), 2), (dict(E=513), 2), (dict(d=96), 2),
    (dict(I=200), 2), (dict(dtype=2), 2), (dict(T=-1), 1), (dict(k=0), 1), (dict(d=0), 1),
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


def test_fill_zero_checks_arguments_before_any_device_call(lib):
    """The write-bandwidth probe wants a 16-byte aligned address and a size
    that is a multiple of 16; a zero size enqueues nothing."""
    assert lib.mok_fill_zero(None, 0, None) == 0
    assert lib.mok_fill_zero(None, 64, None) == 1
    assert lib.mok_fill_zero(ctypes.c_void_p(24), 64, None) == 1
    assert lib.mok_fill_zero(ctypes.c_void_p(32), 40, None) == 1


def test_status_strings(lib):
    for c in (0, 1, 2, 3, 4, 5, 16, 17, 18):
        assert lib.mok_status_string(c).decode()
    assert lib.mok_status_string(999) == b"unknown status"


def test_widths_multiples_of_32(lib):
    """d and I may be any multiples of 32 from 128 on in BF16 (ragged GEMM
    tiles); MXFP8 keeps them multiples of 128, NVFP4 of 256."""
    ok = lambda **kw: _sizes(lib, _desc(**kw))[0]
    assert ok(d=160) == 0 and ok(d=2880) == 0 and ok(d=7168) == 0
    assert ok(I=160) == 0 and ok(I=2880) == 0 and ok(d=2880, I=2880) == 0
    assert ok(d=96) == 2 and ok(d=200) == 2 and ok(I=96) == 2 and ok(I=200) == 2
    assert ok(d=2880, dtype=1) == 2 and ok(I=160, dtype=1) == 2
    assert ok(d=2944, dtype=2, I=256) == 2 and ok(d=256, dtype=2, I=384) == 2
