"""PyTorch-facing wrappers of the C ABI in include/mok.h.

Tensors only provide device memory and the current stream; every step runs in
libmok.so.  Shapes and dtypes are checked here, everything else by the library.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

BF16, MXFP8, NVFP4 = 0, 1, 2
FLAG_BF16_ACT_OUT = 0x1    # y and dx written as bf16 (default fp32)
FLAG_BF16_WGRAD_OUT = 0x2  # weight gradients written as bf16 (default fp32)
FLAG_ACCUMULATE_WGRAD = 0x4  # backward adds into the fp32 weight gradients
FLAG_RECOMPUTE_GATE_UP = 0x8  # g, u not kept by the forward; the backward recomputes them
FLAG_SINGLE_CTA_GEMM = 0x10  # one-CTA 128-row GEMM tiles instead of CTA pairs
FLAG_RECOMPUTE_DISPATCH = 0x20  # dispatched x rows not kept; the backward gathers them again
NOT_KEPT = (1 << 64) - 1  # saved-layout offset of a field the flags leave out


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(T, d, E, I, k, dtype=BF16, flags=0, mb_tokens=0, ring_slots=0) -> _lib.MoeDesc:
    return _lib.MoeDesc(T=T, d=d, E=E, I=I, k=k, dtype=dtype, mb_tokens=mb_tokens,
                        ring_slots=ring_slots, flags=flags, reserved=0)


def workspace_sizes(desc):
    """(forward scratch, saved, backward scratch) bytes."""
    lib = _lib.load()
    f, s, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _lib.check(lib.mok_moe_workspace_size(ctypes.byref(desc), ctypes.byref(f), ctypes.byref(s),
                                          ctypes.byref(b)), "mok_moe_workspace_size")
    return f.value, s.value, b.value


def saved_layout(desc) -> _lib.SavedLayout:
    lib = _lib.load()
    L = _lib.SavedLayout()
    _lib.check(lib.mok_moe_saved_layout(ctypes.byref(desc), ctypes.byref(L)), "mok_moe_saved_layout")
    return L


def stage_workspace_size(desc) -> int:
    lib = _lib.load()
    n = ctypes.c_size_t()
    _lib.check(lib.mok_moe_stage_workspace_size(ctypes.byref(desc), ctypes.byref(n)),
               "mok_moe_stage_workspace_size")
    return n.value


def forward(desc, x, w_router, bias, w_gate_up, w_down, y, saved, workspace, stream=None):
    lib = _lib.load()
    _lib.check(lib.mok_moe_forward(ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(bias),
                                   _ptr(w_gate_up), _ptr(w_down), _ptr(y), _ptr(saved),
                                   saved.numel(), _ptr(workspace), workspace.numel(),
                                   _stream(stream)), "mok_moe_forward")


def backward(desc, dy, x, w_router, bias, w_gate_up, w_down, saved, dx, dw_router, dw_gate_up,
             dw_down, workspace, stream=None):
    lib = _lib.load()
    _lib.check(lib.mok_moe_backward(ctypes.byref(desc), _ptr(dy), _ptr(x), _ptr(w_router),
                                    _ptr(bias), _ptr(w_gate_up), _ptr(w_down), _ptr(saved),
                                    saved.numel(), _ptr(dx), _ptr(dw_router), _ptr(dw_gate_up),
                                    _ptr(dw_down), _ptr(workspace), workspace.numel(),
                                    _stream(stream)), "mok_moe_backward")


def route(desc, x, w_router, bias, topk_idx, topk_w, workspace, stream=None):
    lib = _lib.load()
    _lib.check(lib.mok_moe_route(ctypes.byref(desc), _ptr(x), _ptr(w_router), _ptr(bias),
                                 _ptr(topk_idx), _ptr(topk_w), _ptr(workspace), workspace.numel(),
                                 _stream(stream)), "mok_moe_route")


def dispatch_plan(desc, topk_idx, counts, offsets, pos, token_of_row, workspace, stream=None):
    lib = _lib.load()
    _lib.check(lib.mok_moe_dispatch_plan(ctypes.byref(desc), _ptr(topk_idx), _ptr(counts),
                                         _ptr(offsets), _ptr(pos), _ptr(token_of_row),
                                         _ptr(workspace), workspace.numel(), _stream(stream)),
               "mok_moe_dispatch_plan")


def gemm_bf16(A, a_mn_major, B, b_mn_major, C, workspace, stream=None):
    """C = A @ B with A given as [M,K] (a_mn_major=False) or [K,M] (True) and
    B as [N,K] (b_mn_major=False) or [K,N] (True)."""
    lib = _lib.load()
    M, N = C.shape
    K = A.shape[0] if a_mn_major else A.shape[1]
    _lib.check(lib.mok_gemm_bf16(M, N, K, _ptr(A), int(a_mn_major), _ptr(B), int(b_mn_major),
                                 _ptr(C), _ptr(workspace), workspace.numel(), _stream(stream)),
               "mok_gemm_bf16")


def gemm_mxfp8(A, sa, B, sb, C, workspace, cta_pair=False, stream=None):
    """C[M,N] fp32 = dequant(A) dequant(B)^T for E4M3 codes A [M,K], B [N,K]
    and E8M0 scale bytes sa [M,K/32], sb [N,K/32] (see mok_gemm_mxfp8)."""
    lib = _lib.load()
    M, N = C.shape
    K = A.shape[1]
    _lib.check(lib.mok_gemm_mxfp8(M, N, K, _ptr(A), _ptr(sa), _ptr(B), _ptr(sb), _ptr(C),
                                  int(cta_pair), _ptr(workspace), workspace.numel(),
                                  _stream(stream)),
               "mok_gemm_mxfp8")


def mx_quantize(x, along_rows: bool, out=None, codes=None, scales=None, stream=None):
    """MXFP8 fake quantisation of a 2-D bf16 tensor (see mok_mx_quantize)."""
    lib = _lib.load()
    out = torch.empty_like(x) if out is None else out
    rows, cols = x.shape
    _lib.check(lib.mok_mx_quantize(_ptr(x), rows, cols, int(along_rows), _ptr(out), _ptr(codes),
                                   _ptr(scales), _stream(stream)), "mok_mx_quantize")
    return out


def nvfp4_tensor_scale(x, g=None, stream=None):
    """NVFP4 tensor scale of a bf16 tensor into the device fp32 `g` (see
    mok_nvfp4_tensor_scale)."""
    g = torch.empty(1, dtype=torch.float32, device=x.device) if g is None else g
    _lib.check(_lib.load().mok_nvfp4_tensor_scale(_ptr(x), x.numel(), _ptr(g), _stream(stream)),
               "mok_nvfp4_tensor_scale")
    return g


def nvfp4_quantize(x, g, codes=None, scales=None, stream=None):
    """NVFP4 codes [rows, cols/2] and E4M3 block scales [rows, cols/16] of a
    2-D bf16 tensor with tensor scale g (see mok_nvfp4_quantize)."""
    rows, cols = x.shape
    codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device) if codes is None \
        else codes
    scales = torch.empty(rows, cols // 16, dtype=torch.uint8, device=x.device) if scales is None \
        else scales
    _lib.check(_lib.load().mok_nvfp4_quantize(_ptr(x), rows, cols, _ptr(g), _ptr(codes),
                                              _ptr(scales), _stream(stream)),
               "mok_nvfp4_quantize")
    return codes, scales


def nvfp4_quantize_cols(x, g, codes=None, scales=None, stream=None):
    """NVFP4 of the columns of a bf16 [ng, K, C] (or [K, C]) tensor, blocks of
    16 along K: codes [ng*C, K/2] and E4M3 scales [ng*C, K/16] (see
    mok_nvfp4_quantize_cols)."""
    x3 = x if x.dim() == 3 else x.unsqueeze(0)
    ng, K, C = x3.shape
    codes = torch.empty(ng * C, K // 2, dtype=torch.uint8, device=x.device) if codes is None \
        else codes
    scales = torch.empty(ng * C, K // 16, dtype=torch.uint8, device=x.device) if scales is None \
        else scales
    _lib.check(_lib.load().mok_nvfp4_quantize_cols(_ptr(x3), ng, K, C, _ptr(g), _ptr(codes),
                                                   _ptr(scales), _stream(stream)),
               "mok_nvfp4_quantize_cols")
    return codes, scales


def gemm_nvfp4(A, sa, ga, B, sb, gb, C, workspace, stream=None):
    """C[M,N] fp32 = ga gb dequant(A) dequant(B)^T for NVFP4 codes A [M,K/2],
    B [N,K/2], E4M3 block scales sa [M,K/16], sb [N,K/16] and device tensor
    scales ga, gb (see mok_gemm_nvfp4)."""
    M, N = C.shape
    K = 2 * A.shape[1]
    _lib.check(_lib.load().mok_gemm_nvfp4(M, N, K, _ptr(A), _ptr(sa), _ptr(ga), _ptr(B),
                                          _ptr(sb), _ptr(gb), _ptr(C), _ptr(workspace),
                                          workspace.numel(), _stream(stream)), "mok_gemm_nvfp4")


def device_status(buf, stream=None) -> int:
    """Synchronises the stream and returns the device status word of `buf`."""
    lib = _lib.load()
    code = ctypes.c_int32()
    _lib.check(lib.mok_get_device_status(_ptr(buf), _stream(stream), ctypes.byref(code)),
               "mok_get_device_status")
    return code.value


def fill_zero(buf, stream=None):
    """Zeroes the contiguous device tensor `buf` with the library's bulk-store
    fill (its byte size a multiple of 16, its address 16-byte aligned)."""
    nbytes = buf.numel() * buf.element_size()
    _lib.check(_lib.load().mok_fill_zero(_ptr(buf), nbytes, _stream(stream)), "mok_fill_zero")
    return buf


def last_launch_count() -> int:
    return int(_lib.load().mok_last_launch_count())


def profile_enable(on: bool = True):
    _lib.check(_lib.load().mok_profile_enable(int(on)), "mok_profile_enable")


def profile_reset():
    _lib.check(_lib.load().mok_profile_reset(), "mok_profile_reset")


def profile_collect() -> dict:
    """{kernel name: (launches, total ms)} since the last reset (waits for the events)."""
    lib = _lib.load()
    buf = (_lib.KernelTime * 64)()
    n = ctypes.c_int32()
    _lib.check(lib.mok_profile_collect(buf, 64, ctypes.byref(n)), "mok_profile_collect")
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(n.value)}


class MoELayer:
    """Owns the three buffers of one layer shape and calls forward/backward."""

    def __init__(self, T, d, E, I, k, device="cuda", flags=0, dtype=BF16, mb_tokens=0,
                 ring_slots=0):
        self.desc = make_desc(T, d, E, I, k, dtype=dtype, flags=flags, mb_tokens=mb_tokens,
                              ring_slots=ring_slots)
        self.T, self.d, self.E, self.I, self.k = T, d, E, I, k
        self.act_dtype = torch.bfloat16 if flags & FLAG_BF16_ACT_OUT else torch.float32
        self.wgrad_dtype = torch.bfloat16 if flags & FLAG_BF16_WGRAD_OUT else torch.float32
        f, s, b = workspace_sizes(self.desc)
        self.fwd_ws = torch.empty(max(f, 256), dtype=torch.uint8, device=device)
        self.saved = torch.zeros(max(s, 256), dtype=torch.uint8, device=device)
        self.bwd_ws = torch.empty(max(b, 256), dtype=torch.uint8, device=device)
        self.layout = saved_layout(self.desc)

    def saved_tensor(self, field: str, dtype, shape, micro_batch: int = 0):
        off = getattr(self.layout, field)
        if off == NOT_KEPT:
            raise KeyError(f"{field} is not kept in saved with these flags")
        off += micro_batch * self.layout.mb_stride
        n = 1
        for v in shape:
            n *= v
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.saved[off:off + nbytes].view(dtype).view(*shape)

    def forward(self, x, w_router, bias, w_gate_up, w_down, y=None, stream=None):
        if y is None:
            y = torch.empty(x.shape, dtype=self.act_dtype, device=x.device)
        forward(self.desc, x, w_router, bias, w_gate_up, w_down, y, self.saved, self.fwd_ws,
                stream)
        return y

    def backward(self, dy, x, w_router, bias, w_gate_up, w_down, dx=None, dw_router=None,
                 dw_gate_up=None, dw_down=None, stream=None):
        def out(like, dt, given):
            return torch.empty(like.shape, dtype=dt, device=like.device) if given is None else given
        dx = out(x, self.act_dtype, dx)
        dw_router = out(w_router, self.wgrad_dtype, dw_router)
        dw_gate_up = out(w_gate_up, self.wgrad_dtype, dw_gate_up)
        dw_down = out(w_down, self.wgrad_dtype, dw_down)
        backward(self.desc, dy, x, w_router, bias, w_gate_up, w_down, self.saved, dx, dw_router,
                 dw_gate_up, dw_down, self.bwd_ws, stream)
        return dx, dw_router, dw_gate_up, dw_down

    def status(self, stream=None) -> int:
        return device_status(self.saved, stream)
