"""The block-scaled weights the forward leaves in `saved` for the backward,
bit for bit against the oracle's quantisers: W_gate_up along 2I (the gate/up
dgrad's operand; MXFP8 and NVFP4 codes with their tiled scales) and, for
MXFP8, W_down along d as bf16 values (the down dgrad's operand).  The forward
writes them from the same read of each weight as its own row codes, so these
also pin the tile kernels that do both orientations at once."""
import numpy as np
import pytest
import torch

from oracle import mx_ref, nvfp4_ref
from routing_dispatch_grouped_router_gb300 import api
from routing_dispatch_grouped_router_gb300 import inputs as gen

import _gpu

pytestmark = pytest.mark.gpu

SHAPES = [gen.Shape(T=256, d=256, E=4, I=256, k=2), gen.Shape(T=128, d=512, E=3, I=768, k=2)]


def _untile(buf, rows, nblk):
    """Scale bytes of a [rows, nblk blocks] operand from the GEMMs' tiled
    layout: per 128 rows and 4 consecutive blocks one 512-byte group, row r's
    block j at byte 16 (r % 32) + 4 ((r / 32) % 4) + j % 4 of it."""
    r = np.arange(rows)[:, None]
    j = np.arange(nblk)[None, :]
    off = ((r >> 7) * (nblk // 4) + (j >> 2)) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3) + (j & 3)
    return buf[off]


def _e4m3_values(codes):
    c = codes.astype(np.int64)
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, 2.0 ** (e - 7) * (1 + m / 8))
    return np.where(s == 1, -mag, mag)


def _e2m1_values(codes):
    lo, hi = codes & 15, codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1).astype(np.int64)
    s, e, m = c >> 3, (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, 2.0 ** (e - 1) * (1 + m / 2))
    return np.where(s == 1, -mag, mag)


def _weights(inp):
    f = gen.bf16_bits_to_f32
    return f(inp["w_gate_up"]).astype(np.float64), f(inp["w_down"]).astype(np.float64)


@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_mxfp8_backward_weight_forms(si):
    shape = SHAPES[si]
    inp = gen.make_inputs(shape, seed=5)
    gpu = _gpu.run_gpu(shape, inp, dtype=api.MXFP8)
    assert gpu["status"] == 0
    layer, (E, d, I) = gpu["layer"], (shape.E, shape.d, shape.I)
    wgu, wd = _weights(inp)
    n = E * 2 * I * d
    raw = layer.saved_tensor("w_gate_up_t", torch.uint8, (n + n // 32,)).cpu().numpy()
    codes = raw[:n].reshape(E * d, 2 * I)
    shared = _untile(raw[n:], E * d, 2 * I // 32).astype(np.int64) - 127
    got = _e4m3_values(codes) * np.repeat(np.ldexp(1.0, shared), 32, axis=1)
    ref = mx_ref.mx_fake(wgu, axis=1).transpose(0, 2, 1).reshape(E * d, 2 * I)
    assert np.array_equal(got, ref)
    wdc = layer.saved_tensor("w_down_col", torch.bfloat16, (E * d, I)).float().cpu().numpy()
    assert np.array_equal(wdc.astype(np.float64), mx_ref.mx_fake(wd, axis=1).reshape(E * d, I))


@pytest.mark.parametrize("si", range(len(SHAPES)))
def test_nvfp4_backward_weight_forms(si):
    shape = SHAPES[si]
    inp = gen.make_inputs(shape, seed=6)
    gpu = _gpu.run_gpu(shape, inp, dtype=api.NVFP4)
    assert gpu["status"] == 0
    layer, (E, d, I) = gpu["layer"], (shape.E, shape.d, shape.I)
    wgu, _ = _weights(inp)
    n = E * 2 * I * d
    raw = layer.saved_tensor("w_gate_up_t", torch.uint8, (n // 2 + n // 16,)).cpu().numpy()
    q = _e2m1_values(raw[:n // 2].reshape(E * d, I))
    sb = _untile(raw[n // 2:], E * d, 2 * I // 16)
    _, q_ref, sb_ref, _ = nvfp4_ref.nvfp4_quantize(wgu, 1)     # along 2I, one tensor scale
    assert np.array_equal(q, q_ref.transpose(0, 2, 1).reshape(E * d, 2 * I))
    e, m = (sb.astype(np.int64) >> 3) & 15, sb.astype(np.int64) & 7
    sb_val = np.where(e == 0, m * 2.0 ** -9, 2.0 ** (e - 7) * (1 + m / 8))
    assert np.array_equal(sb_val, sb_ref.reshape(E * d, 2 * I // 16))
    with pytest.raises(KeyError):
        layer.saved_tensor("w_down_col", torch.bfloat16, (1,))
