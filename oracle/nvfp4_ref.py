"""NVFP4 quantisation for the oracle: E2M1 elements, one E4M3 scale per block
of 16 consecutive values, and one float32 scale per tensor.

TEST INFRASTRUCTURE (see the package docstring).

Source: [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by
5.8x", section "Background: solving the MoE bottleneck": Cursor's earlier
training kernels ran the expert GEMMs in MXFP8 and NVFP4.  The pages do not
define NVFP4, so NVIDIA's published format is taken (a reading, listed in the
design notes), with one fixed order of operations, all in float32 (the
kernel's precision, so that both sides take every rounding decision alike);
the block and element steps multiply by rounded reciprocals:
  * tensor scale   g   = amax(|a|) / 2688          (2688 = 6 * 448: the
                   largest E2M1 magnitude times the largest E4M3 one);
                   g = 1 for an all-zero tensor;
  * block scale    s_b = RNE_E4M3(amax_b * r6)     with r6 = RN(1 / RN(6 g));
                   saturating at 448; a positive E4M3 value or 0;
  * element        q   = RNE_E2M1(v * r_b)         with r_b = RN(1 / RN(s_b g))
                   (the largest finite float32 where that overflows);
                   saturating at +-6; 0 where s_b = 0;
  * value          q * s_b * g.
E2M1: sign, two exponent bits (bias 1), one mantissa bit; magnitudes 0, 0.5,
1, 1.5, 2, 3, 4, 6; ties go to the even code (mantissa bit 0).
"""
from __future__ import annotations

import numpy as np

from .mx_ref import e4m3_round

E2M1_MAX = 6.0
E4M3_MAX = 448.0
BLOCK = 16
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_round(v) -> np.ndarray:
    """Nearest E2M1 value (ties to the even code), saturating at +-6.

    The grid is evenly spaced inside three bands: step 0.5 on [0, 2] (codes
    0..4 are the multiples 0..4), step 1 on [2, 4] (codes 4..6 are the
    multiples 2..4) and step 2 on [4, 6] (codes 6, 7 are the multiples 2, 3).
    In each band an even multiple is an even code, so rounding the multiple
    half to even is rounding to the nearest code, ties to the even one."""
    v = np.asarray(v, dtype=np.float64)
    m = np.minimum(np.abs(v), E2M1_MAX)
    step = np.where(m < 2.0, 0.5, np.where(m < 4.0, 1.0, 2.0))
    r = np.round(m / step) * step          # np.round: half to even
    return np.copysign(r, v)


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def nvfp4_quantize(a, axis: int = -1):
    """Fake-quantise `a` to NVFP4 along `axis` (its length a multiple of 16).

    Returns (dequantised float64 array, element values q, block scales s_b
    (float64, E4M3 values), tensor scale g (float))."""
    a = np.asarray(a, dtype=np.float64)
    x = np.moveaxis(a, axis, -1)
    n = x.shape[-1]
    assert n % BLOCK == 0, n
    xf = _f32(x)
    amax_t = np.float32(np.abs(xf).max()) if xf.size else np.float32(0)
    g = np.float32(amax_t / np.float32(6.0 * E4M3_MAX)) if amax_t > 0 else np.float32(1.0)
    blocks = xf.reshape(xf.shape[:-1] + (n // BLOCK, BLOCK))
    amax_b = np.abs(blocks).max(axis=-1)
    six_g = np.float32(np.float32(6.0) * g)
    r6 = np.float32(np.float32(1.0) / six_g)
    sb = e4m3_round((amax_b * r6).astype(np.float32).astype(np.float64))
    sb = np.minimum(sb, E4M3_MAX)
    denom = (_f32(sb) * g).astype(np.float32)                    # s_b g, rounded
    with np.errstate(divide="ignore", over="ignore"):
        rb = (np.float32(1.0) / denom).astype(np.float32)        # inf where s_b = 0
        rb = np.minimum(rb, np.finfo(np.float32).max)
        ratio = (blocks * rb[..., None]).astype(np.float32).astype(np.float64)
    q = np.where(sb[..., None] > 0, e2m1_round(ratio), 0.0)
    deq = q * sb[..., None] * np.float64(g)
    out = np.moveaxis(deq.reshape(x.shape), -1, axis)
    qv = np.moveaxis(q.reshape(x.shape), -1, axis)
    return out, qv, sb, float(g)


def nvfp4_fake(a, axis: int = -1) -> np.ndarray:
    return nvfp4_quantize(a, axis)[0]
