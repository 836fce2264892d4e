"""MX (microscaling) quantisation for the oracle: E4M3 elements with one E8M0
power-of-two scale per block of 32 consecutive values.

TEST INFRASTRUCTURE (see the package docstring).

Source: [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by
5.8x", "MoK technical details", bullet "Precision and scheduling": the
megakernel supports MXFP8.  The pages do not give the scaling rule, so the
public OCP Microscaling (MX) v1.0 rule is taken (a reading, listed in the
design notes):
  * block of 32 consecutive values along the GEMM's reduction dimension;
  * shared exponent = floor(log2(max |v|)) - 8 (8 = exponent of the largest
    E4M3 normal, 448 = 1.75 * 2^8), clamped to the E8M0 range [-127, 127];
    an all-zero block takes the smallest scale;
  * each element v / 2^shared is rounded to nearest, ties to even, onto the
    E4M3 grid (3 mantissa bits, normals down to 2^-6, subnormals in steps of
    2^-9), saturating at +-448;
  * the dequantised value is that grid value times 2^shared.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8
E4M3_MIN_NORMAL_EXP = -6
E4M3_SUBNORMAL_STEP = 2.0 ** -9
BLOCK = 32


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value (ties to even), saturating at +-448 (float64 in/out)."""
    v = np.asarray(v, dtype=np.float64)
    m = np.abs(v)
    _, ex = np.frexp(m)                     # m = f * 2**ex, 0.5 <= f < 1
    e = ex - 1                              # floor(log2 m) for m > 0
    normal = m >= 2.0 ** E4M3_MIN_NORMAL_EXP
    ulp = np.where(normal, np.ldexp(1.0, np.where(normal, e - 3, 0)), E4M3_SUBNORMAL_STEP)
    r = np.round(m / ulp) * ulp             # np.round: half to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v)


def mx_quantize(a, axis: int = -1):
    """Fake-quantise `a` to MXFP8 along `axis` (its length a multiple of 32).

    Returns (dequantised float64 array, shared exponents per block)."""
    a = np.asarray(a, dtype=np.float64)
    x = np.moveaxis(a, axis, -1)
    n = x.shape[-1]
    assert n % BLOCK == 0, n
    blocks = x.reshape(x.shape[:-1] + (n // BLOCK, BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    _, ex = np.frexp(amax)
    shared = np.where(amax > 0, ex - 1 - E4M3_EMAX, -127)
    shared = np.clip(shared, -127, 127)
    scale = np.ldexp(1.0, shared)[..., None]
    q = e4m3_round(blocks / scale) * scale
    out = np.moveaxis(q.reshape(x.shape), -1, axis)
    return out, shared


def mx_fake(a, axis: int = -1) -> np.ndarray:
    return mx_quantize(a, axis)[0]
