"""Pins for the oracle's MXFP8 quantiser and its MXFP8 layer mode.

  * e4m3_round against a brute-force nearest-value search over the 254 finite
    E4M3 codes, decoded here from the code layout (sign, 4 exponent bits with
    bias 7, 3 mantissa bits; subnormals at exponent 0), ties to the even
    mantissa code, saturation at 448;
  * values already on the E4M3 grid times a power of two survive
    quantisation unchanged;
  * every block's scale puts its largest magnitude in [256, 512) before
    rounding, and all-zero blocks stay zero;
  * the MXFP8 layer mode with quantisation switched off is the fp64 mode,
    and with it on differs from fp64 by MXFP8 noise, not more.
"""
import numpy as np
import pytest

import oracle
from oracle import moe_ref, mx_ref
from routing_dispatch_grouped_router_gb300 import inputs as gen


def _e4m3_codes():
    vals = []
    for code in range(256):
        s, e, m = code >> 7, (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue  # NaN
        mag = 2.0 ** (e - 7) * (1 + m / 8) if e > 0 else 2.0 ** -6 * (m / 8)
        vals.append(((-1) ** s * mag, m))
    return vals


def _brute(v, grid):
    best = None
    for g, m in grid:
        dist = abs(v - g)
        if best is None or dist < best[0] - 1e-300 or (dist == best[0] and m % 2 == 0):
            best = (dist, g)
    return best[1]


def test_e4m3_round_is_nearest_code_ties_to_even():
    grid = _e4m3_codes()
    assert len(grid) == 254
    rng = np.random.default_rng(0)
    vs = list(rng.uniform(-470, 470, 400)) + list(rng.uniform(-0.05, 0.05, 300))
    # exact midpoints between neighbouring codes exercise the tie rule
    pos = sorted({g for g, _ in grid if g >= 0})
    vs += [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])][::3]
    vs += [500.0, -1e6, 449.0, 2.0 ** -10, -(2.0 ** -10) * 3]
    got = mx_ref.e4m3_round(np.array(vs))
    for v, q in zip(vs, got):
        want = _brute(v, grid) if abs(v) <= 448 else np.copysign(448.0, v)
        assert q == want, (v, q, want)


def test_mx_grid_values_round_trip():
    rng = np.random.default_rng(1)
    grid = np.array([g for g, _ in _e4m3_codes()])
    top = grid[(np.abs(grid) >= 256)]
    for k in (-20, -3, 0, 5):
        blocks = rng.choice(grid, size=(16, 32))
        blocks[:, 0] = rng.choice(top, size=16)     # largest element in the top binade
        a = blocks * 2.0 ** k
        q, shared = mx_ref.mx_quantize(a, axis=1)
        assert np.array_equal(q, a)
        assert (shared == k).all()


def test_mx_block_scale_range_and_zero_blocks():
    rng = np.random.default_rng(2)
    a = rng.standard_normal((8, 4 * 32)) * np.exp(rng.uniform(-20, 20, (8, 1)))
    a[3, 32:64] = 0.0
    q, shared = mx_ref.mx_quantize(a, axis=1)
    blocks = np.abs(a).reshape(8, 4, 32).max(axis=2)
    nz = blocks > 0
    scale = 2.0 ** shared
    assert ((blocks[nz] >= 256 * scale[nz]) & (blocks[nz] < 512 * scale[nz])).all()
    assert shared[3, 1] == -127 and (q[3, 32:64] == 0).all()
    # each element is off by at most half an ulp of the block's top binade
    # (16 * scale), or by the saturation from below 512 * scale to 448 * scale
    err = np.abs(q - a).reshape(8, 4, 32)
    big = np.abs(a).reshape(8, 4, 32) > 448 * scale[..., None]
    assert (err[~big] <= (16 * scale[..., None] * np.ones_like(err))[~big]).all()
    assert (err[big] < (64 * scale[..., None] * np.ones_like(err))[big]).all()


def test_mx_quantize_along_axis0():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((64, 5))
    q0, _ = mx_ref.mx_quantize(a, axis=0)
    q1, _ = mx_ref.mx_quantize(a.T, axis=1)
    assert np.array_equal(q0, q1.T)


def _tiny(seed=0, T=24, d=64, E=4, I=64, k=2):
    sh = gen.Shape(T=T, d=d, E=E, I=I, k=k)
    return sh, gen.make_inputs(sh, seed)


def test_mxfp8_mode_without_quantisation_is_fp64_mode(monkeypatch):
    sh, inp = _tiny(seed=4)
    args = (inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], sh.k)
    y64, f64 = oracle.moe_forward_ref(*args, keep=True)
    g64 = oracle.moe_backward_ref(*args, inp["dy"], fwd=f64)
    monkeypatch.setattr(moe_ref, "mx_fake", lambda a, axis=-1: np.asarray(a, dtype=np.float64))
    ym, fm = oracle.moe_forward_ref(*args, keep=True, precision="mxfp8")
    gm = oracle.moe_backward_ref(*args, inp["dy"], fwd=fm)
    np.testing.assert_allclose(ym, y64, rtol=1e-12, atol=1e-12)
    for n in ("dx", "dw_router", "dw_gate_up", "dw_down"):
        np.testing.assert_allclose(gm[n], g64[n], rtol=1e-11, atol=1e-11)


def test_mxfp8_mode_is_fp64_plus_mx_noise():
    """E4M3 keeps 3 mantissa bits (elements off by up to 1/16 of their block
    scale's binade), so over K = 512 the outputs move by a few percent of
    their rms, far less than an error of structure would."""
    sh, inp = _tiny(seed=5, T=48, d=512, I=512)
    args = (inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], sh.k)
    y64, f64 = oracle.moe_forward_ref(*args, keep=True)
    g64 = oracle.moe_backward_ref(*args, inp["dy"], fwd=f64)
    ym, fm = oracle.moe_forward_ref(*args, keep=True, precision="mxfp8")
    gm = oracle.moe_backward_ref(*args, inp["dy"], fwd=fm)
    for got, ref in [(ym, y64), (gm["dx"], g64["dx"])]:
        rel = np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2))
        assert 1e-3 < rel < 0.1, rel
