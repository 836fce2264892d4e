"""Pins for the oracle's NVFP4 quantiser (E2M1 elements, E4M3 scale per 16
values, float32 scale per tensor).

  * e2m1_round against a brute-force nearest-value search over the 15 finite
    E2M1 codes, decoded here from the code layout (sign, 2 exponent bits with
    bias 1, 1 mantissa bit; subnormals at exponent 0), ties to the even code,
    saturation at 6;
  * blocks built from E2M1 values, E4M3 block scales and a power-of-two
    tensor scale survive quantisation unchanged;
  * every block whose scale is a normal E4M3 value puts its largest
    magnitude on the code 6, and every element within half a grid step (in
    units of the block's scale) of its value;
  * all-zero blocks and tensors stay zero; quantising along axis 0 is
    quantising the transpose along axis 1.
"""
import numpy as np
import pytest

from oracle import nvfp4_ref, mx_ref


def _e2m1_codes():
    vals = []
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        vals.append(((-1) ** s * mag, m))
    return vals


def _brute(v, grid):
    best = None
    for g, m in grid:
        dist = abs(v - g)
        if best is None or dist < best[0] or (dist == best[0] and m % 2 == 0):
            best = (dist, g)
    return best[1]


def test_e2m1_grid_decodes_to_the_expected_magnitudes():
    mags = sorted({abs(g) for g, _ in _e2m1_codes()})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_round_is_nearest_code_ties_to_even():
    grid = _e2m1_codes()
    rng = np.random.default_rng(0)
    vs = list(rng.uniform(-7, 7, 500))
    pos = sorted({g for g, _ in grid if g >= 0})
    vs += [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]       # every tie
    vs += [-(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]
    vs += [6.0, 6.5, 100.0, -1e9, 0.0, 1e-9]
    got = nvfp4_ref.e2m1_round(np.array(vs))
    for v, q in zip(vs, got):
        want = _brute(v, grid) if abs(v) <= 6 else np.copysign(6.0, v)
        assert q == want, (v, q, want)


def _e4m3_values():
    """Positive normal E4M3 values, decoded from the code layout."""
    out = []
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            out.append(2.0 ** (e - 7) * (1 + m / 8))
    return np.array(out)


@pytest.mark.parametrize("j", [-10, 0, 3])
def test_nvfp4_representable_blocks_round_trip(j):
    rng = np.random.default_rng(j + 20)
    g = 2.0 ** j
    nblk = 12
    sb = rng.choice(_e4m3_values()[(_e4m3_values() >= 2.0 ** -4)], size=nblk)
    sb[0] = 448.0                       # the tensor's largest block: amax = 6 * 448 * g
    q = rng.choice(nvfp4_ref.E2M1_GRID, size=(nblk, 16)) * rng.choice([-1.0, 1.0], (nblk, 16))
    q[:, 3] = 6.0                        # every block's largest magnitude is 6
    a = (q * sb[:, None] * g).reshape(1, -1)
    deq, qv, sbv, gv = nvfp4_ref.nvfp4_quantize(a, axis=1)
    assert gv == g
    assert np.array_equal(sbv.ravel(), sb)
    assert np.array_equal(qv.reshape(nblk, 16), q)
    assert np.array_equal(deq, a)


def test_nvfp4_block_maximum_maps_to_six_and_elements_to_the_nearest_code():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((16, 8 * 16)) * np.exp(rng.uniform(-3, 3, (16, 1)))
    deq, q, sb, g = nvfp4_ref.nvfp4_quantize(a, axis=1)
    blocks = np.abs(a).reshape(16, 8, 16)
    qb = np.abs(q).reshape(16, 8, 16)
    normal = sb >= 2.0 ** -6
    assert normal.sum() > 100
    top = np.take_along_axis(qb, blocks.argmax(axis=2)[..., None], axis=2)[..., 0]
    assert (top[normal] == 6.0).all()
    # each element sits within half a grid step of its value / (s_b g), in
    # units of the block scale (steps 0.5, 1, 2 below 2, 4, 6), or saturates
    r = (blocks / (sb[..., None] * g))
    step = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
    err = np.abs(qb - np.minimum(r, 6.0))
    assert (err[normal] <= step[normal] / 2 + 1e-6).all()


def test_nvfp4_zero_blocks_and_tensor():
    a = np.zeros((2, 32))
    a[1, 16:] = np.linspace(-1, 1, 16)
    deq, q, sb, g = nvfp4_ref.nvfp4_quantize(a, axis=1)
    assert (deq[0] == 0).all() and (deq[1, :16] == 0).all() and sb[0, 0] == 0 and sb[1, 0] == 0
    d0, _, _, g0 = nvfp4_ref.nvfp4_quantize(np.zeros((3, 16)), axis=1)
    assert g0 == 1.0 and (d0 == 0).all()


def test_nvfp4_along_axis0_is_the_transpose():
    rng = np.random.default_rng(4)
    a = rng.standard_normal((48, 5))
    q0 = nvfp4_ref.nvfp4_fake(a, axis=0)
    q1 = nvfp4_ref.nvfp4_fake(a.T, axis=1)
    assert np.array_equal(q0, q1.T)


def test_nvfp4_scales_are_e4m3_values():
    rng = np.random.default_rng(5)
    _, _, sb, _ = nvfp4_ref.nvfp4_quantize(rng.standard_normal((8, 64)), axis=1)
    assert np.array_equal(mx_ref.e4m3_round(sb), sb)
    assert (sb >= 0).all() and (sb <= 448).all()
