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
    quantising the transpose along axis 1;
  * the layer's NVFP4 mode: with quantisation switched off it is the fp64
    mode; W_down scaled by 2^3 scales y by 2^3 (the tensor scale absorbs it);
    and the axis of each forward operand (x and W_gate_up along d, W_down and
    h along I) by power-of-two scale covariance of rows below each tensor's
    maximum, and of the gate/up dgrad's operands (dG/dU and W_gate_up along
    2I); planted wrong axes fail these pins.
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


# ----------------------------------------------------------------------------
# the layer's NVFP4 mode (moe_forward_ref(precision="nvfp4")): forward GEMM
# operands quantised along their reduction dimension with whole-tensor scales;
# h in bf16 before its quantisation; float64 backward with dp = <dy W_down, h>
# ----------------------------------------------------------------------------

import oracle  # noqa: E402
from oracle import moe_ref  # noqa: E402

D, I_ = 64, 96


def _case(seed, T=64, E=2, gate_positive=False):
    """Top-1 routing forced to T // E tokens per expert; the largest value of
    x sits in token 0, of W_gate_up in row 0 and of W_down in row 0 of expert
    0, so scaling other rows down by a power of two leaves every tensor scale
    as it is."""
    rng = np.random.default_rng(seed)
    x = rng.uniform(1, 2, (T, D)) if gate_positive else rng.standard_normal((T, D))
    wgu = rng.standard_normal((E, 2 * I_, D)) / np.sqrt(D)
    if gate_positive:
        wgu[:, :I_] = rng.uniform(1, 2, (E, I_, D))
    wd = rng.standard_normal((E, D, I_)) / np.sqrt(I_)
    x[0, 0] = 3 * np.abs(x).max()
    wgu[0, 0, 0] = 3 * np.abs(wgu).max()
    wd[0, 0, 0] = 3 * np.abs(wd).max()
    idx = rng.permutation(np.repeat(np.arange(E), T // E)).astype(np.int32)[:, None]
    return dict(x=x, w_router=rng.standard_normal((E, D)), w_gate_up=wgu, w_down=wd,
                dy=rng.standard_normal((T, D)), routing=(idx, np.ones((T, 1))))


def _fwd(c, precision="nvfp4"):
    return oracle.moe_forward_ref(c["x"], c["w_router"], None, c["w_gate_up"], c["w_down"], 1,
                                  routing=c["routing"], keep=True, precision=precision)


def _scaled(before, after, mask, f, what):
    want = np.where(mask, before * f, before)
    np.testing.assert_allclose(after, want, rtol=1e-12,
                               atol=1e-12 * float(np.sqrt(np.mean(want ** 2))), err_msg=what)


def test_nvfp4_layer_without_quantisation_is_fp64(monkeypatch):
    c = _case(30)
    y64, f64 = _fwd(c, "fp64")
    g64 = oracle.moe_backward_ref(c["x"], c["w_router"], None, c["w_gate_up"], c["w_down"], 1,
                                  c["dy"], fwd=f64)
    monkeypatch.setattr(moe_ref, "nvfp4_fake", lambda a, axis=-1: np.asarray(a, np.float64))
    monkeypatch.setattr(moe_ref, "bf16_round", lambda a: np.asarray(a, np.float64))
    yn, fn = _fwd(c)
    gn = oracle.moe_backward_ref(c["x"], c["w_router"], None, c["w_gate_up"], c["w_down"], 1,
                                 c["dy"], fwd=fn)
    np.testing.assert_allclose(yn, y64, rtol=1e-12, atol=1e-12)
    for n in ("dx", "dw_router", "dw_gate_up", "dw_down", "dp"):
        np.testing.assert_allclose(gn[n], g64[n], rtol=1e-10, atol=1e-10, err_msg=n)


def test_nvfp4_layer_is_fp64_plus_fp4_noise():
    c = _case(31)
    y64, _ = _fwd(c, "fp64")
    yn, _ = _fwd(c)
    rel = np.sqrt(np.mean((yn - y64) ** 2) / np.mean(y64 ** 2))
    assert 1e-2 < rel < 0.5, rel


def _pin_w_down_global_scale():
    """W_down -> 2^3 W_down: its tensor scale absorbs the factor, so y -> 2^3 y."""
    c = _case(32)
    y0, _ = _fwd(c)
    y1, _ = _fwd(dict(c, w_down=c["w_down"] * 8.0))
    _scaled(y0, y1, True, 8.0, "y")


def _pin_x_rows():
    """Tokens (not token 0) -> 2^-2: x is quantised along d, so their g, u rows
    scale by 2^-2."""
    c = _case(33)
    _, f0 = _fwd(c)
    sel = (np.arange(64) % 3 == 1)
    _, f1 = _fwd(dict(c, x=np.where(sel[:, None], c["x"] / 4, c["x"])))
    rows = np.zeros(f0["G"].shape[0], dtype=bool)
    rows[f0["pos"][sel, 0]] = True
    _scaled(f0["G"], f1["G"], rows[:, None], 0.25, "G")
    _scaled(f0["U"], f1["U"], rows[:, None], 0.25, "U")


def _pin_w_gate_up_rows():
    """W_gate_up rows (not row 0) -> 2^-1: quantised along d, so the matching
    columns of g (or u) scale by 2^-1."""
    c = _case(34)
    _, f0 = _fwd(c)
    n = np.zeros(2 * I_, dtype=bool)
    n[[5, 40, I_ + 3, I_ + 77]] = True
    w = c["w_gate_up"].copy()
    w[:, n] /= 2
    _, f1 = _fwd(dict(c, w_gate_up=w))
    _scaled(f0["G"], f1["G"], n[None, :I_], 0.5, "G")
    _scaled(f0["U"], f1["U"], n[None, I_:], 0.5, "U")


def _pin_w_down_rows():
    """W_down rows j (not 0) -> 2^-1: quantised along I, so y[:, j] scales."""
    c = _case(35)
    y0, _ = _fwd(c)
    j = np.zeros(D, dtype=bool)
    j[[3, 17, 50]] = True
    w = c["w_down"].copy()
    w[:, j] /= 2
    y1, _ = _fwd(dict(c, w_down=w))
    _scaled(y0, y1, j[None, :], 0.5, "y")


def _pin_h_rows():
    """Gate-positive regime (h = g u exactly): tokens (not token 0) -> 2^-1
    scale their h rows by 2^-2; h is quantised along I, so their y rows scale
    by 2^-2."""
    c = _case(36, gate_positive=True)
    y0, f0 = _fwd(c)
    assert f0["G"].min() >= 64
    sel = (np.arange(64) % 4 == 2)
    y1, _ = _fwd(dict(c, x=np.where(sel[:, None], c["x"] / 2, c["x"])))
    _scaled(y0, y1, sel[:, None], 0.25, "y")


def _bwd(c, f):
    return oracle.moe_backward_ref(c["x"], c["w_router"], None, c["w_gate_up"], c["w_down"], 1,
                                   c["dy"], fwd=f)


def _pin_w_gate_up_columns_backward():
    """W_gate_up column j (not 0) -> 2^-1 in the backward only (forward
    intermediates kept): the gate/up dgrad quantises W_gate_up along 2I, so
    feature j of dx scales by 2^-1."""
    c = _case(37)
    _, f = _fwd(c)
    g0 = _bwd(c, f)
    j = np.zeros(D, dtype=bool)
    j[[2, 33, 61]] = True
    w = c["w_gate_up"].copy()
    w[:, :, j] /= 2
    g1 = _bwd(dict(c, w_gate_up=w), f)
    _scaled(g0["dx"], g1["dx"], j[None, :], 0.5, "dx")


def _pin_dgu_rows_backward():
    """dy rows (not token 0, whose huge dy holds the tensor maximum of dG/dU)
    -> 2^-1: dG/dU rows scale by 2^-1 and are quantised along 2I, so those
    tokens' dx rows scale by 2^-1."""
    c = _case(38)
    c["dy"][0] *= 64
    _, f = _fwd(c)
    g0 = _bwd(c, f)
    sel = (np.arange(64) % 5 == 3)
    g1 = _bwd(dict(c, dy=np.where(sel[:, None], c["dy"] / 2, c["dy"])), f)
    _scaled(g0["dx"], g1["dx"], sel[:, None], 0.5, "dx")


NV_PINS = {"w_down_global_scale": _pin_w_down_global_scale, "x_rows": _pin_x_rows,
           "w_gate_up_rows": _pin_w_gate_up_rows, "w_down_rows": _pin_w_down_rows,
           "h_rows": _pin_h_rows, "w_gate_up_columns_backward": _pin_w_gate_up_columns_backward,
           "dgu_rows_backward": _pin_dgu_rows_backward}


@pytest.mark.parametrize("name", sorted(NV_PINS))
def test_nvfp4_layer_quantisation_axes(name):
    NV_PINS[name]()


def _plant(monkeypatch, shape_tail, rows):
    """nvfp4_fake along the rows instead of the columns for arrays whose
    trailing dimension is shape_tail (and row count `rows`, if given)."""
    real = nvfp4_ref.nvfp4_fake

    def fake(a, axis=-1):
        a = np.asarray(a)
        if a.shape[-1] == shape_tail and (rows is None or a.shape[0] == rows) \
                and axis % a.ndim == a.ndim - 1:
            axis = 0
        return real(a, axis)
    monkeypatch.setattr(moe_ref, "nvfp4_fake", fake)


@pytest.mark.parametrize("tail,rows,pin", [
    (D, 64, "x_rows"),                   # x along the tokens
    (D, 2 * 2 * I_, "w_gate_up_rows"),   # W_gate_up along 2I
    (I_, 2 * D, "w_down_rows"),          # W_down along d
    (I_, 64, "h_rows"),                  # h along the tokens
    (2 * I_, 2 * D, "w_gate_up_columns_backward"),  # W_gate_up (transposed) along d
    (2 * I_, 64, "dgu_rows_backward"),              # dG/dU along the tokens
])
def test_planted_nvfp4_axis_is_caught(monkeypatch, tail, rows, pin):
    _plant(monkeypatch, tail, rows)
    with pytest.raises(AssertionError):
        NV_PINS[pin]()
