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
    and with it on differs from fp64 by MXFP8 noise, not more;
  * the axis along which each GEMM operand is quantised, one pin per operand
    (power-of-two scale covariance: quantisation along K commutes with
    scaling the non-K index and not with scaling K), the token-axis blocking
    of the weight-gradient operands (blocks start at each expert's first row,
    zero-padded tail), and the router-weight gradient's dp = <dA, h> form;
    planted wrong axes and blockings show that each pin fails when it should.
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


# ----------------------------------------------------------------------------
# Where the MXFP8 mode quantises: one pin per quantised GEMM operand.
#
# MX quantisation along an axis commutes with scaling by a power of two that
# is constant along that axis (every block's shared exponent shifts, the E4M3
# codes stay), and does not commute with one that varies inside a block.  So
# for each GEMM, scaling an operand along its non-reduction index by 2^a must
# scale exactly the outputs that index reaches, and leave every other output
# bit for bit; quantising that operand along the wrong axis breaks this.  The
# weight-gradient operands along the token dimension are pinned in addition
# by inputs that are exactly representable only in blocks that start at each
# expert's first row.  Sizes: d = 64, I = 96 (2I = 192), so that every
# operand has a shape of its own; top-1 routing forced to 32 tokens per
# expert, so that p = 1, dl = 0 and a token-axis block is well defined.
# ----------------------------------------------------------------------------

D, I_ = 64, 96


def _k1_case(seed, T=64, E=2, gate_positive=False):
    """Float64 inputs with forced top-1 routing, T // E tokens per expert.
    ``gate_positive``: x in [1, 2) and W_gate in [1, 2), so every gate
    pre-activation g >= 64, where sigmoid(g) rounds to 1 in float64 and the
    SwiGLU is exactly h = g * u."""
    rng = np.random.default_rng(seed)
    x = rng.uniform(1, 2, (T, D)) if gate_positive else rng.standard_normal((T, D))
    wgu = rng.standard_normal((E, 2 * I_, D)) / np.sqrt(D)
    if gate_positive:
        wgu[:, :I_] = rng.uniform(1, 2, (E, I_, D))
    idx = rng.permutation(np.repeat(np.arange(E), T // E)).astype(np.int32)[:, None]
    return dict(x=x, w_router=rng.standard_normal((E, D)), w_gate_up=wgu,
                w_down=rng.standard_normal((E, D, I_)) / np.sqrt(I_),
                dy=rng.standard_normal((T, D)), routing=(idx, np.ones((T, 1))), k=1)


def _fwd(c):
    return oracle.moe_forward_ref(c["x"], c["w_router"], None, c["w_gate_up"], c["w_down"],
                                  c["k"], routing=c["routing"], keep=True, precision="mxfp8")


def _bwd(c, fwd):
    return oracle.moe_backward_ref(c["x"], c["w_router"], None, c["w_gate_up"], c["w_down"],
                                   c["k"], c["dy"], fwd=fwd)


def _assert_scaled(before, after, mask, factor, what):
    """after == before * factor where mask holds, == before elsewhere."""
    want = np.where(mask, before * factor, before)
    tol = 1e-12 * float(np.sqrt(np.mean(want * want)))
    np.testing.assert_allclose(after, want, rtol=1e-12, atol=tol, err_msg=what)


def _pin_token_scale_forward():
    """x_t -> 2^5 x_t: the gate/up GEMM (x along d) scales g_t, u_t by 2^5;
    h_t = g_t u_t by 2^10; the down GEMM (h along I) scales y_t by 2^10."""
    c = _k1_case(10, gate_positive=True)
    y0, f0 = _fwd(c)
    assert f0["G"].min() >= 64
    sel = np.arange(c["x"].shape[0]) % 3 == 0
    y1, f1 = _fwd(dict(c, x=np.where(sel[:, None], c["x"] * 32.0, c["x"])))
    rows = np.zeros(f0["G"].shape[0], dtype=bool)
    rows[f0["pos"][sel, 0]] = True
    _assert_scaled(f0["G"], f1["G"], rows[:, None], 32.0, "gate rows")
    _assert_scaled(f0["U"], f1["U"], rows[:, None], 32.0, "up rows")
    _assert_scaled(y0, y1, sel[:, None], 1024.0, "y rows")


def _pin_token_scale_backward():
    """dy_t -> 2^-7 dy_t: the down dgrad (dy along d) scales dA_t, so dG_t,
    dU_t; the gate/up dgrad (dG/dU along 2I) scales dx_t."""
    c = _k1_case(11)
    _, f = _fwd(c)
    g0 = _bwd(c, f)
    sel = np.arange(c["x"].shape[0]) % 4 == 1
    g1 = _bwd(dict(c, dy=np.where(sel[:, None], c["dy"] / 128.0, c["dy"])), f)
    _assert_scaled(g0["dx"], g1["dx"], sel[:, None], 1 / 128.0, "dx rows")
    _assert_scaled(g0["dp"], g1["dp"], sel[:, None], 1 / 128.0, "dp")


def _pin_gate_up_weight_rows():
    """W_gu row n -> 2^6 W_gu row n: the gate/up GEMM (W_gu along d) scales
    output column n of g (n < I) or of u (n >= I)."""
    c = _k1_case(12)
    _, f0 = _fwd(c)
    n = np.zeros(2 * I_, dtype=bool)
    n[[3, 40, 95, I_ + 1, I_ + 70]] = True
    w = c["w_gate_up"].copy()
    w[:, n] *= 64.0
    _, f1 = _fwd(dict(c, w_gate_up=w))
    _assert_scaled(f0["G"], f1["G"], n[None, :I_], 64.0, "gate columns")
    _assert_scaled(f0["U"], f1["U"], n[None, I_:], 64.0, "up columns")


def _pin_down_weight_rows():
    """W_down row j -> 2^-4 W_down row j: the down GEMM (W_down along I)
    scales output feature j of y."""
    c = _k1_case(13)
    y0, _ = _fwd(c)
    j = np.zeros(D, dtype=bool)
    j[[0, 9, 33, 63]] = True
    w = c["w_down"].copy()
    w[:, j] /= 16.0
    y1, _ = _fwd(dict(c, w_down=w))
    _assert_scaled(y0, y1, j[None, :], 1 / 16.0, "y columns")


def _pin_down_weight_columns_backward():
    """W_down column i -> 2^3 W_down column i, forward intermediates kept:
    the down dgrad (W_down along d) scales dA[:, i], so dG[:, i], dU[:, i] and
    rows i, I + i of dW_gate_up; dW_down does not read W_down."""
    c = _k1_case(14)
    _, f = _fwd(c)
    g0 = _bwd(c, f)
    i = np.zeros(I_, dtype=bool)
    i[[2, 31, 32, 80]] = True
    w = c["w_down"].copy()
    w[:, :, i] *= 8.0
    g1 = _bwd(dict(c, w_down=w), f)
    rows = np.concatenate([i, i])
    _assert_scaled(g0["dw_gate_up"], g1["dw_gate_up"], rows[None, :, None], 8.0, "dW_gu rows")
    _assert_scaled(g0["dw_down"], g1["dw_down"], False, 1.0, "dW_down")


def _pin_gate_up_weight_columns_backward():
    """W_gu column j -> 2^5 W_gu column j, forward intermediates kept: the
    gate/up dgrad (W_gu along 2I) scales feature j of dx."""
    c = _k1_case(15)
    _, f = _fwd(c)
    g0 = _bwd(c, f)
    j = np.zeros(D, dtype=bool)
    j[[1, 17, 32, 50]] = True
    w = c["w_gate_up"].copy()
    w[:, :, j] *= 32.0
    g1 = _bwd(dict(c, w_gate_up=w), f)
    _assert_scaled(g0["dx"], g1["dx"], j[None, :], 32.0, "dx columns")


def _pin_upstream_grad_columns_backward():
    """dy[:, j] -> 2^-6 dy[:, j], forward intermediates kept: the down-
    projection weight gradient (dy along the tokens) scales row j of every
    dW_down."""
    c = _k1_case(16)
    _, f = _fwd(c)
    g0 = _bwd(c, f)
    j = np.zeros(D, dtype=bool)
    j[[4, 5, 40]] = True
    g1 = _bwd(dict(c, dy=np.where(j[None, :], c["dy"] / 64.0, c["dy"])), f)
    _assert_scaled(g0["dw_down"], g1["dw_down"], j[None, :, None], 1 / 64.0, "dW_down rows")


def _pin_input_columns_backward():
    """x[:, j] -> 2^4 x[:, j] in the backward only (forward intermediates
    kept): the gate/up weight gradient (x along the tokens) scales column j
    of every dW_gate_up."""
    c = _k1_case(17)
    _, f = _fwd(c)
    g0 = _bwd(c, f)
    j = np.zeros(D, dtype=bool)
    j[[0, 31, 44]] = True
    g1 = _bwd(dict(c, x=np.where(j[None, :], c["x"] * 16.0, c["x"])), f)
    _assert_scaled(g0["dw_gate_up"], g1["dw_gate_up"], j[None, None, :], 16.0, "dW_gu columns")


TOP = 256.0 * (1 + np.arange(7) / 8)      # the E4M3 values in [256, 448]


def _on_grid(rng, shape):
    """Random E4M3 values of the top binade with random signs: a block of
    them times one power of two is quantised exactly (its maximum sits in
    [256, 448], so the shared exponent is that power)."""
    return rng.choice(TOP, size=shape) * rng.choice([-1.0, 1.0], size=shape)


def _pin_wgrad_token_blocks():
    """Token-axis blocks of the weight gradients start at each expert's first
    row and the segment's tail is zero-padded.  Experts get 33 and 40 rows;
    in the backward, the x and dy rows of a token carry 2^0 or 2^-20 by the
    parity of their 32-row block inside the expert's segment (constant along
    d, so the down dgrad's dy operand stays exact).  Blocked that way, both
    token-axis operands are on their MX grid, so from the same forward
    intermediates the MXFP8 weight gradients equal the fp64 ones; blocks
    placed anywhere else put a 2^0 row and a 2^-20 row together and flush the
    small one to zero."""
    rng = np.random.default_rng(18)
    T, E = 73, 2
    idx = rng.permutation(np.r_[np.zeros(33, np.int32), np.ones(40, np.int32)])[:, None]
    seg = np.zeros(T, dtype=np.int64)
    for e in range(E):
        toks = np.nonzero(idx[:, 0] == e)[0]
        seg[toks] = np.arange(len(toks))
    scale = np.where((seg // 32) % 2 == 1, 2.0 ** -20, 1.0)[:, None]
    c = dict(x=rng.standard_normal((T, D)), dy=_on_grid(rng, (T, D)) * scale / 256,
             w_router=rng.standard_normal((E, D)),
             w_gate_up=rng.standard_normal((E, 2 * I_, D)) / np.sqrt(D),
             w_down=_on_grid(rng, (E, D, I_)) * 2.0 ** -12,
             routing=(idx, np.ones((T, 1))), k=1)
    _, f = _fwd(c)
    c["x"] = _on_grid(rng, (T, D)) * scale / 256
    # the fixture discriminates: 32-row blocks of the whole expert-ordered
    # matrix (not restarted per expert) are not exact
    order = np.argsort(idx[:, 0], kind="stable")
    flat = c["dy"][order]
    padded = np.concatenate([flat, np.zeros((96 - T, D))])
    assert not np.array_equal(mx_ref.mx_fake(padded, 0)[:T], flat)
    gm = _bwd(c, f)
    g64 = oracle.moe_backward_ref(c["x"], c["w_router"], None, c["w_gate_up"], c["w_down"], 1,
                                  c["dy"], fwd=f, precision="fp64")
    for n in ("dw_down", "dw_gate_up"):
        _assert_scaled(g64[n], gm[n], False, 1.0, n)


def _pin_router_gradient_form():
    """dp = <dA, h>: with x, dy, W_gate_up and W_down exactly representable
    along d (one power of two per row of x, dy, W_gate_up and per column of
    W_down), the down dgrad dA = dy W_down is exact, so <dA, h> equals the
    fp64 mode's <dy, O> with O = h W_down^T unquantised, while the MXFP8
    expert output O (h and W_down along I, neither exact) does not: dp, dl
    and dW_router of the MXFP8 mode equal the fp64 ones."""
    rng = np.random.default_rng(19)
    T, E, k = 40, 4, 2
    rs = lambda n: 2.0 ** rng.integers(-12, 0, size=n)   # noqa: E731
    x = _on_grid(rng, (T, D)) * rs(T)[:, None] / 256
    dy = _on_grid(rng, (T, D)) * rs(T)[:, None] / 256
    wgu = _on_grid(rng, (E, 2 * I_, D)) * rs(E * 2 * I_).reshape(E, 2 * I_, 1) / 2048
    wd = _on_grid(rng, (E, D, I_)) * rs(E * I_).reshape(E, 1, I_) / 2048
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    p = rng.dirichlet(np.ones(k), size=T)
    c = dict(x=x, dy=dy, w_router=rng.standard_normal((E, D)), w_gate_up=wgu, w_down=wd,
             routing=(idx, p), k=k)
    ym, fm = _fwd(c)
    gm = _bwd(c, fm)
    y64, f64 = oracle.moe_forward_ref(x, c["w_router"], None, wgu, wd, k, routing=(idx, p),
                                      keep=True)
    g64 = oracle.moe_backward_ref(x, c["w_router"], None, wgu, wd, k, dy, fwd=f64)
    assert np.array_equal(fm["H"], f64["H"])
    # the expert output itself is not exact, so <dy, O_mxfp8> would differ
    assert np.abs(fm["O"] - f64["O"]).max() > 1e-3 * np.sqrt(np.mean(f64["O"] ** 2))
    for n in ("dp", "dl", "dw_router"):
        _assert_scaled(g64[n], gm[n], False, 1.0, n)


MX_PINS = {
    "token_scale_forward": _pin_token_scale_forward,
    "token_scale_backward": _pin_token_scale_backward,
    "gate_up_weight_rows": _pin_gate_up_weight_rows,
    "down_weight_rows": _pin_down_weight_rows,
    "down_weight_columns_backward": _pin_down_weight_columns_backward,
    "gate_up_weight_columns_backward": _pin_gate_up_weight_columns_backward,
    "upstream_grad_columns_backward": _pin_upstream_grad_columns_backward,
    "input_columns_backward": _pin_input_columns_backward,
    "wgrad_token_blocks": _pin_wgrad_token_blocks,
    "router_gradient_form": _pin_router_gradient_form,
}


@pytest.mark.parametrize("name", sorted(MX_PINS))
def test_mxfp8_mode_quantisation_axes(name):
    MX_PINS[name]()


# planted mistakes: a wrong quantisation axis in one GEMM operand, identified
# by the operand's shape, the axis and the pass (forward or backward)
def _plant_axis(monkeypatch, phase, shape, wrong_from, wrong_to):
    real_fake = moe_ref.mx_fake
    real_ffn = moe_ref.expert_ffn
    state = {"phase": "bwd"}

    def fake(a, axis=-1):
        a = np.asarray(a)
        if (state["phase"] == phase and a.shape[1:] == shape[1:]
                and (shape[0] is None or a.shape[0] == shape[0])
                and axis % a.ndim == wrong_from % a.ndim):
            axis = wrong_to
        return real_fake(a, axis)

    def ffn(*args, **kw):
        state["phase"] = "fwd"
        try:
            return real_ffn(*args, **kw)
        finally:
            state["phase"] = "bwd"
    monkeypatch.setattr(moe_ref, "mx_fake", fake)
    monkeypatch.setattr(moe_ref, "expert_ffn", ffn)


PLANTED_AXES = [
    # (pass, operand shape, correct axis, wrong axis, pin that must fail)
    ("fwd", (None, D), -1, 0, "token_scale_forward"),            # x rows along tokens
    ("fwd", (2 * I_, D), -1, 0, "gate_up_weight_rows"),          # W_gate_up along 2I
    ("fwd", (None, I_), -1, 0, "token_scale_forward"),           # h along tokens
    ("fwd", (D, I_), -1, 0, "down_weight_rows"),                 # W_down along d
    ("bwd", (None, D), -1, 0, "token_scale_backward"),           # dy rows along tokens
    ("bwd", (D, I_), 0, -1, "down_weight_columns_backward"),     # W_down along I
    ("bwd", (None, 2 * I_), -1, 0, "token_scale_backward"),      # dG/dU along tokens
    ("bwd", (2 * I_, D), 0, -1, "gate_up_weight_columns_backward"),  # W_gate_up along d
]


@pytest.mark.parametrize("plant", PLANTED_AXES, ids=lambda p: f"{p[0]}-{p[1]}-{p[4]}")
def test_planted_wrong_quantisation_axis_is_caught(monkeypatch, plant):
    phase, shape, right, wrong, pin = plant
    _plant_axis(monkeypatch, phase, shape, right, wrong)
    with pytest.raises(AssertionError):
        MX_PINS[pin]()


def _rows_along_d(a):
    return mx_ref.mx_fake(a, -1)


def _rows_front_padded(a):
    n = a.shape[0]
    pad = (-n) % 32
    a = np.concatenate([np.zeros((pad,) + a.shape[1:]), a], axis=0)
    return mx_ref.mx_fake(a, 0)[pad:]


@pytest.mark.parametrize("wrong,pins", [
    (_rows_along_d, ["upstream_grad_columns_backward", "input_columns_backward"]),
    (_rows_front_padded, ["wgrad_token_blocks"]),
], ids=["along-d", "front-padded"])
def test_planted_wgrad_token_blocking_is_caught(monkeypatch, wrong, pins):
    monkeypatch.setattr(moe_ref, "_mx_rows", wrong)
    for pin in pins:
        with pytest.raises(AssertionError):
            MX_PINS[pin]()
