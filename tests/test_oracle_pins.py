"""Pins for the fp64 oracle: each checks it against something other than itself.

  * routing against brute force (python sort of every token's logits), the
    sum-to-one property, and the k = E special case (the full softmax);
  * dispatch against a brute-force nested-loop count, bijectivity and the
    k = E block transpose;
  * the forward against a dense formulation that applies every expert to
    every token and masks by the routing (no dispatch, no permutation), the
    E = 1 plain SwiGLU FFN, exact homogeneity in W_down and token
    permutation equivariance;
  * a worked example small enough to evaluate in closed form;
  * the backward against central finite differences in float64.
Planted-mistake tests at the end show that these pins catch plausible bugs.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import moe_ref
from routing_dispatch_grouped_router_gb300 import inputs as gen


def _tiny(seed=0, T=24, d=16, E=6, I=8, k=2):
    sh = gen.Shape(T=T, d=d, E=E, I=I, k=k)
    return sh, gen.make_inputs(sh, seed)


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------

def _brute_logits(x, wr):
    X = gen.bf16_bits_to_f32(x).astype(np.float64)
    W = gen.bf16_bits_to_f32(wr).astype(np.float64)
    T, E = X.shape[0], W.shape[0]
    out = np.zeros((T, E))
    for t in range(T):
        for e in range(E):
            out[t, e] = math.fsum(float(a) * float(b) for a, b in zip(X[t], W[e]))
    return out


@pytest.mark.parametrize("k", [1, 2, 3, 6])
def test_routing_matches_brute_force(k):
    sh, inp = _tiny(seed=3, k=k)
    idx, w, logits, flagged, inner = oracle.route_ref(inp["x"], inp["w_router"], None, k)
    L = _brute_logits(inp["x"], inp["w_router"])
    np.testing.assert_allclose(logits, L, rtol=0, atol=1e-12)
    for t in range(sh.T):
        l32 = [np.float32(v) for v in L[t]]
        order = sorted(range(sh.E), key=lambda e: (-l32[e], e))[:k]
        assert list(idx[t]) == order
        chosen = [L[t, e] for e in order]
        m = max(chosen)
        den = sum(math.exp(c - m) for c in chosen)
        for s in range(k):
            assert abs(w[t, s] - math.exp(chosen[s] - m) / den) < 1e-14
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (w > 0).all() and (w <= 1).all()
    # slots are in descending-logit order
    sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    assert (np.diff(sel, axis=1) <= 0).all()


def test_routing_k_equals_E_is_full_softmax():
    sh, inp = _tiny(seed=5, E=5, k=5)
    idx, w, logits, flagged, _ = oracle.route_ref(inp["x"], inp["w_router"], None, 5)
    full = scipy.special.softmax(logits, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx.astype(np.int64), axis=1),
                               rtol=1e-13, atol=0)
    assert not flagged.any()


def test_routing_bias_shifts_logits():
    sh, inp = _tiny(seed=2, E=4, k=1)
    bias = np.array([0.0, 0.0, 100.0, 0.0], dtype=np.float32)
    idx, w, logits, _, _ = oracle.route_ref(inp["x"], inp["w_router"], bias, 1)
    assert (idx[:, 0] == 2).all()
    np.testing.assert_allclose(w, 1.0)


def test_exact_tie_goes_to_lower_index_and_is_flagged():
    # experts 1 and 3 have identical router rows: their logits tie exactly
    sh, inp = _tiny(seed=7, E=4, k=1)
    wr = inp["w_router"].copy()
    wr[3] = wr[1]
    bias = np.array([-50.0, 0.0, -50.0, 0.0], dtype=np.float32)
    idx, w, logits, flagged, _ = oracle.route_ref(inp["x"], wr, bias, 1)
    assert (idx[:, 0] == 1).all()
    assert flagged.all()
    idx2, _, _, flagged2, inner2 = oracle.route_ref(inp["x"], wr, bias, 2)
    assert (idx2 == np.array([1, 3])).all()
    assert inner2.all() and not flagged2.any()


# ----------------------------------------------------------------------------
# dispatch
# ----------------------------------------------------------------------------

def _brute_dispatch(idx, E):
    T, k = idx.shape
    counts = [0] * E
    for t in range(T):
        for s in range(k):
            counts[idx[t, s]] += 1
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    pos = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        for s in range(k):
            e = idx[t, s]
            earlier = sum(1 for tt in range(t) if e in list(idx[tt]))
            pos[t, s] = offsets[e] + earlier
    return counts, offsets, pos


@pytest.mark.parametrize("seed,T,E,k", [(0, 40, 5, 2), (1, 33, 8, 3), (2, 17, 4, 4), (3, 1, 3, 2)])
def test_dispatch_matches_brute_force(seed, T, E, k):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, pos, tok = oracle.dispatch_ref(idx, E)
    bc, bo, bp = _brute_dispatch(idx, E)
    assert list(counts) == bc and list(offsets) == bo
    assert (pos == bp).all()
    assert counts.sum() == T * k
    # bijection, and dropless: every (t, s) lands exactly once
    assert sorted(pos.ravel().tolist()) == list(range(T * k))
    for t in range(T):
        for s in range(k):
            assert tok[pos[t, s]] == t
    # rows of one expert are ascending by token
    for e in range(E):
        seg = tok[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()


def test_dispatch_k_equals_E_is_block_transpose():
    T, E = 7, 4
    idx = np.array([np.roll(np.arange(E), t) for t in range(T)], dtype=np.int32)
    counts, offsets, pos, tok = oracle.dispatch_ref(idx, E)
    assert (counts == T).all()
    for t in range(T):
        for s in range(E):
            assert pos[t, s] == idx[t, s] * T + t
    assert (tok == np.tile(np.arange(T), E)).all()


def test_dispatch_empty_expert():
    idx = np.array([[0, 2], [2, 0], [0, 2]], dtype=np.int32)
    counts, offsets, pos, tok = oracle.dispatch_ref(idx, 4)
    assert list(counts) == [3, 0, 3, 0]
    assert list(offsets) == [0, 3, 3, 6, 6]


# ----------------------------------------------------------------------------
# forward
# ----------------------------------------------------------------------------

def _dense_forward(inp, k, bias=None):
    """Every expert on every token, masked by the routing: no dispatch."""
    X = gen.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    Wr = gen.bf16_bits_to_f32(inp["w_router"]).astype(np.float64)
    Wgu = gen.bf16_bits_to_f32(inp["w_gate_up"]).astype(np.float64)
    Wd = gen.bf16_bits_to_f32(inp["w_down"]).astype(np.float64)
    E, I2, d = Wgu.shape
    I = I2 // 2
    T = X.shape[0]
    L = X @ Wr.T
    if bias is not None:
        L = L + bias.astype(np.float64)
    y = np.zeros((T, d))
    for t in range(T):
        l32 = L[t].astype(np.float32)
        chosen = sorted(range(E), key=lambda e: (-l32[e], e))[:k]
        z = np.array([L[t, e] for e in chosen])
        pr = np.exp(z - z.max()); pr /= pr.sum()
        for e in range(E):
            gate = Wgu[e, :I] @ X[t]
            up = Wgu[e, I:] @ X[t]
            h = gate / (1.0 + np.exp(-gate)) * up
            out = Wd[e] @ h
            if e in chosen:
                y[t] += pr[chosen.index(e)] * out
    return y


@pytest.mark.parametrize("seed,k", [(0, 1), (1, 2), (2, 3)])
def test_forward_matches_dense(seed, k):
    sh, inp = _tiny(seed=seed, k=k)
    y = oracle.moe_forward_ref(inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], k)
    np.testing.assert_allclose(y, _dense_forward(inp, k), rtol=1e-12, atol=1e-12)


def test_forward_with_bias_matches_dense():
    sh, inp = _tiny(seed=4, k=2)
    bias = np.linspace(-1, 1, sh.E).astype(np.float32)
    y = oracle.moe_forward_ref(inp["x"], inp["w_router"], bias, inp["w_gate_up"], inp["w_down"], 2)
    np.testing.assert_allclose(y, _dense_forward(inp, 2, bias), rtol=1e-12, atol=1e-12)


def test_single_expert_is_plain_swiglu_ffn():
    sh, inp = _tiny(seed=9, E=1, k=1)
    y = oracle.moe_forward_ref(inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], 1)
    X = gen.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    W = gen.bf16_bits_to_f32(inp["w_gate_up"][0]).astype(np.float64)
    Wd = gen.bf16_bits_to_f32(inp["w_down"][0]).astype(np.float64)
    g = X @ W[:sh.I].T
    u = X @ W[sh.I:].T
    ref = (g * scipy.special.expit(g) * u) @ Wd.T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_forward_homogeneous_in_w_down():
    sh, inp = _tiny(seed=11, k=2)
    y1 = oracle.moe_forward_ref(inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], 2)
    wd2 = 2.0 * gen.bf16_bits_to_f32(inp["w_down"]).astype(np.float64)
    y2 = oracle.moe_forward_ref(inp["x"], inp["w_router"], None, inp["w_gate_up"], wd2, 2)
    assert np.array_equal(y2, 2.0 * y1)


def test_forward_token_permutation_equivariant():
    sh, inp = _tiny(seed=12, k=2)
    perm = np.random.default_rng(0).permutation(sh.T)
    y = oracle.moe_forward_ref(inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], 2)
    yp = oracle.moe_forward_ref(inp["x"][perm], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], 2)
    np.testing.assert_allclose(yp, y[perm], rtol=1e-13, atol=1e-13)


def test_worked_example_closed_form():
    """One token, three experts, I = 1: every quantity has a closed form.

    logits = (2, 1, 0) -> experts {0, 1}, p0 = 1/(1+e^-1), p1 = 1/(1+e).
    Expert e: gate = a_e x_0, up = b_e x_0, out = c_e silu(gate) up on dim 0.
    """
    one = lambda v: gen.f32_to_bf16_bits(np.asarray(v, dtype=np.float32))
    x = one([[1.0, 0.0]])
    wr = one([[2.0, 0.0], [1.0, 0.0], [0.0, 0.0]])
    a, b, c = [1.0, -0.5, 3.0], [2.0, 4.0, 1.0], [0.5, 0.25, 8.0]
    wgu = one([[[a[e], 0.0], [b[e], 0.0]] for e in range(3)])
    wd = one([[[c[e]], [0.0]] for e in range(3)])
    y, st = oracle.moe_forward_ref(x, wr, None, wgu, wd, 2, keep=True)
    p0 = 1.0 / (1.0 + math.exp(-1.0))
    p1 = 1.0 / (1.0 + math.exp(1.0))
    sl = lambda z: z / (1.0 + math.exp(-z))
    expect = p0 * c[0] * sl(a[0]) * b[0] + p1 * c[1] * sl(a[1]) * b[1]
    assert list(st["idx"][0]) == [0, 1]
    assert abs(st["p"][0, 0] - p0) < 1e-15 and abs(st["p"][0, 1] - p1) < 1e-15
    assert abs(y[0, 0] - expect) < 1e-14 and y[0, 1] == 0.0
    # backward with dy = (1, 0): dL/dp_s = out_s,  dL/dl_j = p_j (out_j - sum p out)
    dy = one([[1.0, 0.0]])
    g = oracle.moe_backward_ref(x, wr, None, wgu, wd, 2, dy)
    o0, o1 = c[0] * sl(a[0]) * b[0], c[1] * sl(a[1]) * b[1]
    mean = p0 * o0 + p1 * o1
    assert abs(g["dp"][0, 0] - o0) < 1e-14 and abs(g["dp"][0, 1] - o1) < 1e-14
    dl0, dl1 = p0 * (o0 - mean), p1 * (o1 - mean)
    np.testing.assert_allclose(g["dw_router"][:, 0], [dl0, dl1, 0.0], atol=1e-14)
    # dW_down[e][0,0] = p_e * dy_0 * h_e
    np.testing.assert_allclose(g["dw_down"][0, 0, 0], p0 * sl(a[0]) * b[0], atol=1e-14)
    np.testing.assert_allclose(g["dw_down"][2], 0.0)


# ----------------------------------------------------------------------------
# backward: central finite differences
# ----------------------------------------------------------------------------

def _loss(xf, wrf, wguf, wdf, k, dyf, bias=None):
    y, st = oracle.moe_forward_ref(xf, wrf, bias, wguf, wdf, k, keep=True)
    return float((y * dyf).sum()), st["idx"]


def _fd_check(inp, k, n_coords=12, seed=0, h=1e-6, tol=1e-6, bias=None):
    X = gen.bf16_bits_to_f32(inp["x"]).astype(np.float64)
    Wr = gen.bf16_bits_to_f32(inp["w_router"]).astype(np.float64)
    Wgu = gen.bf16_bits_to_f32(inp["w_gate_up"]).astype(np.float64)
    Wd = gen.bf16_bits_to_f32(inp["w_down"]).astype(np.float64)
    dY = gen.bf16_bits_to_f32(inp["dy"]).astype(np.float64)
    g = oracle.moe_backward_ref(X, Wr, bias, Wgu, Wd, k, dY)
    _, idx0 = _loss(X, Wr, Wgu, Wd, k, dY, bias)
    rng = np.random.default_rng(seed)
    worst = 0.0
    checked = 0
    tensors = dict(x=(X, "dx"), w_router=(Wr, "dw_router"), w_gate_up=(Wgu, "dw_gate_up"),
                   w_down=(Wd, "dw_down"))
    for name, (arr, gname) in tensors.items():
        for _ in range(n_coords):
            c = tuple(int(rng.integers(0, n)) for n in arr.shape)
            args = dict(x=X, w_router=Wr, w_gate_up=Wgu, w_down=Wd)
            vals = []
            same = True
            for sgn in (+1, -1):
                a2 = arr.copy()
                a2[c] += sgn * h
                args[name] = a2
                L, idx = _loss(args["x"], args["w_router"], args["w_gate_up"], args["w_down"], k, dY, bias)
                same &= bool(np.array_equal(idx, idx0))
                vals.append(L)
            if not same:
                continue
            fd = (vals[0] - vals[1]) / (2 * h)
            an = g[gname][c]
            err = abs(fd - an) / (1.0 + abs(an))
            worst = max(worst, err)
            checked += 1
    return worst, checked


@pytest.mark.parametrize("seed,k", [(0, 2), (1, 1), (2, 3)])
def test_backward_matches_finite_differences(seed, k):
    sh, inp = _tiny(seed=seed, T=8, d=16, E=4, I=8, k=k)
    worst, checked = _fd_check(inp, k, seed=seed)
    assert checked >= 40
    assert worst < 1e-6, worst


def test_backward_with_bias_matches_finite_differences():
    sh, inp = _tiny(seed=6, T=8, d=16, E=4, I=8, k=2)
    worst, checked = _fd_check(inp, 2, seed=6, bias=np.array([0.3, -0.2, 0.0, 0.1], dtype=np.float32))
    assert checked >= 40 and worst < 1e-6, worst


def test_backward_zero_row_expert_has_zero_grads():
    sh, inp = _tiny(seed=8, T=8, d=16, E=4, I=8, k=1)
    bias = np.array([0.0, -1e3, 0.0, 0.0], dtype=np.float32)
    g = oracle.moe_backward_ref(inp["x"], inp["w_router"], bias, inp["w_gate_up"], inp["w_down"], 1, inp["dy"])
    assert (g["dw_gate_up"][1] == 0).all() and (g["dw_down"][1] == 0).all()
    assert (g["dw_router"][1] == 0).all()


# ----------------------------------------------------------------------------
# planted mistakes: the pins above must catch each of them
# ----------------------------------------------------------------------------

def test_planted_silu_grad_mistake_is_caught(monkeypatch):
    sh, inp = _tiny(seed=0, T=8, d=16, E=4, I=8, k=2)
    monkeypatch.setattr(moe_ref, "silu_grad", lambda z: 1.0 / (1.0 + np.exp(-z)))  # dropped term
    worst, _ = _fd_check(inp, 2, seed=0)
    assert worst > 1e-3


def test_planted_router_sign_mistake_is_caught(monkeypatch):
    sh, inp = _tiny(seed=1, T=8, d=16, E=4, I=8, k=2)
    orig = moe_ref.moe_backward_ref

    def wrong(*a, **kw):
        g = orig(*a, **kw)
        g["dw_router"] = -g["dw_router"]
        return g
    monkeypatch.setattr(oracle, "moe_backward_ref", wrong)
    worst, _ = _fd_check(inp, 2, seed=1)
    assert worst > 1e-3


def test_planted_unstable_dispatch_is_caught(monkeypatch):
    sh, inp = _tiny(seed=2, k=2)
    orig = moe_ref.dispatch_ref

    def wrong(idx, E):
        c, o, pos, tok = orig(idx, E)
        # swap two slots' rows: a transposition bug in the permutation
        pos = pos.copy()
        pos[0, 0], pos[0, 1] = pos[0, 1], pos[0, 0]
        return c, o, pos, tok
    monkeypatch.setattr(moe_ref, "dispatch_ref", wrong)
    y = oracle.moe_forward_ref(inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], 2)
    assert np.abs(y - _dense_forward(inp, 2)).max() > 1e-3


def test_planted_gate_up_swap_is_caught(monkeypatch):
    sh, inp = _tiny(seed=3, k=2)

    def wrong(X, wgu, wd, rnd=None, mx=False):
        W = moe_ref.widen(wgu)
        I = W.shape[0] // 2
        U = X @ W[:I].T
        G = X @ W[I:].T
        H = moe_ref.silu(G) * U
        return G, U, H, H @ moe_ref.widen(wd).T
    monkeypatch.setattr(moe_ref, "expert_ffn", wrong)
    y = oracle.moe_forward_ref(inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], 2)
    assert np.abs(y - _dense_forward(inp, 2)).max() > 1e-3


# ----------------------------------------------------------------------------
# BF16-operand mode
# ----------------------------------------------------------------------------

def test_bf16_round_matches_bit_level_rounding():
    """The oracle's frexp-based rounding against the generator's integer
    bit-pattern rounding (two independent implementations), including exact
    ties, subnormals and the largest finite values."""
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(20000).astype(np.float32),
            (rng.standard_normal(2000) * 1e-39).astype(np.float32),
            np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.3895313892515355e38,
                      2.0 ** -126, 2.0 ** -133, 0.0, -0.0, 1e-45], dtype=np.float32)]
    ties = (np.arange(1, 2000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    vals.append(ties)
    for v in vals:
        want = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(v)).astype(np.float64)
        got = oracle.bf16_round(v.astype(np.float64))
        assert np.array_equal(got, want)


def test_bf16_mode_is_fp64_mode_plus_operand_rounding(monkeypatch):
    sh, inp = _tiny(seed=1, k=2)
    args = (inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], 2)
    y64, f64 = oracle.moe_forward_ref(*args, keep=True)
    g64 = oracle.moe_backward_ref(*args, inp["dy"], fwd=f64)
    monkeypatch.setattr(moe_ref, "bf16_round", lambda a: a)
    yb, fb = oracle.moe_forward_ref(*args, keep=True, precision="bf16")
    gb = oracle.moe_backward_ref(*args, inp["dy"], fwd=fb)
    assert np.array_equal(y64, yb)
    for n in ("dx", "dw_router", "dw_gate_up", "dw_down"):
        assert np.array_equal(g64[n], gb[n])


def test_bf16_mode_operands_are_nearest_bf16():
    sh, inp = _tiny(seed=2, k=2)
    args = (inp["x"], inp["w_router"], None, inp["w_gate_up"], inp["w_down"], 2)
    y64, f64 = oracle.moe_forward_ref(*args, keep=True)
    yb, fb = oracle.moe_forward_ref(*args, keep=True, precision="bf16")
    G, U, H = fb["G"], fb["U"], fb["H"]
    for t in (G, U, H):
        assert np.array_equal(t, oracle.bf16_round(t))
    # within half an ulp of what the definition gives before rounding
    def half_ulp(v):
        e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
        return 2.0 ** (e - 8)
    assert (np.abs(G - f64["G"]) <= half_ulp(f64["G"])).all()
    hpre = oracle.silu(G) * U
    assert (np.abs(H - hpre) <= half_ulp(hpre)).all()
    # bf16 operands change the result by bf16 noise, not more
    rms = np.sqrt(np.mean(y64 ** 2))
    assert 0 < np.abs(yb - y64).max() / rms < 0.05
