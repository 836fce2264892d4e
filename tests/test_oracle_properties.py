"""Randomised small-shape properties of the fp64 oracle (Hypothesis draws the
shape, the seed and whether a router bias is present).  For every draw:

  * routing: each token's experts are its k largest float32 logits, larger
    first, exact ties to the lower index (checked by sorting, not by the
    oracle's selection), and the weights are positive and sum to one;
  * dispatch: a stable bijection of the T*k (token, slot) pairs onto rows,
    grouped by expert and ascending by token inside each expert, with the
    counts of a brute-force count;
  * forward: equal to the dense formulation (every expert applied to every
    token, masked by the routing; no dispatch, no permutation);
  * backward: the analytic gradients against a central finite difference of
    the loss along one random direction in all four inputs at once, unless
    the routing changes inside the step.

The fixed-shape pins (test_oracle_pins.py) hold the worked example and the
planted mistakes; these widen the same checks to shapes nobody picked.
"""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from routing_dispatch_grouped_router_gb300 import inputs as gen  # noqa: E402
from test_oracle_pins import _dense_forward, _loss  # noqa: E402


@st.composite
def layer_cases(draw):
    E = draw(st.integers(1, 8))
    k = draw(st.integers(1, min(E, 4)))
    shape = gen.Shape(T=draw(st.integers(1, 12)), d=draw(st.sampled_from([4, 8, 12, 16])), E=E,
                      I=draw(st.sampled_from([2, 4, 6, 8])), k=k)
    seed = draw(st.integers(0, 2**16 - 1))
    biased = draw(st.booleans())
    return shape, seed, biased


def _case(shape, seed, biased):
    inp = gen.make_inputs(shape, seed)
    bias = None
    if biased:
        bias = np.random.default_rng(seed + 1).normal(0.0, 0.5, shape.E).astype(np.float32)
    return inp, bias


def _f64(bits):
    return gen.bf16_bits_to_f32(bits).astype(np.float64)


SETTINGS = settings(max_examples=30, deadline=None, derandomize=True)


@SETTINGS
@given(layer_cases())
def test_routing_is_the_sorted_top_k(case):
    shape, seed, biased = case
    inp, bias = _case(shape, seed, biased)
    idx, w, logits, _, _ = oracle.route_ref(inp["x"], inp["w_router"], bias, shape.k)
    L = _f64(inp["x"]) @ _f64(inp["w_router"]).T
    if bias is not None:
        L = L + bias.astype(np.float64)
    np.testing.assert_allclose(logits, L, rtol=0, atol=1e-12)
    for t in range(shape.T):
        l32 = L[t].astype(np.float32)
        assert list(idx[t]) == sorted(range(shape.E), key=lambda e: (-l32[e], e))[:shape.k]
    assert (w > 0).all()
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)


@SETTINGS
@given(layer_cases())
def test_dispatch_is_a_stable_bijection(case):
    shape, seed, biased = case
    inp, bias = _case(shape, seed, biased)
    idx = oracle.route_ref(inp["x"], inp["w_router"], bias, shape.k)[0]
    counts, offsets, pos, tok = oracle.dispatch_ref(idx, shape.E)
    T, k, E = shape.T, shape.k, shape.E
    brute = [sum(1 for t in range(T) for s in range(k) if idx[t, s] == e) for e in range(E)]
    assert list(counts) == brute
    assert offsets[0] == 0 and list(np.diff(offsets)) == brute
    assert sorted(pos.ravel().tolist()) == list(range(T * k))
    for t in range(T):
        for s in range(k):
            r = pos[t, s]
            assert tok[r] == t and offsets[idx[t, s]] <= r < offsets[idx[t, s] + 1]
    for e in range(E):
        assert (np.diff(tok[offsets[e]:offsets[e + 1]]) > 0).all()


@SETTINGS
@given(layer_cases())
def test_forward_is_the_dense_layer(case):
    shape, seed, biased = case
    inp, bias = _case(shape, seed, biased)
    y = oracle.moe_forward_ref(inp["x"], inp["w_router"], bias, inp["w_gate_up"], inp["w_down"],
                               shape.k)
    np.testing.assert_allclose(y, _dense_forward(inp, shape.k, bias), rtol=1e-12, atol=1e-12)


@SETTINGS
@given(layer_cases())
def test_backward_is_the_directional_derivative(case):
    shape, seed, biased = case
    inp, bias = _case(shape, seed, biased)
    args = [_f64(inp[n]) for n in ("x", "w_router", "w_gate_up", "w_down")]
    dY = _f64(inp["dy"])
    g = oracle.moe_backward_ref(*args[:2], bias, *args[2:], shape.k, dY)
    grads = [g[n] for n in ("dx", "dw_router", "dw_gate_up", "dw_down")]
    rng = np.random.default_rng(seed)
    v = [rng.normal(size=a.shape) for a in args]
    h = 1e-6
    L0, idx0 = _loss(*args, shape.k, dY, bias)
    vals = []
    for sgn in (+1, -1):
        moved = [a + sgn * h * dv for a, dv in zip(args, v)]
        L, idx = _loss(*moved, shape.k, dY, bias)
        hypothesis.assume(np.array_equal(idx, idx0))  # no routing change inside the step
        vals.append(L)
    fd = (vals[0] - vals[1]) / (2 * h)
    an = sum(float((gr * dv).sum()) for gr, dv in zip(grads, v))
    assert abs(fd - an) <= 1e-6 * (1.0 + abs(an)), (fd, an)
