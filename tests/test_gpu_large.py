"""Parity at the full sizes of the large (T=8192, d=7168, E=384, I=2048, k=8)
and imbalanced (T=16384, d=4096, E=128, I=1536, k=8, Zipf-biased router)
workloads, in the launch configuration the benchmark uses.

The full fp64 oracle is too slow at these sizes, so the comparison is on
outputs the oracle can compute one by one:
  * routing of every token (the router is cheap), and the dispatch plan;
  * y and dx of sampled tokens: each token's outputs depend on that token
    only, so the oracle runs on the sampled tokens alone;
  * dW_gate_up and dW_down of sampled experts: an expert's weight gradients
    depend only on its own rows, so the oracle runs on the tokens routed to
    it with the routing restricted to that expert;
  * dW_router rows of sampled experts (imbalanced workload): row e depends on
    the tokens routed to e, run through the oracle with their full routing.
Bar: max|diff| <= 2e-2 * rms(oracle) per compared tensor."""
import numpy as np
import pytest
import torch

import oracle
from routing_dispatch_grouped_router_gb300 import inputs as gen

import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routing_dispatch_grouped_router_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _sub(inp, toks):
    return dict(inp, x=inp["x"][toks], dy=inp["dy"][toks])


@pytest.mark.parametrize("name", ["imbalanced", "large"])
def test_full_size_sampled_parity(name):
    shape = gen.workload_shape(name)
    inp = gen.workload_inputs(name, seed=0, parallel=True)
    gpu = _gpu.run_gpu(shape, inp)
    assert gpu["status"] == 0
    bias = inp["bias"]
    k, E = shape.k, shape.E

    # routing of every token, and the plan
    idx, p, _, flagged, inner = oracle.route_ref(inp["x"], inp["w_router"], bias, k)
    decided = _gpu.check_routing(gpu["topk_idx"], gpu["topk_w"], idx, p, flagged, inner)
    counts, offsets, pos, tok = oracle.dispatch_ref(idx, E)
    if decided.all():
        assert np.array_equal(gpu["counts"], counts)
        assert np.array_equal(gpu["offsets"], offsets)
        assert np.array_equal(gpu["pos"], pos)
        assert np.array_equal(gpu["token_of_row"], tok)
    _gpu.check_dispatch_valid(gpu["topk_idx"], gpu["counts"], gpu["offsets"], gpu["pos"],
                              gpu["token_of_row"], E)
    if name == "imbalanced":
        ratio = counts.max() / (shape.R / E)
        assert 7.6 <= ratio <= 8.4, ratio

    rng = np.random.default_rng(1234)
    errs = {}

    # sampled tokens: y and dx
    toks = np.sort(rng.choice(np.nonzero(decided)[0], size=6, replace=False))
    sub = _sub(inp, toks)
    y_ref, fwd = oracle.moe_forward_ref(sub["x"], inp["w_router"], bias, inp["w_gate_up"],
                                        inp["w_down"], k, keep=True)
    g = oracle.moe_backward_ref(sub["x"], inp["w_router"], bias, inp["w_gate_up"],
                                inp["w_down"], k, sub["dy"], fwd=fwd, grad_experts=[])
    errs["y"] = _gpu.rel_err(_gpu.host64(gpu["y"][toks]), y_ref)
    errs["dx"] = _gpu.rel_err(_gpu.host64(gpu["dx"][toks]), g["dx"])

    # sampled experts: the hottest one and a random non-empty one, away from
    # undecided tokens
    touched = np.zeros(E, dtype=bool)
    for t in np.nonzero(~decided)[0]:
        touched[idx[t]] = True
        touched[gpu["topk_idx"][t]] = True
    ok = (counts > 0) & ~touched
    hot = int(np.argmax(np.where(ok, counts, -1)))
    other = int(rng.choice(np.nonzero(ok & (np.arange(E) != hot))[0]))
    for e in (hot, other):
        rows = np.nonzero((idx == e).any(axis=1))[0]
        slot = np.argmax(idx[rows] == e, axis=1)
        pe = p[rows, slot][:, None]
        ie = np.full((len(rows), 1), e, dtype=np.int32)
        sub = _sub(inp, rows)
        _, fe = oracle.moe_forward_ref(sub["x"], inp["w_router"], bias, inp["w_gate_up"],
                                       inp["w_down"], 1, routing=(ie, pe), keep=True)
        ge = oracle.moe_backward_ref(sub["x"], inp["w_router"], bias, inp["w_gate_up"],
                                     inp["w_down"], 1, sub["dy"], fwd=fe, grad_experts=[e])
        errs[f"dw_gate_up[{e}]"] = _gpu.rel_err(_gpu.host64(gpu["dw_gate_up"][e]),
                                                ge["dw_gate_up"][e])
        errs[f"dw_down[{e}]"] = _gpu.rel_err(_gpu.host64(gpu["dw_down"][e]), ge["dw_down"][e])

    # dW_router rows of two sampled experts (imbalanced: its cold experts are cheap)
    if name == "imbalanced":
        cold = np.nonzero(ok & (counts > 0) & (counts < 400))[0]
        for e in rng.choice(cold, size=min(2, len(cold)), replace=False):
            rows = np.nonzero((idx == e).any(axis=1))[0]
            sub = _sub(inp, rows)
            _, fe = oracle.moe_forward_ref(sub["x"], inp["w_router"], bias, inp["w_gate_up"],
                                           inp["w_down"], k, keep=True)
            ge = oracle.moe_backward_ref(sub["x"], inp["w_router"], bias, inp["w_gate_up"],
                                         inp["w_down"], k, sub["dy"], fwd=fe, grad_experts=[])
            errs[f"dw_router[{e}]"] = _gpu.rel_err(_gpu.host64(gpu["dw_router"][e]),
                                                   ge["dw_router"][e])
    print(name, errs)
    for n, v in errs.items():
        assert v <= _gpu.BF16_TOL, (n, v, errs)


def test_mxfp8_workload_sampled_parity():
    """MXFP8 expert GEMMs, T=16384 in 8 micro-batches of 2048 through a ring
    of 2 slots (micro-batches 0..5 are dispatched again in the backward);
    BF16 activation outputs, fp32 weight gradients.  Bar 6e-2 * rms."""
    from routing_dispatch_grouped_router_gb300 import api
    name = "mxfp8"
    w = gen.WORKLOADS[name]
    shape = gen.workload_shape(name)
    inp = gen.workload_inputs(name, seed=0, parallel=True)
    gpu = _gpu.run_gpu(shape, inp, dtype=api.MXFP8, flags=api.FLAG_BF16_ACT_OUT,
                       mb_tokens=w["mb_tokens"], ring_slots=w["ring_slots"])
    assert gpu["status"] == 0 and gpu["nmb"] == 8
    k, E, mb = shape.k, shape.E, gpu["mb"]
    idx, p, _, flagged, inner = oracle.route_ref(inp["x"], inp["w_router"], None, k)
    decided = _gpu.check_routing(gpu["topk_idx"], gpu["topk_w"], idx, p, flagged, inner)
    rng = np.random.default_rng(99)
    errs = {}
    args = (inp["w_router"], None, inp["w_gate_up"], inp["w_down"])
    toks = np.sort(rng.choice(np.nonzero(decided)[0], size=6, replace=False))
    y_ref, fwd = oracle.moe_forward_ref(inp["x"][toks], *args, k, keep=True, precision="mxfp8")
    g = oracle.moe_backward_ref(inp["x"][toks], *args, k, inp["dy"][toks], fwd=fwd,
                                grad_experts=[])
    errs["y"] = _gpu.rel_err(_gpu.host64(gpu["y"][toks]), y_ref)
    errs["dx"] = _gpu.rel_err(_gpu.host64(gpu["dx"][toks]), g["dx"])
    touched = np.zeros(E, dtype=bool)
    for t in np.nonzero(~decided)[0]:
        touched[idx[t]] = True
        touched[gpu["topk_idx"][t]] = True
    counts = np.bincount(idx.ravel(), minlength=E)
    ok = (counts > 0) & ~touched
    for e in rng.choice(np.nonzero(ok)[0], size=2, replace=False):
        dwgu = 0.0
        dwd = 0.0
        for i in range(gpu["nmb"]):
            sl = np.arange(i * mb, (i + 1) * mb)
            rows = sl[(idx[sl] == e).any(axis=1)]
            if len(rows) == 0:
                continue
            slot = np.argmax(idx[rows] == e, axis=1)
            pe = p[rows, slot][:, None]
            ie = np.full((len(rows), 1), e, dtype=np.int32)
            _, fe = oracle.moe_forward_ref(inp["x"][rows], *args, 1, routing=(ie, pe), keep=True,
                                           precision="mxfp8")
            ge = oracle.moe_backward_ref(inp["x"][rows], *args, 1, inp["dy"][rows], fwd=fe,
                                         grad_experts=[e])
            dwgu = dwgu + ge["dw_gate_up"][e]
            dwd = dwd + ge["dw_down"][e]
        errs[f"dw_gate_up[{e}]"] = _gpu.rel_err(_gpu.host64(gpu["dw_gate_up"][e]), dwgu)
        errs[f"dw_down[{e}]"] = _gpu.rel_err(_gpu.host64(gpu["dw_down"][e]), dwd)
    print(name, errs)
    for n, v in errs.items():
        assert v <= _gpu.MX_TOL, (n, v, errs)
