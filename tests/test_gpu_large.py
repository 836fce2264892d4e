"""Parity, determinism and invariants at the full sizes of the large
(T=8192, d=7168, E=384, I=2048, k=8), imbalanced (T=16384, d=4096, E=128,
I=1536, k=8, Zipf-biased router) and MXFP8 (the imbalanced shape without the
bias, 8 micro-batches of 2048 tokens through a 2-slot ring) workloads, in the
launch configuration the benchmark uses.

The full fp64 oracle is too slow at these sizes, so the comparison is on
outputs the oracle can compute one by one, with the routing forced as in
every other parity check (_gpu.forced_routing: the oracle's own top-k, except
where a near-tie leaves it undecided at float32):
  * routing of every token (the router is cheap), and the dispatch plan of
    every token, bit-exact;
  * y and dx of 64 sampled tokens: each token's outputs depend on that token
    only, so the oracle runs on the sampled tokens alone;
  * dW_gate_up and dW_down of sampled experts: an expert's weight gradients
    depend only on its own rows, so the oracle runs on the tokens routed to
    it with the routing restricted to that expert;
  * dW_router rows of sampled experts (on large: two with index >= 128, the
    second and third M tiles of the router-gradient GEMM): row e depends on
    the tokens routed to e, run through the oracle with their full routing.
Bar: max|diff| <= 2e-2 * rms(oracle) per compared tensor (6e-2 for MXFP8).

Properties that hold at any size, checked on whole tensors:
  * ten forward + backward calls give bitwise-identical outputs (compared by
    a wrap-around integer fingerprint of every output's bits);
  * permuting the tokens permutes y and dx bit for bit (each row's K loop is
    position-independent; the weight gradients sum rows in a different order
    and are not compared).
"""
import numpy as np
import pytest
import torch

import oracle
from routing_dispatch_grouped_router_gb300 import api, inputs as gen

import _gpu

pytestmark = pytest.mark.gpu

NAMES = ["imbalanced", "large", "mxfp8"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routing_dispatch_grouped_router_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.fixture(scope="module", params=NAMES)
def workload(request):
    """(name, shape, host inputs, layer options); tests are grouped by workload
    so each workload's inputs are drawn once."""
    name = request.param
    shape = gen.workload_shape(name)
    inp = gen.workload_inputs(name, seed=0, parallel=True)
    w = gen.WORKLOADS[name]
    opts = {}
    if name == "mxfp8":
        opts = dict(dtype=api.MXFP8, mb_tokens=w["mb_tokens"], ring_slots=w["ring_slots"])
    yield name, shape, inp, opts
    del inp
    torch.cuda.empty_cache()


def _sub(inp, toks):
    return dict(inp, x=inp["x"][toks], dy=inp["dy"][toks])


def _tol(name):
    return _gpu.MX_TOL if name == "mxfp8" else _gpu.BF16_TOL


def _prec(name):
    return "mxfp8" if name == "mxfp8" else "fp64"


def test_full_size_sampled_parity(workload):
    name, shape, inp, opts = workload
    gpu = _gpu.run_gpu(shape, inp, **opts)
    assert gpu["status"] == 0
    bias = inp["bias"]
    k, E, mb, nmb = shape.k, shape.E, gpu["mb"], gpu["nmb"]
    prec = _prec(name)
    args = (inp["w_router"], bias, inp["w_gate_up"], inp["w_down"])

    # routing of every token, and the plan of every micro-batch
    idx, p, _, flagged, inner = oracle.route_ref(inp["x"], inp["w_router"], bias, k)
    _gpu.check_routing(gpu["topk_idx"], gpu["topk_w"], idx, p, flagged, inner)
    fidx, fp, _ = _gpu.forced_routing(inp, k, gpu["topk_idx"])
    for i in range(nmb):
        sl = slice(i * mb, (i + 1) * mb)
        ref = oracle.dispatch_ref(fidx[sl], E)
        for n, r in zip(("mb_counts", "mb_offsets", "mb_pos", "mb_token_of_row"), ref):
            assert np.array_equal(gpu[n][i], r), (n, i)
    counts = np.bincount(fidx.ravel(), minlength=E)
    if name == "imbalanced":
        ratio = counts.max() / (shape.R / E)
        assert 7.6 <= ratio <= 8.4, ratio

    rng = np.random.default_rng(1234)
    errs = {"near_tie_tokens": int(flagged.sum())}

    # dW_router rows of the two coldest non-empty experts (large: among those
    # with index >= 128) and y, dx of 64 sampled tokens, in one oracle call on
    # the union of their tokens (a token's outputs and its dl depend on that
    # token only)
    eligible = (counts > 0) & ((np.arange(E) >= 128) if name == "large" else True)
    r_experts = np.argsort(np.where(eligible, counts, np.iinfo(np.int64).max),
                           kind="stable")[:2]
    assert eligible[r_experts].all()
    toks = np.sort(rng.choice(shape.T, size=64, replace=False))
    r_toks = np.nonzero(np.isin(fidx, r_experts).any(axis=1))[0]
    union = np.union1d(toks, r_toks)
    sub = _sub(inp, union)
    y_ref, fwd = oracle.moe_forward_ref(sub["x"], *args, k, routing=(fidx[union], fp[union]),
                                        keep=True, precision=prec)
    g = oracle.moe_backward_ref(sub["x"], *args, k, sub["dy"], fwd=fwd, grad_experts=[])
    at = np.searchsorted(union, toks)
    errs["y"] = _gpu.rel_err(_gpu.host64(gpu["y"][toks]), y_ref[at])
    errs["dx"] = _gpu.rel_err(_gpu.host64(gpu["dx"][toks]), g["dx"][at])
    for e in r_experts:
        errs[f"dw_router[{e}]"] = _gpu.rel_err(_gpu.host64(gpu["dw_router"][e]),
                                               g["dw_router"][e])

    # expert weight gradients: the hottest expert and one other (large: one
    # with index >= 256 as well); micro-batches sum their own rows' gradients
    hot = int(np.argmax(counts))
    others = [int(rng.choice(np.nonzero((counts > 0) & (np.arange(E) != hot))[0]))]
    if name == "large":
        others.append(int(rng.choice(np.nonzero((counts > 0) & (np.arange(E) >= 256))[0])))
    for e in [hot] + others:
        dwgu, dwd = 0.0, 0.0
        for i in range(nmb):
            sl = np.arange(i * mb, (i + 1) * mb)
            rows = sl[(fidx[sl] == e).any(axis=1)]
            if len(rows) == 0:
                continue
            slot = np.argmax(fidx[rows] == e, axis=1)
            pe = fp[rows, slot][:, None]
            ie = np.full((len(rows), 1), e, dtype=np.int32)
            sub = _sub(inp, rows)
            _, fe = oracle.moe_forward_ref(sub["x"], *args, 1, routing=(ie, pe), keep=True,
                                           precision=prec)
            ge = oracle.moe_backward_ref(sub["x"], *args, 1, sub["dy"], fwd=fe, grad_experts=[e])
            dwgu = dwgu + ge["dw_gate_up"][e]
            dwd = dwd + ge["dw_down"][e]
        errs[f"dw_gate_up[{e}]"] = _gpu.rel_err(_gpu.host64(gpu["dw_gate_up"][e]), dwgu)
        errs[f"dw_down[{e}]"] = _gpu.rel_err(_gpu.host64(gpu["dw_down"][e]), dwd)
    print(name, errs)
    for n, v in errs.items():
        if n != "near_tie_tokens":
            assert v <= _tol(name), (n, v, errs)


def fingerprint(t: torch.Tensor) -> tuple:
    """Two wrap-around (mod 2^64) integer sums of a tensor's 32-bit words, one
    of them position-weighted: any change of any bit changes them except by a
    vanishing chance, and integer addition mod 2^64 does not depend on the
    order torch sums in."""
    v = t.contiguous().view(-1).view(torch.int32)
    s1 = torch.zeros((), dtype=torch.int64, device=v.device)
    s2 = torch.zeros((), dtype=torch.int64, device=v.device)
    chunk = 1 << 26
    for i in range(0, v.numel(), chunk):
        c = v[i:i + chunk].to(torch.int64)
        w = torch.arange(i, i + c.numel(), dtype=torch.int64, device=v.device) % 1000003 + 1
        s1 += c.sum()
        s2 += (c * w).sum()
    return int(s1.item()), int(s2.item())


def _device_inputs(inp):
    x, wr, wgu, wd, dy = (_gpu.dev_bf16(inp[n]) for n in ("x", "w_router", "w_gate_up",
                                                          "w_down", "dy"))
    bias = torch.from_numpy(inp["bias"]).cuda() if inp.get("bias") is not None else None
    return x, wr, bias, wgu, wd, dy


def test_full_size_bitwise_deterministic(workload):
    """Ten calls of the benchmark's configuration, every output bitwise equal."""
    name, shape, inp, opts = workload
    layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k, **opts)
    x, wr, bias, wgu, wd, dy = _device_inputs(inp)
    f32 = dict(dtype=torch.float32, device="cuda")
    y, dx = torch.empty(x.shape, **f32), torch.empty(x.shape, **f32)
    dwr, dwgu, dwd = (torch.empty(t.shape, **f32) for t in (wr, wgu, wd))
    first = None
    for _ in range(10):
        layer.forward(x, wr, bias, wgu, wd, y=y)
        layer.backward(dy, x, wr, bias, wgu, wd, dx=dx, dw_router=dwr, dw_gate_up=dwgu,
                       dw_down=dwd)
        cur = [fingerprint(t) for t in (y, dx, dwr, dwgu, dwd)]
        cur.append(fingerprint(layer.saved_tensor("topk_idx", torch.int32, (shape.T // (
            layer.layout.mb_count), shape.k))))
        if first is None:
            first = cur
        assert cur == first
    assert layer.status() == 0


def test_full_size_token_permutation_equivariance(workload):
    """Permuting the tokens permutes y and dx bit for bit, and the routing."""
    name, shape, inp, opts = workload
    if name != "large":
        pytest.skip("checked on the large workload")
    x, wr, bias, wgu, wd, dy = _device_inputs(inp)
    perm = torch.from_numpy(np.random.default_rng(5).permutation(shape.T)).cuda()
    outs = []
    for xs, dys in ((x, dy), (x[perm].contiguous(), dy[perm].contiguous())):
        layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k, **opts)
        y = layer.forward(xs, wr, bias, wgu, wd)
        dx, dwr, dwgu, dwd = layer.backward(dys, xs, wr, bias, wgu, wd)
        del dwr, dwgu, dwd
        assert layer.status() == 0
        idx = layer.saved_tensor("topk_idx", torch.int32, (shape.T, shape.k)).clone()
        outs.append((y, dx, idx))
        del layer
    (y0, dx0, i0), (y1, dx1, i1) = outs
    assert torch.equal(i1, i0[perm])
    assert torch.equal(y1.view(torch.int32), y0[perm].view(torch.int32))
    assert torch.equal(dx1.view(torch.int32), dx0[perm].view(torch.int32))
