"""Helpers of the GPU tests: device copies of the seeded inputs, one layer
call through the C ABI, and the comparisons against the oracle.

The oracle always computes from the same seeded inputs.  Routing has more
than one correct answer only where float32 logits cannot decide it (a near-tie
the oracle flags); there the kernel's choice is checked to be valid and the
checks after the router take it (forced_routing), so every token and expert is
compared.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from routing_dispatch_grouped_router_gb300 import api, inputs as gen

BF16_TOL = 2e-2   # max|diff| <= tol * rms(oracle) for BF16 layers
MX_TOL = 6e-2     # and for MXFP8 layers


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rel_err(got, ref) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    diff = float(np.max(np.abs(got - ref)))
    if rms == 0.0:
        return diff
    return diff / rms


def run_gpu(shape: gen.Shape, inp: dict, layer=None, flags=0, dtype=0, mb_tokens=0, ring_slots=0):
    """Forward + backward of one layer call; returns host copies of the plan of
    every micro-batch and device tensors of the outputs."""
    if layer is None:
        layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k, flags=flags,
                             dtype=dtype, mb_tokens=mb_tokens, ring_slots=ring_slots)
    x = dev_bf16(inp["x"])
    wr = dev_bf16(inp["w_router"])
    wgu = dev_bf16(inp["w_gate_up"])
    wd = dev_bf16(inp["w_down"])
    dy = dev_bf16(inp["dy"])
    bias = torch.from_numpy(inp["bias"]).cuda() if inp.get("bias") is not None else None
    y = layer.forward(x, wr, bias, wgu, wd)
    dx, dwr, dwgu, dwd = layer.backward(dy, x, wr, bias, wgu, wd)
    status = layer.status()
    k, E = shape.k, shape.E
    L = layer.layout
    nmb = int(L.mb_count)
    T = shape.T // nmb if shape.T else 0

    def plan(field, dtype, shp):
        return [layer.saved_tensor(field, dtype, shp, i).cpu().numpy() for i in range(nmb)]
    out = dict(
        status=status,
        y=y, dx=dx, dw_router=dwr, dw_gate_up=dwgu, dw_down=dwd,
        topk_idx=np.concatenate(plan("topk_idx", torch.int32, (T, k))),
        topk_w=np.concatenate(plan("topk_w", torch.float32, (T, k))),
        mb_counts=plan("counts", torch.int32, (E,)),
        mb_offsets=plan("offsets", torch.int32, (E + 1,)),
        mb_pos=plan("pos", torch.int32, (T, k)),
        mb_token_of_row=plan("token_of_row", torch.int32, (T * k,)),
        padded_pos=layer.saved_tensor("padded_pos", torch.int32, (T, k)).cpu().numpy(),
        gate_up=(None if L.gate_up == api.NOT_KEPT else
                 layer.saved_tensor("gate_up", torch.float32, (L.rows_max, 2 * shape.I))),
        layer=layer, nmb=nmb, mb=T,
    )
    out["counts"], out["offsets"] = out["mb_counts"][0], out["mb_offsets"][0]
    out["pos"], out["token_of_row"] = out["mb_pos"][0], out["mb_token_of_row"][0]
    return out


def check_routing(gpu_idx, gpu_w, ref_idx, ref_w, flagged, inner_tie):
    """Bit-exact routing except where the oracle flags a near-tie.
    Returns the mask of tokens whose routing is decided (and equal)."""
    T = ref_idx.shape[0]
    ok = ~flagged
    same_order = (gpu_idx == ref_idx).all(axis=1)
    same_set = (np.sort(gpu_idx, axis=1) == np.sort(ref_idx, axis=1)).all(axis=1)
    # decided tokens: exact slot order unless two chosen logits are within 1e-5
    bad = ok & ~np.where(inner_tie, same_set, same_order)
    assert not bad.any(), f"routing differs on {int(bad.sum())} decided tokens: {np.nonzero(bad)[0][:10]}"
    # routing weights: softmax of fp32 logits whose accumulation over d terms
    # is off by ~1e-6 of |l| (|l| < ~10 here); 1e-4 bounds |dp| with margin
    w_err = np.abs(np.sort(gpu_w, axis=1) - np.sort(ref_w, axis=1))[ok]
    assert w_err.size == 0 or w_err.max() < 1e-4, w_err.max()
    np.testing.assert_allclose(gpu_w.sum(axis=1), 1.0, atol=2e-6)
    return ok & same_order


def check_dispatch_valid(idx, counts, offsets, pos, token_of_row, E):
    """Properties every correct dispatch of `idx` has (used where the exact
    result would need the undecided routing)."""
    T, k = idx.shape
    assert counts.sum() == T * k
    assert offsets[0] == 0 and (np.diff(offsets) == counts).all()
    assert sorted(pos.ravel().tolist()) == list(range(T * k))
    for e in range(E):
        seg = token_of_row[offsets[e]:offsets[e + 1]]
        assert (np.diff(seg) > 0).all()
    tt = np.repeat(np.arange(T), k)
    assert (token_of_row[pos.ravel()] == tt).all()


def check_bf16_intermediate(got_bf16: np.ndarray, ref: np.ndarray, name: str):
    """A stored bf16 value against the oracle's bf16 value of the same
    quantity.  They agree except where the kernel's float32 accumulation and
    the oracle's exact one fall on the two sides of a bf16 rounding boundary:
    then they differ by one bf16 ulp, plus at most the float32 accumulation
    error (which matters only for results near zero, where a bf16 ulp is
    smaller than it).  Returns the fraction of elements that differ."""
    got_bf16 = np.asarray(got_bf16, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    diff = got_bf16 != ref
    frac = float(diff.mean())
    rms = float(np.sqrt(np.mean(ref * ref)))
    if diff.any():
        a = np.abs(ref[diff])
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7)
        excess = np.abs(got_bf16[diff] - ref[diff]) - ulp
        worst = float(excess.max()) / rms if rms else float(excess.max())
        assert worst <= 1e-5, (name, "beyond one ulp by", worst, "x rms; differing fraction", frac)
    assert frac < 1e-2, (name, "differing fraction", frac)
    return frac


def forced_routing(inp: dict, k: int, gpu_idx: np.ndarray):
    """The routing the downstream checks use.

    Routing is one of the results with several correct answers: where the
    float64 gap between the k-th and (k+1)-th logit is below 1e-5 (flagged),
    float32 logits cannot decide the chosen set, and where two chosen logits
    are that close (inner tie) they cannot decide the slot order.  So the
    oracle's own top-k is used for every token, except where the kernel chose
    differently on such a token; there the kernel's choice is first checked
    to be a valid top-k within the tolerance (every chosen logit at least the
    largest unchosen one minus 1e-5, no expert twice) and then taken.  The
    weights are the definition's softmax over the set taken, from the
    oracle's own float64 logits.  Returns (topk_idx, p, flagged)."""
    idx, _, logits, flagged, inner = oracle.route_ref(inp["x"], inp["w_router"], inp.get("bias"),
                                                      k)
    g = np.ascontiguousarray(gpu_idx, dtype=np.int32)
    differs = (g != idx).any(axis=1)
    same_set = (np.sort(g, axis=1) == np.sort(idx, axis=1)).all(axis=1)
    T, E = logits.shape
    in_range = ((g >= 0) & (g < E)).all(axis=1)
    distinct = (np.diff(np.sort(g, axis=1), axis=1) > 0).all(axis=1) if k > 1 else in_range
    chosen = np.zeros((T, E), dtype=bool)
    np.put_along_axis(chosen, np.clip(g, 0, E - 1).astype(np.int64), True, axis=1)
    low = np.where(chosen, logits, np.inf).min(axis=1)
    high = np.where(chosen, -np.inf, logits).max(axis=1) if k < E else np.full(T, -np.inf)
    valid = in_range & distinct & (low >= high - oracle.NEAR_TIE)
    ok = (inner & same_set) | (flagged & valid)
    bad = differs & ~ok
    assert not bad.any(), f"routing differs on decided tokens {np.nonzero(bad)[0][:10]}"
    use = np.where(differs[:, None], g, idx).astype(np.int32)
    return use, oracle.routing_weights(logits, use), flagged


def full_parity(shape: gen.Shape, inp: dict, gpu: dict, tol=BF16_TOL, precision="fp64"):
    """Element-wise comparison of every output against the full oracle (fp64,
    or its mxfp8 definition), every token and expert included.  Routing is
    bit-exact where the oracle decides it; everything after it is checked with
    the oracle forced to the kernel's chosen sets (forced_routing), so the
    dispatch plan is bit-exact with no exclusions.  With micro-batches each
    one is dispatched on its own, so the plan is compared per micro-batch and
    the weight gradients against the sum of the oracle's per-micro-batch
    gradients (MXFP8 blocks along the token dimension are formed inside each
    micro-batch's expert segments)."""
    assert gpu["status"] == 0, gpu["status"]
    bias = inp.get("bias")
    nmb, mb = gpu["nmb"], gpu["mb"]
    idx, p, logits, flagged, inner = oracle.route_ref(inp["x"], inp["w_router"], bias, shape.k)
    check_routing(gpu["topk_idx"], gpu["topk_w"], idx, p, flagged, inner)
    gidx, pf, _ = forced_routing(inp, shape.k, gpu["topk_idx"])
    # the kernel's weights on its own sets: float32 logits and softmax
    assert np.abs(gpu["topk_w"] - pf).max() < 1e-4
    for i in range(nmb):
        sl = slice(i * mb, (i + 1) * mb)
        counts, offsets, pos, tok = oracle.dispatch_ref(gidx[sl], shape.E)
        assert (gpu["mb_counts"][i] == counts).all()
        assert (gpu["mb_offsets"][i] == offsets).all()
        assert (gpu["mb_pos"][i] == pos).all()
        assert (gpu["mb_token_of_row"][i] == tok).all()

    args = (inp["w_router"], bias, inp["w_gate_up"], inp["w_down"], shape.k)
    y, fwd = oracle.moe_forward_ref(inp["x"], *args, routing=(gidx, pf), keep=True,
                                    precision=precision)
    g = oracle.moe_backward_ref(inp["x"], *args, inp["dy"], fwd=fwd)
    if nmb > 1:
        parts, ys = [], []
        for i in range(nmb):
            sl = slice(i * mb, (i + 1) * mb)
            yi, fi = oracle.moe_forward_ref(inp["x"][sl], *args, routing=(gidx[sl], pf[sl]),
                                            keep=True, precision=precision)
            ys.append(yi)
            parts.append(oracle.moe_backward_ref(inp["x"][sl], *args, inp["dy"][sl], fwd=fi))
        for n in ("dw_router", "dw_gate_up", "dw_down"):
            g[n] = sum(q[n] for q in parts)
        if precision == "nvfp4":
            # NVFP4 tensor scales are taken per micro-batch (its x, its h), so
            # y and dx are those of each micro-batch's own forward
            y = np.concatenate(ys)
            g["dx"] = np.concatenate([q["dx"] for q in parts])
    errs = {}
    errs["y"] = rel_err(host64(gpu["y"]), y)
    errs["dx"] = rel_err(host64(gpu["dx"]), g["dx"])
    # fp32 pre-activations saved for the backward (micro-batch 0): fp32
    # accumulation error only
    if gpu["gate_up"] is not None:
        pos0 = oracle.dispatch_ref(gidx[:mb], shape.E)[2]
        gu = host64(gpu["gate_up"])
        rows_gpu = gpu["padded_pos"].ravel()
        rows_ref = pos0.ravel()
        if nmb > 1:
            _, f0 = oracle.moe_forward_ref(inp["x"][:mb], *args, routing=(gidx[:mb], pf[:mb]),
                                           keep=True, precision=precision)
        else:
            f0 = fwd
        errs["gate"] = rel_err(gu[rows_gpu, :shape.I], f0["G"][rows_ref])
        errs["up"] = rel_err(gu[rows_gpu, shape.I:], f0["U"][rows_ref])
        assert errs["gate"] < 1e-4 and errs["up"] < 1e-4, errs
    for n in ("dw_router", "dw_gate_up", "dw_down"):
        errs[n] = rel_err(host64(gpu[n]), g[n])
    for name, v in errs.items():
        assert v <= tol, (name, v, errs)
    # experts that received no rows have exactly zero weight gradients
    empty = np.bincount(gidx.ravel(), minlength=shape.E) == 0
    if empty.any():
        assert (host64(gpu["dw_gate_up"])[empty] == 0).all()
        assert (host64(gpu["dw_down"])[empty] == 0).all()
        assert (host64(gpu["dw_router"])[empty] == 0).all()
    errs["near_tie_tokens"] = int(flagged.sum())
    return errs
