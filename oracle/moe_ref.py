"""fp64 CPU oracle of the deterministic MoE layer: routing, dispatch, experts,
combine and the analytic backward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with
the CUDA path and never calls it.

Sources (page title, section):
  [gtnt]     "MoK揭秘：NVL72上大规模MoE训练工程方案深度解读" (gtnt.cn), §1.1:
             a gating network (router) picks the best few experts per token.
  [dothoosh] "Cursor Mixture-of-Kittens cuts MoE training latency by 5.8x"
             (dothoosh.com), section "MoK technical details":
             bullet "Hybrid communication": forward = dispatch, expert
             compute, combine; backward = reverse-combine then reverse-dispatch;
             bullet "Ring buffer logic": dropless (no token is dropped);
             bullet "Precision and scheduling": SwiGLU experts, BF16/MXFP8,
             router-weight gradients taken inside the SwiGLU backward.

Every float computation here runs in float64 on the bf16 inputs widened
exactly.  The one decision taken in float32 is the top-k selection, because the
CUDA router takes it on float32 logits (the layer's stated logit precision);
tokens whose float64 k-th/(k+1)-th logit gap is below 1e-5 are flagged so a
comparison can leave them out.

Precision.  ``precision="fp64"`` (default) is the layer's plain definition in
float64.  ``precision="bf16"`` is the same definition with the operand
precision the pages fix for the expert GEMMs ([dothoosh] "Precision and
scheduling": the megakernel runs its GEMMs in BF16): every operand of the six
expert GEMMs is a bf16 value, each GEMM accumulates exactly (float64), and
nothing that is not a GEMM operand is rounded.  The rounded operands are
  G, U            (outputs of the gate/up GEMM, stored as bf16)
  H = silu(G) U   (operand of the down GEMM)
  P = p * H       (operand of the down-projection weight gradient,
                   dW_down = sum_r dy_r (p_r h_r)^T)
  dG, dU          (operands of the gate/up dgrad and weight gradient)
each rounded to the nearest bf16 (ties to even).  ``precision="mxfp8"`` is the
MXFP8 definition (E4M3 elements, one E8M0 scale per 32 values along each
GEMM's reduction dimension, see mx_ref.py): every operand of the forward
GEMMs and of the two dgrads is fake-quantised (x rows, W_gate/W_up along d,
h and W_down along I, dy rows along d, W_down along d, [dG dU] along 2I,
W_gate_up along 2I); in the two weight-gradient GEMMs the layer inputs x and
dy are quantised along the token dimension (each expert's rows zero-padded to
a multiple of 32) while the derived operands p*h and [dG dU] are not.  With
quantised GEMMs the identity <dy, O> = <dy W_down, h> no longer holds exactly;
the router-weight gradient is taken the way the pages fuse it into the SwiGLU
backward ([dothoosh] "Precision and scheduling"): dp = <dA, h> with dA the
(quantised) down-projection dgrad of the row and h unquantised.
``precision="nvfp4"`` quantises the forward GEMMs' operands and those of the
gate/up dgrad to NVFP4 (see _nvfp4_experts, _nvfp4_gate_up_dgrad and
nvfp4_ref.py: per-tensor fp32 scales, E4M3 scales per 16 values along K); the
rest of the backward is the float64 one on the forward's g, u, h, with the
router-weight gradient in the same fused form dp = <dy W_down, h>.
dy is itself a bf16 input,
so the down dgrad dH = p * (dy W_down) needs no rounded operand.  The expert
output O, y, dp, the router gradient, dx and the weight gradients are not
rounded.

Readings where the pages say nothing (all are listed again in the design notes):
  * routing weights are a softmax over the k chosen logits (equal to the full
    softmax restricted to the chosen set and renormalised, so they sum to 1);
  * ties in float32 go to the lower expert index; slots are in descending
    logit order;
  * SwiGLU is silu(gate) * up with silu(z) = z*sigmoid(z), gate rows first in
    the stacked [2I, d] weight;
  * rows of one expert are ordered by token id (a stable counting sort);
  * the loss used for the backward is L = sum(y * dy).
"""
from __future__ import annotations

import numpy as np

from .mx_ref import mx_fake
from .nvfp4_ref import nvfp4_fake

NEAR_TIE = 1e-5


# ----------------------------------------------------------------------------
# storage helpers (own copy: the oracle does not import the CUDA package)
# ----------------------------------------------------------------------------

def widen(a) -> np.ndarray:
    """bf16 bit pattern (uint16) or float array -> float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def bf16_round(a) -> np.ndarray:
    """Nearest bfloat16 value (8 significant bits, ties to even, fp32 exponent
    range, subnormal quantum 2^-133, overflow to inf) of float64 values."""
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)                       # a = m * 2**e, 0.5 <= |m| < 1
    r = np.ldexp(np.round(np.ldexp(m, 8)), e - 8)   # np.round: half to even
    tiny = np.abs(a) < 2.0 ** -126
    if tiny.any():
        q = 2.0 ** -133
        r = np.where(tiny, np.round(a / q) * q, r)
    big = np.abs(r) > 3.3895313892515355e38  # largest finite bf16
    if big.any():
        r = np.where(big, np.copysign(np.inf, a), r)
    return r


def _identity(a):
    return a


def _rounder(precision: str):
    if precision in ("fp64", "mxfp8", "nvfp4"):
        return _identity
    if precision == "bf16":
        return bf16_round
    raise ValueError(precision)


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * _sigmoid(z)


def silu_grad(z):
    s = _sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


# ----------------------------------------------------------------------------
# routing  [gtnt] §1.1; reading: softmax over the chosen k, fixed tie rule
# ----------------------------------------------------------------------------

def router_logits(x, w_router, bias=None) -> np.ndarray:
    """l = x W_r^T (+ b), float64 [T, E]."""
    l = widen(x) @ widen(w_router).T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    return l


def routing_weights(logits, topk_idx) -> np.ndarray:
    """Softmax over each token's chosen experts, in the given slot order:
    p_s = exp(l_s - m) / sum_{j in S} exp(l_j - m), m = max over S (float64).
    With a chosen set taken from elsewhere (the kernel's, where a near-tie
    makes the set undecidable), this gives the weights the definition
    assigns to that set."""
    sel = np.take_along_axis(np.asarray(logits, dtype=np.float64),
                             np.asarray(topk_idx, dtype=np.int64), axis=1)
    m = sel.max(axis=1, keepdims=True)
    ex = np.exp(sel - m)
    return ex / ex.sum(axis=1, keepdims=True)


def route_ref(x, w_router, bias, k: int):
    """Top-k routing.

    Returns (topk_idx [T,k] int32, topk_w [T,k] float64, logits [T,E] float64,
    flagged [T] bool, inner_tie [T] bool).

    Selection: the k largest float32-rounded logits; equal values go to the
    lower expert index; slots are ordered by descending logit.
    Weights: p_s = exp(l_s - m) / sum_{j in S} exp(l_j - m), m = max over S.
    ``flagged``: the float64 gap between the k-th and (k+1)-th largest logit is
    below 1e-5, so the chosen set itself is not decidable at the kernel's
    precision.  ``inner_tie``: two adjacent chosen logits are within 1e-5, so
    only the chosen set (not the slot order) is decidable.
    """
    logits = router_logits(x, w_router, bias)
    T, E = logits.shape
    l32 = logits.astype(np.float32)
    # order experts by (-l32, index): lexsort keys are applied last-key-primary
    cols = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((cols, -l32), axis=-1)
    idx = order[:, :k].astype(np.int32)
    w = routing_weights(logits, idx)
    sel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    ranked = np.take_along_axis(logits, order, axis=1)
    if k < E:
        flagged = (ranked[:, k - 1] - ranked[:, k]) < NEAR_TIE
    else:
        flagged = np.zeros(T, dtype=bool)
    if k > 1:
        inner_tie = (np.abs(np.diff(sel, axis=1)) < NEAR_TIE).any(axis=1)
    else:
        inner_tie = np.zeros(T, dtype=bool)
    return idx, w, logits, flagged, inner_tie


# ----------------------------------------------------------------------------
# dispatch  [dothoosh] "Hybrid communication" + "Ring buffer logic" (dropless)
# ----------------------------------------------------------------------------

def dispatch_ref(topk_idx, E: int):
    """Stable counting sort of the T*k (token, slot) pairs by expert.

    counts[e]  = #{(t,s): idx[t,s] = e}
    offsets    = exclusive prefix sum of counts, length E+1
    pos[t,s]   = offsets[e] + #{t' < t routed to e}   (ties by token id)
    token_of_row[pos[t,s]] = t
    """
    idx = np.asarray(topk_idx, dtype=np.int64)
    T, k = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    np.cumsum(counts, out=offsets[1:])
    # flat position f = t*k + s is token-major, so a stable sort by expert
    # keeps token order inside each expert
    order = np.argsort(idx.ravel(), kind="stable")
    pos = np.empty(T * k, dtype=np.int64)
    pos[order] = np.arange(T * k)
    token_of_row = order // k
    return (counts.astype(np.int32), offsets.astype(np.int32),
            pos.reshape(T, k).astype(np.int32), token_of_row.astype(np.int32))


# ----------------------------------------------------------------------------
# forward  ([dothoosh] "Hybrid communication", "Precision and scheduling")
# ----------------------------------------------------------------------------

def expert_ffn(X, w_gate_up_e, w_down_e, rnd=_identity, mx=False):
    """SwiGLU FFN of one expert on rows X (float64).  Returns (G, U, H, O).
    ``rnd`` rounds the GEMM operands (identity in float64 mode); ``mx``
    fake-quantises them to MXFP8 along their reduction dimension."""
    Wgu = widen(w_gate_up_e)
    Wd = widen(w_down_e)
    I = Wgu.shape[0] // 2
    if mx:
        Xq, Wq = mx_fake(X, -1), mx_fake(Wgu, -1)
        G = Xq @ Wq[:I].T
        U = Xq @ Wq[I:].T
        H = silu(G) * U
        return G, U, H, mx_fake(H, -1) @ mx_fake(Wd, -1).T
    G = rnd(X @ Wgu[:I].T)
    U = rnd(X @ Wgu[I:].T)
    H = rnd(silu(G) * U)
    O = H @ Wd.T
    return G, U, H, O


def _mx_rows(a):
    """MXFP8 along the token dimension (axis 0), the rows zero-padded to a
    multiple of 32 as the blocks start at the expert's first row."""
    n = a.shape[0]
    pad = (-n) % 32
    if pad:
        a = np.concatenate([a, np.zeros((pad,) + a.shape[1:])], axis=0)
    return mx_fake(a, 0)[:n]


def _nvfp4_experts(X, w_gate_up, w_down, offsets, tok, R):
    """The experts' GEMMs on NVFP4 operands (nvfp4_ref): every operand is
    quantised along its GEMM's reduction dimension, with its tensor scale
    taken over the whole tensor -- x over all tokens, W_gate_up over all
    experts' stacked [E*2I, d] rows, W_down over all [E*d, I] rows, and h over
    all routed rows.  h = silu(g) u is materialised in bf16 before its
    quantisation (the layer stores it so between the two GEMMs).  Returns
    (G, U, H, O) in expert order; H is silu(G) U before any rounding."""
    Wgu = widen(w_gate_up)
    Wd = widen(w_down)
    E, I2, d = Wgu.shape
    I = I2 // 2
    Xq = nvfp4_fake(X, -1)
    Wgu_q = nvfp4_fake(Wgu.reshape(E * I2, d), -1).reshape(E, I2, d)
    Wd_q = nvfp4_fake(Wd.reshape(E * d, I), -1).reshape(E, d, I)
    G = np.zeros((R, I)); U = np.zeros((R, I)); H = np.zeros((R, I)); O = np.zeros((R, d))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        G[a:b] = Xq[tok[a:b]] @ Wgu_q[e, :I].T
        U[a:b] = Xq[tok[a:b]] @ Wgu_q[e, I:].T
        H[a:b] = silu(G[a:b]) * U[a:b]
    Hq = nvfp4_fake(bf16_round(H), -1) if R else H
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a < b:
            O[a:b] = Hq[a:b] @ Wd_q[e].T
    return G, U, H, O


def _nvfp4_gate_up_dgrad(dGU, w_gate_up, offsets):
    """The gate/up dgrad dX = [dG dU] W_gate_up on NVFP4 operands: [dG dU]
    (as bf16, the layer's stored form) along 2I with its tensor scale over all
    routed rows, W_gate_up along 2I with its tensor scale over all experts
    (the same scale as in the forward: the same tensor)."""
    Wgu = widen(w_gate_up)
    E, I2, d = Wgu.shape
    dGU_q = nvfp4_fake(bf16_round(dGU), -1)
    # each expert's [2I, d] weights as d rows of 2I values, quantised along 2I
    Wt_q = nvfp4_fake(Wgu.transpose(0, 2, 1).reshape(E * d, I2), -1).reshape(E, d, I2)
    dX = np.zeros((dGU.shape[0], d))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a < b:
            dX[a:b] = dGU_q[a:b] @ Wt_q[e].T
    return dX


def moe_forward_ref(x, w_router, bias, w_gate_up, w_down, k: int, routing=None,
                    keep=False, precision="fp64"):
    """y_t = sum_s p[t,s] * FFN_{e[t,s]}(x_t), summed in slot order.

    ``routing`` = (topk_idx, topk_w) forces the routing (e.g. to check the
    later stages on exactly the kernel's selection); otherwise route_ref runs.
    Returns y [T,d] float64, and with keep=True also a dict of intermediates.
    ``precision`` selects the plain float64 definition or the BF16-operand one.
    """
    rnd = _rounder(precision)
    X = widen(x)
    T, d = X.shape
    E = np.asarray(w_gate_up).shape[0]
    if routing is None:
        idx, p, _, _, _ = route_ref(x, w_router, bias, k)
    else:
        idx = np.asarray(routing[0], dtype=np.int32)
        p = np.asarray(routing[1], dtype=np.float64)
    counts, offsets, pos, tok = dispatch_ref(idx, E)
    R = T * k
    I = np.asarray(w_gate_up).shape[1] // 2
    O = np.zeros((R, d))
    G = np.zeros((R, I)); U = np.zeros((R, I)); H = np.zeros((R, I))
    if precision == "nvfp4":
        G, U, H, O = _nvfp4_experts(X, w_gate_up, w_down, offsets, tok, R)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b or precision == "nvfp4":
            continue
        G[a:b], U[a:b], H[a:b], O[a:b] = expert_ffn(X[tok[a:b]], w_gate_up[e], w_down[e], rnd,
                                                     mx=(precision == "mxfp8"))
    y = np.zeros((T, d))
    for s in range(k):
        y += p[:, s:s + 1] * O[pos[:, s]]
    if not keep:
        return y
    return y, dict(idx=idx, p=p, counts=counts, offsets=offsets, pos=pos,
                   token_of_row=tok, G=G, U=U, H=H, O=O, precision=precision)


# ----------------------------------------------------------------------------
# backward of L = sum(y * dy)
# ([dothoosh] "Hybrid communication": reverse-combine then reverse-dispatch;
#  "Precision and scheduling": router-weight gradient from the SwiGLU backward)
# ----------------------------------------------------------------------------

def moe_backward_ref(x, w_router, bias, w_gate_up, w_down, k: int, dy,
                     routing=None, fwd=None, grad_experts=None, precision=None):
    """Analytic gradients of L = sum(y*dy).

    Returns dict with dx [T,d], dw_router [E,d], dw_gate_up [E,2I,d],
    dw_down [E,d,I] (all float64) and dp [T,k] (dL/dp).
    With ``grad_experts`` (an iterable of expert ids), dw_gate_up and dw_down
    are dicts holding only those experts' gradients (large layers).
    The routing (the chosen set S_t) is piecewise constant, so only p carries
    a gradient into the router logits:
      dp[t,s]   = <dy_t, O[pos[t,s]]>
      dl[t,j]   = p_j (dp_j - sum_i p_i dp_i) for j in S_t, 0 elsewhere
      dx       += dl W_r,   dW_r = dl^T x.
    ``precision`` defaults to the one of ``fwd`` (float64 when fwd is None).
    """
    if precision is None:
        precision = fwd.get("precision", "fp64") if fwd is not None else "fp64"
    rnd = _rounder(precision)
    X = widen(x)
    dY = widen(dy)
    T, d = X.shape
    E = np.asarray(w_gate_up).shape[0]
    I = np.asarray(w_gate_up).shape[1] // 2
    if fwd is None:
        _, fwd = moe_forward_ref(x, w_router, bias, w_gate_up, w_down, k,
                                 routing=routing, keep=True, precision=precision)
    idx, p, offsets, pos, tok = fwd["idx"], fwd["p"], fwd["offsets"], fwd["pos"], fwd["token_of_row"]
    G, U, H, O = fwd["G"], fwd["U"], fwd["H"], fwd["O"]
    R = T * k

    # reverse-combine: per routed row, the upstream gradient scaled by p
    row_t = tok
    row_p = np.empty(R)
    for s in range(k):
        row_p[pos[:, s]] = p[:, s]
    dO = row_p[:, None] * dY[row_t]
    if precision in ("mxfp8", "nvfp4"):
        dp_rows = np.zeros(R)
    else:
        dp = np.einsum("tsd,td->ts", O[pos], dY)

    dX_rows = np.zeros((R, d))
    dGU_all = np.zeros((R, 2 * I)) if precision == "nvfp4" else None
    if grad_experts is None:
        dw_gate_up = np.zeros((E, 2 * I, d))
        dw_down = np.zeros((E, d, I))
    else:
        dw_gate_up = {int(e): np.zeros((2 * I, d)) for e in grad_experts}
        dw_down = {int(e): np.zeros((d, I)) for e in grad_experts}
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        Wd = widen(w_down[e])
        Wgu = widen(w_gate_up[e])
        Xe = X[tok[a:b]]
        dYe = dY[row_t[a:b]]
        if precision == "mxfp8":
            dA = mx_fake(dYe, -1) @ mx_fake(Wd, 0)
            dp_rows[a:b] = (dA * H[a:b]).sum(axis=1)
            dH = row_p[a:b, None] * dA
            dG = dH * U[a:b] * silu_grad(G[a:b])
            dU = dH * silu(G[a:b])
            dGU = np.concatenate([dG, dU], axis=1)
            dX_rows[a:b] = mx_fake(dGU, -1) @ mx_fake(Wgu, 0)
            if grad_experts is None or e in dw_down:
                dw_down[e][...] = _mx_rows(dYe).T @ (row_p[a:b, None] * H[a:b])
                dw_gate_up[e][...] = dGU.T @ _mx_rows(Xe)
            continue
        if precision == "nvfp4":
            # router-weight gradient in the fused form, <dA, h> with dA the
            # (unquantised) down dgrad: the forward's O is quantised
            dp_rows[a:b] = ((dYe @ Wd) * H[a:b]).sum(axis=1)
        dH = dO[a:b] @ Wd                       # [rows, I]
        dG = rnd(dH * U[a:b] * silu_grad(G[a:b]))
        dU = rnd(dH * silu(G[a:b]))
        if precision == "nvfp4":
            # the gate/up dgrad runs after every expert's dG/dU exists (its
            # operand's tensor scale covers all rows): kept for below
            dGU_all[a:b] = np.concatenate([dG, dU], axis=1)
        else:
            dX_rows[a:b] = dG @ Wgu[:I] + dU @ Wgu[I:]
        if grad_experts is None or e in dw_down:
            # sum_r p_r dy_r h_r^T, with p applied on the h side
            dw_down[e][...] = dYe.T @ rnd(row_p[a:b, None] * H[a:b])
            dw_gate_up[e][:I] = dG.T @ Xe
            dw_gate_up[e][I:] = dU.T @ Xe

    if precision == "nvfp4" and R:
        dX_rows = _nvfp4_gate_up_dgrad(dGU_all, w_gate_up, offsets)
    if precision in ("mxfp8", "nvfp4"):
        dp = dp_rows[pos]

    # reverse-dispatch: sum each token's k rows in slot order
    dx = np.zeros((T, d))
    for s in range(k):
        dx += dX_rows[pos[:, s]]

    # router: softmax over the chosen set
    c = (p * dp).sum(axis=1, keepdims=True)
    dl_sel = p * (dp - c)
    dl = np.zeros((T, E))
    np.put_along_axis(dl, idx.astype(np.int64), dl_sel, axis=1)
    Wr = widen(w_router)
    dx += dl @ Wr
    dw_router = dl.T @ X
    return dict(dx=dx, dw_router=dw_router, dw_gate_up=dw_gate_up,
                dw_down=dw_down, dp=dp, dl=dl_sel)
