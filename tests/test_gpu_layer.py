"""Parity of the CUDA layer (through the C ABI) against the fp64 oracle, plus
determinism and edge cases.  Bar: routing bit-exact where the oracle decides
it; dispatch plan bit-exact and every output and gradient within
max|diff| <= 2e-2 * rms(oracle) per tensor, with the oracle's routing taking
the kernel's choice only on near-ties (tests/_gpu.py forced_routing);
repeated calls bitwise identical."""
import numpy as np
import pytest
import torch

import oracle
from routing_dispatch_grouped_router_gb300 import api, inputs as gen

import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routing_dispatch_grouped_router_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


# ------------------------------------------------------------------ GEMM ---

@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 512, 320 - 64), (384, 384, 640)])
def test_engine_dense_gemm(a_mn, b_mn, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    A = gen.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    B = gen.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    ref = gen.bf16_bits_to_f32(A).astype(np.float64) @ gen.bf16_bits_to_f32(B).astype(np.float64).T
    At = _gpu.dev_bf16(np.ascontiguousarray(A.T) if a_mn else A)
    Bt = _gpu.dev_bf16(np.ascontiguousarray(B.T) if b_mn else B)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.gemm_bf16(At, a_mn, Bt, b_mn, C, ws)
    assert api.device_status(ws) == 0
    # the bf16 result is the nearest bf16 of the exact product, up to rare
    # one-ulp flips from fp32 accumulation
    _gpu.check_bf16_intermediate(_gpu.host64(C), oracle.bf16_round(ref), "C")


# ------------------------------------------------------------ full layer ---

SMALL = {
    "tiny": gen.Shape(T=256, d=128, E=8, I=256, k=2),
    "ragged": gen.Shape(T=300, d=128, E=5, I=128, k=2),
    "k1_I384": gen.Shape(T=200, d=256, E=4, I=384, k=1),
    "k_eq_E": gen.Shape(T=64, d=128, E=4, I=128, k=4),
    "d384": gen.Shape(T=130, d=384, E=6, I=256, k=3),
    "one_token": gen.Shape(T=1, d=128, E=8, I=128, k=8),
    "many_experts": gen.Shape(T=64, d=128, E=128, I=128, k=8),
    "wide": gen.Shape(T=512, d=512, E=16, I=512, k=4),
    # the widest rows the layer takes: 32 KB per token row, so the dispatch
    # runs one CTA per SM with six row slots
    "d16384": gen.Shape(T=64, d=16384, E=4, I=128, k=2),
    # E > 128: the router-weight gradient GEMM has two 128-row M tiles (E padded
    # to 256), several token chunks and a ragged last chunk
    "e200": gen.Shape(T=300, d=256, E=200, I=128, k=2),
    # d >= 6144 with 256-wide down-dgrad tiles: the SwiGLU backward stores
    # from registers (long K loop, five operand stages)
    "d7168": gen.Shape(T=256, d=7168, E=4, I=512, k=2),
    # d a multiple of 32 but not of 128: ragged K blocks (zero-filled) and
    # ragged N and M tiles (unstored chunks) wherever d is a GEMM dimension
    "d160": gen.Shape(T=300, d=160, E=5, I=128, k=2),
    "d2880": gen.Shape(T=128, d=2880, E=4, I=256, k=2),
    # I a multiple of 32 but not of 128: a ragged last gate/up tile (FFN
    # columns past I unstored), ragged down-dgrad tiles (no outputs, no dp),
    # ragged K blocks in the down projection and the gate/up dgrad, ragged M
    # tiles in the weight gradients
    "i160": gen.Shape(T=200, d=256, E=4, I=160, k=2),
    "d160_i224": gen.Shape(T=150, d=160, E=6, I=224, k=3),
    "d2880_i2880": gen.Shape(T=64, d=2880, E=4, I=2880, k=2),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_parity_small(name):
    shape = SMALL[name]
    inp = gen.make_inputs(shape, seed=0)
    gpu = _gpu.run_gpu(shape, inp)
    _gpu.full_parity(shape, inp, gpu)


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_layer_parity_tiny_seeds(seed):
    shape = gen.workload_shape("tiny")
    inp = gen.make_inputs(shape, seed=seed)
    _gpu.full_parity(shape, inp, _gpu.run_gpu(shape, inp))


def test_layer_parity_empty_expert():
    shape = gen.Shape(T=128, d=128, E=8, I=128, k=2)
    inp = gen.make_inputs(shape, seed=5)
    inp["bias"] = np.zeros(8, dtype=np.float32)
    inp["bias"][2] = -1e4
    gpu = _gpu.run_gpu(shape, inp)
    assert gpu["counts"][2] == 0
    _gpu.full_parity(shape, inp, gpu)
    assert (_gpu.host64(gpu["dw_gate_up"])[2] == 0).all()


def test_layer_zero_tokens():
    shape = gen.Shape(T=0, d=128, E=4, I=128, k=2)
    layer = api.MoELayer(0, 128, 4, 128, 2)
    wr = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    wgu = torch.ones(4, 256, 128, dtype=torch.bfloat16, device="cuda")
    wd = torch.ones(4, 128, 128, dtype=torch.bfloat16, device="cuda")
    x = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    y = layer.forward(x, wr, None, wgu, wd)
    dx, dwr, dwgu, dwd = layer.backward(x, x, wr, None, wgu, wd)
    assert layer.status() == 0
    assert y.numel() == 0 and dx.numel() == 0
    assert (dwgu == 0).all() and (dwd == 0).all() and (dwr == 0).all()


@pytest.mark.parametrize("dtype", [api.MXFP8, api.NVFP4])
def test_layer_zero_tokens_block_scaled(dtype):
    """No tokens in the block-scaled modes: the weights are still quantised
    (and their backward forms written), every GEMM has no rows, and the
    weight gradients come out zero."""
    layer = api.MoELayer(0, 256, 4, 256, 2, dtype=dtype)
    wr = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
    wgu = torch.ones(4, 512, 256, dtype=torch.bfloat16, device="cuda")
    wd = torch.ones(4, 256, 256, dtype=torch.bfloat16, device="cuda")
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    y = layer.forward(x, wr, None, wgu, wd)
    dx, dwr, dwgu, dwd = layer.backward(x, x, wr, None, wgu, wd)
    assert layer.status() == 0
    assert y.numel() == 0 and dx.numel() == 0
    assert (dwgu == 0).all() and (dwd == 0).all() and (dwr == 0).all()


def test_layer_parity_fine_full_size():
    """The fine-grained workload at its full size, every element."""
    shape = gen.workload_shape("fine")
    inp = gen.make_inputs(shape, seed=0)
    gpu = _gpu.run_gpu(shape, inp)
    errs = _gpu.full_parity(shape, inp, gpu)
    print("fine errs", errs)


def test_nan_token_reports_status_and_leaves_other_tokens_finite():
    """A NaN in one token's hidden state makes its router logits NaN: the
    router treats them as -inf (so the token takes experts 0..k-1 with equal
    weights), reports MOK_ERR_DEVICE_NONFINITE, and every other token keeps
    its routing and finite outputs."""
    shape = SMALL["wide"]
    inp = gen.make_inputs(shape, seed=3)
    clean = _gpu.run_gpu(shape, inp)
    assert clean["status"] == 0
    x = inp["x"].copy()
    x[5, 17] = 0x7FC0  # bf16 quiet NaN
    bad = _gpu.run_gpu(shape, dict(inp, x=x))
    assert bad["status"] == 16
    assert list(bad["topk_idx"][5]) == list(range(shape.k))
    np.testing.assert_allclose(bad["topk_w"][5], 1.0 / shape.k, rtol=1e-6)
    others = np.arange(shape.T) != 5
    assert np.array_equal(bad["topk_idx"][others], clean["topk_idx"][others])
    for n in ("y", "dx"):
        got = _gpu.host64(bad[n])[others]
        assert np.isfinite(got).all(), n
        assert _gpu.rel_err(got, _gpu.host64(clean[n])[others]) <= 1e-6, n


@pytest.mark.parametrize("name", ["tiny", "fine"])
def test_bitwise_deterministic(name):
    shape = gen.workload_shape(name)
    inp = gen.make_inputs(shape, seed=0)
    layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k)
    first = None
    for _ in range(10):
        g = _gpu.run_gpu(shape, inp, layer=layer)
        cur = [g[n].view(torch.int32).cpu().numpy().copy() for n in
               ("y", "dx", "dw_router", "dw_gate_up", "dw_down")]
        cur.append(g["topk_idx"].copy())
        if first is None:
            first = cur
        else:
            for a, b in zip(first, cur):
                assert np.array_equal(a, b)


@pytest.mark.parametrize("name,single", [("wide", False), ("wide", True), ("d384", False),
                                         ("ragged", False)])
def test_bf16_output_flags_round_the_fp32_outputs(name, single):
    """With the bf16-output flags every output is the round-to-nearest-even
    of the default fp32 output, bit for bit.  The weight gradients' bf16 TMA
    stores: row-major and transposed (d % 256 == 0), row-major only (d384,
    ragged), on CTA pairs and on single CTAs."""
    shape = SMALL[name]
    inp = gen.make_inputs(shape, seed=1)
    extra = api.FLAG_SINGLE_CTA_GEMM if single else 0
    a = _gpu.run_gpu(shape, inp, flags=extra)
    b = _gpu.run_gpu(shape, inp,
                     flags=api.FLAG_BF16_ACT_OUT | api.FLAG_BF16_WGRAD_OUT | extra)
    assert b["status"] == 0
    for n in ("y", "dx", "dw_router", "dw_gate_up", "dw_down"):
        assert a[n].dtype == torch.float32 and b[n].dtype == torch.bfloat16
        assert torch.equal(a[n].to(torch.bfloat16).view(torch.int16), b[n].view(torch.int16)), n


@pytest.mark.parametrize("shape,dtype,mb", [
    # one 128-row tile per expert: every pair's odd CTA stages rows it never stores
    (gen.Shape(T=256, d=256, E=4, I=256, k=2), 0, 0),
    # 2-3 tiles per expert (odd and even counts), wider N and K
    (gen.Shape(T=1024, d=512, E=16, I=512, k=4), 0, 0),
    (gen.Shape(T=1024, d=512, E=16, I=512, k=4), 1, 256),
])
def test_pair_and_single_cta_engines_agree_bitwise(shape, dtype, mb):
    """256-row tiles on CTA pairs (tcgen05.mma.cta_group::2) and 128-row
    tiles on single CTAs accumulate every element over the same K sequence."""
    inp = gen.make_inputs(shape, seed=6)
    outs = []
    for flags in (0, api.FLAG_SINGLE_CTA_GEMM):
        g = _gpu.run_gpu(shape, inp, flags=flags, dtype=dtype, mb_tokens=mb,
                         ring_slots=2 if mb else 0)
        assert g["status"] == 0
        outs.append([g[n].view(torch.int32).cpu().numpy() for n in
                     ("y", "dx", "dw_router", "dw_gate_up", "dw_down")])
    for n, a, b in zip(("y", "dx", "dw_router", "dw_gate_up", "dw_down"), *outs):
        assert np.array_equal(a, b), n


@pytest.mark.parametrize("dtype,mb,ring", [(0, 0, 0), (0, 256, 1), (1, 256, 2)])
def test_recompute_gate_up_is_bitwise_identical(dtype, mb, ring):
    """The backward's recomputed g, u equal the ones the forward would have
    kept, so every output is bitwise the same as without the flag."""
    shape = gen.Shape(T=1024, d=256, E=8, I=256, k=2)
    inp = gen.make_inputs(shape, seed=5)
    outs = []
    for flags in (0, api.FLAG_RECOMPUTE_GATE_UP):
        g = _gpu.run_gpu(shape, inp, flags=flags, dtype=dtype, mb_tokens=mb, ring_slots=ring)
        assert g["status"] == 0
        assert (g["gate_up"] is None) == bool(flags)
        outs.append([g[n].view(torch.int32).cpu().numpy() for n in
                     ("y", "dx", "dw_router", "dw_gate_up", "dw_down")])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("flags,mb,ring", [
    (0x20, 0, 0),          # dispatch recompute, one pass
    (0x20, 256, 1),        # micro-batches through a 1-slot ring
    (0x20 | 0x8, 0, 0),    # with the gate/up recompute too
])
def test_recompute_dispatch_is_bitwise_identical(flags, mb, ring):
    """The backward's second dispatch of x gives the rows the forward's gave,
    so every output is bitwise the same as with the rows kept in `saved`."""
    shape = gen.Shape(T=1024, d=256, E=8, I=256, k=2)
    inp = gen.make_inputs(shape, seed=7)
    outs = []
    for f in (0, flags):
        g = _gpu.run_gpu(shape, inp, flags=f, mb_tokens=mb, ring_slots=ring)
        assert g["status"] == 0
        assert (g["layer"].layout.x_perm == api.NOT_KEPT) == bool(f & api.FLAG_RECOMPUTE_DISPATCH)
        outs.append([g[n].view(torch.int32).cpu().numpy() for n in
                     ("y", "dx", "dw_router", "dw_gate_up", "dw_down")])
    for n, a, b in zip(("y", "dx", "dw_router", "dw_gate_up", "dw_down"), *outs):
        assert np.array_equal(a, b), n


def test_recompute_dispatch_parity():
    shape = SMALL["wide"]
    inp = gen.make_inputs(shape, seed=4)
    gpu = _gpu.run_gpu(shape, inp, flags=api.FLAG_RECOMPUTE_DISPATCH)
    _gpu.full_parity(shape, inp, gpu)


def test_recompute_gate_up_parity():
    shape = SMALL["wide"]
    inp = gen.make_inputs(shape, seed=1)
    gpu = _gpu.run_gpu(shape, inp, flags=api.FLAG_RECOMPUTE_GATE_UP)
    _gpu.full_parity(shape, inp, gpu)


def test_accumulate_wgrad_flag_adds_into_the_gradients():
    shape = SMALL["wide"]
    inp = gen.make_inputs(shape, seed=2)
    a = _gpu.run_gpu(shape, inp)
    layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k,
                         flags=api.FLAG_ACCUMULATE_WGRAD)
    x, wr, wgu, wd, dy = (_gpu.dev_bf16(inp[n]) for n in ("x", "w_router", "w_gate_up", "w_down",
                                                          "dy"))
    dws = [torch.zeros(t.shape, dtype=torch.float32, device="cuda") for t in (wr, wgu, wd)]
    for _ in range(2):
        layer.forward(x, wr, None, wgu, wd)
        layer.backward(dy, x, wr, None, wgu, wd, dw_router=dws[0], dw_gate_up=dws[1],
                       dw_down=dws[2])
    assert layer.status() == 0
    for got, one in zip(dws, (a["dw_router"], a["dw_gate_up"], a["dw_down"])):
        assert torch.equal(got, 2 * one)


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing completes ends with MOK_ERR_DEVICE_TIMEOUT in the
    status word (no hang, no trap), and the next call runs normally."""
    from routing_dispatch_grouped_router_gb300 import _lib
    import ctypes
    lib = _lib.load()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    code = lib.mok_selftest_bounded_wait(ctypes.c_void_p(ws.data_ptr()), 256,
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    assert api.device_status(ws) == 18  # MOK_ERR_DEVICE_TIMEOUT
    shape = SMALL["tiny"]
    inp = gen.make_inputs(shape, seed=0)
    _gpu.full_parity(shape, inp, _gpu.run_gpu(shape, inp))


@pytest.mark.parametrize("offset,nbytes", [(0, 0), (16, 48), (0, 16384), (32, 3 * 16384 + 4080),
                                           (16, (64 << 20) + 16)])
def test_fill_zero_writes_exactly_its_range(offset, nbytes):
    """The bulk-store fill zeroes whole chunks, the ragged tail and nothing
    outside [dst, dst + bytes)."""
    buf = torch.full((offset + nbytes + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    api.fill_zero(buf[offset:offset + nbytes])
    torch.cuda.synchronize()
    h = buf.cpu().numpy()
    assert not h[offset:offset + nbytes].any()
    assert (h[:offset] == 0xA5).all() and (h[offset + nbytes:] == 0xA5).all()


def test_fill_zero_rejects_unaligned_arguments():
    from routing_dispatch_grouped_router_gb300 import _lib
    import ctypes
    lib = _lib.load()
    buf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.mok_fill_zero(ctypes.c_void_p(buf.data_ptr() + 8), 64, st) != 0
    assert lib.mok_fill_zero(ctypes.c_void_p(buf.data_ptr()), 40, st) != 0


# ------------------------------------------------------------ stage APIs ---

def test_route_stage_matches_oracle():
    shape = gen.workload_shape("fine")
    inp = gen.make_inputs(shape, seed=3)
    desc = api.make_desc(shape.T, shape.d, shape.E, shape.I, shape.k)
    ws = torch.zeros(api.stage_workspace_size(desc), dtype=torch.uint8, device="cuda")
    idx = torch.empty(shape.T, shape.k, dtype=torch.int32, device="cuda")
    w = torch.empty(shape.T, shape.k, dtype=torch.float32, device="cuda")
    api.route(desc, _gpu.dev_bf16(inp["x"]), _gpu.dev_bf16(inp["w_router"]), None, idx, w, ws)
    assert api.device_status(ws) == 0
    ridx, rp, _, flagged, inner = oracle.route_ref(inp["x"], inp["w_router"], None, shape.k)
    _gpu.check_routing(idx.cpu().numpy(), w.cpu().numpy(), ridx, rp, flagged, inner)


@pytest.mark.parametrize("T,E,k", [(1000, 7, 3), (4096, 64, 8), (513, 512, 8), (5, 3, 3)])
def test_dispatch_plan_stage_bit_exact(T, E, k):
    rng = np.random.default_rng(T + E + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    desc = api.make_desc(T, 128, E, 128, k)
    ws = torch.zeros(api.stage_workspace_size(desc), dtype=torch.uint8, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty(T, k, dtype=torch.int32, device="cuda")
    tok = torch.empty(T * k, dtype=torch.int32, device="cuda")
    api.dispatch_plan(desc, torch.from_numpy(idx).cuda(), counts, offsets, pos, tok, ws)
    assert api.device_status(ws) == 0
    c, o, p, t = oracle.dispatch_ref(idx, E)
    assert np.array_equal(counts.cpu().numpy(), c)
    assert np.array_equal(offsets.cpu().numpy(), o)
    assert np.array_equal(pos.cpu().numpy(), p)
    assert np.array_equal(tok.cpu().numpy(), t)


@pytest.mark.parametrize("name", ["tiny", "ragged", "one_token", "many_experts", "e200", "fine"])
def test_fused_front_end_matches_the_stage_kernels(name):
    """The forward runs the router's top-k and the dispatch plan as one
    persistent kernel walking a schedule table; the stage entry points run
    them as four kernels (top-k, histogram, scan, placement).  Same inputs,
    bitwise the same routing weights and plan."""
    shape = SMALL.get(name) or gen.workload_shape(name)
    inp = gen.make_inputs(shape, seed=2)
    layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k)
    x, wr, wgu, wd = (_gpu.dev_bf16(inp[n]) for n in ("x", "w_router", "w_gate_up", "w_down"))
    layer.forward(x, wr, None, wgu, wd)
    assert layer.status() == 0
    T, k, E = shape.T, shape.k, shape.E
    desc = api.make_desc(T, shape.d, E, shape.I, k)
    ws = torch.zeros(api.stage_workspace_size(desc), dtype=torch.uint8, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    api.route(desc, x, wr, None, idx, w, ws)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty(T, k, dtype=torch.int32, device="cuda")
    tok = torch.empty(T * k, dtype=torch.int32, device="cuda")
    api.dispatch_plan(desc, idx, counts, offsets, pos, tok, ws)
    assert api.device_status(ws) == 0
    fused = {n: layer.saved_tensor(n, dt, shp) for n, dt, shp in (
        ("topk_idx", torch.int32, (T, k)), ("topk_w", torch.int32, (T, k)),
        ("counts", torch.int32, (E,)), ("offsets", torch.int32, (E + 1,)),
        ("pos", torch.int32, (T, k)), ("token_of_row", torch.int32, (T * k,)))}
    stages = dict(topk_idx=idx, topk_w=w.view(torch.int32), counts=counts, offsets=offsets,
                  pos=pos, token_of_row=tok)
    for n in stages:
        assert torch.equal(fused[n], stages[n]), n


def test_dispatch_plan_flags_bad_indices():
    T, E, k = 40, 6, 2
    rng = np.random.default_rng(0)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[3, 1] = 6        # out of range
    idx[7, 1] = idx[7, 0]  # repeated
    desc = api.make_desc(T, 128, E, 128, k)
    ws = torch.zeros(api.stage_workspace_size(desc), dtype=torch.uint8, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty(T, k, dtype=torch.int32, device="cuda")
    tok = torch.empty(T * k, dtype=torch.int32, device="cuda")
    api.dispatch_plan(desc, torch.from_numpy(idx).cuda(), counts, offsets, pos, tok, ws)
    assert api.device_status(ws) == 17
    p = pos.cpu().numpy()
    assert p[3, 1] == -1 and p[7, 1] == -1
    assert counts.cpu().numpy().sum() == T * k - 2


# --------------------------------------------------- micro-batches, MXFP8 ---

@pytest.mark.parametrize("ring", [0, 1, 2])
def test_layer_micro_batched_bf16(ring):
    """Four micro-batches of 256 tokens through a ring of `ring` slots
    (0 = one per micro-batch; 1 and 2 re-dispatch evicted slots in backward)."""
    shape = gen.Shape(T=1024, d=256, E=8, I=256, k=2)
    inp = gen.make_inputs(shape, seed=2)
    gpu = _gpu.run_gpu(shape, inp, mb_tokens=256, ring_slots=ring)
    assert gpu["nmb"] == 4
    _gpu.full_parity(shape, inp, gpu)


@pytest.mark.parametrize("name", ["tiny", "wide", "k1_I384", "d16384"])
def test_layer_parity_mxfp8(name):
    shape = SMALL[name]
    inp = gen.make_inputs(shape, seed=0)
    gpu = _gpu.run_gpu(shape, inp, dtype=api.MXFP8, flags=api.FLAG_BF16_ACT_OUT)
    errs = _gpu.full_parity(shape, inp, gpu, tol=_gpu.MX_TOL, precision="mxfp8")
    print(name, errs)


def test_layer_micro_batched_mxfp8():
    shape = gen.Shape(T=1024, d=512, E=16, I=512, k=4)
    inp = gen.make_inputs(shape, seed=3)
    gpu = _gpu.run_gpu(shape, inp, dtype=api.MXFP8, flags=api.FLAG_BF16_ACT_OUT, mb_tokens=256,
                       ring_slots=2)
    errs = _gpu.full_parity(shape, inp, gpu, tol=_gpu.MX_TOL, precision="mxfp8")
    print(errs)


@pytest.mark.parametrize("dtype", [0, 1])
def test_micro_batched_deterministic(dtype):
    shape = gen.Shape(T=1024, d=256, E=8, I=256, k=2)
    inp = gen.make_inputs(shape, seed=4)
    layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k, dtype=dtype,
                         mb_tokens=256, ring_slots=2)
    outs = []
    for _ in range(3):
        g = _gpu.run_gpu(shape, inp, layer=layer)
        outs.append([g[n].view(torch.int32).cpu().numpy().copy() for n in
                     ("y", "dx", "dw_router", "dw_gate_up", "dw_down")])
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
    for a, b in zip(outs[0], outs[2]):
        assert np.array_equal(a, b)


# ------------------------------------------------------------------ MXFP8 ---

@pytest.mark.parametrize("along_rows", [False, True])
@pytest.mark.parametrize("shape", [(96, 160), (352, 1056)])
def test_mx_quantize_bit_exact(along_rows, shape):
    """(352, 1056): the column quantiser's 32 x 256 tiles, eleven row blocks by
    five column tiles, the last 32 columns wide."""
    rows, cols = shape
    rng = np.random.default_rng(7)
    a = rng.standard_normal((rows, cols)).astype(np.float32) * np.exp(
        rng.uniform(-30, 30, (rows, 1)).astype(np.float32))
    a[5, :32] = 0.0
    a[:32, 7] = 0.0
    bits = gen.f32_to_bf16_bits(a)
    x = _gpu.dev_bf16(bits)
    codes = torch.empty(a.shape, dtype=torch.uint8, device="cuda")
    nsc = (rows // 32, cols) if along_rows else (rows, cols // 32)
    scales = torch.empty(nsc, dtype=torch.uint8, device="cuda")
    out = api.mx_quantize(x, along_rows, codes=codes, scales=scales)
    ref, shared = oracle.mx_quantize(gen.bf16_bits_to_f32(bits).astype(np.float64),
                                     axis=0 if along_rows else 1)
    assert np.array_equal(_gpu.host64(out), ref)
    # the oracle lists the blocks of a column along its last axis
    shared = shared.T if along_rows else shared
    assert np.array_equal(scales.cpu().numpy().astype(np.int64), shared + 127)
    # codes decode (sign, exponent bias 7, 3 mantissa bits) to ref / 2^shared
    c = codes.cpu().numpy().astype(np.int64)
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    mag = np.where(e > 0, 2.0 ** (e - 7) * (1 + m / 8), 2.0 ** -6 * (m / 8))
    sh = np.repeat(shared, 32, axis=0) if along_rows else np.repeat(shared, 32, axis=1)
    np.testing.assert_array_equal(np.where(s == 1, -mag, mag) * 2.0 ** sh, ref)


@pytest.mark.parametrize("dtype", [api.BF16, api.MXFP8, api.NVFP4])
def test_layer_step_replays_in_a_cuda_graph(dtype):
    """Forward + backward enqueue only stream-ordered work (no allocation, no
    host read-back), so a whole step can be captured in a CUDA graph; replays
    give the eager results bit for bit."""
    shape = SMALL["wide"]
    inp = gen.make_inputs(shape, seed=4)
    eager = _gpu.run_gpu(shape, inp, dtype=dtype)
    assert eager["status"] == 0
    layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k, dtype=dtype)
    x, wr, wgu, wd, dy = (_gpu.dev_bf16(inp[n]) for n in ("x", "w_router", "w_gate_up", "w_down",
                                                          "dy"))
    f32 = dict(dtype=torch.float32, device="cuda")
    y, dx = torch.empty(x.shape, **f32), torch.empty(x.shape, **f32)
    dws = [torch.empty(t.shape, **f32) for t in (wr, wgu, wd)]

    def step():
        layer.forward(x, wr, None, wgu, wd, y=y)
        layer.backward(dy, x, wr, None, wgu, wd, dx=dx, dw_router=dws[0], dw_gate_up=dws[1],
                       dw_down=dws[2])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # first calls outside the capture (kernel attributes, descriptors)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in [y, dx] + dws:
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert layer.status() == 0
    for got, n in zip([y, dx] + dws, ("y", "dx", "dw_router", "dw_gate_up", "dw_down")):
        assert torch.equal(got, eager[n]), n


def test_expert_relabelling_equivariance_fine():
    """Relabelling the experts (their router rows, bias entries and weights
    permuted together) leaves y and dx bitwise unchanged and permutes the
    weight gradients, bit for bit: each expert's GEMMs see the same rows in the
    same order wherever the expert sits, and the combine and the reverse
    dispatch add the slots in logit order, not expert order."""
    shape = gen.workload_shape("fine")
    inp = gen.make_inputs(shape, seed=8)
    perm = np.random.default_rng(8).permutation(shape.E)
    relabelled = dict(inp)
    for n in ("w_router", "w_gate_up", "w_down"):
        relabelled[n] = np.ascontiguousarray(inp[n][perm])
    if inp.get("bias") is not None:
        relabelled["bias"] = np.ascontiguousarray(inp["bias"][perm])
    a = _gpu.run_gpu(shape, inp)
    b = _gpu.run_gpu(shape, relabelled)
    assert a["status"] == 0 and b["status"] == 0
    # expert i of the second run is expert perm[i] of the first
    assert np.array_equal(perm[b["topk_idx"]], a["topk_idx"])
    for n in ("y", "dx"):
        assert torch.equal(b[n].view(torch.int32), a[n].view(torch.int32)), n
    p = torch.from_numpy(perm).cuda()
    for n in ("dw_router", "dw_gate_up", "dw_down"):
        assert torch.equal(b[n].view(torch.int32), a[n][p].view(torch.int32)), n


@pytest.mark.parametrize("mode", ["single_cta", "micro_batched", "recompute"])
def test_ragged_widths_in_every_layer_mode(mode):
    """Ragged d and I (multiples of 32, not of the tiles) through the other
    kernel paths: single-CTA tiles, micro-batches with deferred weight
    gradients over a two-slot ring, and the recompute flags."""
    shape = gen.Shape(T=150, d=160, E=6, I=224, k=3)
    inp = gen.make_inputs(shape, seed=12)
    kw = {"single_cta": dict(flags=api.FLAG_SINGLE_CTA_GEMM),
          "micro_batched": dict(mb_tokens=50, ring_slots=2),
          "recompute": dict(flags=api.FLAG_RECOMPUTE_GATE_UP | api.FLAG_RECOMPUTE_DISPATCH)}[mode]
    gpu = _gpu.run_gpu(shape, inp, **kw)
    assert gpu["status"] == 0
    _gpu.full_parity(shape, inp, gpu)


# ------------------------------------------- padding rows that nothing reads ---

@pytest.mark.parametrize("T,mb,ring", [(480, 0, 0), (640, 160, 1)])
def test_unread_padding_rows_reach_no_output(T, mb, ring):
    """Rows of an expert's segment past its real rows rounded up to 64 (the
    plan's token -2 rows) are read only by whole-tile GEMMs, for output rows
    that nothing reads: the dispatch leaves them unwritten and the grouped
    GEMMs skip their epilogue there.  With the dispatched x rows and the saved
    fp32 g, u filled with NaN before the call instead of zeros, every output is
    bitwise the same.  (About 160 and 53 rows per expert: 64 such rows each.)"""
    shape = gen.Shape(T=T, d=256, E=6, I=256, k=2)
    inp = gen.make_inputs(shape, seed=7)
    outs = []
    for poison in (False, True):
        layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k, mb_tokens=mb,
                             ring_slots=ring)
        L = layer.layout
        nmb = int(L.mb_count)
        if poison:
            # only float row arrays: NaN bytes (0xFF) in bf16 and fp32
            rows = int(L.rows_max)
            for s in range(max(int(L.ring_slots), 1)):
                off = int(L.x_perm) + s * int(L.ring_slot_bytes)
                layer.saved[off:off + rows * shape.d * 2].fill_(0xFF)
            for i in range(nmb):
                off = int(L.gate_up) + i * int(L.mb_stride)
                layer.saved[off:off + rows * 2 * shape.I * 4].fill_(0xFF)
        gpu = _gpu.run_gpu(shape, inp, layer=layer)
        assert gpu["status"] == 0
        counts = np.concatenate(gpu["mb_counts"])
        assert ((counts % 128 >= 1) & (counts % 128 <= 64)).any()  # such rows exist
        outs.append([gpu[n].clone() for n in ("y", "dx", "dw_router", "dw_gate_up", "dw_down")])
    for a, b in zip(*outs):
        assert torch.equal(a, b)
