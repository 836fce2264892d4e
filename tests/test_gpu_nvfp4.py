"""NVFP4 (E2M1 elements, E4M3 scale per 16 values, fp32 tensor scale) through
the C ABI: the quantiser bit for bit against the oracle's, and the dense GEMM
on the block-scaled FP4 tensor cores (tcgen05.mma.kind::mxf4nvf4) against an
fp64 product of the dequantised operands.  The crafted GEMM cases put
all-ones codes under block scales that vary by row, by column and by 16-wide
K block, so a scale byte read from the wrong place shows up as a wrong
entry."""
import numpy as np
import pytest
import torch

import oracle
from oracle import nvfp4_ref
from routing_dispatch_grouped_router_gb300 import api
from routing_dispatch_grouped_router_gb300 import inputs as gen

import _gpu

pytestmark = pytest.mark.gpu

E2M1_ONE = 0x2        # sign 0, exponent 1 (bias 1), mantissa 0
E2M1_ONES = E2M1_ONE | (E2M1_ONE << 4)


def _decode_e2m1(codes):
    """Packed codes [rows, n/2] -> values [rows, n] (low nibble first)."""
    lo, hi = codes & 15, codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1).astype(np.int64)
    s, e, m = c >> 3, (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, 2.0 ** (e - 1) * (1 + m / 2))
    return np.where(s == 1, -mag, mag)


def _decode_e4m3(b):
    b = b.astype(np.int64)
    e, m = (b >> 3) & 15, b & 7
    return np.where(e == 0, m * 2.0 ** -9, 2.0 ** (e - 7) * (1 + m / 8))


def _quantize(bits):
    x = _gpu.dev_bf16(bits)
    g = api.nvfp4_tensor_scale(x)
    codes, scales = api.nvfp4_quantize(x, g)
    return g, codes, scales


@pytest.mark.parametrize("shape", [(96, 256), (160, 1088)])
def test_nvfp4_quantize_bit_exact(shape):
    rows, cols = shape
    rng = np.random.default_rng(rows + cols)
    a = rng.standard_normal(shape).astype(np.float32) * np.exp(
        rng.uniform(-12, 12, (rows, 1)).astype(np.float32))
    a[3, 16:32] = 0.0                       # an all-zero block
    a[7, :16] *= 1e-20                      # a block whose scale underflows to 0
    bits = gen.f32_to_bf16_bits(a)
    g, codes, scales = _quantize(bits)
    deq, q, sb, gr = nvfp4_ref.nvfp4_quantize(gen.bf16_bits_to_f32(bits).astype(np.float64), 1)
    assert np.float32(g.item()) == np.float32(gr)
    assert np.array_equal(_decode_e4m3(scales.cpu().numpy()), sb)
    assert np.array_equal(_decode_e2m1(codes.cpu().numpy()), q)
    assert (scales.cpu().numpy()[7, 0] == 0) and (codes.cpu().numpy()[7, :8] == 0).all()


@pytest.mark.parametrize("ng,K,C", [(1, 128, 128), (3, 256, 384)])
def test_nvfp4_quantize_cols_bit_exact(ng, K, C):
    """The column quantiser (blocks of 16 down each column of each stacked
    matrix) against the oracle's quantiser along K, bit for bit."""
    rng = np.random.default_rng(ng * K + C)
    a = rng.standard_normal((ng, K, C)).astype(np.float32) * np.exp(
        rng.uniform(-10, 10, (ng, 1, C)).astype(np.float32))
    a[0, 16:32, 5] = 0.0                    # an all-zero block
    a[-1, :16, 7] *= 1e-20                  # a block whose scale underflows to 0
    bits = gen.f32_to_bf16_bits(a)
    x = _gpu.dev_bf16(bits)
    g = api.nvfp4_tensor_scale(x)
    codes, scales = api.nvfp4_quantize_cols(x, g)
    vals = gen.bf16_bits_to_f32(bits).astype(np.float64)
    _, q, sb, gr = nvfp4_ref.nvfp4_quantize(vals, 1)     # along K, one tensor scale
    assert np.float32(g.item()) == np.float32(gr)
    got_q = _decode_e2m1(codes.cpu().numpy()).reshape(ng, C, K)
    got_s = _decode_e4m3(scales.cpu().numpy()).reshape(ng, C, K // 16)
    assert np.array_equal(got_s, sb)
    assert np.array_equal(got_q, q.transpose(0, 2, 1))
    assert got_s[0, 5, 1] == 0 and got_s[-1, 7, 0] == 0


def _gemm(ca, sa, ga, cb, sb, gb):
    dev = [torch.from_numpy(np.ascontiguousarray(v)).cuda() for v in (ca, sa, cb, sb)]
    gad = torch.tensor([ga], dtype=torch.float32, device="cuda")
    gbd = torch.tensor([gb], dtype=torch.float32, device="cuda")
    M, N = ca.shape[0], cb.shape[0]
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.gemm_nvfp4(dev[0], dev[1], gad, dev[2], dev[3], gbd, C, ws)
    assert api.device_status(ws) == 0
    return C.cpu().numpy().astype(np.float64)


def _e4m3_byte(v):
    """E4M3 bytes of exactly representable positive values."""
    v = np.asarray(v, dtype=np.float64)
    e = np.floor(np.log2(v)).astype(np.int64)
    m = np.round((v / 2.0 ** e - 1) * 8).astype(np.int64)
    return ((e + 7) << 3 | m).astype(np.uint8)


@pytest.mark.parametrize("pattern", ["rows", "cols", "kblocks", "mixed"])
def test_nvfp4_gemm_scale_placement(pattern):
    M, N, K = 256, 256, 512
    kb = K // 16
    rng = np.random.default_rng(12)
    vals = 2.0 ** np.arange(-4, 5)         # exact E4M3 scales 1/16 .. 16
    sa = np.ones((M, kb))
    sb = np.ones((N, kb))
    if pattern == "rows":
        sa[:] = vals[np.arange(M) % 9][:, None] * (1 + (np.arange(M) % 3)[:, None] / 8)
    elif pattern == "cols":
        sb[:] = vals[np.arange(N) % 9][:, None] * (1 + (np.arange(N) % 5)[:, None] / 8)
    elif pattern == "kblocks":
        sa[:] = vals[np.arange(kb) % 9][None, :]
        sb[:] = vals[(np.arange(kb) * 5) % 9][None, :] * 1.5
    else:
        sa = rng.choice(vals, (M, kb)) * rng.choice([1.0, 1.25, 1.5, 1.875], (M, kb))
        sb = rng.choice(vals, (N, kb)) * rng.choice([1.0, 1.125, 1.75], (N, kb))
    ca = np.full((M, K // 2), E2M1_ONES, np.uint8)
    cb = np.full((N, K // 2), E2M1_ONES, np.uint8)
    got = _gemm(ca, _e4m3_byte(sa), 1.0, cb, _e4m3_byte(sb), 0.5)
    ref = 0.5 * 16.0 * sa @ sb.T
    # every term is positive: fp32 accumulation stays within a few ulps
    np.testing.assert_allclose(got, ref, rtol=2e-5, atol=0)


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 1024), (384, 256, 2048)])
def test_nvfp4_gemm_matches_dequantised_product(M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = rng.standard_normal((M, K)).astype(np.float32) * np.exp(rng.uniform(-3, 3, (M, 1)))
    b = rng.standard_normal((N, K)).astype(np.float32) * np.exp(rng.uniform(-3, 3, (N, 1)))
    out = {}
    for name, v in (("a", a), ("b", b)):
        bits = gen.f32_to_bf16_bits(v.astype(np.float32))
        g, codes, scales = _quantize(bits)
        deq = nvfp4_ref.nvfp4_fake(gen.bf16_bits_to_f32(bits).astype(np.float64), 1)
        out[name] = (codes.cpu().numpy(), scales.cpu().numpy(), float(g.item()), deq)
    got = _gemm(out["a"][0], out["a"][1], out["a"][2], out["b"][0], out["b"][1], out["b"][2])
    ref = out["a"][3] @ out["b"][3].T
    scale = np.abs(out["a"][3]) @ np.abs(out["b"][3]).T
    # fp32 accumulation and the fp32 product of the two tensor scales
    assert np.all(np.abs(got - ref) <= 4e-6 * scale + 1e-30)


# ------------------------------------------------------------ the layer ---

NV_TOL = 6e-2  # as for MXFP8: E2M1 flips where the kernel's fp32 h and the
               # oracle's fp64 h fall on two sides of a rounding boundary

NV_SHAPES = {
    "small": gen.Shape(T=256, d=256, E=8, I=256, k=2),
    "ragged": gen.Shape(T=300, d=256, E=5, I=256, k=2),
    "wide": gen.Shape(T=512, d=512, E=16, I=512, k=4),
    "many_experts": gen.Shape(T=200, d=256, E=64, I=256, k=8),
}


@pytest.mark.parametrize("name", list(NV_SHAPES))
def test_layer_parity_nvfp4(name):
    """Forward expert GEMMs on NVFP4 operands, every output against the
    oracle's NVFP4 mode (the same quantisation of x, the weights and h; the
    float64 backward on the forward's g, u)."""
    shape = NV_SHAPES[name]
    inp = gen.make_inputs(shape, seed=0)
    gpu = _gpu.run_gpu(shape, inp, dtype=api.NVFP4)
    assert gpu["layer"].layout.x_perm == api.NOT_KEPT
    errs = _gpu.full_parity(shape, inp, gpu, tol=NV_TOL, precision="nvfp4")
    print(name, errs)


def test_layer_nvfp4_micro_batched_and_deterministic():
    shape = gen.Shape(T=1024, d=256, E=8, I=256, k=2)
    inp = gen.make_inputs(shape, seed=3)
    outs = []
    for _ in range(3):
        g = _gpu.run_gpu(shape, inp, dtype=api.NVFP4, mb_tokens=256, ring_slots=2)
        assert g["status"] == 0 and g["nmb"] == 4
        outs.append([g[n].view(torch.int32).cpu().numpy() for n in
                     ("y", "dx", "dw_router", "dw_gate_up", "dw_down")])
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
    for a, b in zip(outs[0], outs[2]):
        assert np.array_equal(a, b)
    print(_gpu.full_parity(shape, inp, g, tol=NV_TOL, precision="nvfp4"))


def test_layer_nvfp4_rejects_what_it_does_not_support():
    from routing_dispatch_grouped_router_gb300 import _lib
    import ctypes
    lib = _lib.load()
    f, s, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    for kw in (dict(d=128), dict(I=128), dict(flags=api.FLAG_SINGLE_CTA_GEMM),
               dict(flags=api.FLAG_RECOMPUTE_GATE_UP)):
        args = dict(T=64, d=256, E=4, I=256, k=2, dtype=api.NVFP4)
        args.update(kw)
        desc = api.make_desc(**args)
        assert lib.mok_moe_workspace_size(ctypes.byref(desc), ctypes.byref(f), ctypes.byref(s),
                                          ctypes.byref(b)) == 2


@pytest.mark.parametrize("dtype", [api.MXFP8, api.NVFP4])
def test_block_scaled_accumulate_and_bf16_outputs(dtype):
    """The output flags in the block-scaled modes: accumulating weight
    gradients over two calls gives exactly twice one call (the forward writes
    the same quantised weights again), and bf16 activations are the fp32 ones
    rounded once."""
    shape = NV_SHAPES["wide"]
    inp = gen.make_inputs(shape, seed=9)
    one = _gpu.run_gpu(shape, inp, dtype=dtype)
    x, wr, wgu, wd, dy = (_gpu.dev_bf16(inp[n]) for n in ("x", "w_router", "w_gate_up", "w_down",
                                                          "dy"))
    layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k, dtype=dtype,
                         flags=api.FLAG_ACCUMULATE_WGRAD)
    dws = [torch.zeros(t.shape, dtype=torch.float32, device="cuda") for t in (wr, wgu, wd)]
    for _ in range(2):
        layer.forward(x, wr, None, wgu, wd)
        layer.backward(dy, x, wr, None, wgu, wd, dw_router=dws[0], dw_gate_up=dws[1],
                       dw_down=dws[2])
    assert layer.status() == 0
    for got, ref in zip(dws, (one["dw_router"], one["dw_gate_up"], one["dw_down"])):
        assert torch.equal(got, 2 * ref)
    bf = _gpu.run_gpu(shape, inp, dtype=dtype, flags=api.FLAG_BF16_ACT_OUT)
    assert bf["status"] == 0
    for n in ("y", "dx"):
        assert torch.equal(bf[n], one[n].to(torch.bfloat16))
