"""Block-scaled MXFP8 GEMM (tcgen05.mma.kind::mxf8f6f4) through the C ABI,
against the oracle's MX quantiser and an fp64 product of the dequantised
operands.  The crafted cases put all-ones codes under scales that vary by
row, by column and by 32-wide K block, so a mistake in where the hardware
finds a scale byte shows up as a wrong entry."""
import numpy as np
import pytest
import torch

import oracle
from routing_dispatch_grouped_router_gb300 import api
from routing_dispatch_grouped_router_gb300 import inputs as gen

import _gpu

pytestmark = pytest.mark.gpu

E4M3_ONE = 0x38  # sign 0, exponent 7 (bias 7), mantissa 0


def _run(codes_a, sc_a, codes_b, sc_b, pair=False):
    M, K = codes_a.shape
    N = codes_b.shape[0]
    dev = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (codes_a, sc_a, codes_b, sc_b)]
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.gemm_mxfp8(*dev, C, ws, cta_pair=pair)
    assert api.device_status(ws) == 0
    return C.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("pattern", ["rows", "cols", "kblocks", "mixed"])
def test_mxfp8_gemm_scale_placement(pattern, pair):
    M, N, K = 256, 256, 512
    kb = K // 32
    rng = np.random.default_rng(11)
    sa = np.full((M, kb), 127, np.uint8)
    sb = np.full((N, kb), 127, np.uint8)
    if pattern == "rows":
        sa[:] = (120 + np.arange(M) % 13)[:, None]
    elif pattern == "cols":
        sb[:] = (118 + np.arange(N) % 17)[:, None]
    elif pattern == "kblocks":
        sa[:] = 121 + np.arange(kb)[None, :] % 11
        sb[:] = 124 + (np.arange(kb)[None, :] * 5) % 7
    else:
        sa = rng.integers(115, 135, (M, kb)).astype(np.uint8)
        sb = rng.integers(115, 135, (N, kb)).astype(np.uint8)
    ca = np.full((M, K), E4M3_ONE, np.uint8)
    cb = np.full((N, K), E4M3_ONE, np.uint8)
    got = _run(ca, sa, cb, sb, pair)
    ref = 32.0 * (2.0 ** (sa.astype(np.float64) - 127)) @ (2.0 ** (sb.astype(np.float64) - 127)).T
    # every term is positive, so fp32 accumulation of the K/32 block sums is
    # within (K/32) * 2^-24 * ref (plus rounding slack); a scale byte read from
    # the wrong row, column or K block changes a term by a factor of 2 or more
    np.testing.assert_allclose(got, ref, rtol=2e-5, atol=0)


@pytest.mark.parametrize("M,N,K,pair", [(128, 128, 128, False), (256, 384, 1024, False),
                                        (512, 256, 2048, False), (256, 256, 128, True),
                                        (512, 768, 1024, True)])
def test_mxfp8_gemm_matches_dequantised_product(M, N, K, pair):
    rng = np.random.default_rng(M + N + K)
    a = rng.standard_normal((M, K)).astype(np.float32) * np.exp(rng.uniform(-3, 3, (M, 1)))
    b = rng.standard_normal((N, K)).astype(np.float32) * np.exp(rng.uniform(-3, 3, (N, 1)))
    out = {}
    for name, v in (("a", a), ("b", b)):
        bits = gen.f32_to_bf16_bits(v.astype(np.float32))
        x = _gpu.dev_bf16(bits)
        codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        scales = torch.empty(x.shape[0], x.shape[1] // 32, dtype=torch.uint8, device="cuda")
        api.mx_quantize(x, False, codes=codes, scales=scales)
        deq, _ = oracle.mx_quantize(gen.bf16_bits_to_f32(bits).astype(np.float64), axis=1)
        out[name] = (codes.cpu().numpy(), scales.cpu().numpy(), deq)
    got = _run(out["a"][0], out["a"][1], out["b"][0], out["b"][1], pair)
    ref = out["a"][2] @ out["b"][2].T
    scale = np.abs(out["a"][2]) @ np.abs(out["b"][2]).T
    # fp32 accumulation: each entry within a few ulps of its absolute sum
    assert np.all(np.abs(got - ref) <= 4e-6 * scale + 1e-30)
