"""bench.py's per-launch accounting: the algorithmic FLOP of each grouped GEMM
and the bytes of each data-movement kernel, with and without micro-batches."""
import pytest

import bench
from routing_dispatch_grouped_router_gb300 import inputs as gen


def test_gemm_flops_fine():
    s = gen.workload_shape("fine")
    f = bench.gemm_flops(s)
    R, d, I = s.T * s.k, s.d, s.I
    assert f["fwd_gate_up_swiglu"] == 2 * R * d * 2 * I == pytest.approx(274.9e9, rel=1e-3)
    assert f["fwd_down"] == f["bwd_down_dgrad_swiglu"] == f["bwd_down_wgrad"] == 2 * R * d * I
    assert f["bwd_gate_up_dgrad"] == f["bwd_gate_up_wgrad"] == 2 * R * d * 2 * I
    # the step's expert GEMMs: 18 R d I
    total = sum(v for n, v in f.items() if n != "router_logits")
    assert total == 18 * R * d * I


def test_micro_batches_divide_the_work_of_a_launch():
    s = gen.workload_shape("mxfp8")
    nmb = s.T // gen.WORKLOADS["mxfp8"]["mb_tokens"]
    whole, part = bench.gemm_flops(s), bench.gemm_flops(s, nmb)
    for n in whole:
        if n in bench.DEFERRED_WGRADS:  # one launch per step over all micro-batches
            assert part[n] == pytest.approx(whole[n])
        else:
            assert part[n] * nmb == pytest.approx(whole[n])
    mw, mp = bench.mover_bytes(s), bench.mover_bytes(s, nmb)
    for n in ("dispatch_rows", "combine"):
        assert mp[n] * nmb == pytest.approx(mw[n], rel=1e-9)


def test_mover_bytes_follow_the_fp32_row_layout():
    s = gen.workload_shape("fine")
    m = bench.mover_bytes(s)
    R, T, d = s.T * s.k, s.T, s.d
    assert m["combine"] == R * d * 4 + T * d * 4 + R * 8
    # unique bytes: x read once, R rows written
    assert m["dispatch_rows"] == T * d * 2 + R * d * 2 + R * 4


def test_workload_options():
    class FakeApi:
        MXFP8 = 1
        NVFP4 = 2
        FLAG_BF16_WGRAD_OUT = 2
    assert bench.WORKLOAD == "large"  # the default: the configuration the targets name
    assert bench.PRECISION == "bf16"

    def opts(workload, precision=None):
        bench.WORKLOAD = workload
        bench.PRECISION = precision or bench.workload_precision(workload)
        try:
            return (bench.layer_options(FakeApi),
                    bench.workload_config(gen.workload_shape(workload))["workload"])
        finally:
            bench.WORKLOAD, bench.PRECISION = "large", "bf16"
    o, cfg = opts("mxfp8")
    assert o == dict(dtype=1, mb_tokens=2048, ring_slots=2) and "MXFP8" in cfg
    # the same micro-batched ring at another precision
    o, cfg = opts("mxfp8", "bf16")
    assert o == dict(mb_tokens=2048, ring_slots=2)
    assert "8 micro-batches of 2048 tokens" in cfg and "at this precision" in cfg
    o, cfg = opts("nvfp4")
    assert o == dict(dtype=2) and "NVFP4" in cfg
    o, cfg = opts("large")
    assert o == {} and cfg.startswith("large: T=8192 d=7168 E=384 I=2048 top-8")
    assert bench.workload_precision("imbalanced") == "bf16"


def test_router_wgrad_reduce_folds_into_the_router_gradient():
    k = {"router_wgrad": (4, 1.0), "router_wgrad_reduce": (4, 0.25), "combine": (4, 0.5)}
    assert bench.fold_kernels(k) == {"router_wgrad": (4, 1.25), "combine": (4, 0.5)}


def test_mx_quantiser_bytes_average_over_launches():
    s = gen.workload_shape("mxfp8")
    nmb = 8
    # per step: one two-orientation launch per weight; per micro-batch the x
    # rows (codes), and column launches for dy (both directions) and for x;
    # the activation bytes count the routed rows (2048 tokens x top-8 per
    # micro-batch), not the padding rows
    kernels = {"mx_quant_2d": (2 * 20, 1.0), "mx_quant_cols": (16 * 20, 1.0),
               "mx_quant_rows": (8 * 20, 1.0)}
    got = bench.mx_quant_bytes(s, nmb, kernels, steps=20)
    w_gu, w_d = s.E * 2 * s.I * s.d, s.E * s.I * s.d
    act, tok = 2048 * 8 * s.d, s.T // nmb * s.d
    c8 = 1 + 1 / 32
    assert got["mx_quant_2d"] * 2 == pytest.approx(
        2 * w_gu + 2 * c8 * w_gu + 2 * w_d + c8 * w_d + 2 * w_d)
    assert got["mx_quant_cols"] * 16 == pytest.approx(
        nmb * (2 * tok + 4 * act) + nmb * (2 * tok + 2 * act))
    assert got["mx_quant_rows"] * 8 == pytest.approx(nmb * (2 * tok + act * c8))


def test_nv_quantiser_bytes_average_over_launches():
    s = gen.workload_shape("nvfp4")
    kernels = {"nvfp4_quantize_2d": (20, 1.0), "nvfp4_quantize": (80, 1.0),
               "nvfp4_amax": (100, 1.0)}
    got = bench.nv_quant_bytes(s, kernels, steps=20)
    w_gu, w_d = s.E * 2 * s.I * s.d, s.E * s.I * s.d
    c4 = 0.5 + 1 / 16
    assert got["nvfp4_quantize_2d"] == pytest.approx(w_gu * 2 + 2 * c4 * w_gu)
    # four row launches: W_down, then x, h and dG/dU over the routed rows
    assert got["nvfp4_quantize"] * 4 == pytest.approx(
        w_d * (2 + c4) + s.T * s.d * 2 + s.R * s.d * c4 + s.R * s.I * (2 + c4)
        + s.R * 2 * s.I * (2 + c4))
    assert got["nvfp4_amax"] * 5 == pytest.approx(
        2 * (w_gu + w_d + s.T * s.d + s.R * s.I + s.R * 2 * s.I))


def test_reference_arm_prints_one_json_line():
    """`bench.py --impl reference` times the fp64 oracle on the host and prints
    the contract's line (tiny workload here to keep it quick)."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3", "--workload", "tiny"],
                         capture_output=True, text=True, timeout=300, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["workload"].startswith("tiny")


def test_mover_roofline_takes_the_tighter_bound():
    # 1 GB moved, 0.9 GB of it written: at 6.7 TB/s copy and 4 TB/s writes
    # the writes bind (225 us > 149 us)
    assert bench.mover_roofline_us(1e9, 0.9e9, 6700.0, 4000.0) == pytest.approx(225.0)
    assert bench.mover_roofline_us(2e9, 0.2e9, 6700.0, 4000.0) == pytest.approx(2e9 / 6700.0 / 1e3)
    s = gen.workload_shape("fine")
    w, m = bench.mover_write_bytes(s), bench.mover_bytes(s)
    for n in w:
        assert 0 < w[n] < m[n]


def test_gemm_bytes_fine_weight_gradients_are_hbm_bound():
    """On the fine workload the gate/up weight gradient reads its operands and
    writes 1.07 GB of fp32 dW, 1.48 GB in all: at the 6.69 TB/s copy bandwidth
    that takes longer (221 us) than its 275 GFLOP at the sustained bf16 rate
    (157 us), and with writes as fast as the bulk-store fill measures them
    (6.4 TB/s) the copy term is the binding one."""
    s = gen.workload_shape("fine")
    b = bench.gemm_bytes(s)
    tot, wr = b["bwd_gate_up_wgrad"]
    assert wr == s.E * 2 * s.I * s.d * 4
    assert tot == 32768 * 2 * s.I * 4 + 32768 * s.d * 2 + wr
    t_mem = bench.mover_roofline_us(tot, wr, 6688.8, 6400.0)
    assert t_mem == pytest.approx(tot / 6688.8 / 1e3)
    t_tc = bench.gemm_flops(s)["bwd_gate_up_wgrad"] / 1748.6e12 * 1e6
    assert t_mem > t_tc
    # bf16 dW halves the write; the deferred form reads every micro-batch
    assert bench.gemm_bytes(s, wgrad_elem_bytes=2)["bwd_gate_up_wgrad"][1] == wr // 2
    m = gen.workload_shape("mxfp8")
    one, eight = bench.gemm_bytes(m, 1), bench.gemm_bytes(m, 8)
    assert eight["bwd_gate_up_wgrad"][1] == one["bwd_gate_up_wgrad"][1]
    assert eight["bwd_gate_up_wgrad"][0] == pytest.approx(one["bwd_gate_up_wgrad"][0])
    for n, (t, w) in b.items():
        assert 0 < w < t, n


def test_router_wgrad_bytes_algorithmic_and_executed():
    """Algorithmic: x read once, fp32 dW_r written.  Executed (fine: 16
    chunks of 256 tokens, E padded to 128): plus the dl hi/lo operand and the
    fp32 partials written and read back."""
    s = gen.workload_shape("fine")
    T, d, E = s.T, s.d, s.E
    assert bench.mover_bytes(s)["router_wgrad"] == T * d * 2 + E * d * 4
    part = 16 * 128 * d * 4
    assert bench.router_wgrad_executed_bytes(s) == T * d * 2 + 2 * T * 128 * 2 + 2 * part + E * d * 4


def test_ncu_traffic_is_per_workload():
    t, src = bench.ncu_traffic("fine", "bwd_gate_up_wgrad")
    assert t > 1e9 and src.startswith("profiles/")
    assert bench.ncu_traffic("tiny", "bwd_gate_up_wgrad") == (None, None)


def test_large_traffic_scales_the_slice_capture_to_the_algorithmic_bytes():
    """The large workload's traffic comes from a capture of its slice scaled by
    the expert ratio; the slice must keep the large workload's per-expert
    shape, and the scaled weight-gradient traffic sits at its algorithmic
    bytes (dW written once, its operands read once)."""
    big, sl = gen.workload_shape("large"), gen.workload_shape("large_slice")
    assert (big.d, big.I, big.k) == (sl.d, sl.I, sl.k)
    assert big.E == 16 * sl.E and big.T == 16 * sl.T
    t, src = bench.ncu_traffic("large", "bwd_gate_up_wgrad")
    alg = bench.gemm_bytes(big)["bwd_gate_up_wgrad"][0]
    assert 0.95 < t / alg < 1.05 and "large_slice" in src


def test_low_precision_peaks_and_bytes():
    """FP8 GEMMs against 2x and FP4 GEMMs against 6x the measured bf16 peak
    (GB300's nominal dense ratios); NVFP4 operands (the forward GEMMs' and
    the gate/up dgrad's) are half a byte plus a sixteenth of a scale byte per
    value."""
    assert bench.peak_ratio("mxfp8", "fwd_down") == 2.0
    assert bench.peak_ratio("nvfp4", "fwd_down") == 6.0
    assert bench.peak_ratio("nvfp4", "bwd_gate_up_dgrad") == 6.0
    assert bench.peak_ratio("nvfp4", "bwd_down_dgrad_swiglu") == 1.0
    assert bench.peak_ratio("large", "fwd_down") == 1.0
    s = gen.workload_shape("nvfp4")
    R, d, I, E = s.R, s.d, s.I, s.E
    nv, bf = bench.gemm_bytes(s, nv=True), bench.gemm_bytes(s)
    q4 = 0.5 + 1 / 16
    assert nv["fwd_down"][0] == R * I * q4 + E * d * I * q4 + R * d * 4
    assert nv["bwd_gate_up_dgrad"][0] == R * 2 * I * q4 + E * 2 * I * d * q4 + R * d * 4
    assert nv["bwd_down_dgrad_swiglu"] == bf["bwd_down_dgrad_swiglu"]


def test_gemm_peak_fraction_takes_each_gemm_at_its_own_peak():
    # two GEMMs of 1 TFLOP each, one launch, 1 ms each, bf16 peak 1000 TFLOP/s
    flops = {"fwd_gate_up_swiglu": 1e12, "bwd_gate_up_wgrad": 1e12}
    kernels = {"fwd_gate_up_swiglu": (1, 1.0), "bwd_gate_up_wgrad": (1, 1.0)}
    names = list(flops)
    # bf16: both at the bf16 peak -> 1 ms each at peak, 2 ms measured
    assert bench.gemm_peak_fraction(flops, kernels, names, 1000.0, "bf16") == pytest.approx(1.0)
    # NVFP4: the forward GEMM's peak is 6x, so its FLOPs take 1/6 ms at peak
    got = bench.gemm_peak_fraction(flops, kernels, names, 1000.0, "nvfp4")
    assert got == pytest.approx((1 / 6 + 1) / 2)
    assert bench.gemm_peak_fraction(flops, {n: (1, 0.0) for n in names}, [], 1000.0, "bf16") == 0.0
