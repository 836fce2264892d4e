#!/usr/bin/env python
"""Throughput of one deterministic MoE layer, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mok|reference]

A step is one forward + backward of the layer (router, dispatch, grouped
SwiGLU GEMMs, combine, and the mirrored backward) over one batch of the large
fine-grained workload by default: T=8192 tokens, d=7168, E=384 experts,
I=2048, top-8, bf16, seeded synthetic inputs (`--workload` selects the fine,
imbalanced, MXFP8 or tiny one).  The weights (33.8 GB) and activations read
per step are far larger than the 129 MB L2, so no flush is needed between
steps.

Printed (rank 0, one JSON line): tokens/s over all ranks, per-kernel times
from CUDA events recorded around each kernel on one in four steps of the timed
region, the
dominant kernel's roofline, the end-to-end number through the C ABI with
pinned-host inputs and outputs, the fp64 oracle's CPU throughput on a small
sample, and the SM clocks sampled during the timed region.

With N > 1 (torchrun) every rank runs its own replica of the layer on its own
GPU: the layer has no cross-GPU exchange on one node, so scaling is weak.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routing_dispatch_grouped_router_gb300 import inputs as gen  # noqa: E402

METRIC = "MoE layer fwd+bwd tokens/s on 1 GB300; grouped-GEMM % of tensor-core peak"
WORKLOAD = "large"
# operand precision of the expert GEMMs: the workload's own, or --precision
PRECISION = "bf16"


def workload_precision(name: str) -> str:
    """The precision a workload is defined with: mxfp8, nvfp4 or bf16."""
    w = gen.WORKLOADS[name]
    return "mxfp8" if name == "mxfp8" else ("nvfp4" if w.get("nvfp4") else "bf16")
PROFILE_EVERY = 4  # per-kernel events on one timed step in this many

# Algorithmic work per launch of each kernel (R = T*k routed rows).
#   GEMMs: 2*M*N*K flops with M summed over the experts' real rows.
#   Row movers: bytes that must cross HBM once.


# GEMMs that run on the block-scaled FP8 tensor cores in the MXFP8 workload
MX_GEMMS = ("fwd_gate_up_swiglu", "fwd_down", "bwd_gate_up_dgrad")
# ... and on the block-scaled FP4 tensor cores in the NVFP4 workload
NV_GEMMS = ("fwd_gate_up_swiglu", "fwd_down", "bwd_gate_up_dgrad")


def peak_ratio(precision: str, gemm: str) -> float:
    """A GEMM's tensor peak relative to the measured bf16 one: the nominal
    dense ratios of GB300 (fp8 4.5 / bf16 2.25 PFLOP/s = 2, fp4 13.5 / 2.25 = 6)
    for the GEMMs that run on those operands."""
    if precision == "mxfp8" and gemm in MX_GEMMS:
        return 2.0
    if precision == "nvfp4" and gemm in NV_GEMMS:
        return 6.0
    return 1.0


def gemm_peak_fraction(flops: dict, kernels: dict, names, bf16_tflops: float,
                       precision: str) -> float:
    """Fraction of the tensor peak the GEMMs `names` reach together: the time
    their algorithmic FLOPs take at each one's own operands' peak (FP8 and FP4
    GEMMs at the nominal 2x and 6x of the bf16 one) over their measured time.
    `kernels[name]` = (launches, total ms), `flops[name]` = FLOP per launch."""
    ms = sum(kernels[n][1] for n in names)
    at_peak = sum(flops[n] * kernels[n][0] / (bf16_tflops * 1e12 * peak_ratio(precision, n))
                  for n in names) * 1e3
    return at_peak / ms if ms else 0.0


# Weight-gradient GEMMs: with micro-batches the layer defers them and launches
# each once per step over every micro-batch's rows
DEFERRED_WGRADS = ("bwd_down_wgrad", "bwd_gate_up_wgrad")


def gemm_flops(shape: gen.Shape, micro_batches: int = 1) -> dict:
    """Algorithmic FLOP of one launch of each GEMM; with micro-batching a
    launch covers T / micro_batches tokens, except the deferred weight
    gradients, whose one launch per step covers all T."""
    R, d, I, T, E = (shape.R // micro_batches, shape.d, shape.I, shape.T // micro_batches,
                     shape.E)
    f = {
        "router_logits": 2.0 * T * d * E,
        "fwd_gate_up_swiglu": 2.0 * R * d * 2 * I,
        "fwd_down": 2.0 * R * I * d,
        "bwd_down_dgrad_swiglu": 2.0 * R * d * I,
        "bwd_down_wgrad": 2.0 * R * d * I,
        "bwd_gate_up_dgrad": 2.0 * R * 2 * I * d,
        "bwd_gate_up_wgrad": 2.0 * R * 2 * I * d,
    }
    for n in DEFERRED_WGRADS:
        f[n] *= micro_batches
    return f


def gemm_bytes(shape: gen.Shape, micro_batches: int = 1, mx: bool = False,
               wgrad_elem_bytes: int = 4, nv: bool = False) -> dict:
    """Algorithmic HBM bytes of one launch of each grouped GEMM in the layer's
    layout, as (total, written): every operand read once, every output written
    once.  Forward: bf16 rows, weights, fp32 g/u and O, bf16 h.  Backward:
    the SwiGLU backward reads fp32 g/u and writes dG/dU and p*h as bf16 hi/lo
    pairs; the dgrads write fp32 rows; the weight gradients read their hi/lo
    operand and write dW (fp32 by default).  MXFP8: E4M3 codes (+1/32 scale
    byte) for the block-scaled GEMMs' operands.  A deferred weight gradient
    reads every micro-batch's operands and writes dW once.  NVFP4: the
    forward GEMMs and the gate/up dgrad read E2M1 codes (half a byte, +1/16
    scale byte per value)."""
    R, d, I, E = shape.R // micro_batches, shape.d, shape.I, shape.E
    wgu, wd = E * 2 * I * d, E * d * I
    q8 = 1 + 1 / 32
    q4 = 0.5 + 1 / 16
    a_gu, w_gu = (R * d * q8, wgu * q8) if mx else (R * d * 2, wgu * 2)
    if nv:
        a_gu, w_gu = R * d * q4, wgu * q4
    h_out = R * I * q8 if mx else R * I * 2
    f = {
        "fwd_gate_up_swiglu": (a_gu + w_gu + R * 2 * I * 4 + h_out, R * 2 * I * 4 + h_out),
        "fwd_down": ((R * I * q8 + wd * q8) if mx else
                     ((R * I * q4 + wd * q4) if nv else (R * I * 2 + wd * 2))) + R * d * 4,
        "bwd_down_dgrad_swiglu": R * d * 2 + wd * 2 + R * 2 * I * 4 + R * 2 * I * 4 + R * I * 4
                                 + (R * 2 * I * q8 if mx else 0),
        "bwd_gate_up_dgrad": ((R * 2 * I * q8 + wgu * q8) if mx else
                              ((R * 2 * I * q4 + wgu * q4) if nv else (R * 2 * I * 2 + wgu * 2)))
                             + R * d * 4,
    }
    w = {
        "fwd_gate_up_swiglu": f["fwd_gate_up_swiglu"][1],
        "fwd_down": R * d * 4,
        "bwd_down_dgrad_swiglu": R * 2 * I * 4 + R * I * 4 + (R * 2 * I * q8 if mx else 0),
        "bwd_gate_up_dgrad": R * d * 4,
    }
    out = {n: (v[0] if isinstance(v, tuple) else v, w[n]) for n, v in f.items()}
    mb = micro_batches
    out["bwd_down_wgrad"] = (mb * (R * d * 2 + R * I * 4) + wd * wgrad_elem_bytes,
                             wd * wgrad_elem_bytes)
    out["bwd_gate_up_wgrad"] = (mb * (R * 2 * I * 4 + R * d * 2) + wgu * wgrad_elem_bytes,
                                wgu * wgrad_elem_bytes)
    return out


# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of the
# grouped GEMMs, per workload, from the ncu captures summarised in profiles/
# (kernels as of the commit each file names); a kernel changed since its
# capture has no entry.
NCU_TRAFFIC_FINE = {
    "fwd_gate_up_swiglu": 689.183232e6 + 312.882e6,
    "fwd_down": 343.459072e6 + 240.195e6,
    "bwd_down_dgrad_swiglu": 781.232640e6 + 383.957e6,
    "bwd_down_wgrad": 284.840960e6 + 479.524e6,
    "bwd_gate_up_dgrad": 688.372224e6 + 257.197e6,
    "bwd_gate_up_wgrad": 427.129344e6 + 1013.322e6,
}
# The large workload's GEMMs from a capture of its slice (1/16 of its experts and
# tokens, the same widths and rows per expert): per-expert work, so 16x the bytes.
NCU_TRAFFIC_LARGE = {k: 16 * v for k, v in {
    "fwd_gate_up_swiglu": 1.511265e9 + 0.078212e9,
    "fwd_down": 0.733215e9 + 0.112134e9,
    "bwd_down_dgrad_swiglu": 0.908464e9 + 0.092401e9,
    "bwd_down_wgrad": 0.103909e9 + 1.347131e9,
    "bwd_gate_up_dgrad": 1.474287e9 + 0.122661e9,
    "bwd_gate_up_wgrad": 0.142005e9 + 2.757084e9,
}.items()}
NCU_TRAFFIC = {"fine": (NCU_TRAFFIC_FINE, "profiles/grouped_gemms_fine.txt"),
               "large": (NCU_TRAFFIC_LARGE,
                         "profiles/grouped_gemms_large_slice.txt (slice launch x 16)")}


def ncu_traffic(workload: str, kernel: str):
    """(bytes per launch or None, source file) of a kernel's committed capture."""
    table, src = NCU_TRAFFIC.get(workload, ({}, None))
    return table.get(kernel), src


def mx_quant_bytes(shape: gen.Shape, nmb: int, kernels: dict, steps: int) -> dict:
    """Average bytes per launch of the MXFP8 quantisers in one step.  Once per
    call, one launch per weight reads it and writes both orientations: W_gate_up
    as E4M3 codes + scales along d (the forward) and along 2I (the gate/up
    dgrad), W_down as codes + scales along I and as bf16 MX values along d (the
    down dgrad).  Per micro-batch: the dispatched x rows as codes (row
    launch), dy in both block directions as bf16 values and x along the rows
    as bf16 values (two column launches).  The activation launches read the
    token rows through the row -> token map: each token row once, each
    routed row written (algorithmic bytes: the padding rows the kernels also
    write, up to the plan's padded total, are not counted)."""
    E, d, I = shape.E, shape.d, shape.I
    w_gu, w_d = E * 2 * I * d, E * d * I       # weight elements
    act = shape.T // nmb * shape.k * d         # one micro-batch's routed rows
    tok = shape.T // nmb * d                   # one micro-batch's token rows
    c8 = 1 + 1 / 32                            # E4M3 code + 1/32 scale byte
    two_d = w_gu * (2 + 2 * c8) + w_d * (2 + c8 + 2)
    rows_bytes = nmb * (tok * 2 + act * c8)
    cols_bytes = nmb * (tok * 2 + act * 4) + nmb * (tok * 2 + act * 2)
    out = {}
    for name, total in (("mx_quant_2d", two_d), ("mx_quant_rows", rows_bytes),
                        ("mx_quant_cols", cols_bytes)):
        if name in kernels:
            n, _ = kernels[name]
            out[name] = total / (n / steps)
    return out


def nv_quant_bytes(shape: gen.Shape, kernels: dict, steps: int) -> dict:
    """Average bytes per launch of the NVFP4 quantisers in one step (one call,
    no micro-batches).  W_gate_up: one launch reads it and writes E2M1 codes
    + E4M3 scales along d and along 2I.  Row launches: W_down, x (token rows
    through the row map, each read once), h and dG/dU, over the routed rows
    (algorithmic bytes: the padding rows up to the plan's padded total are
    not counted).  Tensor scales: one read of W_gate_up, W_down and x, and of
    h and dG/dU over the routed rows."""
    E, d, I, R = shape.E, shape.d, shape.I, shape.R
    w_gu, w_d = E * 2 * I * d, E * d * I
    c4 = 0.5 + 1 / 16                          # E2M1 code + 1/16 scale byte
    two_d = w_gu * (2 + 2 * c4)
    rows = (w_d * (2 + c4) + (shape.T * d * 2 + R * d * c4)
            + R * I * (2 + c4) + R * 2 * I * (2 + c4))
    amax = 2 * (w_gu + w_d + shape.T * d + R * I + R * 2 * I)
    out = {}
    for name, total in (("nvfp4_quantize_2d", two_d), ("nvfp4_quantize", rows),
                        ("nvfp4_amax", amax)):
        if name in kernels:
            n, _ = kernels[name]
            out[name] = total / (n / steps)
    return out


def mover_bytes(shape: gen.Shape, micro_batches: int = 1) -> dict:
    """Bytes one launch of each data-movement kernel must move in the layer's
    layout: bf16 token rows, fp32 expert-output and dX rows, fp32 y and dx
    (the default); with micro-batching a launch covers T / micro_batches tokens."""
    R, d, T, E, I = (shape.R // micro_batches, shape.d, shape.T // micro_batches, shape.E,
                     shape.I)
    np_ = 2 * I // (256 if I % 256 == 0 else 128)
    return {
        # read each token row once, write its k bf16 rows, read the positions
        "dispatch_rows": T * d * 2 + R * d * 2 + R * 4,
        # read k fp32 expert rows + weights per token, write the fp32 token row
        "combine": R * 4 * d + T * 4 * d + R * 8,
        # read k fp32 dX rows and the dp partials, write fp32 dx (router rows from L2)
        "reverse_dispatch": R * 4 * d + T * 4 * d + R * (12 + 4 * np_),
        # algorithmic: read each token row once, write dW_r (fp32); the executed
        # form moves more (router_wgrad_executed_bytes)
        "router_wgrad": T * d * 2 + E * d * 4,
    }


def router_wgrad_executed_bytes(shape: gen.Shape, micro_batches: int = 1) -> float:
    """Bytes the router-weight gradient moves as executed: the tensor-core
    GEMM reads x once and the dense dl operand as a bf16 hi/lo pair [T, E
    padded to 128] and writes one fp32 partial [E padded, d] per token chunk;
    the reduce reads the partials and writes dW_r (fp32).  The chunk count
    follows the library's split: ks = 152 // (M tiles x N tiles) chunks of
    whole 64-token blocks, at least 1 and at most the block count."""
    T, d, E = shape.T // micro_batches, shape.d, shape.E
    e_pad = -(-E // 128) * 128
    bn = 256 if d % 256 == 0 else 128
    tiles = (e_pad // 128) * (d // bn)
    nkb = max(1, -(-T // 64))
    ks = min(max(1, 152 // tiles), nkb)
    kb = -(-nkb // ks)
    ks = -(-nkb // kb)
    part = ks * e_pad * d * 4
    return T * d * 2 + 2 * T * e_pad * 2 + 2 * part + E * d * 4


# kernels whose time belongs to another one's step: the router-weight
# gradient is a tensor-core GEMM over token chunks plus the in-order sum of
# its chunks' partial products
FOLDED = {"router_wgrad_reduce": "router_wgrad"}


def fold_kernels(kernels: dict) -> dict:
    """{name: (launches, ms)} with each FOLDED kernel's time added to the
    kernel it completes; the launch count stays that kernel's own."""
    out = {n: v for n, v in kernels.items() if n not in FOLDED}
    for n, (_, ms) in kernels.items():
        if n in FOLDED:
            launches, total = out.get(FOLDED[n], (0, 0.0))
            out[FOLDED[n]] = (launches, total + ms)
    return out


def mover_write_bytes(shape: gen.Shape, micro_batches: int = 1) -> dict:
    """Bytes each data-movement launch writes (part of mover_bytes)."""
    R, d, T, E = shape.R // micro_batches, shape.d, shape.T // micro_batches, shape.E
    return {"dispatch_rows": R * d * 2, "combine": T * d * 4, "reverse_dispatch": T * d * 4,
            "router_wgrad": E * d * 4}


def mover_roofline_us(total_bytes: float, write_bytes: float, copy_gbs: float,
                      write_gbs: float) -> float:
    """Shortest time for a launch that moves total_bytes, write_bytes of them
    written: HBM moves at most copy_gbs in both directions together and
    write_gbs of writes alone."""
    return max(total_bytes / copy_gbs, write_bytes / write_gbs) / 1e3


def measure_write_gbs(torch, api) -> tuple:
    """HBM write bandwidth on this GPU: 1 GiB set to zero by torch's fill
    kernel and by the library's bulk-store fill (the store path of the row
    dispatch), best of 5 CUDA-event timings each after one warm-up.  Returns
    (the faster one's GB/s, {fill: GB/s})."""
    buf = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    fills = {"torch zero_": lambda: buf.zero_(), "bulk-store fill": lambda: api.fill_zero(buf)}
    rates = {}
    for name, fill in fills.items():
        fill()
        best = None
        for _ in range(5):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fill()
            b.record()
            torch.cuda.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        rates[name] = (1 << 30) / (best / 1e3) / 1e9
    del buf
    return max(rates.values()), rates


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=j.get("hbm_gbs", 6800.0), bf16=j.get("bf16_tflops", 1900.0),
                    bf16_sustained=j.get("bf16_tflops_sustained", 1700.0), source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ clocks --

CLOCK_FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + CLOCK_FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append(parts)
        bus = {r[1].lower() for r in rows}
        if self.bus_id and any(self.bus_id[-12:] in b for b in bus):
            rows = [r for r in rows if self.bus_id[-12:] in r[1].lower()]
        elif len(bus) > 1:
            rows = [r for r in rows if r[0] == rows[0][0]]
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for i, n in enumerate(names):
                if r[6 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": sorted(reasons)}


# ------------------------------------------------------- CPU (oracle) side --

def oracle_sample(inp: dict, shape: gen.Shape, tokens: np.ndarray):
    """fp64 oracle forward + backward on a slice of the workload's tokens
    (every token is independent in the layer; the expert gradients of the
    experts the slice touches are complete for that slice)."""
    import oracle
    xs = inp["x"][tokens]
    dys = inp["dy"][tokens]
    _, fwd = oracle.moe_forward_ref(xs, inp["w_router"], inp["bias"], inp["w_gate_up"],
                                    inp["w_down"], shape.k, keep=True)
    experts = np.unique(fwd["idx"])
    oracle.moe_backward_ref(xs, inp["w_router"], inp["bias"], inp["w_gate_up"], inp["w_down"],
                            shape.k, dys, fwd=fwd, grad_experts=experts)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# tokens per oracle slice: a slice touches up to k x tokens experts, and the
# oracle widens each touched expert's weights to float64 (0.35 GB per expert on
# the large workload), so slices are sized to a few seconds each
SLICE_TOKENS = {"tiny": 32, "fine": 32, "imbalanced": 2, "mxfp8": 2, "nvfp4": 2, "large": 1,
                "large_slice": 1, "nvfp4_slice": 2}


def cpu_baseline(inp: dict, shape: gen.Shape, budget_s: float = 12.0,
                 tokens_per_sample: int | None = None):
    tokens_per_sample = tokens_per_sample or SLICE_TOKENS.get(WORKLOAD, 1)
    t0 = time.perf_counter()
    done = 0
    n = 0
    while True:
        tok = (np.arange(tokens_per_sample) + n * tokens_per_sample) % shape.T
        oracle_sample(inp, shape, tok)
        done += tokens_per_sample
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} x {tokens_per_sample}-token slices of the {WORKLOAD} workload, fp64 "
                      f"numpy oracle forward+backward (all routing, dispatch, expert FFNs and "
                      f"gradients of the touched experts), {dt:.1f} s"}


# Timed-step budget of the reference arm (the fp64 oracle on the host)
REFERENCE_BUDGET_S = 120.0


def run_reference(args, shape: gen.Shape, rank: int):
    if rank != 0:
        return
    inp = gen.workload_inputs(WORKLOAD, seed=0, parallel=True)
    tok_per_step = 1  # the smallest unit the oracle runs: one token's forward + backward
    for i in range(args.warmup):
        oracle_sample(inp, shape, np.array([i % shape.T]))
    # a step of the large workload takes seconds on the host: past the time
    # budget the remaining steps are not run, and the line says how many were
    t0 = time.perf_counter()
    done = 0
    for i in range(args.steps):
        oracle_sample(inp, shape, np.array([(args.warmup + i) % shape.T]))
        done += 1
        if time.perf_counter() - t0 > REFERENCE_BUDGET_S:
            break
    dt = time.perf_counter() - t0
    value = tok_per_step * done / dt
    sample = f"one token of the {WORKLOAD} workload per step"
    if done < args.steps:
        sample += f"; {done} of the {args.steps} requested steps ({REFERENCE_BUDGET_S:.0f} s budget)"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": done, "warmup": args.warmup, "ms_per_step": 1e3 * dt / done,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": workload_config(shape),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(shape: gen.Shape) -> dict:
    w = gen.WORKLOADS[WORKLOAD]
    prec = {"bf16": "bf16",
            "mxfp8": "MXFP8 operands (E4M3, E8M0 per 32) for the forward GEMMs and the gate/up "
                     "dgrad",
            "nvfp4": "NVFP4 operands (E2M1, E4M3 per 16, fp32 per tensor) for the forward "
                     "GEMMs and the gate/up dgrad"}[PRECISION]
    if PRECISION != workload_precision(WORKLOAD):
        prec += f" (the {WORKLOAD} workload run at this precision)"
    if w.get("mb_tokens"):
        prec += (f", {shape.T // w['mb_tokens']} micro-batches of {w['mb_tokens']} tokens "
                 f"through a {w['ring_slots']}-slot ring")
    if w.get("zipf_s"):
        prec += f", Zipf({w['zipf_s']}) router bias"
    wbytes = shape.E * 3 * shape.I * shape.d * 2
    cfg = {"workload": f"{WORKLOAD}: T={shape.T} d={shape.d} E={shape.E} I={shape.I} "
                       f"top-{shape.k} {prec} forward+backward",
           "T": shape.T, "d": shape.d, "E": shape.E, "I": shape.I, "k": shape.k,
           "l2": f"inputs larger than L2 ({wbytes / 1e9:.1f} GB of expert weights read per step), "
                 "no flush",
           "parallelism": "replicas (one independent layer per GPU)"}
    return cfg


def layer_options(api, bf16_wgrad: bool = False) -> dict:
    """MoELayer keyword arguments of the selected workload (bf16_wgrad: weight
    gradients returned in bf16, rounded once from the fp32 accumulation)."""
    w = gen.WORKLOADS[WORKLOAD]
    opts = {}
    if w.get("mb_tokens"):
        if bf16_wgrad:
            raise SystemExit("--bf16-wgrad: a micro-batched workload accumulates dW in fp32")
        opts.update(mb_tokens=w["mb_tokens"], ring_slots=w["ring_slots"])
    elif bf16_wgrad:
        opts["flags"] = api.FLAG_BF16_WGRAD_OUT
    if PRECISION != "bf16":
        opts["dtype"] = {"mxfp8": api.MXFP8, "nvfp4": api.NVFP4}[PRECISION]
    return opts


# ------------------------------------------------------------- multi-rank --

def max_over_ranks(value: float, dist, device) -> float:
    """The largest `value` of all ranks (the slowest rank's time)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_rank: int, steps: int, t_max_ms: float) -> float:
    """Tokens/s of the whole job: every rank runs its own replica on its own
    tokens, and the job takes as long as its slowest rank."""
    return world * tokens_per_rank * steps / (t_max_ms / 1e3)


# --------------------------------------------------------------- GPU side --

def e2e_pipelined(layer, inp, x, dy, wr, bias, wgu, wd, dwr, dwgu, dwd, stream, steps, world,
                  dist):
    """Milliseconds for `steps` layer steps through the public API, each with
    its inputs uploaded from and its outputs read back to pinned host memory
    inside the timed region (uploads and read-backs on two side streams, so
    both directions of the host link run at once; two buffer sets)."""
    import torch
    xh = torch.from_numpy(inp["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    dyh = torch.from_numpy(inp["dy"].view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = [torch.empty(xh.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    dxh = [torch.empty(xh.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    dyd = [torch.empty_like(dy) for _ in range(2)]
    yd = [torch.empty(x.shape, dtype=torch.float32, device=x.device) for _ in range(2)]
    dxd = [torch.empty(x.shape, dtype=torch.float32, device=x.device) for _ in range(2)]
    copy = torch.cuda.Stream()  # uploads
    back = torch.cuda.Stream()  # read-backs
    inputs_in = [torch.cuda.Event() for _ in range(2)]      # upload into set b done
    inputs_free = [torch.cuda.Event() for _ in range(2)]    # the step that read set b finished
    outputs_out = [torch.cuda.Event() for _ in range(2)]    # read-back of set b done
    outputs_ready = [torch.cuda.Event() for _ in range(2)]  # the step that wrote set b finished

    def run(n):
        with torch.cuda.stream(copy):
            xd[0].copy_(xh, non_blocking=True)
            dyd[0].copy_(dyh, non_blocking=True)
            inputs_in[0].record(copy)
        for i in range(n):
            b = i % 2
            if i + 1 < n:  # upload the next step's inputs into the other set
                with torch.cuda.stream(copy):
                    if i >= 1:
                        copy.wait_event(inputs_free[1 - b])
                    xd[1 - b].copy_(xh, non_blocking=True)
                    dyd[1 - b].copy_(dyh, non_blocking=True)
                    inputs_in[1 - b].record(copy)
            stream.wait_event(inputs_in[b])
            if i >= 2:
                stream.wait_event(outputs_out[b])  # y, dx of step i-2 read back
            layer.forward(xd[b], wr, bias, wgu, wd, y=yd[b])
            layer.backward(dyd[b], xd[b], wr, bias, wgu, wd, dx=dxd[b], dw_router=dwr,
                           dw_gate_up=dwgu, dw_down=dwd)
            inputs_free[b].record(stream)
            outputs_ready[b].record(stream)
            with torch.cuda.stream(back):
                back.wait_event(outputs_ready[b])
                yh[b].copy_(yd[b], non_blocking=True)
                dxh[b].copy_(dxd[b], non_blocking=True)
                outputs_out[b].record(back)
        stream.wait_stream(copy)
        stream.wait_stream(back)

    run(3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run(steps)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)

def graph_steps(torch, step, steps: int, stream, world: int, dist) -> float:
    """Milliseconds for `steps` replays of one step captured in a CUDA graph
    (the same kernels, without per-launch host work or launch gaps)."""
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mok", choices=["mok", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--bf16-wgrad", action="store_true",
                    help="return the weight gradients in bf16 (default fp32)")
    ap.add_argument("--workload", default="large", choices=sorted(gen.WORKLOADS),
                    help="large (default: the configuration the targets are stated on), "
                         "fine, imbalanced, mxfp8, nvfp4 or tiny")
    ap.add_argument("--precision", default=None, choices=["bf16", "mxfp8", "nvfp4"],
                    help="expert-GEMM operands (default: the workload's own)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    global WORKLOAD, PRECISION
    WORKLOAD = args.workload
    PRECISION = args.precision or workload_precision(WORKLOAD)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    shape = gen.workload_shape(WORKLOAD)

    if args.impl == "reference":
        run_reference(args, shape, rank)
        return

    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    from routing_dispatch_grouped_router_gb300 import api, build
    build.build()

    inp = gen.workload_inputs(WORKLOAD, seed=0, parallel=True)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    x, wr, wgu, wd, dy = (dev(inp[n]) for n in ("x", "w_router", "w_gate_up", "w_down", "dy"))
    bias = torch.from_numpy(inp["bias"]).cuda() if inp.get("bias") is not None else None
    layer = api.MoELayer(shape.T, shape.d, shape.E, shape.I, shape.k,
                         **layer_options(api, args.bf16_wgrad))
    f32 = dict(dtype=torch.float32, device="cuda")
    y = torch.empty(x.shape, **f32)
    dx = torch.empty(x.shape, **f32)
    wg = dict(dtype=layer.wgrad_dtype, device="cuda")
    dwr = torch.empty(wr.shape, **wg)
    dwgu = torch.empty(wgu.shape, **wg)
    dwd = torch.empty(wd.shape, **wg)
    stream = torch.cuda.current_stream()

    def step():
        layer.forward(x, wr, bias, wgu, wd, y=y)
        layer.backward(dy, x, wr, bias, wgu, wd, dx=dx, dw_router=dwr, dw_gate_up=dwgu,
                       dw_down=dwd)

    for _ in range(args.warmup):
        step()
    status = layer.status()
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")
    launches_per_step = api.last_launch_count()

    bus = None
    try:
        bus = torch.cuda.get_device_properties(local).pci_bus_id
    except Exception:
        bus = None
    sampler = ClockSampler(str(bus) if bus is not None else None)

    # ---- timed region: K steps.  Per-kernel events are recorded on the stream
    # in one step of every PROFILE_EVERY (steps 0, 4, 8, ...): each event is a
    # stream operation between two kernels, and recording them on every step
    # would slow the very region they measure.
    api.profile_reset()
    prof_steps = (args.steps + PROFILE_EVERY - 1) // PROFILE_EVERY
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        api.profile_enable(i % PROFILE_EVERY == 0)
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    api.profile_enable(False)
    elapsed_ms = ev0.elapsed_time(ev1)
    kernels = fold_kernels(api.profile_collect())
    if layer.status() != 0:
        raise RuntimeError("device status set during the timed region")
    t_max = max_over_ranks(elapsed_ms, dist, "cuda") if world > 1 else elapsed_ms
    value = job_throughput(world, shape.T, args.steps, t_max)

    # ---- per-kernel summary and the dominant kernel's roofline
    peaks = load_peaks()
    write_gbs, write_rates = measure_write_gbs(torch, api)
    flops = gemm_flops(shape, int(layer.layout.mb_count))
    gbytes = gemm_bytes(shape, int(layer.layout.mb_count), mx=PRECISION == "mxfp8",
                        wgrad_elem_bytes=2 if args.bf16_wgrad else 4,
                        nv=PRECISION == "nvfp4")

    def gemm_roofline_us(n):
        """(bound, shortest time in us) of GEMM n: tensor time at the measured
        (FP8: x2) peak against HBM time at the copy and write bandwidths."""
        t_tc = flops[n] / (peaks["bf16_sustained"] * peak_ratio(PRECISION, n) * 1e12) * 1e6
        if n not in gbytes:
            return "tensor", t_tc
        t_mem = mover_roofline_us(gbytes[n][0], gbytes[n][1], peaks["hbm"], write_gbs)
        return ("hbm", t_mem) if t_mem > t_tc else ("tensor", t_tc)
    movers = mover_bytes(shape, int(layer.layout.mb_count))
    if PRECISION == "mxfp8":
        movers.update(mx_quant_bytes(shape, int(layer.layout.mb_count), kernels, prof_steps))
    if PRECISION == "nvfp4":
        movers.update(nv_quant_bytes(shape, kernels, prof_steps))
    total_k = sum(v[1] for v in kernels.values())
    ksum = {}
    for name, (n, ms) in kernels.items():
        ksum[name] = {"launches": n, "avg_us": 1e3 * ms / n, "share": ms / total_k}
        if name in flops:
            b, t_us = gemm_roofline_us(name)
            ksum[name].update({"bound": b, "roofline_us": t_us,
                               "frac_roofline": t_us / ksum[name]["avg_us"]})
    # the dominant kernel among those whose work per launch is known
    dom = max((n for n in kernels if n in flops or n in movers), key=lambda n: kernels[n][1])
    n_dom, ms_dom = kernels[dom]
    avg_s = ms_dom / n_dom / 1e3
    if dom in flops and gemm_roofline_us(dom)[0] == "hbm":
        # bound by HBM: its fp32 outputs (dW, g/u, rows) outweigh its tensor time
        tb, tw = gbytes[dom]
        ach = tb / avg_s / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm"],
                "unit": "GB/s", "frac": ach / peaks["hbm"],
                "frac_roofline": gemm_roofline_us(dom)[1] / (avg_s * 1e6),
                "written_per_launch": tw, "write_bw_gbs": write_gbs,
                "traffic": ncu_traffic(WORKLOAD if PRECISION == workload_precision(WORKLOAD) else "", dom)[0],
                "traffic_source": ncu_traffic(WORKLOAD if PRECISION == workload_precision(WORKLOAD) else "", dom)[1],
                "peak_source": f"hbm_gbs of {peaks['source']}; write bandwidth measured here "
                               "(1 GiB zero fill: the faster of torch's and the bulk-store one)",
                "write_bw_fills_gbs": write_rates,
                "algorithmic_per_launch": tb,
                "tensor": {"achieved_tflops": flops[dom] / avg_s / 1e12,
                           "peak_tflops": peaks["bf16_sustained"],
                           "frac": flops[dom] / avg_s / 1e12 / peaks["bf16_sustained"]}}
    elif dom in flops:
        ach = flops[dom] / avg_s / 1e12
        # block-scaled GEMMs run on the FP8 / FP4 tensor rates: their peak is the
        # measured bf16 one times the nominal ratio (peak_ratio)
        ratio = peak_ratio(PRECISION, dom)
        peak = peaks["bf16_sustained"] * ratio
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak,
                "traffic": ncu_traffic(WORKLOAD if PRECISION == workload_precision(WORKLOAD) else "", dom)[0],
                "traffic_source": ncu_traffic(WORKLOAD if PRECISION == workload_precision(WORKLOAD) else "", dom)[1],
                "peak_source": f"bf16_tflops_sustained of {peaks['source']}"
                               + (f" x {ratio:g} (nominal low-precision/bf16 ratio)"
                                  if ratio != 1.0 else ""),
                "algorithmic_per_launch": flops[dom]}
    else:
        ach = movers.get(dom, 0) / avg_s / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": peaks["hbm"],
                "unit": "GB/s", "frac": ach / peaks["hbm"], "traffic": None,
                "peak_source": f"hbm_gbs of {peaks['source']}",
                "algorithmic_per_launch": movers.get(dom, 0)}
    gemm_ms = sum(kernels[n][1] for n in flops if n in kernels)
    gemm_fl = sum(flops[n] * kernels[n][0] for n in flops if n in kernels)
    gg = [n for n in flops if n != "router_logits" and n in kernels]
    gg_ms = sum(kernels[n][1] for n in gg)
    gg_fl = sum(flops[n] * kernels[n][0] for n in gg)
    gg_tflops = gg_fl / (gg_ms / 1e3) / 1e12 if gg_ms else 0.0
    gg_frac = gemm_peak_fraction(flops, kernels, gg, peaks["bf16_sustained"], PRECISION)
    movers_perf = {}
    wbytes = mover_write_bytes(shape, int(layer.layout.mb_count))
    for n, b in movers.items():
        if n in kernels:
            avg_us = kernels[n][1] / kernels[n][0] * 1e3
            gbs = b / (avg_us / 1e6) / 1e9
            movers_perf[n] = {"GB/s": gbs, "frac_hbm": gbs / peaks["hbm"]}
            if n == "router_wgrad":
                ex = router_wgrad_executed_bytes(shape, int(layer.layout.mb_count))
                movers_perf[n].update({"bytes_algorithmic": b, "bytes_executed": ex,
                                       "GB/s_executed": ex / (avg_us / 1e6) / 1e9})
            if n in wbytes:
                # against the copy bandwidth and the measured write bandwidth
                # together: write-heavy movers (the dispatch) are bound by the latter
                roof_us = mover_roofline_us(b, wbytes[n], peaks["hbm"], write_gbs)
                movers_perf[n]["frac_roofline"] = roof_us / avg_us
    movers_perf["write_bw_gbs"] = write_gbs
    movers_perf["write_bw_fills_gbs"] = write_rates

    # ---- end to end through the C ABI: every step's x, dy uploaded from
    # pinned host memory and its y, dx read back to pinned host memory.  The
    # copies run on a second stream, double-buffered, so that step i+1's
    # upload and step i's read-back overlap the layer's kernels; events order
    # every reuse of a buffer.
    e2e_ms = e2e_pipelined(layer, inp, x, dy, wr, bias, wgu, wd, dwr, dwgu, dwd, stream,
                           args.e2e_steps, world, dist)
    xh_bytes = x.numel() * 2
    if world > 1:
        e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")
    e2e = {"value": job_throughput(world, shape.T, args.e2e_steps, e2e_ms), "unit": "tokens/s",
           "h2d_bytes_per_step": 2 * xh_bytes, "d2h_bytes_per_step": 2 * x.numel() * 4,
           "steps": args.e2e_steps}

    # ---- the same step replayed from a CUDA graph (after the timed region)
    g_ms = graph_steps(torch, step, args.steps, stream, world, dist)
    if world > 1:
        g_ms = max_over_ranks(g_ms, dist, "cuda")
    if layer.status() != 0:
        raise RuntimeError("device status set during the graph replays")
    graph_line = {"ms_per_step": g_ms / args.steps, "steps": args.steps,
                  "value": job_throughput(world, shape.T, args.steps, g_ms), "unit": "tokens/s"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, shape)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": PRECISION,
            "dtype_detail": {
                "mxfp8": "E4M3 + E8M0 per 32: block-scaled FP8 MMAs for the forward GEMMs and "
                         "the gate/up dgrad; bf16 MMAs on MX-valued operands for the down "
                         "dgrad; weight gradients on bf16 hi/lo operands",
                "nvfp4": "E2M1 + E4M3 per 16 + fp32 per tensor: block-scaled FP4 MMAs for "
                         "the forward GEMMs and the gate/up dgrad; the down dgrad and the "
                         "weight gradients on the BF16 engine"}.get(PRECISION),
            "data": "synthetic",
            "config": dict(workload_config(shape),
                           weight_grad_out="bf16" if args.bf16_wgrad else "fp32"),
            "grouped_gemm_tflops": gg_tflops,
            "grouped_gemm_frac_of_peak": gg_frac,
            "grouped_gemm_peak": "sustained bf16 of " + peaks["source"] + "; FP8 and FP4 GEMMs "
                                 "at the nominal 2x and 6x of it",
            "all_gemm_tflops": gemm_fl / (gemm_ms / 1e3) / 1e12 if gemm_ms else 0.0,
            "roofline": roof, "movers": movers_perf, "cpu_baseline": cpu, "e2e": e2e,
            "graph": graph_line,
            "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
            "clocks": clocks, "kernels": ksum,
            "kernel_timing": f"CUDA events around each kernel on {prof_steps} of the "
                             f"{args.steps} timed steps (one in {PROFILE_EVERY})",
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
