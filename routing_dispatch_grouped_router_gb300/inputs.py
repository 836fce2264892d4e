"""Seeded synthetic inputs for the MoE layer.

This module only draws numbers and stores them. It holds none of the layer's
arithmetic, so that both the CUDA path and the fp64 oracle can consume the same
inputs without sharing any code that computes the method.

Recipe (one seed per workload):
  * numpy ``Generator(PCG64(SeedSequence(seed)))`` spawned into sub-streams in
    a fixed order: x, W_r, then for every expert e (W_gate_e, W_up_e, W_down_e),
    then dy, then the Zipf rank permutation.  Experts therefore can be drawn
    one at a time and independently of each other.
  * x ~ N(0,1); W_r, W_gate, W_up ~ N(0, 1/d); W_down ~ N(0, 1/I); dy ~ N(0,1).
  * Values are drawn in float32 and stored as bfloat16 bit patterns (uint16),
    rounded to nearest even.
  * The imbalanced workload adds a per-expert router offset
    ``b_e = -beta * s * ln(rank_e)`` with s = 1.1 (a Zipf exponent) and
    ``rank`` a seeded permutation of 1..E; ``beta`` is a stored constant.

Arrays are returned as numpy arrays; bfloat16 tensors are uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import numpy as np

# Workload shapes.  Names describe the workload; sizes are the ones the layer
# is benchmarked and tested on.
WORKLOADS = {
    "tiny":       dict(T=256,   d=128,  E=8,   I=256,  k=2),
    "fine":       dict(T=4096,  d=2048, E=64,  I=1024, k=8),
    "large":      dict(T=8192,  d=7168, E=384, I=2048, k=8),
    "imbalanced": dict(T=16384, d=4096, E=128, I=1536, k=8, zipf_s=1.1),
    "mxfp8":      dict(T=16384, d=4096, E=128, I=1536, k=8, mb_tokens=2048, ring_slots=2),
    # the large workload's widths and rows per expert (T*k/E = 170.7) with 1/16
    # of its experts and tokens: its kernels at a size a full profiler capture
    # can replay (2 GB of weights); per-expert work scales by 16 to the large one
    "large_slice": dict(T=512, d=7168, E=24, I=2048, k=8),
    # the imbalanced workload's shape without its router bias, with the forward
    # expert GEMMs on NVFP4 operands
    "nvfp4":      dict(T=16384, d=4096, E=128, I=1536, k=8, nvfp4=True),
    # the nvfp4 workload's widths and rows per expert with 1/8 of its experts
    # and tokens (0.6 GB of weights): its kernels at a size a full profiler
    # capture can replay
    "nvfp4_slice": dict(T=2048, d=4096, E=16, I=1536, k=8, nvfp4=True),
}

# Scale of the Zipf offsets for the imbalanced workload (seed 0), found by
# bisection so that the hottest expert receives 8x the mean number of rows
# (tests/golden/zipf_beta.json, written by tests/golden/make_zipf_beta.py).
ZIPF_BETA = {"imbalanced": 0.391659}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); return bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    out = ((u + rounding) >> 16).astype(np.uint16)
    # keep NaN as a quiet NaN
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Shape:
    T: int
    d: int
    E: int
    I: int
    k: int

    @property
    def R(self) -> int:
        return self.T * self.k


def _streams(seed: int, E: int):
    root = np.random.SeedSequence(seed)
    # fixed spawn order: x, W_r, 3 per expert, dy, zipf permutation
    kids = root.spawn(2 + 3 * E + 2)
    return kids


def _normal_bf16(ss: np.random.SeedSequence, shape, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(ss))
    v = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return f32_to_bf16_bits(v)


def make_x(shape: Shape, seed: int) -> np.ndarray:
    return _normal_bf16(_streams(seed, shape.E)[0], (shape.T, shape.d), 1.0)


def make_router(shape: Shape, seed: int) -> np.ndarray:
    return _normal_bf16(_streams(seed, shape.E)[1], (shape.E, shape.d), shape.d ** -0.5)


def make_expert(shape: Shape, seed: int, e: int, kids=None):
    """(W_gate_e [I,d], W_up_e [I,d], W_down_e [d,I]) as bf16 bits."""
    kids = kids if kids is not None else _streams(seed, shape.E)
    base = 2 + 3 * e
    wg = _normal_bf16(kids[base + 0], (shape.I, shape.d), shape.d ** -0.5)
    wu = _normal_bf16(kids[base + 1], (shape.I, shape.d), shape.d ** -0.5)
    wd = _normal_bf16(kids[base + 2], (shape.d, shape.I), shape.I ** -0.5)
    return wg, wu, wd


def make_dy(shape: Shape, seed: int) -> np.ndarray:
    return _normal_bf16(_streams(seed, shape.E)[2 + 3 * shape.E], (shape.T, shape.d), 1.0)


def make_zipf_bias(shape: Shape, seed: int, s: float, beta: float) -> np.ndarray:
    """Per-expert float32 router offsets b_e = -beta*s*ln(rank_e)."""
    g = np.random.Generator(np.random.PCG64(_streams(seed, shape.E)[3 + 3 * shape.E]))
    rank = g.permutation(shape.E).astype(np.float64) + 1.0
    return (-beta * s * np.log(rank)).astype(np.float32)


def make_inputs(shape: Shape, seed: int, zipf_s: float | None = None,
                zipf_beta: float | None = None, experts=None) -> dict:
    """All inputs of one layer call.

    Returns a dict with ``x [T,d]``, ``w_router [E,d]``, ``w_gate_up [E,2I,d]``
    (gate rows 0..I-1 then up rows I..2I-1), ``w_down [E,d,I]``, ``dy [T,d]``
    as bf16 bits, and ``bias`` ([E] float32 or None).
    """
    kids = _streams(seed, shape.E)
    E, I, d = shape.E, shape.I, shape.d
    w_gu = np.empty((E, 2 * I, d), dtype=np.uint16)
    w_dn = np.empty((E, d, I), dtype=np.uint16)
    for e in range(E):
        wg, wu, wd = make_expert(shape, seed, e, kids)
        w_gu[e, :I] = wg
        w_gu[e, I:] = wu
        w_dn[e] = wd
    bias = None
    if zipf_s is not None:
        bias = make_zipf_bias(shape, seed, zipf_s, zipf_beta if zipf_beta is not None else 1.0)
    return dict(
        x=_normal_bf16(kids[0], (shape.T, d), 1.0),
        w_router=_normal_bf16(kids[1], (E, d), d ** -0.5),
        w_gate_up=w_gu,
        w_down=w_dn,
        dy=_normal_bf16(kids[2 + 3 * E], (shape.T, d), 1.0),
        bias=bias,
    )


def _expert_worker(args):
    """Pool worker: draws experts [e0, e1) into the shared-memory weights."""
    from multiprocessing import shared_memory
    name_gu, name_dn, shape_t, seed, e0, e1 = args
    shape = Shape(*shape_t)
    E, I, d = shape.E, shape.I, shape.d
    sgu = shared_memory.SharedMemory(name=name_gu)
    sdn = shared_memory.SharedMemory(name=name_dn)
    try:
        w_gu = np.ndarray((E, 2 * I, d), dtype=np.uint16, buffer=sgu.buf)
        w_dn = np.ndarray((E, d, I), dtype=np.uint16, buffer=sdn.buf)
        kids = _streams(seed, E)
        for e in range(e0, e1):
            wg, wu, wd = make_expert(shape, seed, e, kids)
            w_gu[e, :I] = wg
            w_gu[e, I:] = wu
            w_dn[e] = wd
        del w_gu, w_dn
    finally:
        sgu.close()
        sdn.close()
    return e1 - e0


class _SharedArrays:
    """Keeps shared-memory segments mapped while their arrays are alive."""

    def __init__(self, segs):
        self.segs = segs

    def __del__(self):
        for s in self.segs:
            try:
                s.close()
            except Exception:
                pass


def make_inputs_parallel(shape: Shape, seed: int, zipf_s: float | None = None,
                         zipf_beta: float | None = None, workers: int | None = None) -> dict:
    """make_inputs with the experts drawn by a pool of processes (spawned, so
    it is safe after CUDA initialisation).  Same values as make_inputs."""
    import multiprocessing as mp
    import os
    from multiprocessing import shared_memory
    E, I, d = shape.E, shape.I, shape.d
    n_gu = E * 2 * I * d * 2
    n_dn = E * d * I * 2
    sgu = shared_memory.SharedMemory(create=True, size=max(n_gu, 1))
    sdn = shared_memory.SharedMemory(create=True, size=max(n_dn, 1))
    try:
        workers = workers or min(E, len(os.sched_getaffinity(0)), 32)
        bounds = np.linspace(0, E, workers + 1).astype(int)
        jobs = [(sgu.name, sdn.name, (shape.T, shape.d, shape.E, shape.I, shape.k), seed,
                 int(bounds[i]), int(bounds[i + 1])) for i in range(workers) if bounds[i] < bounds[i + 1]]
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            assert sum(pool.map(_expert_worker, jobs)) == E
    finally:
        sgu.unlink()
        sdn.unlink()
    keep = _SharedArrays([sgu, sdn])
    w_gu = np.ndarray((E, 2 * I, d), dtype=np.uint16, buffer=sgu.buf)
    w_dn = np.ndarray((E, d, I), dtype=np.uint16, buffer=sdn.buf)
    kids = _streams(seed, E)
    bias = None
    if zipf_s is not None:
        bias = make_zipf_bias(shape, seed, zipf_s, zipf_beta if zipf_beta is not None else 1.0)
    return dict(
        x=_normal_bf16(kids[0], (shape.T, d), 1.0),
        w_router=_normal_bf16(kids[1], (E, d), d ** -0.5),
        w_gate_up=w_gu,
        w_down=w_dn,
        dy=_normal_bf16(kids[2 + 3 * E], (shape.T, d), 1.0),
        bias=bias,
        _shared=keep,
    )


def workload_inputs(name: str, seed: int = 0, parallel: bool = False) -> dict:
    """Inputs of a named workload (with its Zipf offsets where it has them)."""
    shape = workload_shape(name)
    w = WORKLOADS[name]
    zs = w.get("zipf_s")
    zb = ZIPF_BETA.get(name) if zs is not None else None
    if parallel:
        return make_inputs_parallel(shape, seed, zs, zb)
    return make_inputs(shape, seed, zs, zb)


def workload_shape(name: str) -> Shape:
    w = WORKLOADS[name]
    return Shape(T=w["T"], d=w["d"], E=w["E"], I=w["I"], k=w["k"])
