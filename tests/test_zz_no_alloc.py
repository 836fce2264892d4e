"""The dispatch plan entry point that allocates nothing
(mok_moe_dispatch_plan_noalloc), called through the C ABI, against the
workspace entry point (mok_moe_dispatch_plan): two calls in a row with
different shapes, outputs bit-identical (the plan's outputs are integers).

Some callers cannot allocate device memory where they call the plan, so this
variant keeps its scratch in a fixed array inside the library.  This file is
collected last so that a run stopping at the first failure has already run
every other test."""
import ctypes

import numpy as np
import pytest
import torch

from routing_dispatch_grouped_router_gb300 import _lib, api, build

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _plan(lib, idx, E, k, noalloc):
    T = idx.shape[0]
    desc = api.make_desc(T, 128, E, 128, k)
    dev = torch.from_numpy(idx).cuda()
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    pos = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    tok = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if noalloc:
        status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        code = lib.mok_moe_dispatch_plan_noalloc(ctypes.byref(desc), _ptr(dev), _ptr(counts),
                                                 _ptr(offsets), _ptr(pos), _ptr(tok),
                                                 _ptr(status), stream)
        assert code == 0, lib.mok_status_string(code)
        torch.cuda.synchronize()
        st = int(status.item())
    else:
        ws = torch.zeros(api.stage_workspace_size(desc), dtype=torch.uint8, device="cuda")
        code = lib.mok_moe_dispatch_plan(ctypes.byref(desc), _ptr(dev), _ptr(counts),
                                         _ptr(offsets), _ptr(pos), _ptr(tok), _ptr(ws),
                                         ws.numel(), stream)
        assert code == 0, lib.mok_status_string(code)
        st = api.device_status(ws)
    return st, [t.cpu().numpy() for t in (counts, offsets, pos, tok)]


def test_noalloc_plan_matches_workspace_plan_twice_in_a_row():
    build.build()
    lib = _lib.load()
    rng = np.random.default_rng(11)
    # a large plan first, then a small one over whatever the first left behind
    for T, E, k in [(16384, 128, 8), (1000, 7, 3)]:
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        st_ref, ref = _plan(lib, idx, E, k, noalloc=False)
        st_new, new = _plan(lib, idx, E, k, noalloc=True)
        assert st_ref == 0 and st_new == 0
        for a, b in zip(ref, new):
            assert np.array_equal(a, b)


def test_noalloc_plan_reports_a_bad_index_in_the_callers_status():
    """An expert index outside [0, E) is skipped on the device and reported as
    MOK_ERR_DEVICE_INDEX (17) in the caller's status word, as the workspace
    plan reports it in its workspace; both plans agree on every output."""
    lib = _lib.load()
    T, E, k = 200, 9, 3
    rng = np.random.default_rng(12)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    idx[17, 2] = E
    st_ref, ref = _plan(lib, idx, E, k, noalloc=False)
    st_new, new = _plan(lib, idx, E, k, noalloc=True)
    assert st_ref == 17 and st_new == 17
    for a, b in zip(ref, new):
        assert np.array_equal(a, b)
    assert new[2][17, 2] == -1


def test_noalloc_plan_rejects_problems_beyond_its_scratch():
    lib = _lib.load()
    desc = api.make_desc(200000, 128, 64, 128, 8)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    code = lib.mok_moe_dispatch_plan_noalloc(ctypes.byref(desc), _ptr(dummy), _ptr(dummy),
                                             _ptr(dummy), _ptr(dummy), _ptr(dummy), None, None)
    assert code == 6  # MOK_ERR_SCRATCH_LIMIT, nothing enqueued
