"""The allocation-free decode entry point (mla_decode_noalloc), called
through the C ABI, against the workspace entry points (mla_decode_plan +
mla_decode) on the same inputs: same results within the parity tolerance,
on two calls in a row (the shared scratch keeps the previous call's bytes).
This file sorts last so that a run stopping at the first failure has run
every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import mla_workloads as mw
from mla_testlib import DeviceWorkload, f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,heads,lens", [("v3", 128, [3000, 17, 900, 2500, 0, 64]),
                                             ("v2lite", 16, [2992, 130, 1333, 3992]),
                                             ("fp8", 128, [4096, 33, 1500, 0])])
def test_noalloc_decode_matches_workspace_decode_twice(name, heads, lens):
    import paged_mla_decode_04_gb300 as m
    lib = m.load_library()
    wl = mw.make(name, num_heads=heads, context_lens=lens)
    dw = DeviceWorkload(wl, m)
    ref_out, ref_lse = dw.step()          # writes the new rows, then plan + decode
    stream = torch.cuda.current_stream().cuda_stream
    pool = dw.pool._c()
    for call in range(2):
        out = torch.full_like(dw.out, float("nan"))
        lse = torch.full_like(dw.lse, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = lib.mla_decode_noalloc(ctypes.byref(pool), wl.layer, dw.q.data_ptr(), None,
                                    dw.block_table.data_ptr(), dw.block_table.shape[1],
                                    dw.lens.data_ptr(), wl.batch, wl.num_heads,
                                    ctypes.c_float(wl.softmax_scale), wl.window, 0,
                                    out.data_ptr(), lse.data_ptr(), status.data_ptr(), stream)
        assert rc == 0, "call %d returned %d" % (call, rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        # the same plan and kernels as the workspace path: identical bits
        assert np.array_equal(f64(out), ref_out), "call %d" % call
        assert np.array_equal(lse.cpu().numpy().astype(np.float64), ref_lse), "call %d" % call


def test_noalloc_rejects_calls_beyond_its_scratch():
    import paged_mla_decode_04_gb300 as m
    lib = m.load_library()
    wl = mw.make("tiny")
    dw = DeviceWorkload(wl, m)
    pool = dw.pool._c()
    too_many = 1 << 20                    # far beyond what the fixed scratch holds
    rc = lib.mla_decode_noalloc(ctypes.byref(pool), 0, dw.q.data_ptr(), None,
                                dw.block_table.data_ptr(), dw.block_table.shape[1],
                                dw.lens.data_ptr(), too_many, 128, ctypes.c_float(0.07), 0, 0,
                                dw.out.data_ptr(), None, None, 0)
    assert rc == -3                       # MLA_ERR_WORKSPACE, nothing launched


def test_noalloc_rejected_call_leaves_the_previous_call_intact():
    """A call with a bad argument (here a layer out of range) is refused before
    it touches the shared scratch: an earlier call still in flight on the same
    stream finishes with its own schedule and result."""
    import paged_mla_decode_04_gb300 as m
    lib = m.load_library()
    wl = mw.make("v3", num_heads=128, context_lens=[3000, 17, 900])
    dw = DeviceWorkload(wl, m)
    ref_out, ref_lse = dw.step()
    stream = torch.cuda.current_stream().cuda_stream
    pool = dw.pool._c()
    out = torch.full_like(dw.out, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    args = (dw.q.data_ptr(), None, dw.block_table.data_ptr(), dw.block_table.shape[1],
            dw.lens.data_ptr(), wl.batch, wl.num_heads, ctypes.c_float(wl.softmax_scale), wl.window, 0)
    rc = lib.mla_decode_noalloc(ctypes.byref(pool), wl.layer, *args, out.data_ptr(), None,
                                status.data_ptr(), stream)
    assert rc == 0
    bad_out = torch.empty_like(dw.out)
    rc = lib.mla_decode_noalloc(ctypes.byref(pool), wl.num_layers, *args, bad_out.data_ptr(), None,
                                None, stream)
    assert rc == -1                       # MLA_ERR_ARG, nothing enqueued
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(f64(out), ref_out)
