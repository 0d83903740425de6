"""The bounded wait every kernel of the library uses on its mbarriers, made
to run out on purpose: a wait on a phase that nothing completes (an
mbarrier no thread arrives on) gives up after its limit, the kernel records
MLA_STATUS_TIMEOUT in the status word and returns, and the context stays
usable for a decode that is then checked against the oracle. No GPU fault,
trap or hang is involved: the wait has a 2 ms limit."""
import numpy as np
import pytest
import torch

import mla_workloads as mw
from mla_testlib import DeviceWorkload, check_outputs, oracle_step

pytestmark = pytest.mark.gpu

MLA_STATUS_TIMEOUT = 0x8


@pytest.fixture(scope="module")
def lib():
    import paged_mla_decode_04_gb300 as m
    m.load_library()
    return m


def test_a_wait_nothing_completes_runs_out_and_reports_it(lib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.selftest_bounded_wait(status, arrive=False, limit_us=2000)
    torch.cuda.synchronize()
    assert int(status.item()) & MLA_STATUS_TIMEOUT


def test_a_completed_phase_returns_at_once(lib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    lib.selftest_bounded_wait(status, arrive=True, limit_us=1000000)
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert e0.elapsed_time(e1) < 100.0  # ms: far below the 1 s limit


def test_the_context_is_usable_after_a_wait_ran_out(lib):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.selftest_bounded_wait(status, arrive=False, limit_us=2000)
    wl = mw.make("v2lite", num_heads=16, context_lens=[0, 70, 300])
    dw = DeviceWorkload(wl, lib)
    out, lse = dw.step()
    assert int(status.item()) & MLA_STATUS_TIMEOUT
    assert lib.get_error(dw.ws) == 0
    ref_out, ref_lse = oracle_step(wl)
    check_outputs(out, lse, ref_out, ref_lse)
