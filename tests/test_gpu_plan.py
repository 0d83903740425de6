"""The split-KV schedule written by the device plan, read back from the
workspace and checked for what any valid schedule must satisfy: every
64-token block of every (request, row group) lies in exactly one item, the
items of a request are contiguous in block order, items are grouped by
cluster behind the per-cluster start table, and a split request's partial
slots are consecutive and match its merge record (the plan/run split of
SGLang PR #32972 "Let Kimi-Linear use the paged MLA attention backends",
Correction; windows per FastDeploy PR #8049 "Support MLA_SWA", Motivation).

The plan keeps the cheaper of two schedules for batches of up to 1024
requests: the equal cut of the concatenated blocks, and a packed one that
splits only requests heavier than a cluster's share. Lognormal lengths (the
V3-shaped batch) take the packed one with few split requests; equal lengths
and a few very long requests keep the cut. Index work: checked exactly.

The workspace regions are read at the offsets the library's layout gives
them (header, items, cluster starts, split records, each 256-byte aligned)."""
from __future__ import annotations

from collections import defaultdict

import numpy as np
import pytest
import torch

import mla_workloads as mw
from mla_testlib import DeviceWorkload, check_outputs, oracle_step
from test_gpu_multi_query import oracle_q, run_q

pytestmark = pytest.mark.gpu

# 24 requests of 319-3195 tokens (a lognormal-like mix): at 16 clusters the
# equal cut would leave 22 fp32 partials, the packed schedule 8, with the
# same largest cluster load; the plan picks the packed one, single- and
# two-position alike (128 rows per request either way).
MIXED_LENS = [1849, 2840, 2008, 455, 339, 943, 1644, 1285, 3195, 1522, 1408, 539, 414, 2543, 931, 1588,
              343, 663, 364, 522, 1693, 319, 619, 1009]

HEADER = ["status", "batch", "num_heads", "page_size", "window", "num_clusters", "total_blocks",
          "num_items", "num_partials", "num_split", "planned", "q_len", "schedule"]
CUT, PACKED = 0, 1


@pytest.fixture(scope="module")
def lib():
    import paged_mla_decode_04_gb300 as m
    m.load_library()
    return m


def _align(x, a=256):
    return (x + a - 1) // a * a


def read_schedule(lib, ws, V):
    cmax = lib.num_clusters()
    w = ws.cpu().numpy()
    head = dict(zip(HEADER, w[:64].view(np.int32)[:len(HEADER)].tolist()))
    items_off = _align(64)
    cs_off = _align(items_off + 32 * (V + cmax))
    split_off = _align(cs_off + 4 * (cmax + 1))
    items = w[items_off:items_off + 32 * head["num_items"]].view(np.int32).reshape(-1, 8)
    cstart = w[cs_off:cs_off + 4 * (cmax + 1)].view(np.int32)
    split = w[split_off:split_off + 16 * head["num_split"]].view(np.int32).reshape(-1, 4)
    return head, items, cstart, split, cmax


def plan_and_check(lib, lens, heads, q_len=1, window=0, clusters=0):
    lens = np.asarray(lens, np.int32)
    G = (q_len * heads + 127) // 128
    V = len(lens) * G
    ws = lib.alloc_workspace_q(len(lens), q_len, heads)
    lib.plan_q(torch.from_numpy(lens).cuda(), q_len, heads, 64, window, ws, clusters)
    torch.cuda.synchronize()
    head, items, cstart, split, cmax = read_schedule(lib, ws, V)
    assert head["planned"] == 1 and head["status"] == 0 and head["schedule"] in (CUT, PACKED)
    C = head["num_clusters"]
    assert 1 <= C <= (clusters or cmax)
    assert head["num_items"] <= V + cmax and head["num_partials"] <= 2 * cmax
    # items grouped by cluster behind the start table (entries up to the
    # requested cluster count are written)
    cstart = cstart[:(clusters or cmax) + 1]
    assert cstart[0] == 0 and np.all(np.diff(cstart) >= 0)
    assert np.all(cstart[C:] == head["num_items"])
    for c in range(C):
        assert np.all(items[cstart[c]:cstart[c + 1], 6] == c)
    # every block of every (request, row group) exactly once
    expect = {}
    for b, L in enumerate(lens.tolist()):
        s = max(0, L + 1 - window) if window > 0 else 0
        first = s // 64
        n = (L + q_len - 1) // 64 - first + 1
        for g in range(G):
            expect[(b, 128 * g)] = (first, n, s, L + q_len)
    by_req = defaultdict(list)
    for it in items:
        by_req[(int(it[0]), int(it[7]))].append(it)
    assert set(by_req) == set(expect)
    records = {(int(r[0]), int(r[3])): r for r in split}
    assert len(records) == head["num_split"]
    slots = []
    for key, its in by_req.items():
        first, n, s, hi = expect[key]
        its = sorted(its, key=lambda x: x[1])
        assert its[0][1] == first and its[-1][2] == first + n
        assert all(a[2] == nxt[1] for a, nxt in zip(its, its[1:]))
        assert all(x[2] > x[1] and x[4] == s and x[5] == hi for x in its)
        if len(its) == 1:
            assert its[0][3] == -1 and key not in records
        else:
            r = records[key]
            assert r[1] == len(its)
            assert sorted(int(x[3]) for x in its) == list(range(r[2], r[2] + len(its)))
            slots += [int(x[3]) for x in its]
    assert len(slots) == len(set(slots)) == head["num_partials"]
    return head


@pytest.mark.parametrize("case", ["v3", "v3_7", "v3_window", "v2lite", "fp8", "long", "long_window",
                                  "tiny", "mtp", "ragged_small", "batch_1100"])
def test_schedule_covers_every_block_once(lib, case):
    if case.startswith("v3"):
        lens = mw.make("v3").context_lens
        head = plan_and_check(lib, lens, 128, clusters=7 if case == "v3_7" else 0,
                              window=300 if case == "v3_window" else 0)
    elif case in ("v2lite", "fp8", "long", "long_window"):
        wl = mw.make(case)
        head = plan_and_check(lib, wl.context_lens, wl.num_heads, window=wl.window)
    elif case == "tiny":
        head = plan_and_check(lib, [0, 5], 128)
    elif case == "mtp":
        rng = np.random.default_rng(7)
        head = plan_and_check(lib, rng.integers(0, 3000, size=40), 64, q_len=3)
    elif case == "ragged_small":
        head = plan_and_check(lib, [3000, 17, 900, 2500, 63, 64, 65, 8191], 128, clusters=5)
    else:
        rng = np.random.default_rng(1100)
        head = plan_and_check(lib, rng.integers(0, 200, size=1100), 16)
        assert head["schedule"] == CUT  # beyond 1024 requests only the cut is formed


def test_mixed_lengths_take_the_packed_schedule(lib):
    """Lognormal lengths: the packed schedule splits only the few requests
    heavier than a cluster's share, where the cut splits at nearly every
    cluster boundary."""
    head = plan_and_check(lib, mw.make("v3").context_lens, 128)
    assert head["schedule"] == PACKED
    assert head["num_split"] <= 20


def test_equal_lengths_keep_the_cut(lib):
    """256 equal requests over the clusters: whole requests cannot balance,
    so the cut (every cluster the same share) is kept."""
    head = plan_and_check(lib, mw.make("fp8").context_lens, 128)
    assert head["schedule"] == CUT


def test_packed_schedule_decode_matches_the_oracle(lib):
    """Decode under the packed schedule (whole requests written directly,
    the heavy ones split and merged): every request against the oracle."""
    wl = mw.make("v3", context_lens=MIXED_LENS)
    dw = DeviceWorkload(wl, lib)
    out, lse = dw.step(num_clusters=16)
    head = read_schedule(lib, dw.ws, wl.batch)[0]
    assert head["schedule"] == PACKED and 0 < head["num_partials"] < 22
    ref_out, ref_lse = oracle_step(wl)
    check_outputs(out, lse, ref_out, ref_lse)
    assert lib.get_error(dw.ws) == 0


def test_packed_schedule_with_two_positions_matches_the_oracle(lib):
    """The same mix with two query positions per request at 64 heads (one
    128-row group per request), through mla_decode_q."""
    wl = mw.make("v3", num_heads=64, context_lens=MIXED_LENS, q_len=2)
    head = plan_and_check(lib, MIXED_LENS, 64, q_len=2, clusters=16)
    assert head["schedule"] == PACKED
    out, lse = run_q(lib, wl, num_clusters=16)
    ref_out, ref_lse = oracle_q(wl)
    check_outputs(out, lse, ref_out, ref_lse)
