"""Per-role event trace of the decode kernel (a developer tool).

Builds the library with -DMLA_TRACE into ``_build/trace/`` (the default build
carries no trace code), runs one plan + decode of a named workload after a
few untraced warm-up calls with L2 flushed, reads the per-CTA, per-role
records through ``mla_trace_read`` and prints, for the first CTAs, the medians
over 64-token tiles of the intervals between the roles' events and the tile
period, then the global-timer span of the whole grid. Event ids are read from
``csrc/trace.cuh`` so the two cannot drift apart.

    python -m paged_mla_decode_04_gb300.tracing v3 [v2lite fp8 long long_window]

Clock stamps are SM cycles (per SM, not comparable across SMs); the kernel
start and end stamps are global nanoseconds. Tracing adds stores to the
roles' loops, so absolute times run somewhat above an untraced launch. The
softmax events come from the first and last softmax warps, which hold no
rows when a row group has fewer than 128 (16 heads: only the producer, QK
and PV intervals are meaningful there).
"""
from __future__ import annotations

import ctypes
import os
import re
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
TRACE_DIR = os.path.join(HERE, "_build", "trace")
TRACE_LIB = os.path.join(TRACE_DIR, "libmla_decode_trace.so")
CTAS, ROLES, CAP = 160, 6, 2048   # kTraceCtas, kTraceRoles, kTraceCap in trace.cuh
PRODUCER, QK, PV, SM_FIRST, SM_LAST, KERNEL = range(6)


def event_ids() -> dict:
    """Name -> id of the TraceEvent enum in csrc/trace.cuh."""
    text = open(os.path.join(HERE, "csrc", "trace.cuh")).read()
    body = text[text.index("enum TraceEvent"):]
    body = body[body.index("{") + 1:body.index("};")]
    names = re.findall(r"^\s*kEv(\w+)", body, flags=re.M)
    first = int(re.search(r"kEv\w+\s*=\s*(\d+)", body).group(1))
    return {n: first + i for i, n in enumerate(names)}


def build_traced() -> str:
    from . import _build
    return _build.build(defines=["-DMLA_TRACE"], lib_path=TRACE_LIB, build_dir=TRACE_DIR)


def records(rec: np.ndarray, cnt: np.ndarray) -> dict:
    """(cta, role) -> (stamp, event, tile) arrays."""
    out = {}
    for c in range(rec.shape[0]):
        for r in range(rec.shape[1]):
            n = int(cnt[c, r])
            if n:
                x = rec[c, r, :n]
                out[(c, r)] = ((x & 0xFFFFFFFFFF).astype(np.int64), ((x >> 40) & 0xFF).astype(int),
                               ((x >> 48) & 0xFFFF).astype(int))
    return out


def times(tr: dict, cta: int, role: int, ev: int) -> dict:
    """tile -> stamp of `ev` recorded by `role` of `cta`."""
    if (cta, role) not in tr:
        return {}
    clk, e, t = tr[(cta, role)]
    m = e == ev
    return dict(zip(t[m].tolist(), clk[m].tolist()))


def summarize(tr: dict, ids: dict, ctas=(0, 1)) -> str:
    lines = []
    steps = [  # (label, (role, event) from, (role, event) to) per tile
        ("slot acquired -> copy issued", (PRODUCER, "SlotAcquired"), (PRODUCER, "TileIssued")),
        ("copy issued -> tile ready", (PRODUCER, "TileIssued"), (QK, "QkTileReady")),
        ("tile ready -> S free", (QK, "QkTileReady"), (QK, "QkSFree")),
        ("S free -> QK issued", (QK, "QkSFree"), (QK, "QkIssued")),
        ("QK issued -> S full", (QK, "QkIssued"), (SM_FIRST, "SmSFull")),
        ("S full -> partials sent", (SM_FIRST, "SmSFull"), (SM_FIRST, "SmSent")),
        ("sent -> peer partials in", (SM_FIRST, "SmSent"), (SM_FIRST, "SmXFull")),
        ("peer partials in -> P computed", (SM_FIRST, "SmXFull"), (SM_FIRST, "SmComputed")),
        ("P computed -> previous PV done", (SM_FIRST, "SmComputed"), (SM_FIRST, "SmPvDone")),
        ("previous PV done -> P in TMEM", (SM_FIRST, "SmPvDone"), (SM_FIRST, "SmOFixed")),
        ("P in TMEM -> PV issued", (PV, "PvOFixed"), (PV, "PvIssued")),
    ]
    for c in ctas:
        qk = times(tr, c, QK, ids["QkIssued"])
        if not qk:
            continue
        lines.append("CTA %d: %d tiles" % (c, len(qk)))
        for label, (r0, e0), (r1, e1) in steps:
            a, b = times(tr, c, r0, ids[e0]), times(tr, c, r1, ids[e1])
            d = [b[g] - a[g] for g in a if g in b]
            if d:
                lines.append("  %-32s median %7.0f cycles" % (label, np.median(d)))
        k = sorted(qk)
        if len(k) > 2:
            lines.append("  %-32s median %7.0f cycles" % ("tile period (QK issue)", np.median(np.diff([qk[g] for g in k]))))
    start = [v for c in range(CTAS) for v in times(tr, c, KERNEL, ids["GlobalStart"]).values()]
    end = [v for c in range(CTAS) for v in times(tr, c, KERNEL, ids["GlobalEnd"]).values()]
    if start and end:
        lines.append("grid: first CTA start to last CTA end %.1f us (median CTA end %.1f us)"
                     % ((max(end) - min(start)) / 1e3, (np.median(end) - min(start)) / 1e3))
    return "\n".join(lines)


def main(names) -> None:
    sys.path.insert(0, ROOT)
    import torch
    import mla_workloads as mw
    import paged_mla_decode_04_gb300 as m

    lib = m.load_library(build_traced())
    lib.mla_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.mla_trace_read.restype = ctypes.c_int
    ids = event_ids()
    dev = torch.device("cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    for name in names:
        wl = mw.make(name)
        if wl.dtype == mw.BF16:
            pool = m.KVPool(bf16(wl.pool_bf16))
        else:
            pool = m.KVPool(torch.zeros(wl.pool_bf16.shape, dtype=torch.uint8, device=dev), wl.kv_scale)
            rows = wl.pool_bf16.reshape(wl.num_layers, -1, mw.D_ROW)
            slots = torch.arange(rows.shape[1], dtype=torch.int64, device=dev)
            for layer in range(wl.num_layers):
                m.kv_write(pool, layer, bf16(rows[layer]), slots)
        q = bf16(wl.q)
        lens = torch.from_numpy(wl.context_lens).to(dev)
        table = torch.from_numpy(wl.block_table).to(dev)
        ws = m.alloc_workspace(wl.batch, wl.num_heads, dev)
        out = torch.empty(wl.batch, wl.num_heads, mw.D_CKV, dtype=torch.bfloat16, device=dev)

        def step():
            m.plan(lens, wl.num_heads, wl.page_size, wl.window, ws)
            m.decode(pool, wl.layer, q, lens, wl.softmax_scale, ws, out, block_table=table, window=wl.window)

        rec = np.zeros((CTAS, ROLES, CAP), np.uint64)
        cnt = np.zeros((CTAS, ROLES), np.uint32)
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        assert lib.mla_trace_read(rec.ctypes.data, cnt.ctypes.data) == 0  # drop the warm-up records
        flush.fill_(1)
        step()
        torch.cuda.synchronize()
        assert lib.mla_trace_read(rec.ctypes.data, cnt.ctypes.data) == 0
        assert m.get_error(ws) == 0
        print("== %s (%d records)" % (name, int(cnt.sum())))
        print(summarize(records(rec, cnt), ids))


if __name__ == "__main__":
    main(sys.argv[1:] or ["v3"])
