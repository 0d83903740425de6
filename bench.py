"""Paged MLA decode bench on GB300.

One step = the whole decode hot path for one batch: latent write of the new
tokens through slot_mapping, split-KV plan, decode (split kernel + merge),
and the W_UV projection, on the DeepSeek-V3-shaped workload (128 heads,
batch 128, lognormal context lengths, page size 64, bf16 576-d latent cache).
Inputs are seeded synthetic data; L2 is flushed between timed steps.

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]
                  [--config v3|v2lite|fp8|long|long_window]

Prints one JSON line. `--impl reference` times the CPU oracle (the reference
arm of this workload) on the host cores on a bounded sample of requests.
Under torchrun (N > 1) each rank runs an independent replica (the path does
not shard across GPUs), timing is max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_workloads as mw  # noqa: E402

# dram__bytes_read.sum + dram__bytes_write.sum of one mla_decode_kernel launch
# from an ncu capture, keyed by workload and by the digest of the decode
# kernel's sources at capture time (decode_source_digest): the figure is
# printed only for the kernel it was measured on, null for any other.
MEASURED_TRAFFIC = {("v3", "1b30d15897f2214c"): 365.50e6, ("fp8", "1b30d15897f2214c"): 666.80e6}
DECODE_SOURCES = ["decode_sm103.cu", "ptx.cuh", "mla_internal.h", "trace.cuh"]
METRIC = "paged MLA decode µs/step, KV GB/s & TFLOP/s as % of GB300 roofline"
UNIT = "us/step"
L2_FLUSH_BYTES = 512 << 20


def decode_source_digest() -> str:
    """Short digest of the decode kernel's source files."""
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, "paged_mla_decode_04_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, ws, device):
    """Element-wise max of per-rank timings (each rank runs its own replica:
    the job's step takes as long as its slowest rank)."""
    if ws <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_sample_requests(wl: mw.Workload, target_tokens: int):
    """A deterministic, length-representative subset: every k-th request."""
    att = wl.attended
    k = max(1, int(np.ceil(att.sum() / max(target_tokens, 1))))
    return list(range(0, wl.batch, k))


def run_oracle_sample(wl: mw.Workload, requests):
    import oracle
    q = oracle.bf16_bits_to_f64(wl.q)
    t0 = time.perf_counter()
    oracle.decode(wl.pool_bf16 if wl.dtype == mw.BF16 else wl.extra["pool_fp8"], wl.dtype,
                  wl.num_layers, wl.num_pages, wl.page_size, wl.kv_scale, wl.layer, q,
                  wl.context_lens, wl.softmax_scale, wl.window, block_table=wl.block_table,
                  requests=requests)
    return time.perf_counter() - t0


def prepare_fp8_host_pool(wl: mw.Workload):
    """The oracle's own quantised pool (only needed by the CPU legs)."""
    import oracle
    pool = np.zeros(wl.pool_bf16.shape, np.uint8)
    for li in range(wl.num_layers):
        rows = wl.pool_bf16[li].reshape(-1, mw.D_ROW)
        oracle.kv_write(pool, wl.dtype, wl.num_layers, wl.num_pages, wl.page_size, wl.kv_scale,
                        li, rows, np.arange(rows.shape[0], dtype=np.int64))
    wl.extra["pool_fp8"] = pool


def cpu_leg(wl: mw.Workload, sample_tokens: int):
    """Oracle time on a bounded sample, scaled by attended tokens to the full
    batch (us/step)."""
    req = cpu_sample_requests(wl, sample_tokens)
    secs = run_oracle_sample(wl, req)
    att = wl.attended
    scale = float(att.sum()) / float(att[req].sum())
    return secs * scale * 1e6, req, secs


def bench_reference(args, wl, ws, rank):
    if rank != 0:
        return
    if wl.dtype != mw.BF16:
        prepare_fp8_host_pool(wl)
    times = []
    req = None
    for i in range(args.warmup + args.steps):
        us, req, secs = cpu_leg(wl, args.cpu_sample_tokens)
        if i >= args.warmup:
            times.append(us)
    v = float(np.mean(times))
    sample = "requests %s (%d of %d, %d attended tokens of %d), extrapolated by tokens" % (
        req[:4] + ["..."] if len(req) > 4 else req, len(req), wl.batch,
        int(wl.attended[req].sum()), int(wl.attended.sum()))
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(wl, args),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_dict(wl, args):
    return {"workload": mw.DESCRIPTIONS[args.config], "batch": wl.batch, "heads": wl.num_heads,
            "page_size": wl.page_size, "kv_dtype": "bf16" if wl.dtype == mw.BF16 else "fp8_e4m3",
            "window": wl.window, "attended_tokens": int(wl.attended.sum()),
            "num_layers": wl.num_layers, "seed": mw.SEEDS[args.config],
            "l2": "flushed (512 MB write) before every timed step"}


def bench_ours(args, wl, ws, rank, local):
    import torch
    import paged_mla_decode_04_gb300 as m

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    m.load_library()
    stream = torch.cuda.current_stream()

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    if wl.dtype == mw.BF16:
        pool = m.KVPool(bf16(wl.pool_bf16))
    else:
        pool = m.KVPool(torch.zeros(wl.pool_bf16.shape, dtype=torch.uint8, device=dev), wl.kv_scale)
        rows = wl.pool_bf16.reshape(wl.num_layers, -1, mw.D_ROW)
        slots_all = torch.arange(rows.shape[1], dtype=torch.int64, device=dev)
        for li in range(wl.num_layers):
            m.kv_write(pool, li, bf16(rows[li]), slots_all)
    B, H = wl.batch, wl.num_heads
    q = bf16(wl.q)
    new_rows = bf16(wl.new_rows)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    lens = torch.from_numpy(wl.context_lens).to(dev)
    table = torch.from_numpy(wl.block_table).to(dev)
    wsb = m.alloc_workspace(B, H, dev)
    out = torch.empty(B, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, dtype=torch.float32, device=dev)
    w_uv = bf16(wl.w_uv) if wl.w_uv is not None else None
    y = torch.empty(B, H, 128, dtype=torch.bfloat16, device=dev) if w_uv is not None else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def prep():
        m.kv_write(pool, wl.layer, new_rows, slots, wsb)
        m.plan(lens, H, wl.page_size, wl.window, wsb)

    def attend():
        m.decode(pool, wl.layer, q, lens, wl.softmax_scale, wsb, out, block_table=table,
                 window=wl.window, lse=lse)

    def project():
        if w_uv is not None:
            m.uv_project(out, w_uv, y, wsb)

    parts = [prep, attend, project]

    def whole():
        for f in parts:
            f()

    for _ in range(2):                      # eager warm-up (loads, first-call set-up)
        whole()
    torch.cuda.synchronize()
    if not args.eager:
        # The step as a serving loop runs it: captured once as a CUDA graph
        # (the library neither allocates nor synchronises, and its tensor
        # maps hold these fixed buffers) and replayed every step. Each part
        # is also captured alone, for the breakdown.
        def capture(f):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                f()
            return g.replay
        whole_fn = capture(whole)
        # (without W_UV the projection part is empty: nothing to capture)
        parts = [capture(f) if (f is not project or w_uv is not None) else f for f in parts]
    else:
        whole_fn = whole

    def step(marks=None):
        if marks:
            marks[0].record(stream)
        whole_fn()
        if marks:
            marks[1].record(stream)

    def step_parts(marks):
        for k, f in enumerate(parts):
            marks[k].record(stream)
            f()
        marks[3].record(stream)

    launches_per_step = 4 + (1 if w_uv is not None else 0)   # write, plan, split, merge (+uv)
    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    assert m.get_error(wsb) == 0, "device status set during warm-up"

    marks = [[ev() for _ in range(2)] for _ in range(args.steps)]
    pmarks = [[ev() for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(1)
        step(marks[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    # The breakdown: the same steps run part by part (one graph each).
    for i in range(args.steps):
        flush.fill_(1)
        step_parts(pmarks[i])
    torch.cuda.synchronize()
    # The decode call's own duration (split + merge kernels), for the
    # roofline: launched eagerly behind the L2 flush, which runs long
    # enough for the host to queue both launches, with events on the
    # launching stream on both sides (no graph-launch gap inside).
    dmarks = [(ev(), ev()) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(1)
        dmarks[i][0].record(stream)
        attend()
        dmarks[i][1].record(stream)
    torch.cuda.synchronize()
    step_ms = [mk[0].elapsed_time(mk[1]) for mk in marks]
    prep_ms = [mk[0].elapsed_time(mk[1]) for mk in pmarks]
    part_ms = [mk[1].elapsed_time(mk[2]) for mk in pmarks]
    uv_ms = [mk[2].elapsed_time(mk[3]) for mk in pmarks]
    dec_ms = [a.elapsed_time(b) for a, b in dmarks]
    t_step = float(np.mean(step_ms))
    t_dec = float(np.mean(dec_ms))
    t_step, t_dec = max_over_ranks([t_step, t_dec], ws, dev)
    assert m.get_error(wsb) == 0, "device status set during the timed steps"

    # End to end through the public API: pinned host inputs copied in, the
    # step's result copied out, every step.
    h_q = torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_rows = torch.from_numpy(wl.new_rows.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_slots = torch.from_numpy(wl.slot_mapping).pin_memory()
    h_lens = torch.from_numpy(wl.context_lens).pin_memory()
    h_table = torch.from_numpy(wl.block_table).pin_memory()
    res = y if y is not None else out
    h_res = torch.empty(res.shape, dtype=res.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_rows, h_slots, h_lens, h_table))
    d2h = h_res.numel() * h_res.element_size()

    def e2e_step():
        q.copy_(h_q, non_blocking=True)
        new_rows.copy_(h_rows, non_blocking=True)
        slots.copy_(h_slots, non_blocking=True)
        lens.copy_(h_lens, non_blocking=True)
        table.copy_(h_table, non_blocking=True)
        step()
        h_res.copy_(res, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e_marks = [(ev(), ev()) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(1)
        e_marks[i][0].record(stream)
        e2e_step()
        e_marks[i][1].record(stream)
    torch.cuda.synchronize()
    t_e2e = float(np.mean([a.elapsed_time(b) for a, b in e_marks]))
    (t_e2e,) = max_over_ranks([t_e2e], ws, dev)

    if rank != 0:
        return
    hbm, tc_burst, tc_sust, peak_src = load_peaks()
    byts, flops = mw.alg_bytes_flops(wl)
    kv_gbs = byts / (t_dec * 1e-3) / 1e9
    tflops = flops / (t_dec * 1e-3) / 1e12
    t_roof_ms = max(byts / (hbm * 1e9), flops / (tc_burst * 1e12)) * 1e3
    bound = "hbm" if byts / (hbm * 1e9) >= flops / (tc_burst * 1e12) else "tensor"
    achieved = kv_gbs if bound == "hbm" else tflops
    peak = hbm if bound == "hbm" else tc_burst
    cpu = None
    if ws == 1 and not args.no_cpu_baseline:
        if wl.dtype != mw.BF16:
            prepare_fp8_host_pool(wl)
        us, req, secs = cpu_leg(wl, args.cpu_sample_tokens)
        cpu = {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "%d of %d requests (every %d-th; %d of %d attended tokens), %.1f s of "
                         "single-thread fp64 work, extrapolated by attended tokens" % (
                             len(req), wl.batch, req[1] - req[0] if len(req) > 1 else 1,
                             int(wl.attended[req].sum()), int(wl.attended.sum()), secs)}
    line = {
        "metric": METRIC, "value": t_step * 1e3, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        # tensor-core operand type: bf16 pools as stored, e4m3 pools widened to f16
        "dtype": "bf16" if wl.dtype == mw.BF16 else "f16",
        "data": "synthetic", "config": config_dict(wl, args),
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                     "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": achieved / peak,
                     "traffic": args.traffic if args.traffic is not None else MEASURED_TRAFFIC.get(
                         (args.config, decode_source_digest())),
                     "kernel_digest": decode_source_digest(),
                     "kernel": "mla_decode (split + merge kernels)",
                     "peak_source": peak_src + " (burst)" + (
                         "" if wl.dtype == mw.BF16 or bound == "hbm" else "; dense f16 rate = bf16 rate")},
        "launch": "eager ctypes calls" if args.eager else "the step replayed as one CUDA graph",
        "decode_us": t_dec * 1e3, "kv_gbs": kv_gbs, "tflops": tflops,
        "roofline_time_us": t_roof_ms * 1e3, "roofline_frac_of_step": t_roof_ms / t_step,
        "roofline_frac_of_decode": t_roof_ms / t_dec,
        "breakdown_us": {"write+plan": float(np.mean(prep_ms)) * 1e3, "decode": float(np.mean(part_ms)) * 1e3,
                         "uv_project": float(np.mean(uv_ms)) * 1e3,
                         "note": "each part replayed alone as its own graph (launch gaps included)"},
        "alg_bytes": byts, "alg_flops": flops,
        "cpu_baseline": cpu,
        "e2e": {"value": t_e2e * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="v3", choices=list(mw.CONFIGS))
    ap.add_argument("--cpu-sample-tokens", type=int, default=30000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="launch every call from Python each step instead of replaying CUDA graphs")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per decode launch from an ncu capture of this kernel "
                         "(default: the committed capture for this workload, if any)")
    args = ap.parse_args()
    ws, rank, local = dist_env()
    if ws > 1:
        import torch
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    wl = mw.make(args.config)
    if args.impl == "reference":
        bench_reference(args, wl, ws, rank)
    else:
        bench_ours(args, wl, ws, rank, local)
    if ws > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
