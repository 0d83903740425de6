"""The oracle's decode of every request of a workload, the requests spread
over spawned processes. The oracle itself stays single-threaded (each
process decodes whole requests); the pool and q are shared through files
that every process maps. Spawned, not forked: a process forked after CUDA
initialisation can hang. This module imports no torch, so the workers start
quickly."""
from __future__ import annotations

import os

import numpy as np

import mla_workloads as mw
import oracle


def _oracle_worker(args):
    """Runs in a spawned process: map the saved pool and q, decode a subset
    of requests with the oracle as it stands."""
    meta, requests = args
    pool = np.load(meta["pool_file"], mmap_mode="r")
    q = np.load(meta["q_file"], mmap_mode="r")
    out, lse = oracle.decode(pool, meta["dtype"], meta["num_layers"], meta["num_pages"],
                             meta["page_size"], meta["kv_scale"], meta["layer"], q,
                             meta["context_lens"], meta["softmax_scale"], meta["window"],
                             block_table=meta["block_table"], requests=requests)
    return requests, out, lse


def oracle_decode_all(wl: mw.Workload, pool: np.ndarray, procs: int = 0, layer=None,
                      window=None):
    """The oracle's decode of every request of `wl` on `pool` (the oracle's own
    pool bytes after the step's write): (out [B, H, 512], lse [B, H])."""
    import multiprocessing as mp
    import tempfile
    layer = wl.layer if layer is None else layer
    window = wl.window if window is None else window
    procs = procs or min(16, os.cpu_count() or 1)
    with tempfile.TemporaryDirectory(prefix="mla_oracle_") as tmp:
        pool_file = os.path.join(tmp, "pool.npy")
        q_file = os.path.join(tmp, "q.npy")
        np.save(pool_file, np.ascontiguousarray(pool))
        np.save(q_file, oracle.bf16_bits_to_f64(wl.q))
        meta = dict(pool_file=pool_file, q_file=q_file, dtype=wl.dtype,
                    num_layers=wl.num_layers, num_pages=wl.num_pages, page_size=wl.page_size,
                    kv_scale=wl.kv_scale, layer=layer, context_lens=wl.context_lens,
                    softmax_scale=wl.softmax_scale, window=window, block_table=wl.block_table)
        # longest requests first, dealt round-robin, so the processes finish together
        order = np.argsort(-wl.attended, kind="stable")
        chunks = [sorted(order[k::procs].tolist()) for k in range(procs)]
        chunks = [c for c in chunks if c]
        out = np.zeros((wl.batch, wl.num_heads, mw.D_CKV), np.float64)
        lse = np.zeros((wl.batch, wl.num_heads), np.float64)
        with mp.get_context("spawn").Pool(len(chunks)) as p:
            for req, o, l in p.imap_unordered(_oracle_worker, [(meta, c) for c in chunks]):
                out[req] = o
                lse[req] = l
        return out, lse
