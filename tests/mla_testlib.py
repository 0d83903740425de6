"""Shared helpers of the GPU parity tests: move a seeded workload to the
device, run the library's step (write, plan, decode) and the oracle's, and
compare."""
from __future__ import annotations

import numpy as np
import torch

import mla_workloads as mw
import oracle

TOL_BF16 = 1e-2   # max|gpu - ref| <= TOL * max|ref| for a bf16 cache
TOL_FP8 = 4e-2    # same, fp8 e4m3 cache


def check_outputs(gpu_out, gpu_lse, ref_out, ref_lse, tol=TOL_BF16):
    """Outputs within the stated tolerance of max|ref|; returns the error.
    lse: the two CTAs of a pair exchange their partial scores, scaled to
    log2 units, as fp16 (relative error 2^-11 of a partial), so lse moves
    by up to ~1e-3 of the score magnitude: 2e-3 relative for bf16 caches,
    1e-2 for fp8 ones (their scores are larger)."""
    err = rel_err(gpu_out, ref_out)
    assert err <= tol, "out rel err %.3e" % err
    lerr = np.abs(gpu_lse - ref_lse).max() if ref_lse.size else 0.0
    ltol = 1e-2 if tol == TOL_FP8 else 2e-3
    assert lerr <= ltol * max(1.0, np.abs(ref_lse).max() if ref_lse.size else 1.0), \
        "lse err %.3e" % lerr
    return err


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    if ref.size == 0:
        return 0.0
    return float(np.abs(gpu - ref).max() / max(np.abs(ref).max(), 1e-30))


class DeviceWorkload:
    """Device copies of a workload; the pool is filled by the library's own
    latent write for fp8 (bf16 pools are uploaded as is)."""

    def __init__(self, wl: mw.Workload, lib, device="cuda"):
        self.wl = wl
        self.lib = lib
        if wl.dtype == mw.BF16:
            self.pool = lib.KVPool(bf16_tensor(wl.pool_bf16, device))
        else:
            data = torch.zeros(wl.pool_bf16.shape, dtype=torch.uint8, device=device)
            self.pool = lib.KVPool(data, wl.kv_scale)
            rows = wl.pool_bf16.reshape(wl.num_layers, -1, mw.D_ROW)
            slots = torch.arange(rows.shape[1], dtype=torch.int64, device=device)
            for layer in range(wl.num_layers):
                lib.kv_write(self.pool, layer, bf16_tensor(rows[layer], device), slots)
        self.q = bf16_tensor(wl.q, device)
        self.new_rows = bf16_tensor(wl.new_rows, device)
        self.slots = torch.from_numpy(wl.slot_mapping).to(device)
        self.lens = torch.from_numpy(wl.context_lens).to(device)
        self.block_table = torch.from_numpy(wl.block_table).to(device)
        self.indptr = torch.from_numpy(wl.page_indptr).to(device)
        self.ids = torch.from_numpy(wl.page_ids).to(device)
        self.ws = lib.alloc_workspace(wl.batch, wl.num_heads, device)
        self.out = torch.empty(wl.batch, wl.num_heads, mw.D_CKV, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(wl.batch, wl.num_heads, dtype=torch.float32, device=device)

    def step(self, layer=None, window=None, num_clusters=0, csr=False, write=True):
        wl, lib = self.wl, self.lib
        layer = wl.layer if layer is None else layer
        window = wl.window if window is None else window
        if write:
            lib.kv_write(self.pool, layer, self.new_rows, self.slots, self.ws)
        lib.plan(self.lens, wl.num_heads, wl.page_size, window, self.ws, num_clusters)
        kw = dict(page_indptr=self.indptr, page_ids=self.ids) if csr else \
            dict(block_table=self.block_table)
        lib.decode(self.pool, layer, self.q, self.lens, wl.softmax_scale, self.ws, self.out,
                   window=window, lse=self.lse, **kw)
        torch.cuda.synchronize()
        return f64(self.out), self.lse.cpu().numpy().astype(np.float64)


def oracle_pool_after_write(wl: mw.Workload, layer=None, write=True, pages=None) -> np.ndarray:
    """The oracle's pool bytes after this step's latent write. For fp8 the
    oracle quantises the pool itself (every row, or only `pages`)."""
    layer = wl.layer if layer is None else layer
    if wl.dtype == mw.BF16:
        pool = wl.pool_bf16.copy()
    else:
        pool = np.zeros(wl.pool_bf16.shape, np.uint8)
        ps = wl.page_size
        for li in range(wl.num_layers):
            if pages is None:
                rows = wl.pool_bf16[li].reshape(-1, mw.D_ROW)
                slots = np.arange(rows.shape[0], dtype=np.int64)
            else:
                pg = np.asarray(sorted(set(int(p) for p in pages)), np.int64)
                rows = wl.pool_bf16[li][pg].reshape(-1, mw.D_ROW)
                slots = (pg[:, None] * ps + np.arange(ps)[None, :]).reshape(-1)
            oracle.kv_write(pool, wl.dtype, wl.num_layers, wl.num_pages, ps, wl.kv_scale, li,
                            rows, slots)
    if write:
        oracle.kv_write(pool, wl.dtype, wl.num_layers, wl.num_pages, wl.page_size, wl.kv_scale,
                        layer, wl.new_rows, wl.slot_mapping)
    return pool


def oracle_step(wl: mw.Workload, layer=None, window=None, requests=None, write=True,
                pool=None):
    layer = wl.layer if layer is None else layer
    window = wl.window if window is None else window
    if pool is None:
        pages = None
        if requests is not None and wl.dtype != mw.BF16:
            pages = np.concatenate([wl.block_table[b][wl.block_table[b] >= 0] for b in requests])
        pool = oracle_pool_after_write(wl, layer, write, pages)
    q = oracle.bf16_bits_to_f64(wl.q)
    return oracle.decode(pool, wl.dtype, wl.num_layers, wl.num_pages, wl.page_size, wl.kv_scale,
                         layer, q, wl.context_lens, wl.softmax_scale, window,
                         block_table=wl.block_table, requests=requests)

