"""Seeded synthetic inputs for paged MLA decode.

This module is shared by the tests, the bench and the oracle checks. It only
draws random numbers and lays them out (lengths, page permutations, block
tables, slot numbers, bf16 bit patterns); it holds none of the attention,
quantisation or absorption arithmetic.

Workload shapes follow the configurations this library is measured on:
DeepSeek-V2-Lite-shaped (16 heads), DeepSeek-V3-shaped (128 heads), an fp8
latent cache, and long contexts with and without a sliding window. Every
pool has two layers sharing one buffer with layer-indexed slots (the
per-layer cache dimension of MoE-Infinity PR #195 "DeepSeek-V2/V3
paged-attention shim (MLA)", Root causes 5), and physical pages handed out in
a random permutation. No public dataset or trained weight is involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

D_CKV = 512
D_ROPE = 64
D_ROW = D_CKV + D_ROPE
D_NOPE = 128
D_V = 128
BF16 = 0
FP8_E4M3 = 1
SPARE_PAGES = 16


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest even) and return the bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


@dataclass
class Workload:
    name: str
    batch: int
    num_heads: int
    page_size: int
    dtype: int                      # BF16 or FP8_E4M3 (cache storage type)
    context_lens: np.ndarray        # int32 [B]: tokens cached before this step
    window: int                     # 0 = full attention
    num_layers: int
    layer: int                      # layer the step writes and decodes
    num_pages: int                  # pages per layer in the pool
    block_table: np.ndarray         # int32 [B, max_blocks], -1 past the end
    page_indptr: np.ndarray         # int32 [B+1]  (CSR form of the same table)
    page_ids: np.ndarray            # int32 [nnz]
    pool_bf16: np.ndarray           # uint16 bf16 bits [NL, P, ps, 576]: cache values
    kv_scale: float                 # fp8 only: per-pool scale (amax / 448); 1.0 for bf16
    q: np.ndarray                   # uint16 bf16 bits [B, H, 576]: absorbed query
    new_rows: np.ndarray            # uint16 bf16 bits [B, 576]: this step's latent rows
    slot_mapping: np.ndarray        # int64 [B]: slot (within the layer) of position L_b
    softmax_scale: float = 192.0 ** -0.5
    w_uv: Optional[np.ndarray] = None   # uint16 bf16 bits [H, 512, 128]
    extra: dict = field(default_factory=dict)
    q_len: int = 1                  # query positions per request (q is [B, q_len, H, 576] if > 1)

    @property
    def attended(self) -> np.ndarray:
        """Tokens each request attends over all its query positions (new
        tokens included)."""
        L = self.context_lens.astype(np.int64)
        end = L + self.q_len
        if self.window > 0:
            return end - np.maximum(0, L + 1 - self.window)
        return end

    @property
    def row_bytes(self) -> int:
        return D_ROW * (2 if self.dtype == BF16 else 1)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    chunk = 1 << 26
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[s:e] = f32_to_bf16_bits(x)
    return out.reshape(shape)


def _lengths(name: str, rng: np.random.Generator, batch: int) -> np.ndarray:
    if name == "tiny":
        return np.array([37, 61][:batch] + [49] * max(0, batch - 2), np.int32)
    if name == "v2lite":
        return rng.integers(512, 4096, size=batch, endpoint=True).astype(np.int32)
    if name == "v3":
        z = rng.standard_normal(batch)
        L = np.exp(np.log(2048.0) + 0.6 * z)
        return np.clip(np.rint(L), 256, 8192).astype(np.int32)
    if name == "fp8":
        return np.full(batch, 4096, np.int32)
    if name in ("long", "long_window"):
        return rng.integers(32768, 131072, size=batch, endpoint=True).astype(np.int32)
    raise KeyError(name)


# name -> (batch, heads, page_size, dtype, window, value std, has W_UV)
CONFIGS = {
    "tiny": (2, 16, 16, BF16, 0, 0.1, True),
    "v2lite": (64, 16, 64, BF16, 0, 0.1, False),
    "v3": (128, 128, 64, BF16, 0, 0.1, True),
    "fp8": (256, 128, 64, FP8_E4M3, 0, 1.0, False),
    "long": (8, 128, 64, BF16, 0, 0.1, False),
    "long_window": (8, 128, 64, BF16, 4096, 0.1, False),
}

DESCRIPTIONS = {
    "tiny": "tiny MLA decode: B2 H16 L{37,61} ps16, bf16 576-d latent",
    "v2lite": "DeepSeek-V2-Lite-shaped decode: B64 H16 L~U[512,4096] ps64 bf16",
    "v3": "DeepSeek-V3-shaped decode: B128 H128 L~lognormal(median 2048, sigma 0.6) "
          "clipped [256,8192] ps64 bf16, + W_UV to v_head_dim 128",
    "fp8": "FP8 latent cache: B256 H128 L=4096 ps64 e4m3 + per-tensor scale",
    "long": "long-context split-KV: B8 H128 L~U[32768,131072] ps64 bf16, full",
    "long_window": "long-context split-KV: B8 H128 L~U[32768,131072] ps64 bf16, window 4096",
}

SEEDS = {"tiny": 1235, "v2lite": 1236, "v3": 1237, "fp8": 1238, "long": 1239,
         "long_window": 1239}


def make(name: str, seed: Optional[int] = None, batch: Optional[int] = None,
         num_heads: Optional[int] = None, context_lens=None, page_size: Optional[int] = None,
         window: Optional[int] = None, num_layers: int = 2, layer: int = 1,
         spare_pages: int = SPARE_PAGES, value_std: Optional[float] = None,
         q_std: float = 1.0, q_len: int = 1) -> Workload:
    """Build one seeded workload. Overrides shrink a configuration for tests;
    value_std and q_std change the spread of the cache values and of q (for
    score scales like a trained model's, where the softmax is peaked). q_len >
    1 gives each request q_len new tokens at positions L .. L + q_len - 1
    (q [B, q_len, H, 576], new_rows and slot_mapping [B * q_len])."""
    B0, H0, ps0, dtype, W0, std, has_uv = CONFIGS[name]
    std = std if value_std is None else value_std
    seed = SEEDS[name] if seed is None else seed
    rng = np.random.default_rng(seed)
    H = H0 if num_heads is None else num_heads
    ps = ps0 if page_size is None else page_size
    W = W0 if window is None else window
    if context_lens is not None:
        L = np.asarray(context_lens, np.int32)
        B = len(L)
    else:
        B = B0 if batch is None else batch
        L = _lengths(name, rng, B)
    n_blocks = ((L.astype(np.int64) + q_len - 1) // ps) + 1   # blocks holding positions 0..L+q_len-1
    P = int(n_blocks.sum()) + spare_pages
    perm = rng.permutation(P).astype(np.int32)
    max_blocks = int(n_blocks.max()) if B else 1
    block_table = np.full((B, max_blocks), -1, np.int32)
    indptr = np.zeros(B + 1, np.int32)
    indptr[1:] = np.cumsum(n_blocks)
    ids = perm[: int(n_blocks.sum())].copy()
    for b in range(B):
        block_table[b, : n_blocks[b]] = ids[indptr[b]: indptr[b + 1]]
    pool = _normal_bf16(rng, (num_layers, P, ps, D_ROW), std)
    q = _normal_bf16(rng, (B, H, D_ROW) if q_len == 1 else (B, q_len, H, D_ROW), q_std)
    new_rows = _normal_bf16(rng, (B * q_len, D_ROW), std)
    slots = np.array([int(block_table[b, (L[b] + i) // ps]) * ps + (int(L[b]) + i) % ps
                      for b in range(B) for i in range(q_len)], np.int64)
    kv_scale = 1.0
    if dtype == FP8_E4M3:
        amax = max(float(np.abs(bf16_bits_to_f32(pool)).max()),
                   float(np.abs(bf16_bits_to_f32(new_rows)).max()) if B else 0.0)
        kv_scale = float(np.float32(amax / 448.0))
    w_uv = _normal_bf16(rng, (H, D_CKV, D_V), 0.02) if has_uv else None
    wl = Workload(name=name, batch=B, num_heads=H, page_size=ps, dtype=dtype,
                  context_lens=L, window=W, num_layers=num_layers, layer=layer,
                  num_pages=P, block_table=block_table, page_indptr=indptr, page_ids=ids,
                  pool_bf16=pool, kv_scale=kv_scale, q=q, new_rows=new_rows,
                  slot_mapping=slots, w_uv=w_uv, q_len=q_len)
    if name == "tiny":
        # Unabsorbed-form parameters: q_nope, q_rope ~ N(0,1); W_UK ~ N(0, 1/128)
        # so that W_UK^T q_nope has unit variance; W_UV ~ N(0, 0.02^2).
        wl.extra["q_nope"] = rng.standard_normal((B, H, D_NOPE))
        wl.extra["q_rope"] = rng.standard_normal((B, H, D_ROPE))
        wl.extra["w_uk"] = rng.standard_normal((H, D_NOPE, D_CKV)) * (128 ** -0.5)
        wl.extra["w_uv"] = rng.standard_normal((H, D_CKV, D_V)) * 0.02
    return wl


def alg_bytes_flops(wl: Workload):
    """Algorithmic bytes and flops of one decode step (write + attend).

    bytes = N * row_bytes (latent rows read) + q + out + the new rows written
    (read bf16 + written in the cache type) + the page ids read;
    flops = N * 2 * H * (576 + 512), N = attended tokens summed over requests.
    """
    N = int(wl.attended.sum())
    B, H = wl.batch, wl.num_heads
    pages_read = int(sum(((L) // wl.page_size) - (max(0, L + 1 - wl.window) // wl.page_size
                                                   if wl.window else 0) + 1
                         for L in wl.context_lens.tolist()))
    byts = (N * wl.row_bytes + B * H * D_ROW * 2 + B * H * D_CKV * 2
            + B * (D_ROW * 2 + wl.row_bytes) + 4 * pages_read + 4 * B)
    flops = N * 2 * H * (D_ROW + D_CKV)
    return byts, flops
