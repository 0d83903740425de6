"""Paged MLA decode for GB300: thin Python binding of libmla_decode.so.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and streams. If the library is missing or
cannot be loaded this module raises; there is no fallback path.

Calls (same names as the C ABI in include/mla_decode.h):
  kv_write(pool, layer, new_rows, slot_mapping, workspace=None)
  workspace_size(batch, num_heads) / num_clusters()
  plan(context_lens, num_heads, page_size, window, workspace, num_clusters=0)
  decode(pool, layer, q, context_lens, softmax_scale, workspace, out,
         block_table=None | page_indptr + page_ids, window=0, lse=None)
  workspace_size_q / plan_q / decode_q: several query positions per request
  (q [batch, q_len, heads, 576]; causal within the step)
  uv_project(attn_out, w_uv, y, workspace=None)
  get_error(workspace, clear=False)
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_decode.so")

MLA_OK = 0
ERRORS = {-1: "MLA_ERR_ARG", -2: "MLA_ERR_UNSUPPORTED", -3: "MLA_ERR_WORKSPACE", -4: "MLA_ERR_CUDA"}
STATUS_BAD_PAGE = 0x1
STATUS_BAD_SLOT = 0x2
STATUS_PLAN_MISMATCH = 0x4
STATUS_TIMEOUT = 0x8
STATUS_BAD_LENGTH = 0x10
DTYPE_BF16 = 0
DTYPE_FP8_E4M3 = 1
LATENT_DIM = 576
KV_LORA_RANK = 512
V_HEAD_DIM = 128

EXPORTED = ["mla_kv_write", "mla_decode_workspace_size", "mla_decode_num_clusters",
            "mla_decode_plan", "mla_decode", "mla_uv_project", "mla_get_error",
            "mla_decode_noalloc", "mla_decode_workspace_size_q", "mla_decode_plan_q",
            "mla_decode_q", "mla_selftest_bounded_wait"]
NOALLOC_SCRATCH_BYTES = 48 << 20


class MlaError(RuntimeError):
    pass


class _Pool(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("num_layers", ctypes.c_int),
                ("num_pages", ctypes.c_int), ("page_size", ctypes.c_int),
                ("dtype", ctypes.c_int), ("kv_scale", ctypes.c_float)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmla_decode.so (raises if it is missing: build it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise MlaError("libmla_decode.so not built; run paged_mla_decode_04_gb300._build.build()")
    lib = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.mla_kv_write.argtypes = [ctypes.POINTER(_Pool), I, P, P, I, P, P]
    lib.mla_kv_write.restype = I
    lib.mla_decode_workspace_size.argtypes = [I, I]
    lib.mla_decode_workspace_size.restype = Z
    lib.mla_decode_num_clusters.argtypes = []
    lib.mla_decode_num_clusters.restype = I
    lib.mla_decode_plan.argtypes = [P, I, I, I, I, I, P, Z, P]
    lib.mla_decode_plan.restype = I
    lib.mla_decode.argtypes = [ctypes.POINTER(_Pool), I, P, P, P, I, P, I, I, ctypes.c_float, I,
                               P, P, P, P]
    lib.mla_decode.restype = I
    lib.mla_uv_project.argtypes = [P, P, P, I, I, P, P]
    lib.mla_uv_project.restype = I
    lib.mla_get_error.argtypes = [P, ctypes.POINTER(I), I, P]
    lib.mla_get_error.restype = I
    lib.mla_selftest_bounded_wait.argtypes = [I, ctypes.c_uint, P, P]
    lib.mla_selftest_bounded_wait.restype = I
    lib.mla_decode_noalloc.argtypes = [ctypes.POINTER(_Pool), I, P, P, P, I, P, I, I, ctypes.c_float,
                                       I, I, P, P, P, P]
    lib.mla_decode_noalloc.restype = I
    lib.mla_decode_workspace_size_q.argtypes = [I, I, I]
    lib.mla_decode_workspace_size_q.restype = Z
    lib.mla_decode_plan_q.argtypes = [P, I, I, I, I, I, I, P, Z, P]
    lib.mla_decode_plan_q.restype = I
    lib.mla_decode_q.argtypes = [ctypes.POINTER(_Pool), I, P, P, P, I, P, I, I, I, ctypes.c_float, I,
                                 P, P, P, P]
    lib.mla_decode_q.restype = I
    _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != MLA_OK:
        raise MlaError("%s failed: %s (%d)" % (what, ERRORS.get(rc, "unknown"), rc))


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


@dataclass
class KVPool:
    """A paged latent pool [num_layers, num_pages, page_size, 576] of bf16 or
    e4m3 codes (torch.uint8), with the fp8 per-pool scale."""
    data: torch.Tensor
    kv_scale: float = 1.0

    @property
    def dtype_code(self) -> int:
        return DTYPE_BF16 if self.data.dtype == torch.bfloat16 else DTYPE_FP8_E4M3

    def _c(self) -> _Pool:
        d = self.data
        if d.dim() != 4 or d.shape[3] != LATENT_DIM:
            raise ValueError("pool must be [num_layers, num_pages, page_size, 576]")
        if d.dtype not in (torch.bfloat16, torch.uint8):
            raise ValueError("pool dtype must be bfloat16 or uint8 (e4m3 codes)")
        _dev(d, "pool")
        return _Pool(d.data_ptr(), d.shape[0], d.shape[1], d.shape[2], self.dtype_code,
                     float(self.kv_scale))


def kv_write(pool: KVPool, layer: int, new_rows: torch.Tensor, slot_mapping: torch.Tensor,
             workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    lib = load_library()
    n = new_rows.shape[0]
    if new_rows.dim() != 2 or new_rows.shape[1] != LATENT_DIM or slot_mapping.shape != (n,):
        raise ValueError("new_rows [n, 576] and slot_mapping [n] expected")
    c = pool._c()
    rc = lib.mla_kv_write(ctypes.byref(c), layer, _dev(new_rows, "new_rows", torch.bfloat16),
                          _dev(slot_mapping, "slot_mapping", torch.int64), n,
                          None if workspace is None else _dev(workspace, "workspace"),
                          _stream(stream))
    _check(rc, "mla_kv_write")


def num_clusters() -> int:
    rc = load_library().mla_decode_num_clusters()
    if rc < 0:
        _check(rc, "mla_decode_num_clusters")
    return rc


def workspace_size(batch: int, num_heads: int) -> int:
    n = load_library().mla_decode_workspace_size(batch, num_heads)
    if n == 0:
        raise MlaError("mla_decode_workspace_size: unsupported arguments")
    return n


def alloc_workspace(batch: int, num_heads: int, device=None) -> torch.Tensor:
    """A zeroed workspace tensor (torch allocations are 256-byte aligned)."""
    return torch.zeros(workspace_size(batch, num_heads), dtype=torch.uint8,
                       device=device or torch.device("cuda"))


def plan(context_lens: torch.Tensor, num_heads: int, page_size: int, window: int,
         workspace: torch.Tensor, num_clusters: int = 0, stream=None) -> None:
    lib = load_library()
    rc = lib.mla_decode_plan(_dev(context_lens, "context_lens", torch.int32), context_lens.numel(),
                             num_heads, page_size, window, num_clusters,
                             _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                             _stream(stream))
    _check(rc, "mla_decode_plan")


def decode(pool: KVPool, layer: int, q: torch.Tensor, context_lens: torch.Tensor,
           softmax_scale: float, workspace: torch.Tensor, out: torch.Tensor,
           block_table: Optional[torch.Tensor] = None, page_indptr: Optional[torch.Tensor] = None,
           page_ids: Optional[torch.Tensor] = None, window: int = 0,
           lse: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    lib = load_library()
    if q.dim() != 3 or q.shape[2] != LATENT_DIM:
        raise ValueError("q must be [batch, heads, 576]")
    B, H, _ = q.shape
    if out.shape != (B, H, KV_LORA_RANK):
        raise ValueError("out must be [batch, heads, 512]")
    if block_table is not None:
        if block_table.dim() != 2 or block_table.shape[0] != B:
            raise ValueError("block_table must be [batch, max_blocks]")
        indptr_p, ids_p, max_blocks = None, _dev(block_table, "block_table", torch.int32), \
            block_table.shape[1]
    else:
        if page_indptr is None or page_ids is None or page_indptr.shape != (B + 1,):
            raise ValueError("give block_table, or page_indptr [batch+1] and page_ids")
        indptr_p = _dev(page_indptr, "page_indptr", torch.int32)
        ids_p, max_blocks = _dev(page_ids, "page_ids", torch.int32), 0
    if context_lens.shape != (B,):
        raise ValueError("context_lens must be [batch]")
    c = pool._c()
    rc = lib.mla_decode(ctypes.byref(c), layer, _dev(q, "q", torch.bfloat16), indptr_p, ids_p,
                        max_blocks, _dev(context_lens, "context_lens", torch.int32), B, H,
                        float(softmax_scale), window, _dev(workspace, "workspace"),
                        _dev(out, "out", torch.bfloat16),
                        None if lse is None else _dev(lse, "lse", torch.float32), _stream(stream))
    _check(rc, "mla_decode")
    return out


def uv_project(attn_out: torch.Tensor, w_uv: torch.Tensor, y: torch.Tensor,
               workspace: Optional[torch.Tensor] = None, stream=None):
    lib = load_library()
    B, H, D = attn_out.shape
    if D != KV_LORA_RANK or w_uv.shape != (H, KV_LORA_RANK, V_HEAD_DIM) or \
            y.shape != (B, H, V_HEAD_DIM):
        raise ValueError("attn_out [B,H,512], w_uv [H,512,128], y [B,H,128] expected")
    rc = lib.mla_uv_project(_dev(attn_out, "attn_out", torch.bfloat16),
                            _dev(w_uv, "w_uv", torch.bfloat16), _dev(y, "y", torch.bfloat16), B, H,
                            None if workspace is None else _dev(workspace, "workspace"),
                            _stream(stream))
    _check(rc, "mla_uv_project")
    return y


def decode_noalloc(pool: KVPool, layer: int, q: torch.Tensor, context_lens: torch.Tensor,
                   softmax_scale: float, out: torch.Tensor, block_table: torch.Tensor,
                   window: int = 0, num_clusters: int = 0, lse: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """mla_decode_plan + mla_decode without a caller workspace: the library's
    fixed scratch array holds the schedule and partials (see the C header for
    the size limit and the one-stream rule)."""
    lib = load_library()
    B, H, _ = q.shape
    c = pool._c()
    rc = lib.mla_decode_noalloc(ctypes.byref(c), layer, _dev(q, "q", torch.bfloat16), None,
                                _dev(block_table, "block_table", torch.int32), block_table.shape[1],
                                _dev(context_lens, "context_lens", torch.int32), B, H,
                                float(softmax_scale), window, num_clusters,
                                _dev(out, "out", torch.bfloat16),
                                None if lse is None else _dev(lse, "lse", torch.float32),
                                None if status is None else _dev(status, "status", torch.int32),
                                _stream(stream))
    _check(rc, "mla_decode_noalloc")
    return out


def get_error(workspace: torch.Tensor, clear: bool = False, stream=None) -> int:
    code = ctypes.c_int(0)
    rc = load_library().mla_get_error(_dev(workspace, "workspace"), ctypes.byref(code),
                                      1 if clear else 0, _stream(stream))
    _check(rc, "mla_get_error")
    return code.value


def selftest_bounded_wait(status: torch.Tensor, arrive: bool, limit_us: int, stream=None) -> None:
    """One thread waits on a fresh mbarrier for at most limit_us; without the
    arrival the wait runs out and MLA_STATUS_TIMEOUT is OR-ed into status
    (a device int32 tensor)."""
    if status.dtype != torch.int32 or status.numel() < 1:
        raise MlaError("mla_selftest_bounded_wait: status must be a device int32 tensor")
    rc = load_library().mla_selftest_bounded_wait(1 if arrive else 0, int(limit_us),
                                                  _dev(status, "status"), _stream(stream))
    _check(rc, "mla_selftest_bounded_wait")


# ----------------------------------------------------------------- several query positions per request

def workspace_size_q(batch: int, q_len: int, num_heads: int) -> int:
    n = load_library().mla_decode_workspace_size_q(batch, q_len, num_heads)
    if n == 0:
        raise MlaError("mla_decode_workspace_size_q: unsupported arguments")
    return n


def alloc_workspace_q(batch: int, q_len: int, num_heads: int, device=None) -> torch.Tensor:
    return torch.zeros(workspace_size_q(batch, q_len, num_heads), dtype=torch.uint8,
                       device=device or torch.device("cuda"))


def plan_q(context_lens: torch.Tensor, q_len: int, num_heads: int, page_size: int, window: int,
           workspace: torch.Tensor, num_clusters: int = 0, stream=None) -> None:
    lib = load_library()
    rc = lib.mla_decode_plan_q(_dev(context_lens, "context_lens", torch.int32), context_lens.numel(), q_len,
                               num_heads, page_size, window, num_clusters, _dev(workspace, "workspace"),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mla_decode_plan_q")


def decode_q(pool: KVPool, layer: int, q: torch.Tensor, context_lens: torch.Tensor,
             softmax_scale: float, workspace: torch.Tensor, out: torch.Tensor,
             block_table: Optional[torch.Tensor] = None, page_indptr: Optional[torch.Tensor] = None,
             page_ids: Optional[torch.Tensor] = None, window: int = 0,
             lse: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q [batch, q_len, heads, 576] -> out [batch, q_len, heads, 512] (lse
    [batch, q_len, heads]); query position i of request b attends positions
    up to context_lens[b] + i."""
    lib = load_library()
    if q.dim() != 4 or q.shape[3] != LATENT_DIM:
        raise ValueError("q must be [batch, q_len, heads, 576]")
    B, QL, H, _ = q.shape
    if out.shape != (B, QL, H, KV_LORA_RANK):
        raise ValueError("out must be [batch, q_len, heads, 512]")
    if lse is not None and lse.shape != (B, QL, H):
        raise ValueError("lse must be [batch, q_len, heads]")
    if block_table is not None:
        if block_table.dim() != 2 or block_table.shape[0] != B:
            raise ValueError("block_table must be [batch, max_blocks]")
        indptr_p, ids_p, max_blocks = None, _dev(block_table, "block_table", torch.int32), \
            block_table.shape[1]
    else:
        if page_indptr is None or page_ids is None or page_indptr.shape != (B + 1,):
            raise ValueError("give block_table, or page_indptr [batch+1] and page_ids")
        indptr_p = _dev(page_indptr, "page_indptr", torch.int32)
        ids_p, max_blocks = _dev(page_ids, "page_ids", torch.int32), 0
    if context_lens.shape != (B,):
        raise ValueError("context_lens must be [batch]")
    c = pool._c()
    rc = lib.mla_decode_q(ctypes.byref(c), layer, _dev(q, "q", torch.bfloat16), indptr_p, ids_p, max_blocks,
                          _dev(context_lens, "context_lens", torch.int32), B, QL, H, float(softmax_scale),
                          window, _dev(workspace, "workspace"), _dev(out, "out", torch.bfloat16),
                          None if lse is None else _dev(lse, "lse", torch.float32), _stream(stream))
    _check(rc, "mla_decode_q")
    return out
