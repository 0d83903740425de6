"""CPU oracle for paged MLA decode (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. It wraps a
plain single-threaded C++17 fp64 implementation (``mla_oracle.cpp``) through
ctypes. It imports nothing from the CUDA library package and the library
imports nothing from here.

Each wrapper states what it computes; the C++ file cites the pages that define
each step (MoE-Infinity PR #195 "DeepSeek-V2/V3 paged-attention shim (MLA)",
SGLang PR #32972 "Let Kimi-Linear use the paged MLA attention backends",
FastDeploy PR #8049 "Support MLA_SWA functionality").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

BF16 = 0
FP8_E4M3 = 1
D_CKV = 512
D_ROPE = 64
D_ROW = 576
D_NOPE = 128
D_V = 128

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_kv_write.restype = I
        lib.oracle_kv_write.argtypes = [P, I, I, I, I, ctypes.c_float, I, P, P, I]
        lib.oracle_decode.restype = I
        lib.oracle_decode.argtypes = [P, I, I, I, I, ctypes.c_float, I, P, P, P, I, P,
                                      I, I, ctypes.c_double, I, P, I, P, P]
        lib.oracle_absorb_query.restype = I
        lib.oracle_absorb_query.argtypes = [P, P, P, I, I, P]
        lib.oracle_uv_project.restype = I
        lib.oracle_uv_project.argtypes = [P, P, I, I, P]
        lib.oracle_decode_unabsorbed.restype = I
        lib.oracle_decode_unabsorbed.argtypes = [P, I, I, I, I, ctypes.c_float, I, P, P,
                                                 P, P, P, P, I, P, I, I, ctypes.c_double,
                                                 I, P]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


def _check(rc):
    if rc != 0:
        raise OracleError("oracle rejected its input (code %d)" % rc)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (OCP FP8 definition)."""
    return _load().oracle_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    """fp32 value -> E4M3 code, round to nearest even, saturate to +-448."""
    return int(_load().oracle_e4m3_encode(float(x)))


def kv_write(pool: np.ndarray, dtype: int, num_layers: int, num_pages: int,
             page_size: int, kv_scale: float, layer: int, new_rows: np.ndarray,
             slot_mapping: np.ndarray) -> None:
    """In-place latent write of ``new_rows`` (bf16 bits [n,576]) into ``pool``
    (raw bytes viewed as uint8 or uint16) at ``slot_mapping`` of ``layer``."""
    assert pool.flags.c_contiguous
    rows = _c(new_rows, np.uint16)
    slots = _c(slot_mapping, np.int64)
    _check(_load().oracle_kv_write(_ptr(pool), dtype, num_layers, num_pages, page_size,
                                   kv_scale, layer, _ptr(rows), _ptr(slots), len(slots)))


def decode(pool, dtype, num_layers, num_pages, page_size, kv_scale, layer, q,
           context_lens, softmax_scale, window=0, page_indptr=None, page_ids=None,
           block_table=None, requests=None):
    """Absorbed paged MLA decode in fp64.

    q: float64 [B, H, 576]. Pages given either as CSR (page_indptr [B+1],
    page_ids) or as block_table [B, max_blocks]. Returns (out [R, H, 512],
    lse [R, H]) for the requests in ``requests`` (all when None), natural-log lse.
    """
    q = _c(q, np.float64)
    B, H, D = q.shape
    assert D == D_ROW
    cl = _c(context_lens, np.int32)
    if block_table is not None:
        bt = _c(block_table, np.int32)
        indptr, ids, max_blocks = None, bt, bt.shape[1]
    else:
        indptr, ids, max_blocks = _c(page_indptr, np.int32), _c(page_ids, np.int32), 0
    req = None if requests is None else _c(requests, np.int32)
    R = B if req is None else len(req)
    out = np.zeros((R, H, D_CKV), np.float64)
    lse = np.zeros((R, H), np.float64)
    _check(_load().oracle_decode(_ptr(pool), dtype, num_layers, num_pages, page_size,
                                 kv_scale, layer, _ptr(q), _ptr(indptr), _ptr(ids),
                                 max_blocks, _ptr(cl), B, H, softmax_scale, window,
                                 _ptr(req), 0 if req is None else len(req),
                                 _ptr(out), _ptr(lse)))
    return out, lse


def absorb_query(q_nope, q_rope, w_uk):
    """q_abs = [W_UK^T q_nope ; q_rope] per (b, h); W_UK is [H, 128, 512]."""
    q_nope = _c(q_nope, np.float64)
    q_rope = _c(q_rope, np.float64)
    w_uk = _c(w_uk, np.float64)
    B, H, _ = q_nope.shape
    out = np.zeros((B, H, D_ROW), np.float64)
    _check(_load().oracle_absorb_query(_ptr(q_nope), _ptr(q_rope), _ptr(w_uk), B, H,
                                       _ptr(out)))
    return out


def uv_project(attn, w_uv):
    """y[b,h,:] = attn[b,h,:] @ W_UV[h]; W_UV is [H, 512, 128]."""
    attn = _c(attn, np.float64)
    w_uv = _c(w_uv, np.float64)
    B, H, _ = attn.shape
    y = np.zeros((B, H, D_V), np.float64)
    _check(_load().oracle_uv_project(_ptr(attn), _ptr(w_uv), B, H, _ptr(y)))
    return y


def decode_unabsorbed(pool, dtype, num_layers, num_pages, page_size, kv_scale, layer,
                      q_nope, q_rope, w_uk, w_uv, context_lens, softmax_scale,
                      window=0, page_indptr=None, page_ids=None, block_table=None):
    """Unabsorbed MHA form (qk 192 = 128 nope + 64 rope, v 128) -> y [B, H, 128]."""
    q_nope = _c(q_nope, np.float64)
    q_rope = _c(q_rope, np.float64)
    w_uk = _c(w_uk, np.float64)
    w_uv = _c(w_uv, np.float64)
    B, H, _ = q_nope.shape
    cl = _c(context_lens, np.int32)
    if block_table is not None:
        bt = _c(block_table, np.int32)
        indptr, ids, max_blocks = None, bt, bt.shape[1]
    else:
        indptr, ids, max_blocks = _c(page_indptr, np.int32), _c(page_ids, np.int32), 0
    y = np.zeros((B, H, D_V), np.float64)
    _check(_load().oracle_decode_unabsorbed(_ptr(pool), dtype, num_layers, num_pages,
                                            page_size, kv_scale, layer, _ptr(q_nope),
                                            _ptr(q_rope), _ptr(w_uk), _ptr(w_uv),
                                            _ptr(indptr), _ptr(ids), max_blocks, _ptr(cl),
                                            B, H, softmax_scale, window, _ptr(y)))
    return y
