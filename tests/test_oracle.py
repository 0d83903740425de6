"""Pins for the CPU oracle: each test checks it against something other than
itself (closed forms, invariants, library routines, an independent
formulation, brute force on tiny inputs), so that a dropped term, a wrong
sign or index or a transposed operand in the oracle fails at least one."""
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import mla_workloads as mw

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _pool_f64(wl, pool_bytes=None):
    """Dense float64 view of a bf16 pool [NL, P, ps, 576]."""
    bits = wl.pool_bf16 if pool_bytes is None else pool_bytes.view(np.uint16)
    return oracle.bf16_bits_to_f64(bits).reshape(wl.num_layers, wl.num_pages, wl.page_size,
                                                 mw.D_ROW)


def _rows_of(wl, pool64, b, layer, start, end):
    """Rows of positions [start, end] of request b, gathered through the table."""
    ps = wl.page_size
    return np.stack([pool64[layer, wl.block_table[b, t // ps], t % ps] for t in
                     range(start, end + 1)])


def _q64(wl):
    return oracle.bf16_bits_to_f64(wl.q)


def _dec(wl, pool_bytes=None, q=None, layer=None, window=None, requests=None, csr=False,
         block_table=None):
    pool_bytes = wl.pool_bf16 if pool_bytes is None else pool_bytes
    kw = dict(page_indptr=wl.page_indptr, page_ids=wl.page_ids) if csr else \
        dict(block_table=wl.block_table if block_table is None else block_table)
    return oracle.decode(pool_bytes, wl.dtype, wl.num_layers, wl.num_pages, wl.page_size,
                         wl.kv_scale, wl.layer if layer is None else layer,
                         _q64(wl) if q is None else q, wl.context_lens, wl.softmax_scale,
                         wl.window if window is None else window, requests=requests, **kw)


# --- fp8 E4M3 codec (OCP FP8 definition) -------------------------------------

def test_e4m3_decode_closed_forms():
    # Closed forms of the OCP E4M3 format: bias 7, 3 mantissa bits,
    # subnormal step 2^-9, smallest normal 2^-6, largest finite 448, S.1111.111 NaN.
    closed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
              0x38: 1.0, 0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0,
              0xB8: -1.0, 0xFE: -448.0}
    for code, val in closed.items():
        assert oracle.e4m3_decode(code) == val, hex(code)
    assert np.isnan(oracle.e4m3_decode(0x7F)) and np.isnan(oracle.e4m3_decode(0xFF))
    vals = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:])), "codes 0x00..0x7E increase"
    for c in range(0x80):
        a, b = oracle.e4m3_decode(c), oracle.e4m3_decode(c | 0x80)
        assert (np.isnan(a) and np.isnan(b)) or a == -b


def test_e4m3_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_decode(c) for c in range(256)])
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.all(both_nan | (ref == ours))


def test_e4m3_roundtrip_all_finite_codes():
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if np.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == c, hex(c)


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1, 30, 150)])
    x = x[np.abs(x) < 448].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.e4m3_encode(v) for v in x], np.uint8)
    assert np.array_equal(ours, ref)


def test_e4m3_encode_ties_to_even_and_saturates():
    # Midpoint between 1.0 (0x38) and 1.125 (0x39) rounds to the even code 0x38;
    # midpoint between 1.125 and 1.25 (0x3A) rounds to 0x3A.
    assert oracle.e4m3_encode(1.0625) == 0x38
    assert oracle.e4m3_encode(1.1875) == 0x3A
    # Subnormal midpoint 1.5 * 2^-9 rounds to 2 * 2^-9 (code 0x02).
    assert oracle.e4m3_encode(1.5 * 2 ** -9) == 0x02
    assert oracle.e4m3_encode(0.5 * 2 ** -9) == 0x00
    assert oracle.e4m3_encode(1e6) == 0x7E and oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(460.0) == 0x7E


# --- latent write through slot_mapping ---------------------------------------

def test_kv_write_bf16_matches_fancy_index_and_isolates_layers():
    wl = mw.make("tiny")
    pool = wl.pool_bf16.copy()
    ref = wl.pool_bf16.copy().reshape(wl.num_layers, -1, mw.D_ROW)
    slots = wl.slot_mapping.copy()
    slots[0] = -1                                  # pad row: no write
    oracle.kv_write(pool, mw.BF16, wl.num_layers, wl.num_pages, wl.page_size, 1.0, 0,
                    wl.new_rows, slots)
    ref[0, slots[1]] = wl.new_rows[1]
    assert np.array_equal(pool.reshape(ref.shape), ref)
    assert np.array_equal(pool[1], wl.pool_bf16[1]), "layer 1 untouched"


def test_kv_write_rejects_out_of_range_slot():
    wl = mw.make("tiny")
    pool = wl.pool_bf16.copy()
    with pytest.raises(oracle.OracleError):
        oracle.kv_write(pool, mw.BF16, wl.num_layers, wl.num_pages, wl.page_size, 1.0, 1,
                        wl.new_rows[:1], np.array([wl.num_pages * wl.page_size]))


def test_kv_write_fp8_matches_torch_quantiser():
    wl = mw.make("tiny")
    NL, P, ps = wl.num_layers, wl.num_pages, wl.page_size
    pool = np.zeros((NL, P, ps, mw.D_ROW), np.uint8)
    scale = 0.0123
    oracle.kv_write(pool, mw.FP8_E4M3, NL, P, ps, scale, 1, wl.new_rows, wl.slot_mapping)
    x = torch.from_numpy(mw.bf16_bits_to_f32(wl.new_rows)) / torch.tensor(scale,
                                                                          dtype=torch.float32)
    x = x.clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    flat = pool.reshape(NL, P * ps, mw.D_ROW)
    assert np.array_equal(flat[1, wl.slot_mapping], ref)
    assert not flat[0].any()


# --- decode -------------------------------------------------------------------

def test_decode_single_token_is_the_row():
    wl = mw.make("tiny", context_lens=[0, 0])
    out, lse = _dec(wl)
    pool64 = _pool_f64(wl)
    for b in range(wl.batch):
        row = _rows_of(wl, pool64, b, wl.layer, 0, 0)[0]
        assert np.array_equal(out[b], np.broadcast_to(row[:512], out[b].shape))
        s = wl.softmax_scale * (_q64(wl)[b] @ row)
        np.testing.assert_allclose(lse[b], s, rtol=0, atol=1e-13)


def test_decode_zero_query_is_uniform_mean():
    wl = mw.make("tiny")
    out, lse = _dec(wl, q=np.zeros((wl.batch, wl.num_heads, mw.D_ROW)))
    pool64 = _pool_f64(wl)
    for b in range(wl.batch):
        L = int(wl.context_lens[b])
        rows = _rows_of(wl, pool64, b, wl.layer, 0, L)
        np.testing.assert_allclose(out[b], np.broadcast_to(rows[:, :512].mean(0), out[b].shape),
                                   rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(lse[b], np.log(L + 1), rtol=1e-14)


def test_decode_matches_scipy_softmax_brute_force():
    wl = mw.make("tiny")
    out, lse = _dec(wl)
    pool64 = _pool_f64(wl)
    q = _q64(wl)
    for b in range(wl.batch):
        K = _rows_of(wl, pool64, b, wl.layer, 0, int(wl.context_lens[b]))
        s = wl.softmax_scale * (q[b] @ K.T)                 # [H, n]
        ref = scipy.special.softmax(s, axis=1) @ K[:, :512]
        np.testing.assert_allclose(out[b], ref, rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(lse[b], scipy.special.logsumexp(s, axis=1), rtol=1e-13)


def test_decode_needle_sweep_pins_indexing():
    """q_rope = c * e_j, k_rope[t*] = e_j, everything else zero in that rope dim:
    the softmax collapses on t*, so out = c_kv[t*] for every position t*."""
    wl = mw.make("tiny", context_lens=[37, 20], page_size=16)
    j, c = 5, 2048.0
    base = wl.pool_bf16.copy()
    pool64 = None
    q = np.zeros((wl.batch, wl.num_heads, mw.D_ROW))
    q[:, :, 512 + j] = c
    one = mw.f32_to_bf16_bits(np.float32([1.0]))[0]
    for b, L in enumerate(wl.context_lens.tolist()):
        for t_star in range(L + 1):
            pool = base.copy()
            pool[:, :, :, 512 + j] = 0
            pool[wl.layer, wl.block_table[b, t_star // wl.page_size],
                 t_star % wl.page_size, 512 + j] = one
            out, _ = _dec(wl, pool_bytes=pool, q=q, requests=[b])
            pool64 = _pool_f64(wl, pool)
            row = pool64[wl.layer, wl.block_table[b, t_star // wl.page_size],
                         t_star % wl.page_size]
            np.testing.assert_allclose(out[0], np.broadcast_to(row[:512], out[0].shape),
                                       rtol=1e-12, atol=1e-12)


def test_decode_page_permutation_invariance_is_exact():
    wl = mw.make("tiny")
    out, lse = _dec(wl)
    rng = np.random.default_rng(7)
    perm = rng.permutation(wl.num_pages)       # new physical id of old page p
    pool = np.empty_like(wl.pool_bf16)
    pool[:, perm] = wl.pool_bf16
    bt = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1)
    out2, lse2 = _dec(wl, pool_bytes=pool, block_table=bt)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_decode_csr_equals_block_table():
    wl = mw.make("tiny")
    a = _dec(wl)
    b = _dec(wl, csr=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_decode_layers_do_not_alias():
    wl = mw.make("tiny")
    out1, _ = _dec(wl, layer=1)
    pool = wl.pool_bf16.copy()
    pool[0] = mw.f32_to_bf16_bits(np.full(pool[0].shape, 3.0, np.float32))
    out1b, _ = _dec(wl, pool_bytes=pool, layer=1)
    out0b, _ = _dec(wl, pool_bytes=pool, layer=0)
    assert np.array_equal(out1, out1b)
    assert np.allclose(out0b, 3.0)


def test_decode_window_reduces_to_full_and_to_truncated_request():
    wl = mw.make("tiny", context_lens=[37, 61])
    full, _ = _dec(wl, window=0)
    same, _ = _dec(wl, window=62)
    assert np.array_equal(full, same)
    W = 20
    win, win_lse = _dec(wl, window=W)
    pool64 = _pool_f64(wl)
    q = _q64(wl)
    for b in range(wl.batch):
        L = int(wl.context_lens[b])
        K = _rows_of(wl, pool64, b, wl.layer, L + 1 - W, L)      # the last W tokens
        assert K.shape[0] == W
        s = wl.softmax_scale * (q[b] @ K.T)
        np.testing.assert_allclose(win[b], scipy.special.softmax(s, 1) @ K[:, :512],
                                   rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(win_lse[b], scipy.special.logsumexp(s, 1), rtol=1e-13)


def test_decode_reads_only_needed_page_prefix():
    wl = mw.make("tiny")
    bt = wl.block_table.copy()
    extra = np.full((wl.batch, 3), 10 ** 6, np.int32)          # garbage past the prefix
    out, _ = _dec(wl)
    out2, _ = _dec(wl, block_table=np.concatenate([bt, extra], 1))
    assert np.array_equal(out, out2)


def test_decode_rejects_bad_page_id():
    wl = mw.make("tiny")
    bt = wl.block_table.copy()
    bt[0, 0] = wl.num_pages
    with pytest.raises(oracle.OracleError):
        _dec(wl, block_table=bt)


def test_decode_fp8_matches_library_dequant():
    wl = mw.make("tiny")
    NL, P, ps = wl.num_layers, wl.num_pages, wl.page_size
    scale = float(np.float32(0.1 * 4 / 448))
    pool = np.zeros((NL, P, ps, mw.D_ROW), np.uint8)
    rows = wl.pool_bf16.reshape(-1, mw.D_ROW)
    for layer in range(NL):
        slots = np.arange(P * ps, dtype=np.int64)
        oracle.kv_write(pool, mw.FP8_E4M3, NL, P, ps, scale, layer,
                        rows[layer * P * ps:(layer + 1) * P * ps], slots)
    out, lse = oracle.decode(pool, mw.FP8_E4M3, NL, P, ps, scale, wl.layer, _q64(wl),
                             wl.context_lens, wl.softmax_scale, block_table=wl.block_table)
    deq = torch.from_numpy(pool).view(torch.float8_e4m3fn).to(torch.float64).numpy() * scale
    q = _q64(wl)
    for b in range(wl.batch):
        K = _rows_of(wl, deq, b, wl.layer, 0, int(wl.context_lens[b]))
        s = wl.softmax_scale * (q[b] @ K.T)
        np.testing.assert_allclose(out[b], scipy.special.softmax(s, 1) @ K[:, :512],
                                   rtol=1e-11, atol=1e-14)


def test_absorbed_equals_unabsorbed_mha_form():
    """MLA with qk_head_dim 192 = 128 nope + 64 rope and v_head_dim 128, run
    as plain multi-head attention over up-projected keys and values, equals the
    absorbed 576/512 latent decode followed by the W_UV projection."""
    wl = mw.make("tiny")
    e = wl.extra
    q_abs = oracle.absorb_query(e["q_nope"], e["q_rope"], e["w_uk"])
    np.testing.assert_allclose(q_abs[..., :512], np.einsum("bhe,hed->bhd", e["q_nope"],
                                                           e["w_uk"]), rtol=1e-12, atol=1e-12)
    out, _ = oracle.decode(wl.pool_bf16, mw.BF16, wl.num_layers, wl.num_pages, wl.page_size,
                           1.0, wl.layer, q_abs, wl.context_lens, wl.softmax_scale,
                           block_table=wl.block_table)
    y_abs = oracle.uv_project(out, e["w_uv"])
    y_mha = oracle.decode_unabsorbed(wl.pool_bf16, mw.BF16, wl.num_layers, wl.num_pages,
                                     wl.page_size, 1.0, wl.layer, e["q_nope"], e["q_rope"],
                                     e["w_uk"], e["w_uv"], wl.context_lens, wl.softmax_scale,
                                     block_table=wl.block_table)
    err = np.abs(y_abs - y_mha).max() / np.abs(y_mha).max()
    assert err <= 1e-10, err
    # The identity must be sensitive: dropping the rope term breaks it.
    y_no_rope = oracle.decode_unabsorbed(wl.pool_bf16, mw.BF16, wl.num_layers, wl.num_pages,
                                         wl.page_size, 1.0, wl.layer, e["q_nope"],
                                         np.zeros_like(e["q_rope"]), e["w_uk"], e["w_uv"],
                                         wl.context_lens, wl.softmax_scale,
                                         block_table=wl.block_table)
    assert np.abs(y_no_rope - y_abs).max() / np.abs(y_abs).max() > 1e-3


def test_uv_project_matches_einsum():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((3, 4, 512))
    w = rng.standard_normal((4, 512, 128))
    np.testing.assert_allclose(oracle.uv_project(a, w), np.einsum("bhd,hde->bhe", a, w),
                               rtol=1e-12, atol=1e-12)


def test_geometry_golden_matches_workloads():
    g = json.load(open(os.path.join(GOLDEN, "mla_geometry.json")))
    assert g["kv_lora_rank"] + g["qk_rope_head_dim"] == mw.D_ROW == oracle.D_ROW
    assert g["qk_nope_head_dim"] + g["qk_rope_head_dim"] == g["qk_head_dim"]
    assert g["v_head_dim"] == oracle.D_V and g["qk_nope_head_dim"] == oracle.D_NOPE
    assert mw.make("tiny").softmax_scale == g["qk_head_dim"] ** -0.5
    # Decode convention: context_length excludes the just-generated token, so
    # the new token's slot is position L, the first position not yet cached.
    ex = g["context_length_example"]
    assert ex["num_computed_tokens"] - ex["len_input_token"] == ex["context_length"]
    wl = mw.make("tiny")
    for b in range(wl.batch):
        L = int(wl.context_lens[b])
        assert wl.slot_mapping[b] == wl.block_table[b, L // wl.page_size] * wl.page_size + \
            L % wl.page_size
