"""Several query positions per request (mla_decode_q): multi-token decode
(speculative / multi-token-prediction steps, LightLLM PR #1593 "Support dsv4
model", Summary and Validation) and the absorbed form of chunked prefill
over the paged latent (vLLM #12639 "[Attention] MLA with chunked prefill",
Future work), against the oracle.

Request b has L_b cached tokens and q_len new ones at positions L_b ..
L_b + q_len - 1; query position i attends [start_i, L_b + i]. By that
definition query i of request b is the single-query decode of a request with
L_b + i cached tokens over the same page list, which is how the oracle is
asked (its decode is the pinned plain definition)."""
import numpy as np
import pytest
import torch

import mla_workloads as mw
import oracle
from mla_testlib import (TOL_BF16, TOL_FP8, DeviceWorkload, bf16_tensor, check_outputs, f64,
                         oracle_pool_after_write)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import paged_mla_decode_04_gb300 as m
    m.load_library()
    return m


def run_q(lib, wl, num_clusters=0, window=None, write=True):
    """Write the q_len new rows of every request, plan and decode through
    mla_decode_q; returns (out [B, q_len, H, 512], lse [B, q_len, H])."""
    window = wl.window if window is None else window
    dw = DeviceWorkload(wl, lib)
    if write:
        lib.kv_write(dw.pool, wl.layer, dw.new_rows, dw.slots, dw.ws)
    ws = lib.alloc_workspace_q(wl.batch, wl.q_len, wl.num_heads)
    lib.plan_q(dw.lens, wl.q_len, wl.num_heads, wl.page_size, window, ws, num_clusters)
    out = torch.full((wl.batch, wl.q_len, wl.num_heads, mw.D_CKV), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((wl.batch, wl.q_len, wl.num_heads), float("nan"), dtype=torch.float32, device="cuda")
    lib.decode_q(dw.pool, wl.layer, dw.q, dw.lens, wl.softmax_scale, ws, out,
                 block_table=dw.block_table, window=window, lse=lse)
    torch.cuda.synchronize()
    assert lib.get_error(ws) == 0
    assert lib.get_error(dw.ws) == 0
    return f64(out), lse.cpu().numpy().astype(np.float64)


def oracle_q(wl, window=None):
    """Query i of request b = a single-query request with L_b + i cached
    tokens and the same pages."""
    window = wl.window if window is None else window
    pool = oracle_pool_after_write(wl)
    B, QL, H = wl.batch, wl.q_len, wl.num_heads
    q = oracle.bf16_bits_to_f64(wl.q).reshape(B * QL, H, mw.D_ROW)
    lens = (wl.context_lens.astype(np.int64)[:, None] + np.arange(QL)[None, :]).reshape(-1).astype(np.int32)
    table = np.repeat(wl.block_table, QL, axis=0)
    out, lse = oracle.decode(pool, wl.dtype, wl.num_layers, wl.num_pages, wl.page_size, wl.kv_scale,
                             wl.layer, q, lens, wl.softmax_scale, window, block_table=table)
    return out.reshape(B, QL, H, mw.D_CKV), lse.reshape(B, QL, H)


@pytest.mark.parametrize("heads,q_len", [(16, 2), (16, 4), (32, 3), (64, 2), (16, 8)])
@pytest.mark.parametrize("clusters", [0, 7])
def test_multi_token_decode(lib, heads, q_len, clusters):
    lens = [0, 1, 62, 63, 64, 200, 777, 1500]
    wl = mw.make("v2lite", num_heads=heads, context_lens=lens, q_len=q_len)
    out, lse = run_q(lib, wl, num_clusters=clusters)
    ref_out, ref_lse = oracle_q(wl)
    check_outputs(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("window", [1, 3, 64, 100])
def test_multi_token_decode_sliding_window(lib, window):
    lens = [0, 5, 64, 130, 999]
    wl = mw.make("v2lite", num_heads=32, context_lens=lens, window=window, q_len=3)
    out, lse = run_q(lib, wl)
    ref_out, ref_lse = oracle_q(wl)
    check_outputs(out, lse, ref_out, ref_lse)


@pytest.mark.parametrize("heads,q_len,lens", [
    (16, 24, [0, 100, 2000]),          # 384 rows: three full row groups
    (64, 5, [10, 300, 4000]),          # 320 rows: the last group half used
    (128, 3, [0, 777, 3000]),          # 384 rows at 128 heads
    (16, 64, [0, 1000]),               # a 64-token chunk, 1024 rows
])
@pytest.mark.parametrize("clusters", [0, 3])
def test_chunked_prefill_absorbed(lib, heads, q_len, lens, clusters):
    wl = mw.make("v3", num_heads=heads, context_lens=lens, q_len=q_len)
    out, lse = run_q(lib, wl, num_clusters=clusters)
    ref_out, ref_lse = oracle_q(wl)
    check_outputs(out, lse, ref_out, ref_lse)


def test_chunked_prefill_fp8_cache(lib):
    wl = mw.make("fp8", num_heads=32, context_lens=[0, 500, 1300], q_len=6, window=256)
    out, lse = run_q(lib, wl, num_clusters=5)
    ref_out, ref_lse = oracle_q(wl)
    check_outputs(out, lse, ref_out, ref_lse, tol=TOL_FP8)


def test_q_len_one_is_mla_decode_bit_for_bit(lib):
    wl = mw.make("v3", num_heads=128, context_lens=[3000, 17, 900, 2500, 0])
    dw = DeviceWorkload(wl, lib)
    ref_out, ref_lse = dw.step()
    wl1 = mw.make("v3", num_heads=128, context_lens=[3000, 17, 900, 2500, 0])
    wl1.q = wl1.q.reshape(wl1.batch, 1, wl1.num_heads, mw.D_ROW)
    out, lse = run_q(lib, wl1, write=True)
    assert np.array_equal(out[:, 0], ref_out) and np.array_equal(lse[:, 0], ref_lse)


def test_causality_with_needles(lib):
    """Head h of query position i carries a needle dim; the token just after
    position L + i (which query i + 1 attends) holds the needle. Query i must
    not pick it up; query i + 1 must return that row exactly."""
    H, QL = 16, 4
    lens = [5, 70, 200]
    wl = mw.make("v2lite", num_heads=H, context_lens=lens, page_size=16, q_len=QL)
    rng = np.random.default_rng(3)
    dims = rng.choice(mw.D_ROW, H, replace=False)
    c = mw.f32_to_bf16_bits(np.float32([2048.0]))[0]
    one = mw.f32_to_bf16_bits(np.float32([1.0]))[0]
    wl.q[:] = 0
    for i in range(QL):
        wl.q[:, i, np.arange(H), dims] = c
    wl.pool_bf16[wl.layer][..., dims] = 0
    wl.new_rows[:, dims] = 0
    # new token at position L + j (j >= 1) carries the needle of every head
    for b in range(len(lens)):
        for j in range(1, QL):
            wl.new_rows[b * QL + j, dims] = one
    out, _ = run_q(lib, wl)
    pool = oracle_pool_after_write(wl)
    for b, L in enumerate(lens):
        for i in range(QL):
            vis = [j for j in range(1, QL) if j <= i]        # needle tokens query i may see
            row_first = pool[wl.layer, wl.block_table[b, (L + 1) // 16], (L + 1) % 16]
            if vis:
                # several needles of equal score: their rows are averaged; with
                # one (i = 1) the output is that row exactly
                if len(vis) == 1:
                    np.testing.assert_array_equal(out[b, i], np.broadcast_to(
                        oracle.bf16_bits_to_f64(row_first)[:512], out[b, i].shape))
            else:
                # query 0 sees no needle: the uniform mean of its L + 1 rows
                assert not np.array_equal(out[b, 0, 0], oracle.bf16_bits_to_f64(row_first)[:512])
    ref_out, _ = oracle_q(wl)
    assert np.abs(out - ref_out).max() <= TOL_BF16 * np.abs(ref_out).max()


def test_rejected_draft_slots_are_rewritten(lib):
    """A speculative step writes q_len = 4 draft tokens; only 2 are accepted,
    so the next step starts at L + 2 and writes its 3 new tokens over the
    rejected slots (L + 2, L + 3) and one more. The pool after both steps is
    bit-exact against the oracle's two writes in order, and the second
    step's outputs see the rewritten rows, never the rejected ones."""
    H = 32
    lens = [40, 300, 63]
    wl = mw.make("v2lite", num_heads=H, context_lens=lens, page_size=16, q_len=6)
    # step 1: 4 draft tokens at L .. L + 3
    wl1 = mw.make("v2lite", num_heads=H, context_lens=lens, page_size=16, q_len=4)
    dw = DeviceWorkload(wl, lib)            # the pool with room for L + 5 in every request
    def slots_of(L_list, q_len):
        return np.array([int(wl.block_table[b, (L + i) // 16]) * 16 + (L + i) % 16
                         for b, L in enumerate(L_list) for i in range(q_len)], np.int64)
    s1 = slots_of(lens, 4)
    lib.kv_write(dw.pool, wl.layer, bf16_tensor(wl1.new_rows), torch.from_numpy(s1).cuda(), dw.ws)
    # step 2: 2 accepted, context L + 2, new tokens at L + 2 .. L + 4 (rewrites two rejected slots)
    lens2 = [L + 2 for L in lens]
    wl2 = mw.make("v2lite", seed=77, num_heads=H, context_lens=lens2, page_size=16, q_len=3)
    s2 = slots_of(lens2, 3)
    lib.kv_write(dw.pool, wl.layer, bf16_tensor(wl2.new_rows), torch.from_numpy(s2).cuda(), dw.ws)
    ref_pool = wl.pool_bf16.copy()
    oracle.kv_write(ref_pool, mw.BF16, wl.num_layers, wl.num_pages, 16, 1.0, wl.layer, wl1.new_rows, s1)
    oracle.kv_write(ref_pool, mw.BF16, wl.num_layers, wl.num_pages, 16, 1.0, wl.layer, wl2.new_rows, s2)
    got = dw.pool.data.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref_pool)
    # decode step 2 on that pool
    lens2_t = torch.tensor(lens2, dtype=torch.int32, device="cuda")
    q2 = bf16_tensor(wl2.q)
    ws = lib.alloc_workspace_q(len(lens), 3, H)
    lib.plan_q(lens2_t, 3, H, 16, 0, ws)
    out = torch.empty(len(lens), 3, H, mw.D_CKV, dtype=torch.bfloat16, device="cuda")
    lib.decode_q(dw.pool, wl.layer, q2, lens2_t, wl.softmax_scale, ws, out, block_table=dw.block_table)
    torch.cuda.synchronize()
    assert lib.get_error(ws) == 0
    q = oracle.bf16_bits_to_f64(wl2.q).reshape(len(lens) * 3, H, mw.D_ROW)
    lens_e = np.array([L + i for L in lens2 for i in range(3)], np.int32)
    table = np.repeat(wl.block_table, 3, axis=0)
    ref, _ = oracle.decode(ref_pool, mw.BF16, wl.num_layers, wl.num_pages, 16, 1.0, wl.layer, q, lens_e,
                           wl.softmax_scale, 0, block_table=table)
    got_out = f64(out).reshape(len(lens) * 3, H, mw.D_CKV)
    assert np.abs(got_out - ref).max() <= TOL_BF16 * np.abs(ref).max()


@pytest.mark.parametrize("name,q_len,clusters", [("v3", 2, 0), ("v3", 4, 0), ("fp8", 2, 0), ("fp8", 2, 75),
                                                 ("v2lite", 4, 0)])
def test_full_size_multi_token_decode_sampled(lib, name, q_len, clusters):
    """Multi-token decode at the full-size workloads' shapes (V3: 128 heads,
    so q_len x 128 rows run as q_len row groups, each split across clusters;
    fp8; V2-Lite: 16 heads, one row group), in the launch configuration of
    the bench (all clusters). Every query position of sampled requests
    against the oracle.

    fp8 over 75 clusters: the schedule then starts a cluster with a
    single-block split piece followed by more items, under full load, the
    case in which a barrier shared by all items' q chunks could complete two
    phases before the widening warps waited on it (now one barrier per ring
    slot); run_q also requires a clean status word (no timed-out wait)."""
    wl = mw.make(name, q_len=q_len)
    out, lse = run_q(lib, wl, num_clusters=clusters)
    B, QL, H = wl.batch, wl.q_len, wl.num_heads
    sample = sorted(set([0, B // 3, B // 2, B - 1]))
    # fp8: the oracle quantises only the sampled requests' pages
    pages = None if wl.dtype == mw.BF16 else np.concatenate(
        [wl.block_table[b][wl.block_table[b] >= 0] for b in sample])
    pool = oracle_pool_after_write(wl, pages=pages)
    q = oracle.bf16_bits_to_f64(wl.q)[sample].reshape(len(sample) * QL, H, mw.D_ROW)
    lens = (wl.context_lens.astype(np.int64)[sample][:, None] + np.arange(QL)[None, :]).reshape(-1).astype(np.int32)
    table = np.repeat(wl.block_table[sample], QL, axis=0)
    ref_out, ref_lse = oracle.decode(pool, wl.dtype, wl.num_layers, wl.num_pages, wl.page_size, wl.kv_scale,
                                     wl.layer, q, lens, wl.softmax_scale, wl.window, block_table=table)
    tol = TOL_FP8 if wl.dtype != mw.BF16 else TOL_BF16
    check_outputs(out[sample].reshape(-1, H, mw.D_CKV), lse[sample].reshape(-1, H),
                  ref_out, ref_lse, tol=tol)


@pytest.mark.parametrize("ps,window,clusters", [(16, 100, 7), (32, 0, 3), (128, 40, 0)])
def test_fp8_pages_windows_and_splits_with_several_positions(lib, ps, window, clusters):
    """fp8 pools at page sizes below and above the 64-token tile (several raw
    copies per ring slot, widened in place), with a window and split items,
    for three query positions per request."""
    wl = mw.make("fp8", num_heads=32, context_lens=[0, 15, 64, 333, 1500], page_size=ps, window=window,
                 q_len=3)
    out, lse = run_q(lib, wl, num_clusters=clusters)
    ref_out, ref_lse = oracle_q(wl)
    check_outputs(out, lse, ref_out, ref_lse, tol=TOL_FP8)


@pytest.mark.parametrize("name", ["v2lite", "fp8"])
def test_csr_page_lists_equal_block_tables_for_several_positions(lib, name):
    """The CSR page lists (kv_indptr / kv_indices) give the same bits as the
    block table for several query positions per request."""
    wl = mw.make(name, num_heads=32, context_lens=[0, 63, 64, 700, 2100], q_len=3)
    out_t, lse_t = run_q(lib, wl, num_clusters=5)
    dw = DeviceWorkload(wl, lib)
    lib.kv_write(dw.pool, wl.layer, dw.new_rows, dw.slots, dw.ws)
    ws = lib.alloc_workspace_q(wl.batch, wl.q_len, wl.num_heads)
    lib.plan_q(dw.lens, wl.q_len, wl.num_heads, wl.page_size, wl.window, ws, 5)
    out = torch.empty(wl.batch, wl.q_len, wl.num_heads, mw.D_CKV, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(wl.batch, wl.q_len, wl.num_heads, dtype=torch.float32, device="cuda")
    lib.decode_q(dw.pool, wl.layer, dw.q, dw.lens, wl.softmax_scale, ws, out, page_indptr=dw.indptr,
                 page_ids=dw.ids, window=wl.window, lse=lse)
    torch.cuda.synchronize()
    assert lib.get_error(ws) == 0
    assert np.array_equal(f64(out), out_t) and np.array_equal(lse.cpu().numpy().astype(np.float64), lse_t)
