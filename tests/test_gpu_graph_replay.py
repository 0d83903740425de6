"""CUDA-graph replay of a decode step: latent write + plan + decode captured
once at a fixed maximum batch, then replayed with the inputs changed in place
between replays (new page tables, new lengths, fewer real requests with the
rest as pad rows of slot -1). Every replay is checked against the oracle, and
the whole pool bit for bit: pad rows write nothing, so no stale slot is
scattered into (SGLang PR #32972 "Let Kimi-Linear use the paged MLA attention
backends", Cuda-graph safety; the plan/run split of its Correction section)."""
import numpy as np
import pytest
import torch

import mla_workloads as mw
import oracle
from mla_testlib import TOL_BF16, bf16_tensor, f64, rel_err

pytestmark = pytest.mark.gpu

B, H, PS, MAX_BLOCKS = 8, 16, 16, 48


def _scenario(rng, num_pages, real, max_len):
    """Lengths, block table and slots for `real` requests on distinct pages;
    the other rows are pads (length 0, one valid page, slot -1)."""
    lens = np.zeros(B, np.int32)
    lens[:real] = rng.integers(0, max_len + 1, size=real)
    ext = [max_len, 0][:real]                   # the extremes every time
    lens[:len(ext)] = ext
    table = np.full((B, MAX_BLOCKS), -1, np.int32)
    pages = rng.permutation(num_pages).astype(np.int32)
    slots = np.full(B, -1, np.int64)
    k = 0
    for b in range(B):
        n = int(lens[b]) // PS + 1
        table[b, :n] = pages[k:k + n]
        k += n
        if b < real:
            slots[b] = int(table[b, lens[b] // PS]) * PS + int(lens[b]) % PS
    q = mw.f32_to_bf16_bits(rng.standard_normal((B, H, mw.D_ROW)).astype(np.float32))
    rows = mw.f32_to_bf16_bits((rng.standard_normal((B, mw.D_ROW)) * 0.1).astype(np.float32))
    return lens, table, slots, q, rows


def test_graph_replay_with_changed_tables_lengths_and_pad_rows():
    import paged_mla_decode_04_gb300 as m
    m.load_library()
    # pool of 8 x 48 + spare pages: any scenario below fits on distinct pages
    wl = mw.make("v2lite", num_heads=H, context_lens=[PS * MAX_BLOCKS - 1] * B, page_size=PS)
    P, NL, layer = wl.num_pages, wl.num_layers, wl.layer
    pool_ref = wl.pool_bf16.copy()
    pool = m.KVPool(bf16_tensor(pool_ref))
    q = torch.empty(B, H, mw.D_ROW, dtype=torch.bfloat16, device="cuda")
    rows = torch.empty(B, mw.D_ROW, dtype=torch.bfloat16, device="cuda")
    slots = torch.full((B,), -1, dtype=torch.int64, device="cuda")
    lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    table = torch.zeros(B, MAX_BLOCKS, dtype=torch.int32, device="cuda")
    ws = m.alloc_workspace(B, H)
    out = torch.empty(B, H, mw.D_CKV, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, dtype=torch.float32, device="cuda")

    def step():
        m.kv_write(pool, layer, rows, slots, ws)
        m.plan(lens, H, PS, 0, ws)
        m.decode(pool, layer, q, lens, wl.softmax_scale, ws, out, block_table=table, lse=lse)

    q.zero_()
    rows.zero_()
    step()                                  # eager first call: every slot -1, nothing written
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    assert np.array_equal(pool.data.view(torch.int16).cpu().numpy().view(np.uint16), pool_ref)

    rng = np.random.default_rng(2024)
    for real, max_len in [(B, 700), (5, 300), (B, 767), (1, 40)]:
        s_lens, s_table, s_slots, s_q, s_rows = _scenario(rng, P, real, max_len)
        lens.copy_(torch.from_numpy(s_lens))
        table.copy_(torch.from_numpy(s_table))
        slots.copy_(torch.from_numpy(s_slots))
        q.copy_(bf16_tensor(s_q))
        rows.copy_(bf16_tensor(s_rows))
        g.replay()
        torch.cuda.synchronize()
        oracle.kv_write(pool_ref, mw.BF16, NL, P, PS, 1.0, layer, s_rows, s_slots)
        got_pool = pool.data.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got_pool, pool_ref), "pool after replay with %d real rows" % real
        ref_out, ref_lse = oracle.decode(pool_ref, mw.BF16, NL, P, PS, 1.0, layer,
                                         oracle.bf16_bits_to_f64(s_q), s_lens, wl.softmax_scale, 0,
                                         block_table=s_table)
        got = f64(out)[:real]
        assert rel_err(got, ref_out[:real]) <= TOL_BF16, "replay with %d real rows" % real
        got_lse = lse.cpu().numpy().astype(np.float64)[:real]
        assert np.abs(got_lse - ref_lse[:real]).max() <= 2e-3 * max(1.0, np.abs(ref_lse).max())
    assert m.get_error(ws) == 0
