"""Parity pins on the shapes the library is measured on (128 heads, page
sizes 64 and 128, bf16 and fp8 e4m3 pools, lengths up to 70k tokens):

- peaked softmaxes: scores scale * q . K with a spread of 6-8 units, as a
  trained model gives, against the oracle at the stated tolerances (the
  default workloads' scores are ~0.2, where score errors hardly move the
  output);
- needles: each head h carries one query dim d_h = c and every row is 0 at
  d_h except the needle row t*_h, where it is 1. The softmax then collapses
  on t*_h and the output of head h is that row, exactly (bf16 rows, or fp8
  codes times a power-of-two scale). The positions cover every page
  boundary, tile edge (hence every split boundary), window edge and the new
  token; needles just outside the attended range (before a window, past the
  last token in its page) must not be picked up;
- every request of the full-size workloads against the oracle, the oracle's
  requests spread over processes.

Sources: the absorbed 512 + 64 latent of SGLang PR #32972 "Let Kimi-Linear
use the paged MLA attention backends" (Validation), its bounded page-prefix
reads (Correction), the window of FastDeploy PR #8049 "Support MLA_SWA"
(Motivation), and the context-length convention of MoE-Infinity PR #195
"DeepSeek-V2/V3 paged-attention shim (MLA)" (Root causes 4)."""
import numpy as np
import pytest
import torch

import mla_workloads as mw
import oracle
from mla_testlib import (TOL_BF16, TOL_FP8, DeviceWorkload, check_outputs,
                         oracle_pool_after_write, oracle_step)
from oracle_fanout import oracle_decode_all

pytestmark = pytest.mark.gpu

SCALE = 192.0 ** -0.5


@pytest.fixture(scope="module")
def lib():
    import paged_mla_decode_04_gb300 as m
    m.load_library()
    return m


# ----------------------------------------------------------------- peaked softmax

def _score_std(wl, b):
    """Spread of scale * q . K over the heads and attended tokens of request b
    (from the bf16 values before any quantisation): confirms the regime."""
    L = int(wl.context_lens[b])
    pos = np.arange(L)
    pages = wl.block_table[b, pos // wl.page_size]
    K = mw.bf16_bits_to_f32(wl.pool_bf16[wl.layer, pages, pos % wl.page_size]).astype(np.float64)
    q = mw.bf16_bits_to_f32(wl.q[b]).astype(np.float64)
    return float((SCALE * q @ K.T).std())


@pytest.mark.parametrize("name,logit_std,clusters", [("v3", 6.0, 0), ("v3", 8.0, 0), ("v3", 6.0, 7),
                                                     ("fp8", 6.0, 0), ("fp8", 8.0, 7)])
def test_peaked_softmax_at_v3_shape(lib, name, logit_std, clusters):
    lens = [1023, 2500, 4000, 1500, 64, 3071, 0, 777]
    q_std = logit_std / (SCALE * 576 ** 0.5)       # cache values ~N(0, 1)
    wl = mw.make(name, num_heads=128, context_lens=lens, page_size=64, value_std=1.0, q_std=q_std)
    std = _score_std(wl, 2)
    assert 0.8 * logit_std < std < 1.25 * logit_std, std
    dw = DeviceWorkload(wl, lib)
    out, lse = dw.step(num_clusters=clusters)
    ref_out, ref_lse = oracle_step(wl)
    tol = TOL_FP8 if wl.dtype == mw.FP8_E4M3 else TOL_BF16
    err = check_outputs(out, lse, ref_out, ref_lse, tol)
    print("peaked softmax %s logit std %.1f clusters %d: max err %.3e of max|ref|" % (
        name, std, clusters, err))
    assert lib.get_error(dw.ws) == 0


# ----------------------------------------------------------------- needles

NEEDLE_C = 2048.0          # q value at a head's needle dim (exact in bf16 and f16)
FP8_NEEDLE_SCALE = 2.0 ** -4   # fp8 pools: codes * 2^-4 are exact in bf16


def _boundary_positions(L, start, ps):
    """Attended positions next to every tile edge (64 tokens), every page
    boundary and both ends of the attended range [start, L]."""
    s = {start, start + 1, L - 1, L}
    for step in (64, ps):
        for k in range(start // step, L // step + 2):
            s.update((step * k - 1, step * k))
    return sorted(p for p in s if start <= p <= L)


def _outside_positions(L, start, ps):
    """Positions next to the attended range that must not be attended: the one
    before a window, and the one after the last token when it is in the same
    page (a stale slot of the request's last page)."""
    out = []
    if start > 0:
        out.append(start - 1)
    if (L + 1) // ps == L // ps:
        out.append(L + 1)
    return out


@pytest.mark.parametrize("kv,ps,window,clusters", [
    ("bf16", 64, 0, 0), ("bf16", 64, 0, 7), ("bf16", 128, 0, 0), ("bf16", 64, 4096, 0),
    ("bf16", 16, 4096, 7), ("fp8", 64, 0, 0), ("fp8", 64, 0, 7), ("fp8", 128, 4096, 0)])
def test_needles_pin_indexing_bit_exact(lib, kv, ps, window, clusters):
    H = 128
    lens = [69_999, 10_000, 33_001, 555]
    wl = mw.make("long" if kv == "bf16" else "fp8", num_heads=H, context_lens=lens,
                 page_size=ps, window=window)
    fp8 = wl.dtype == mw.FP8_E4M3
    if fp8:
        wl.kv_scale = FP8_NEEDLE_SCALE
    rng = np.random.default_rng(ps + window + clusters)
    dims = rng.choice(mw.D_ROW, H, replace=False)     # one needle dim per head, both ranks' halves
    wl.q[:] = 0
    wl.q[:, np.arange(H), dims] = mw.f32_to_bf16_bits(np.float32([NEEDLE_C]))[0]
    wl.pool_bf16[wl.layer][..., dims] = 0
    wl.new_rows[:, dims] = 0
    dw = DeviceWorkload(wl, lib)
    data = dw.pool.data
    if fp8:
        one = torch.tensor([1.0 / FP8_NEEDLE_SCALE]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    else:
        one = 1.0
    dims_t = torch.from_numpy(dims).cuda()
    starts = [max(0, L + 1 - window) if window else 0 for L in lens]
    inside_pos, outside_pos = [], []
    for L, s in zip(lens, starts):
        inside_pos.append(_boundary_positions(L, s, ps))
        outside_pos.append(_outside_positions(L, s, ps))
    # per request: the positions that must not be attended first, then the
    # attended ones; heads beyond the list repeat attended positions
    tasks = [[(p, False) for p in o] + [(p, True) for p in i] for i, o in zip(inside_pos, outside_pos)]
    launches = max((len(t) + H - 1) // H for t in tasks)
    checked = 0
    for k in range(launches):
        plan = []                                     # (b, h, pos, attended)
        for b, t in enumerate(tasks):
            for h in range(H):
                i = k * H + h
                p, inside = t[i] if i < len(t) else (inside_pos[b][i % len(inside_pos[b])], True)
                plan.append((b, h, p, inside))
        bs = np.array([x[0] for x in plan])
        hs = np.array([x[1] for x in plan])
        ps_ = np.array([x[2] for x in plan])
        new_tok = ps_ == np.asarray(lens)[bs]
        pages = wl.block_table[bs, ps_ // ps]
        offs = ps_ % ps
        # needles in the pool, and in the new rows for the new-token position
        pt = torch.from_numpy(pages[~new_tok]).cuda()
        ot = torch.from_numpy(offs[~new_tok]).cuda()
        dt = dims_t[torch.from_numpy(hs[~new_tok]).cuda()]
        data[wl.layer, pt, ot, dt] = one
        nb = torch.from_numpy(bs[new_tok]).cuda()
        nd = dims_t[torch.from_numpy(hs[new_tok]).cuda()]
        dw.new_rows[nb, nd] = 1.0
        out, _ = dw.step(num_clusters=clusters, window=window)
        rows = data[wl.layer, torch.from_numpy(pages).cuda(), torch.from_numpy(offs).cuda(), :mw.D_CKV]
        if fp8:
            rows = rows.view(torch.float8_e4m3fn).float() * FP8_NEEDLE_SCALE
        expect = rows.to(torch.bfloat16).float().cpu().numpy().astype(np.float64)
        got = out[bs, hs]
        ins = np.array([x[3] for x in plan])
        same = (got == expect).all(axis=1)
        bad = np.nonzero(ins & ~same)[0]
        assert bad.size == 0, "needle not returned exactly: (b, h, pos) %s" % [
            (int(bs[i]), int(hs[i]), int(ps_[i])) for i in bad[:8]]
        leak = np.nonzero(~ins & same)[0]
        assert leak.size == 0, "position outside the attended range was attended: %s" % [
            (int(bs[i]), int(hs[i]), int(ps_[i])) for i in leak[:8]]
        checked += int(ins.sum())
        data[wl.layer, pt, ot, dt] = 0
        dw.new_rows[nb, nd] = 0
    assert lib.get_error(dw.ws) == 0
    assert checked >= sum(len(i) for i in inside_pos)


# ----------------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("name", ["v2lite", "v3", "fp8", "long", "long_window"])
def test_full_size_every_request(lib, name):
    """Full batch and lengths in the launch configuration the bench times
    (every cluster, several items per cluster, split requests merged); every
    request of the batch checked against the oracle."""
    wl = mw.make(name)
    dw = DeviceWorkload(wl, lib)
    out, lse = dw.step()
    assert lib.get_error(dw.ws) == 0
    assert np.isfinite(out).all()
    pool = oracle_pool_after_write(wl)
    ref_out, ref_lse = oracle_decode_all(wl, pool)
    tol = TOL_FP8 if wl.dtype == mw.FP8_E4M3 else TOL_BF16
    err = check_outputs(out, lse, ref_out, ref_lse, tol)
    print("%s: %d requests, max err %.3e of max|ref|" % (name, wl.batch, err))


# ----------------------------------------------------------------- equal scores

@pytest.mark.parametrize("name,window,clusters", [("v3", 0, 0), ("v3", 0, 1), ("v3", 300, 7), ("fp8", 0, 0),
                                                  ("fp8", 300, 5)])
def test_equal_scores_give_the_uniform_average(lib, name, window, clusters):
    """q = 0 makes every score 0: the softmax is uniform, so each head's
    output is the plain mean of the attended rows' first 512 dims and its
    lse is ln(n) for n attended positions (the closed form of the
    definition, MoE-Infinity PR #195 "DeepSeek-V2/V3 paged-attention shim
    (MLA)", Root causes 4 for the length convention). The mean is taken here
    directly from the pool, in fp64; the kernel sums n rows with weight 1 in
    fp32 and rounds the mean to bf16."""
    lens = [0, 1, 63, 64, 650, 2999]
    wl = mw.make(name, num_heads=128, context_lens=lens, window=window)
    wl.q[:] = 0
    dw = DeviceWorkload(wl, lib)
    out, lse = dw.step(num_clusters=clusters)
    assert lib.get_error(dw.ws) == 0
    pool = oracle_pool_after_write(wl)
    ps = wl.page_size
    for b, L in enumerate(lens):
        lo = max(0, L + 1 - window) if window > 0 else 0
        pos = np.arange(lo, L + 1)
        rows = pool[wl.layer, wl.block_table[b, pos // ps], pos % ps][:, :mw.D_CKV]
        if wl.dtype == mw.BF16:
            vals = oracle.bf16_bits_to_f64(rows)
        else:
            table = np.array([oracle.e4m3_decode(c) for c in range(256)])
            vals = table[rows] * wl.kv_scale
        mean = vals.mean(axis=0)
        err = np.abs(out[b] - mean[None, :])
        assert np.all(err <= 2.0 ** -8 * np.abs(mean)[None, :] + 1e-6), (b, float(err.max()))
        np.testing.assert_allclose(lse[b], np.log(len(pos)), rtol=0, atol=2e-6 * max(1.0, np.log(len(pos))))
