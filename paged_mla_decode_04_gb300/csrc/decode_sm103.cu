// Absorbed paged MLA decode on sm_103a tensor cores.
//
// What it computes (MoE-Infinity PR #195 "DeepSeek-V2/V3 paged-attention
// shim (MLA)" and SGLang PR #32972 "Let Kimi-Linear use the paged MLA
// attention backends"): for request b and head h, softmax over the attended
// positions of scale * q[b,h,:576] . K_t, and the weighted sum of K_t[:512],
// where K_t is the request's 576-d latent row at position t, fetched through
// its page list. Every head shares each latent row, so S = Q K^T (heads x
// tokens, contraction 576) and O = P V (heads x 512, contraction over tokens)
// are dense tensor-core contractions.
//
// GB300 mapping. A fp32 O for 128 heads x 512 dims fills a whole SM's tensor
// memory, so one work unit is a cluster of two CTAs (rank r = 0, 1):
//   - both ranks gather the full 576-d rows of each 32-token tile by TMA
//     (one box per page and 64-dim chunk, 128-byte swizzle, 3-stage ring);
//   - rank r computes S for its half of the heads over all 576 dims with
//     tcgen05.mma M=64 (heads) x N=32 (tokens) into TMEM, runs the online
//     softmax for those heads (base 2, lazy rescale: a head's reference max
//     moves only when its running max grows by more than 8, i.e. a factor
//     256; the final 1/l makes the result exact) and writes its P rows (bf16)
//     into its own shared memory and, with st.async, into the peer's;
//   - rank r accumulates O for all heads but only its half of the value
//     dims (c_kv[256r, 256r+256)) with tcgen05.mma M=128 x N=256 x K=32,
//     V read MN-major straight from the gathered tile.
// Only P rows, rescale factors and final row sums cross between the two SMs
// (about 136 bytes per token at 128 heads); distributed shared memory is far
// slower than HBM on this part, so scores never cross.
// Warp roles per CTA (224 threads): warp 0 TMA producer (which also runs
// bulk L2 prefetches a few tiles ahead, each rank fetching half of every
// tile, so HBM latency is hidden beyond what the shared-memory ring holds),
// warp 1 TMEM owner and QK issuer, warps 2-5 softmax, O correction and
// epilogue, warp 6 PV issuer (separate issuers, so a QK waiting for data
// never holds back a PV).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kTile = kBlockTokens;                 // 32 tokens per tile
constexpr int kStages = 3;
constexpr int kChunks = kDimRow / 64;               // 9 chunks of 64 dims
constexpr int kKvChunkBytes = kTile * 128;          // [32 tokens][64 dims] bf16
constexpr int kStageBytes = kChunks * kKvChunkBytes;
constexpr int kQChunkBytes = 64 * 128;              // [64 heads][64 dims] bf16
constexpr int kPBytes = 128 * 128;                  // [128 heads][32 tokens] bf16, 128-byte rows
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kChunks * kQChunkBytes;
constexpr int kOffP = kOffKV + kStages * kStageBytes;
constexpr int kOffAlpha = kOffP + 2 * kPBytes;      // [2][128] fp32 rescale factors
constexpr int kOffL = kOffAlpha + 2 * 128 * 4;      // [128] fp32 final row sums
constexpr int kOffBar = kOffL + 128 * 4;
constexpr int kSmemBytes = kOffBar + 512 + 1024;    // barriers + alignment slack
constexpr int kThreads = 224;
constexpr int kPrefetchTiles = 8;  // L2 prefetch distance of the producer, in tiles
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;                       // O: columns [0, 256), lanes = heads
constexpr uint32_t kColS = 256;                     // S[b]: columns 256 + 32 b, M=64 layout
constexpr float kRescaleThreshold = 8.0f;
constexpr int kPRowBytes = kTile * 2;               // 64 bytes of P per head row
constexpr int kPeerBytesPerRow = kPRowBytes + 4;    // P row + rescale factor

static_assert(kOffKV % 1024 == 0 && kOffP % 1024 == 0 && kStageBytes % 1024 == 0, "swizzle alignment");

enum Bar {
  kBarKvFull = 0,                  // [kStages]
  kBarKvEmpty = kBarKvFull + kStages,
  kBarQFull = kBarKvEmpty + kStages,
  kBarQFree,
  kBarSFull,                       // [2]
  kBarSFree = kBarSFull + 2,       // [2]
  kBarPFull = kBarSFree + 2,       // [2] local arrivals + peer st.async bytes
  kBarPvDone = kBarPFull + 2,      // [2] PV on that P buffer done in both ranks
  kBarOFixed = kBarPvDone + 2,     // [2] O rows rescaled for this tile
  kBarLFull = kBarOFixed + 2,      // final row sums landed
  kBarDrain,
  kBarDrainPv,
  kNumBars
};
static_assert(kNumBars * 8 + 16 <= 512, "barrier area");

struct Params {
  CUtensorMap kv_map;  // pool rows [NL*P*ps][576] bf16, box {64, min(ps, 32)}
  CUtensorMap q_map;   // q rows [B*H][576] bf16, box {64, 64}
  DecodeArgs a;
};

__device__ __forceinline__ void flag_status(int* status, int bits) { atomicOr(status, bits); }

// 2^x with the hardware approximation (exact at -inf: returns +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + kNumBars * 8 + 4);
  const float* alpha_s = reinterpret_cast<const float*>(smem + kOffAlpha);
  float* l_s = reinterpret_cast<float*>(smem + kOffL);

  const DecodeArgs& a = p.a;
  uint8_t* ws = a.ws;
  WsHeader* hd = reinterpret_cast<WsHeader*>(ws);
  int* status = &hd->status;
  const WorkItem* items = reinterpret_cast<const WorkItem*>(ws + a.lay.items);
  const int* cstart = reinterpret_cast<const int*>(ws + a.lay.cluster_start);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int cluster_id = blockIdx.x >> 1;
  const int H = a.num_heads;
  const int Hh = H >> 1;  // heads whose scores this rank computes
  const int ps = a.page_size;

  const bool plan_ok = hd->planned == 1 && hd->batch == a.batch && hd->num_heads == a.num_heads &&
                       hd->page_size == a.page_size && hd->window == a.window;
  int it_begin = 0, it_end = 0;
  if (plan_ok && cluster_id < hd->num_clusters) {
    it_begin = cstart[cluster_id];
    it_end = cstart[cluster_id + 1];
  }
  if (!plan_ok && threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, MLA_STATUS_PLAN_MISMATCH);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKvFull + i), 1);
      mbar_init(bar(kBarKvEmpty + i), 1);
    }
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQFree), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSFree + i), 128);
      mbar_init(bar(kBarPFull + i), 128);
      mbar_init(bar(kBarPvDone + i), 2);
      mbar_init(bar(kBarOFixed + i), 128);
    }
    mbar_init(bar(kBarLFull), 128);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrainPv), 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.kv_map);
    tma_prefetch_map(&p.q_map);
  }
  tc_fence_before();
  cluster_sync();  // barriers of both ranks initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the tiles; lane 0 issues the copies. Page ids are
    // fetched 32 at a time by the warp (one coalesced load) and handed out
    // by shuffle, so a tile waits on no global load. A second cursor runs
    // kPrefetchTiles ahead and pulls this rank's half of each tile's rows
    // into L2.
    const uint64_t kv_policy = l2_policy_evict_first();
    const int64_t layer_row0 = static_cast<int64_t>(a.layer) * a.num_pages * ps;
    const int oob_row = a.num_layers * a.num_pages * ps;  // reads as zeros
    const int rows_per_box = ps < kTile ? ps : kTile;
    const int boxes = kTile / rows_per_box;
    const uint8_t* pool_bytes = static_cast<const uint8_t*>(a.pool);
    uint32_t g = 0;
    int last_q_item = -1;
    uint32_t n_items = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it, ++n_items) {
      const WorkItem w = items[it];
      const int first_page = max(w.tok_lo, w.blk_begin * kTile) / ps;
      const int last_page = (min(w.tok_hi, w.blk_end * kTile) - 1) / ps;
      const int nb = a.page_indptr ? a.page_indptr[w.b + 1] - a.page_indptr[w.b] : a.max_blocks;
      const int32_t* ids = a.page_indptr ? a.page_ids + a.page_indptr[w.b]
                                         : a.page_ids + static_cast<int64_t>(w.b) * a.max_blocks;
      // Page-id windows of 32 pages: one for the copies, one for prefetches.
      int batch0 = -64, my_id = -1, pbatch0 = -64, pmy_id = -1;
      auto page_id = [&](int j, int& b0, int& mine) -> int {
        if (j - b0 >= 32 || j < b0) {
          b0 = j;
          const int jj = j + lane;
          mine = (jj <= last_page && jj < nb) ? ids[jj] : -1;
        }
        return __shfl_sync(0xffffffffu, mine, j - b0);
      };
      auto prefetch_tile = [&](int pblk) {
        if (pblk >= w.blk_end) return;
        for (int bx = 0; bx < boxes; ++bx) {
          const int pos0 = pblk * kTile + bx * rows_per_box;
          const int j = pos0 / ps;
          if (j < first_page || j > last_page || j >= nb) continue;
          const int pid = page_id(j, pbatch0, pmy_id);
          if (lane != 0 || pid < 0 || pid >= a.num_pages) continue;
          const int64_t row = layer_row0 + static_cast<int64_t>(pid) * ps + pos0 % ps;
          const uint8_t* src = pool_bytes + row * (kDimRow * 2);
          const uint32_t bytes = static_cast<uint32_t>(rows_per_box * kDimRow * 2);
          if (boxes == 1) {  // this rank's half of the tile's contiguous rows
            prefetch_l2_bulk(src + rank * (bytes / 2), bytes / 2);
          } else if (bx == static_cast<int>(rank)) {
            prefetch_l2_bulk(src, bytes);
          }
        }
      };
      for (int pblk = w.blk_begin; pblk < w.blk_begin + kPrefetchTiles; ++pblk) prefetch_tile(pblk);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarQFree), (n_items & 1u) ^ 1u, abort_flag));
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(kBarQFull), kChunks * kQChunkBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &p.q_map, bar(kBarQFull), c * 64,
                      w.b * H + static_cast<int>(rank) * Hh);
      }
      last_q_item = static_cast<int>(n_items);
      for (int blk = w.blk_begin; blk < w.blk_end; ++blk, ++g) {
        const uint32_t stage = g % kStages, use = g / kStages;
        prefetch_tile(blk + kPrefetchTiles);
        int rows[2];
        int nbox = 0;
#pragma unroll
        for (int bx = 0; bx < 2; ++bx) {
          rows[bx] = -1;
          if (bx >= boxes) continue;
          const int pos0 = blk * kTile + bx * rows_per_box;
          const int j = pos0 / ps;
          if (j < first_page || j > last_page) continue;
          int row;
          if (j >= nb) {
            if (lane == 0) flag_status(status, MLA_STATUS_BAD_LENGTH);
            row = oob_row;
          } else {
            const int pid = page_id(j, batch0, my_id);
            if (pid < 0 || pid >= a.num_pages) {
              if (lane == 0) flag_status(status, MLA_STATUS_BAD_PAGE);
              row = oob_row;
            } else {
              row = static_cast<int>(layer_row0 + static_cast<int64_t>(pid) * ps + pos0 % ps);
            }
          }
          rows[bx] = row;
          ++nbox;
        }
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarKvEmpty + stage), (use & 1u) ^ 1u, abort_flag));
        if (!ok) break;
        if (lane == 0) {
          const uint32_t kvbar = bar(kBarKvFull + stage);
          mbar_arrive_expect_tx(kvbar, static_cast<uint32_t>(nbox * kChunks * rows_per_box * 128));
          const uint32_t dst0 = sbase + kOffKV + stage * kStageBytes;
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) {
            if (rows[bx] < 0) continue;
            for (int c = 0; c < kChunks; ++c)
              tma_load_2d_hint(dst0 + c * kKvChunkBytes + bx * rows_per_box * 128, &p.kv_map, kvbar, c * 64,
                               rows[bx], kv_policy);
          }
        }
      }
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        flag_status(status, MLA_STATUS_TIMEOUT);
      }
      if (*abort_flag) {
        // Let every copy already issued land before the CTA can exit.
        for (uint32_t k = (g > kStages ? g - kStages : 0); k < g; ++k)
          mbar_wait(bar(kBarKvFull + k % kStages), (k / kStages) & 1u, nullptr);
        if (last_q_item >= 0) mbar_wait(bar(kBarQFull), last_q_item & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16(64, kTile, false, false);
      uint32_t g = 0, n_items = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it, ++n_items) {
        const WorkItem w = items[it];
        const int nt = w.blk_end - w.blk_begin;
        if (!mbar_wait(bar(kBarQFull), n_items & 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        for (int t = 0; t < nt; ++t, ++g) {
          const uint32_t stage = g % kStages, use = g / kStages;
          const uint32_t b = g & 1u, u = g >> 1;
          if (!mbar_wait(bar(kBarKvFull + stage), use & 1u, abort_flag)) { ok = false; break; }
          if (!mbar_wait(bar(kBarSFree + b), (u & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kv = sbase + kOffKV + stage * kStageBytes;
          const uint32_t tS = tmem + kColS + 32u * b;
          for (int c = 0; c < kChunks; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sdesc_sw128(sbase + kOffQ + c * kQChunkBytes + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(kv + c * kKvChunkBytes + k * 32, 16, 1024);
              mma_bf16_ss(tS, ad, bd, idesc_qk, (c | k) != 0);
            }
          mma_commit(bar(kBarSFull + b));
        }
        if (ok) mma_commit(bar(kBarQFree));  // every QK of this item issued
      }
      if (!ok) {
        *abort_flag = 1;
        flag_status(status, MLA_STATUS_TIMEOUT);
      }
      mma_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, nullptr);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      const uint32_t idesc_pv = idesc_bf16(128, 256, false, true);
      const uint32_t tO = tmem + kColO;
      uint32_t g = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it) {
        const WorkItem w = items[it];
        const int nt = w.blk_end - w.blk_begin;
        for (int t = 0; t < nt; ++t, ++g) {
          const uint32_t b = g & 1u, u = g >> 1;
          if (!mbar_wait<true>(bar(kBarPFull + b), u & 1u, abort_flag)) { ok = false; break; }
          if (!mbar_wait(bar(kBarOFixed + b), u & 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          fence_proxy_async_smem();
          const uint32_t v0 = sbase + kOffKV + (g % kStages) * kStageBytes + 4 * rank * kKvChunkBytes;
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) {
            const uint64_t ad = sdesc_sw128(sbase + kOffP + b * kPBytes + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(v0 + k * 16 * 128, kKvChunkBytes, 1024);
            mma_bf16_ss(tO, ad, bd, idesc_pv, (t | k) != 0);
          }
          mma_commit(bar(kBarKvEmpty + g % kStages));
          mma_commit_both(bar(kBarPvDone + b));
        }
      }
      if (!ok) {
        *abort_flag = 1;
        flag_status(status, MLA_STATUS_TIMEOUT);
      }
      mma_commit(bar(kBarDrainPv));
      mbar_wait(bar(kBarDrainPv), 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax, correction, epilogue
    // Each S row (one head of this rank) is split over lanes i and i + 16 of
    // its warp (16 tokens each); every lane also owns O row 32 q4 + lane.
    // Per tile g: (A) scores -> P in registers; (B) once PV(g-2) is done in
    // both ranks, P rows go to both ranks' P buffer; (C) once the peer's rows
    // have landed, rescale the owned O rows and release PV(g).
    const int q4 = warp & 3;
    const int half = lane >> 4;
    const int srow = q4 * 16 + (lane & 15);
    const bool s_active = srow < Hh;
    const int gh = static_cast<int>(rank) * Hh + srow;
    const int orow = q4 * 32 + lane;
    const bool o_warp = q4 * 32 < H;
    const int peer_rows = min(max(Hh - q4 * 16, 0), 16);
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tO = tmem + lane_base + kColO;
    const uint32_t dim0 = 256u * rank;
    const int tid_sm = threadIdx.x - 64;
    auto wwait = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, abort_flag));
    };
    auto wwait_cluster = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait<true>(b, parity, abort_flag));
    };
    // Step C for tile gp: rescale owned O rows by the factors both ranks
    // sent, then let the PV issuer run PV(gp).
    auto finish_tile = [&](uint32_t gp, bool first_of_item) -> bool {
      const uint32_t bp = gp & 1u, up = gp >> 1;
      if (!wwait_cluster(bar(kBarPFull + bp), up & 1u)) return false;
      if (!first_of_item && o_warp) {
        const float ao = orow < H ? alpha_s[bp * 128 + orow] : 1.f;
        if (__any_sync(0xffffffffu, ao != 1.f)) {
          // O must hold PV(gp - 1) before it is rescaled.
          if (!wwait(bar(kBarPvDone + ((gp - 1) & 1u)), ((gp - 1) >> 1) & 1u)) return false;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 256 / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(tO + c * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * ao);
            tmem_st16(tO + c * 16, r);
          }
          tmem_wait_st();
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarOFixed + bp));
      return true;
    };
    uint32_t g = 0, n_items = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it, ++n_items) {
      const WorkItem w = items[it];
      const int lo = max(w.blk_begin * kTile, w.tok_lo);
      const int hi = min(w.blk_end * kTile, w.tok_hi);
      float m = -CUDART_INF_F, l = 0.f;
      for (int blk = w.blk_begin; blk < w.blk_end; ++blk, ++g) {
        const int base = blk * kTile;
        const uint32_t b = g & 1u, u = g >> 1;
        // (A) scores of this tile, 16 per lane.
        if (!wwait(bar(kBarSFull + b), u & 1u)) { ok = false; break; }
        tc_fence_after();
        float s[16];
        {
          uint32_t r[16];
          tmem_ld16x2(tmem + lane_base + kColS + 32u * b, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) s[i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(bar(kBarSFree + b));
        const int pos0 = base + 16 * half;
        float mx = -CUDART_INF_F;
        if (lo <= base && hi >= base + kTile) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            s[i] *= a.scale_log2;
            mx = fmaxf(mx, s[i]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int pos = pos0 + i;
            s[i] = (pos >= lo && pos < hi) ? s[i] * a.scale_log2 : -CUDART_INF_F;
            mx = fmaxf(mx, s[i]);
          }
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        float alpha = 1.f;
        if (mx > m + kRescaleThreshold) {  // same decision in both halves
          alpha = fast_exp2(m - mx);       // 0 on the first tile (m = -inf)
          l *= alpha;
          m = mx;
        }
        uint32_t pk[8];
        float rs = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float p0 = fast_exp2(s[2 * i] - m), p1 = fast_exp2(s[2 * i + 1] - m);
          rs += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        l += rs;
        // Value rows of this tile outside [lo, hi) may hold anything (stale
        // or unwritten slots): zero this rank's value dims there so that
        // 0 * garbage cannot reach O. QK of the tile is complete here.
        if (lo > base || hi < base + kTile) {
          const uint32_t v0 = sbase + kOffKV + (g % kStages) * kStageBytes + 4 * rank * kKvChunkBytes;
          for (int e = tid_sm; e < kTile * 4 * 8; e += 128) {
            const int r = e >> 5, c = (e >> 3) & 3, piece = e & 7;
            const int pos = base + r;
            if (pos < lo || pos >= hi) st_shared_v4(v0 + c * kKvChunkBytes + r * 128 + piece * 16, 0, 0, 0, 0);
          }
        }
        // (B) P buffer b is free in both ranks once PV(g-2) is done in both.
        if (!wwait(bar(kBarPvDone + b), (u & 1u) ^ 1u)) { ok = false; break; }
        if (s_active) {
          const uint32_t prow = sbase + kOffP + b * kPBytes + gh * 128;
          const uint32_t prow_peer = mapa(prow, peer);
          const uint32_t pfull_peer = mapa(bar(kBarPFull + b), peer);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t off = ((2 * half + j) ^ (gh & 7)) * 16;
            st_shared_v4(prow + off, pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            st_async_v4(prow_peer + off, pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3], pfull_peer);
          }
          if (half == 0) {
            const uint32_t aaddr = sbase + kOffAlpha + (b * 128 + gh) * 4;
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(aaddr), "r"(__float_as_uint(alpha)) : "memory");
            st_async_b32(mapa(aaddr, peer), __float_as_uint(alpha), pfull_peer);
          }
        }
        fence_proxy_async_smem();
        if (lane == 0)
          mbar_arrive_expect_tx(bar(kBarPFull + b), static_cast<uint32_t>(peer_rows * kPeerBytesPerRow));
        else
          mbar_arrive(bar(kBarPFull + b));
        // (C) once the peer's rows have landed: rescale, release PV(g).
        if (!finish_tile(g, blk == w.blk_begin)) { ok = false; break; }
      }
      if (!ok) break;
      // Epilogue: final row sums of both ranks, wait for the last PV,
      // normalise, store.
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (s_active && half == 0) {
        l_s[gh] = l;
        st_async_b32(mapa(sbase + kOffL + gh * 4, peer), __float_as_uint(l), mapa(bar(kBarLFull), peer));
      }
      if (lane == 0)
        mbar_arrive_expect_tx(bar(kBarLFull), static_cast<uint32_t>(peer_rows * 4));
      else
        mbar_arrive(bar(kBarLFull));
      if (!wwait_cluster(bar(kBarLFull), n_items & 1u)) { ok = false; break; }
      if (!wwait(bar(kBarPvDone + ((g - 1) & 1u)), ((g - 1) >> 1) & 1u)) { ok = false; break; }
      tc_fence_after();
      if (s_active && half == 0) {
        const float lse2 = m + log2f(l);
        if (w.slot < 0) {
          if (a.lse) a.lse[static_cast<size_t>(w.b) * H + gh] = lse2 * 0.69314718055994531f;
        } else {
          reinterpret_cast<float*>(ws + a.lay.partial_lse)[static_cast<size_t>(w.slot) * H + gh] = lse2;
        }
      }
      if (o_warp) {
        const float inv_l = orow < H ? 1.f / l_s[orow] : 0.f;
#pragma unroll 1
        for (int c = 0; c < 256 / 32; ++c) {
          uint32_t r[32];
          tmem_ld16(tO + c * 32, r);
          tmem_ld16(tO + c * 32 + 16, r + 16);
          tmem_wait_ld();
          if (orow < H) {
            if (w.slot < 0) {
              __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                                   (static_cast<size_t>(w.b) * H + orow) * kDimCkv + dim0 + c * 32;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l);
                o.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l);
                o.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l);
                o.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l);
                reinterpret_cast<uint4*>(dst)[v] = o;
              }
            } else {
              float* dst = reinterpret_cast<float*>(ws + a.lay.partial_o) +
                           (static_cast<size_t>(w.slot) * H + orow) * kDimCkv + dim0 + c * 32;
#pragma unroll
              for (int v = 0; v < 8; ++v)
                reinterpret_cast<float4*>(dst)[v] =
                    make_float4(__uint_as_float(r[4 * v]) * inv_l, __uint_as_float(r[4 * v + 1]) * inv_l,
                                __uint_as_float(r[4 * v + 2]) * inv_l, __uint_as_float(r[4 * v + 3]) * inv_l);
            }
          }
        }
      }
      tc_fence_before();
    }
    if (!ok) {
      *abort_flag = 1;
      flag_status(status, MLA_STATUS_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();  // the peer may still address this CTA's shared memory
}

}  // namespace

int decode_max_active_clusters() {
  static int cached = -1;
  if (cached > 0) return cached;
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return -1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cfg.gridDim = dim3(2 * (sms / 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel, &cfg);
  if (e != cudaSuccess || n <= 0) return -1;
  cached = n;
  return n;
}

cudaError_t launch_decode(const CUtensorMap& kv_map, const CUtensorMap& q_map, const DecodeArgs& a,
                          int clusters, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  Params p;
  p.kv_map = kv_map;
  p.q_map = q_map;
  p.a = a;
  mla_decode_kernel<<<dim3(2 * clusters), dim3(kThreads), kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
