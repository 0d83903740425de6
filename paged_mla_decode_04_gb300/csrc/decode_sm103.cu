// Absorbed paged MLA decode on sm_103a tensor cores.
//
// What it computes (MoE-Infinity PR #195 "DeepSeek-V2/V3 paged-attention
// shim (MLA)" and SGLang PR #32972 "Let Kimi-Linear use the paged MLA
// attention backends"): for request b and head h, softmax over the attended
// positions of scale * q[b,h,:576] . K_t, weighted sum of K_t[:512], where
// K_t is the request's 576-d latent row at position t, fetched through its
// page list. Every head shares each latent row, so S = Q K^T (heads x tokens,
// K = 576) and O = P V (heads x 512, K = tokens) are dense contractions.
//
// GB300 mapping. A 128-head fp32 O of width 512 is a whole SM's tensor
// memory (128 lanes x 512 columns), so one work unit is a cluster of two
// CTAs that split the latent dimension: rank 0 holds c_kv[0:256), rank 1
// holds c_kv[256:512) and the 64 rope dims. Each rank
//   - gathers its slice of every 64-token tile by TMA (one box per page and
//     64-dim chunk, 128-byte swizzle) into a 2-stage ring;
//   - computes a partial S over its dims with tcgen05.mma (M=128 heads,
//     N=64 tokens) into TMEM;
//   - swaps partial S with the peer through distributed shared memory, so
//     both ranks hold the same full S, and runs the same online softmax
//     (base 2, lazy rescale: O is rescaled only when the running max grows by
//     more than 8, i.e. a factor 256; the final 1/l makes the result exact);
//   - accumulates its half of O = P V with tcgen05.mma (M=128, N=256, K=64)
//     in TMEM, V read straight from the gathered tile (MN-major operand).
// Warp roles per CTA (192 threads): warp 0 TMA producer, warp 1 TMEM owner
// and MMA issuer, warps 2-5 softmax and epilogue (thread = head row).
// Heads beyond num_heads (16/32/64) are padding rows of the M=128 MMA.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kTile = kBlockTokens;  // 64 tokens per tile
constexpr int kStages = 2;
constexpr int kChunkDims = 64;                       // one 128-byte swizzle row of bf16
constexpr int kKvChunkBytes = kTile * 128;           // [64 tokens][64 dims] bf16
constexpr int kQChunkBytes = 128 * 128;              // [128 heads][64 dims] bf16
constexpr int kMaxChunks = 5;                        // rank 1: 4 c_kv chunks + rope
constexpr int kStageBytes = kMaxChunks * kKvChunkBytes;
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kMaxChunks * kQChunkBytes;
constexpr int kOffP = kOffKV + kStages * kStageBytes;
constexpr int kOffX = kOffP + 128 * kTile * 2;
constexpr int kOffBar = kOffX + 128 * kTile * 4;
constexpr int kSmemBytes = kOffBar + 512 + 1024;  // barriers + alignment slack
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // O half: columns [0, 256)
constexpr uint32_t kColS = 256;  // S: columns [256, 320)
constexpr float kRescaleThreshold = 8.0f;

// Barrier slots (8 bytes each) at kOffBar.
enum Bar {
  kBarKvFull = 0,                 // [kStages]
  kBarKvEmpty = kBarKvFull + kStages,
  kBarQFull = kBarKvEmpty + kStages,
  kBarQFree,
  kBarSFull,
  kBarSFree,
  kBarPFull,
  kBarPFree,
  kBarXFull,                      // [4] one per softmax warp quarter
  kBarXFree = kBarXFull + 4,      // [4]
  kBarDrain = kBarXFree + 4,
  kNumBars
};
static_assert(kNumBars * 8 + 16 <= 512, "barrier area");

struct Params {
  CUtensorMap kv_map;  // pool rows [NL*P*ps][576] bf16, box {64, min(ps, 64)}
  CUtensorMap q_map;   // q rows [B*H][576] bf16, box {64, 128}
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
  const int nchunks = rank == 0 ? 4 : 5;
  const int dim0 = rank == 0 ? 0 : 256;

  // The plan must describe this call; otherwise do nothing.
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
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 128);
    mbar_init(bar(kBarPFull), 128);
    mbar_init(bar(kBarPFree), 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(kBarXFull + i), 32);
      mbar_init(bar(kBarXFree + i), 32);
    }
    mbar_init(bar(kBarDrain), 1);
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

  const int H = a.num_heads;
  const int ps = a.page_size;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t kv_policy = l2_policy_evict_first();
      const int64_t layer_row0 = static_cast<int64_t>(a.layer) * a.num_pages * ps;
      const int oob_row = a.num_layers * a.num_pages * ps;  // reads as zeros
      const int rows_per_box = ps < kTile ? ps : kTile;
      const int boxes = kTile / rows_per_box;
      uint32_t g = 0;
      int last_q_item = -1;
      uint32_t n_items = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it, ++n_items) {
        const WorkItem w = items[it];
        if (!mbar_wait(bar(kBarQFree), (n_items & 1u) ^ 1u, abort_flag)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(kBarQFull), nchunks * kQChunkBytes);
        for (int c = 0; c < nchunks; ++c)
          tma_load_2d(sbase + kOffQ + c * kQChunkBytes, &p.q_map, bar(kBarQFull), dim0 + c * kChunkDims,
                      w.b * H);
        last_q_item = static_cast<int>(n_items);
        const int L = w.tok_hi - 1;
        const int first_page = w.tok_lo / ps, last_page = L / ps;
        const int nb = a.page_indptr ? a.page_indptr[w.b + 1] - a.page_indptr[w.b] : a.max_blocks;
        const int32_t* ids = a.page_indptr ? a.page_ids + a.page_indptr[w.b]
                                           : a.page_ids + static_cast<int64_t>(w.b) * a.max_blocks;
        for (int blk = w.blk_begin; blk < w.blk_end; ++blk, ++g) {
          const uint32_t stage = g % kStages, use = g / kStages;
          if (!mbar_wait(bar(kBarKvEmpty + stage), (use & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          // Which boxes of this tile hold attended positions.
          int rows[kTile / 16];
          int nbox = 0;
          for (int bx = 0; bx < boxes; ++bx) {
            const int pos0 = blk * kTile + bx * rows_per_box;
            const int j = pos0 / ps;
            if (j < first_page || j > last_page) { rows[bx] = -1; continue; }
            int row;
            if (j >= nb) {
              flag_status(status, MLA_STATUS_BAD_LENGTH);
              row = oob_row;
            } else {
              const int pid = ids[j];
              if (pid < 0 || pid >= a.num_pages) {
                flag_status(status, MLA_STATUS_BAD_PAGE);
                row = oob_row;
              } else {
                row = static_cast<int>(layer_row0 + static_cast<int64_t>(pid) * ps + pos0 % ps);
              }
            }
            rows[bx] = row;
            ++nbox;
          }
          const uint32_t kvbar = bar(kBarKvFull + stage);
          mbar_arrive_expect_tx(kvbar, static_cast<uint32_t>(nbox * nchunks * rows_per_box * 128));
          const uint32_t dst0 = sbase + kOffKV + stage * kStageBytes;
          for (int bx = 0; bx < boxes; ++bx) {
            if (rows[bx] < 0) continue;
            for (int c = 0; c < nchunks; ++c)
              tma_load_2d_hint(dst0 + c * kKvChunkBytes + bx * rows_per_box * 128, &p.kv_map, kvbar,
                               dim0 + c * kChunkDims, rows[bx], kv_policy);
          }
        }
      }
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
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16(128, kTile, false, false);
      const uint32_t idesc_pv = idesc_bf16(128, 256, false, true);
      const uint32_t tS = tmem + kColS, tO = tmem + kColO;
      uint32_t g = 0, n_items = 0;
      bool ok = true;
      auto issue_qk = [&](uint32_t gq) -> bool {
        const uint32_t stage = gq % kStages, use = gq / kStages;
        if (!mbar_wait(bar(kBarKvFull + stage), use & 1u, abort_flag)) return false;
        if (!mbar_wait(bar(kBarSFree), (gq & 1u) ^ 1u, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kv = sbase + kOffKV + stage * kStageBytes;
        for (int c = 0; c < nchunks; ++c)
#pragma unroll
          for (int k = 0; k < kChunkDims / 16; ++k) {
            const uint64_t ad = sdesc_sw128(sbase + kOffQ + c * kQChunkBytes + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(kv + c * kKvChunkBytes + k * 32, 16, 1024);
            mma_bf16_ss(tS, ad, bd, idesc_qk, (c | k) != 0);
          }
        mma_commit(bar(kBarSFull));
        return true;
      };
      for (int it = it_begin; it < it_end && ok; ++it, ++n_items) {
        const WorkItem w = items[it];
        const int nt = w.blk_end - w.blk_begin;
        if (!mbar_wait(bar(kBarQFull), n_items & 1u, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (!issue_qk(g)) { ok = false; break; }
        for (int t = 0; t < nt; ++t) {
          const uint32_t gc = g + t;
          if (t + 1 < nt) {
            if (!issue_qk(gc + 1)) { ok = false; break; }
          } else {
            mma_commit(bar(kBarQFree));  // every QK of this item issued
          }
          if (!mbar_wait(bar(kBarPFull), gc & 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kv = sbase + kOffKV + (gc % kStages) * kStageBytes;
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) {
            const uint64_t ad = sdesc_sw128(sbase + kOffP + k * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(kv + k * 16 * 128, kKvChunkBytes, 1024);
            mma_bf16_ss(tO, ad, bd, idesc_pv, (t | k) != 0);
          }
          mma_commit(bar(kBarKvEmpty + gc % kStages));
          mma_commit(bar(kBarPFree));
        }
        g += nt;
      }
      if (!ok) {
        *abort_flag = 1;
        flag_status(status, MLA_STATUS_TIMEOUT);
      }
      // Wait for every MMA issued so far before TMEM can be released.
      mma_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q4 * 32 + lane;
    const bool active = q4 * 32 < H;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS;
    const uint32_t tO = tmem + lane_base + kColO;
    const uint32_t x_local = sbase + kOffX;
    const uint32_t x_peer = mapa(x_local, peer);
    const uint32_t xfull_peer = mapa(bar(kBarXFull + q4), peer);
    const uint32_t xfree_peer = mapa(bar(kBarXFree + q4), peer);
    const int tid_sm = threadIdx.x - 64;  // 0..127 across the softmax warps
    // Waits of these warps are made warp-uniform, since the tcgen05.ld/st
    // that follow them are warp-collective.
    auto wwait = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, abort_flag));
    };
    auto wwait_cluster = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait<true>(b, parity, abort_flag));
    };
    uint32_t g = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const WorkItem w = items[it];
      const int lo = max(w.blk_begin * kTile, w.tok_lo);
      const int hi = min(w.blk_end * kTile, w.tok_hi);
      float m = -CUDART_INF_F, l = 0.f;
      for (int blk = w.blk_begin; blk < w.blk_end; ++blk, ++g) {
        const int base = blk * kTile;
        if (!wwait(bar(kBarSFull), g & 1u)) { ok = false; break; }
        tc_fence_after();
        float s[kTile];
        {
          uint32_t r[kTile];
#pragma unroll
          for (int c = 0; c < kTile / 16; ++c) tmem_ld16(tS + c * 16, r + c * 16);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kTile; ++i) s[i] = __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(bar(kBarSFree));
        // Swap partial scores with the peer rank (row-wise, 16-byte pieces
        // XOR-swizzled by row to spread banks).
        if (!wwait_cluster(bar(kBarXFree + q4), (g & 1u) ^ 1u)) { ok = false; break; }
        if (active) {
#pragma unroll
          for (int j = 0; j < kTile / 4; ++j) {
            const uint32_t off = row * (kTile * 4) + ((j ^ (row & 15)) * 16);
            st_cluster_v4(x_peer + off, __float_as_uint(s[4 * j]), __float_as_uint(s[4 * j + 1]),
                          __float_as_uint(s[4 * j + 2]), __float_as_uint(s[4 * j + 3]));
          }
        }
        mbar_arrive_remote(xfull_peer);
        if (!wwait_cluster(bar(kBarXFull + q4), g & 1u)) { ok = false; break; }
        if (active) {
#pragma unroll
          for (int j = 0; j < kTile / 4; ++j) {
            const uint32_t off = row * (kTile * 4) + ((j ^ (row & 15)) * 16);
            uint32_t x0, x1, x2, x3;
            ld_shared_v4(x_local + off, x0, x1, x2, x3);
            s[4 * j] += __uint_as_float(x0);
            s[4 * j + 1] += __uint_as_float(x1);
            s[4 * j + 2] += __uint_as_float(x2);
            s[4 * j + 3] += __uint_as_float(x3);
          }
        }
        mbar_arrive_remote(xfree_peer);
        // Online softmax in base 2 over the valid positions [lo, hi).
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int i = 0; i < kTile; ++i) {
          const int pos = base + i;
          s[i] = (pos >= lo && pos < hi) ? s[i] * a.scale_log2 : -CUDART_INF_F;
          mx = fmaxf(mx, s[i]);
        }
        const bool first_tile = blk == w.blk_begin;
        const bool need = active && mx > m + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
          alpha = fast_exp2(m - mx);  // 0 on the first tile (m = -inf)
          l *= alpha;
          m = mx;
        }
        // PV of the previous tile must be done before O or P change.
        if (!wwait(bar(kBarPFree), (g & 1u) ^ 1u)) { ok = false; break; }
        tc_fence_after();
        if (!first_tile && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < 256 / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(tO + c * 16, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st16(tO + c * 16, r);
          }
          tmem_wait_st();
        }
        // P = 2^(s - m) as bf16, K-major with the 128-byte swizzle.
        if (active) {
          float rs = 0.f;
#pragma unroll
          for (int j = 0; j < kTile / 8; ++j) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float p0 = fast_exp2(s[8 * j + 2 * e] - m);
              const float p1 = fast_exp2(s[8 * j + 2 * e + 1] - m);
              rs += p0 + p1;
              pk[e] = pack_bf16x2(p0, p1);
            }
            const uint32_t off = kOffP + row * 128 + ((j ^ (row & 7)) * 16);
            st_shared_v4(sbase + off, pk[0], pk[1], pk[2], pk[3]);
          }
          l += rs;
        }
        // Rows of this tile outside [lo, hi) may hold anything (stale or
        // unwritten slots): zero their value part so that 0 * garbage can
        // not reach O.
        if (lo > base || hi < base + kTile) {
          const uint32_t kv = sbase + kOffKV + (g % kStages) * kStageBytes;
          for (int e = tid_sm; e < kTile * 4 * 8; e += 128) {
            const int r = e >> 5;           // row of the tile
            const int c = (e >> 3) & 3;     // value chunk
            const int piece = e & 7;
            const int pos = base + r;
            if (pos < lo || pos >= hi) st_shared_v4(kv + c * kKvChunkBytes + r * 128 + piece * 16, 0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull));
      }
      if (!ok) break;
      // Epilogue: wait for the last PV, normalise, store.
      if (!wwait(bar(kBarPFree), (g - 1) & 1u)) { ok = false; break; }
      tc_fence_after();
      const float inv_l = active ? 1.f / l : 0.f;
      const float lse2 = m + log2f(l);
#pragma unroll 1
      for (int c = 0; c < 256 / 32 && active; ++c) {
        uint32_t r[32];
        tmem_ld16(tO + c * 32, r);
        tmem_ld16(tO + c * 32 + 16, r + 16);
        tmem_wait_ld();
        if (row < H) {
          if (w.slot < 0) {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                                 (static_cast<size_t>(w.b) * H + row) * kDimCkv + dim0 + c * 32;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 pk;
              pk.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l);
              pk.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l);
              pk.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l);
              pk.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l);
              reinterpret_cast<uint4*>(dst)[v] = pk;
            }
          } else {
            float* dst = reinterpret_cast<float*>(ws + a.lay.partial_o) +
                         (static_cast<size_t>(w.slot) * H + row) * kDimCkv + dim0 + c * 32;
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(dst)[v] =
                  make_float4(__uint_as_float(r[4 * v]) * inv_l, __uint_as_float(r[4 * v + 1]) * inv_l,
                              __uint_as_float(r[4 * v + 2]) * inv_l, __uint_as_float(r[4 * v + 3]) * inv_l);
          }
        }
      }
      if (active && row < H && rank == 0) {
        if (w.slot < 0) {
          if (a.lse) a.lse[static_cast<size_t>(w.b) * H + row] = lse2 * 0.69314718055994531f;
        } else {
          reinterpret_cast<float*>(ws + a.lay.partial_lse)[static_cast<size_t>(w.slot) * H + row] = lse2;
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
