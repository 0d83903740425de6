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
// GB300 mapping (measured constraints: a fp32 O for 128 heads x 512 dims
// fills one SM's tensor memory; a tcgen05.mma M=128 K=16 costs ~45 cycles
// at N=64 and 128 at N=256, so only M=128 instructions pay; SM-to-SM shared memory
// moves ~13 bytes/cycle, well below an SM's share of HBM). One work unit is a
// cluster of two CTAs, rank r, that split the latent dimension evenly:
//   - rank r holds c_kv[256r, 256r+256) and rope[32r, 32r+32) of every row
//     (288 dims) and of q. Per item its q slice goes to TMEM (tcgen05.cp,
//     staged through two ring slots), so shared memory holds a 5-stage ring
//     of 64-token tiles gathered by TMA (for pages of 64 tokens or more one
//     3-D box covers the rank's four c_kv chunks, else one box per page and
//     chunk; the rope part is one more box), and
//     the partial S_r = Q_r K_r^T for all heads comes from tcgen05.mma
//     M=128 x N=64 with A read from TMEM;
//   - each rank scales its partial scores to log2 units, rounds them to
//     fp16 and sends them to the peer (st.async, 16 KB per tile), so both
//     ranks form the same sum f16(S_0) + f16(S_1) (fp32 addition commutes)
//     and run the same online softmax for all heads (base 2, lazy rescale:
//     the reference max moves only when the running max grows by more than
//     8, the final 1/l makes the result exact), each keeping P in its own
//     TMEM. One exchange per tile and no P traffic. The rounding puts a
//     relative error of at most 2^-11 of each partial on each score;
//   - each rank accumulates O for all heads over its 256 value dims with
//     tcgen05.mma M=128 x N=256 x K=64, P read from TMEM and V read MN-major
//     straight from the gathered tile.
// TMEM columns: O [0, 256) fp32, q [256, 400), S [400, 464) fp32, P [464,
// 496) 16-bit pairs; S and P are single-buffered (the next QK waits for S to be
// read, the next P for the previous PV).
// Warp roles per CTA. bf16 pools (352 threads): warp 0 TMA producer, warp 1
// TMEM owner and QK issuer, warps 2-9 exchange / softmax / correction /
// epilogue, warp 10 PV issuer. fp8 pools (512 threads, one role group per
// warpgroup so that setmaxnreg can move registers to the softmax warps):
// warps 0, 1, 2 producer, QK issuer, PV issuer (warp 3 idle), warps 4-11
// softmax, warps 12-15 widen fp8 tiles to f16 in place in their ring slot.
// A softmax warp w works on 16 lanes of TMEM lane quarter w & 3; a head's row
// belongs to two threads, tokens [0, 32) and [32, 64) of each tile.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace mla {
namespace {

constexpr int kTile = kBlockTokens;                 // 64 tokens per tile
constexpr int kMaxStages = 5;
constexpr int kWideChunks = 4;                      // c_kv chunks of 64 dims per rank
constexpr int kWideBytes = kTile * 128;             // [64 tokens][64 dims] bf16, 128B swizzle
constexpr int kNarrowBytes = kTile * 64;            // [64 tokens][32 rope dims], 64B swizzle
constexpr int kStageBytes = kWideChunks * kWideBytes + kNarrowBytes;   // 36 KB
constexpr int kQWideBytes = 128 * 128;              // [128 heads][64 dims], 16 KB
constexpr int kQNarrowBytes = 128 * 64;             // [128 heads][32 rope dims], 8 KB
constexpr int kXBytes = 128 * kTile * 2;            // the peer's partial S of 128 rows, bf16
constexpr int kF8WideBytes = kTile * 256;           // fp8 tile: [64 tokens][256 c_kv dims], unswizzled
constexpr int kF8Bytes = kF8WideBytes + kTile * 32;  // + [64 tokens][32 rope dims]
constexpr int kRawOff = kStageBytes - kF8Bytes;      // fp8 pools: the raw tile lands in the slot's back half

// Shared-memory plan of the two variants: q rope part | 5-stage ring of
// 16-bit tiles | exchange | barriers. fp8 pools: a raw tile (18 KB) lands in
// the back half of its ring slot and is widened to f16 in place (every code
// is read into registers before any is overwritten).
template <bool kFp8>
struct Cfg {
  static constexpr int kStages = 5;
  static constexpr int kOffQn = 0;                            // q rope part, staged for TMEM
  static constexpr int kOffKV = kOffQn + kQNarrowBytes;
  static constexpr int kOffX = kOffKV + kStages * kStageBytes;  // [2 buffers]
  static constexpr int kOffBar = kOffX + 2 * kXBytes;
  static constexpr int kSmemBytes = kOffBar + 1024 + 1024;  // barriers + alignment slack
  static constexpr int kThreads = kFp8 ? 512 : 352;
  static constexpr int kSmWarp0 = kFp8 ? 4 : 2;    // first of the 8 softmax warps
  static constexpr int kPvWarp = kFp8 ? 2 : 10;
  static constexpr int kCvtWarp0 = 12;             // fp8 pools: warps 12-15 widen fp8 tiles to f16
  // fp8 pools: registers per thread by warpgroup after setmaxnreg (producer
  // and issuers, softmax, softmax, converters); they add up to the launch's
  // 512 threads x 128.
  static constexpr int kRegsIssue = 64, kRegsSoftmax = 176, kRegsCvt = 96;
  static_assert(!kFp8 || kRegsIssue + 2 * kRegsSoftmax + kRegsCvt == 4 * 128, "register split");
  static_assert(kOffKV % 1024 == 0 && kOffX % 1024 == 0, "alignment");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kStages <= kMaxStages, "barrier arrays");
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;                       // O: [0, 256) fp32
constexpr uint32_t kColQ = 256;                     // q: [256, 400) 16-bit pairs (wide 128 + rope 16)
constexpr uint32_t kColS = 400;                     // S: [400, 464) fp32
constexpr uint32_t kColP = 464;                     // P: [464, 496) 16-bit pairs (bf16, f16 for fp8 pools)
constexpr float kRescaleThreshold = 8.0f;

static_assert(kStageBytes % 1024 == 0 && kF8Bytes % 1024 == 0 && kRawOff % 1024 == 0, "alignment");
static_assert(2 * kQWideBytes <= kStageBytes, "a ring slot holds two wide q chunks");

enum Bar {
  kBarKvFull = 0,                  // [stages] tile (or q chunks) ready for the tensor core
  kBarKvEmpty = kBarKvFull + kMaxStages,
  // [stages] fp8 pools: the slot's raw contents landed (a tile's codes, or
  // two bf16 q chunks), not yet f16. One barrier per slot: its phases follow
  // the slot's uses, which the slot's release keeps in order. (A barrier
  // shared by all items' q chunks could complete twice before the widening
  // warps wait on it when an item has a single tile.)
  kBarRawFull = kBarKvEmpty + kMaxStages,
  kBarCvtRead = kBarRawFull + kMaxStages,  // fp8 pools: every converter holds the raw tile in registers
  kBarQnFull,                              // q rope part ready
  kBarQnRaw,                       // fp8 pools: q rope part landed, not yet f16
  kBarQnFree,                      // q rope part copied into TMEM
  kBarQDone,                       // every QK of the item complete: TMEM q may be replaced
  kBarSFull,
  kBarSFree,
  kBarXFull,                       // [2 buffers][4 quarters][2 halves]: the peer's partial rows landed
  kBarXFree = kBarXFull + 16,      // [2 buffers][4 quarters][2 halves]: the peer read this rank's partial rows
  kBarOFixed = kBarXFree + 16,     // P in TMEM and O rescaled for this tile
  kBarPvDone,                      // PV of the tile done
  kBarDrain,
  kBarDrainPv,
  kNumBars
};
static_assert(kNumBars * 8 + 8 <= 1024, "barrier area");  // + TMEM address, abort flag

struct Params {
  CUtensorMap kv_wide;    // pool rows [NL*P*ps][576]: bf16 box {64, rows} 128B swizzle; fp8 box {256, rows}
  CUtensorMap kv_narrow;  // same rows: bf16 box {32, rows} 64B swizzle; fp8 box {32, rows}
  CUtensorMap q_wide;     // q rows [B*H][576] bf16, box {64, 128}, 128B swizzle
  CUtensorMap q_narrow;   // box {32, 128}, 64B swizzle
  CUtensorMap kv_chunks;  // bf16 pools, page size >= 64: pool as [chunk 0-7][row][64 dims], box {64, 64, 4}
  DecodeArgs a;
};

__device__ __forceinline__ void flag_status(int* status, int bits) { atomicOr(status, bits); }

// 2^x with the hardware approximation (exact at -inf: returns +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<kFp8>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ Params p) {
  using C = Cfg<kFp8>;
  constexpr int kStages = C::kStages;
  constexpr int kOffQn = C::kOffQn;
  constexpr int kOffKV = C::kOffKV;
  constexpr int kOffX = C::kOffX;
  constexpr int kOffBar = C::kOffBar;
  // fp8 pools run the tensor core on f16 (q and P converted, codes exact).
  constexpr uint32_t kIdescQk = kFp8 ? idesc_f16(128, kTile, false, false) : idesc_bf16(128, kTile, false, false);
  constexpr uint32_t kIdescPv = kFp8 ? idesc_f16(128, 256, false, true) : idesc_bf16(128, 256, false, true);
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
  const int H = a.num_heads;
  const int ps = a.page_size;
  MLA_TRACER(trc5);  // kernel-level events (thread 0)
  MLA_TRACER(trc);   // this thread's role events
  if (threadIdx.x == 0) MLA_TRACE_EVENT(trc5, 5, kEvKernelStart, 0);
  if (threadIdx.x == 0) MLA_TRACE_EVENT(trc5, 5, kEvGlobalStart, 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKvFull + i), kFp8 ? 128 : 1);  // fp8: every converter thread arrives
      mbar_init(bar(kBarKvEmpty + i), 1);
    }
    for (int i = 0; i < kMaxStages; ++i) mbar_init(bar(kBarRawFull + i), 1);
    mbar_init(bar(kBarCvtRead), 128);
    mbar_init(bar(kBarQnFull), kFp8 ? 128 : 1);
    mbar_init(bar(kBarQnRaw), 1);
    mbar_init(bar(kBarQnFree), 1);
    mbar_init(bar(kBarQDone), 1);
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 256);
    mbar_init(bar(kBarOFixed), 256);
    mbar_init(bar(kBarPvDone), 1);
    for (int i = 0; i < 16; ++i) {
      mbar_init(bar(kBarXFull + i), 1);
      mbar_init(bar(kBarXFree + i), 1);
    }
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
    tma_prefetch_map(&p.kv_wide);
    tma_prefetch_map(&p.kv_narrow);
    tma_prefetch_map(&p.q_wide);
    tma_prefetch_map(&p.q_narrow);
    if (!kFp8 && ps >= kTile) tma_prefetch_map(&p.kv_chunks);
  }
  tc_fence_before();
  cluster_sync();  // barriers of both ranks initialised before any remote access
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Set-up above overlaps the previous kernel (the plan); from here on the
  // workspace, the pool and q are read.
  pdl_wait();
  // The cluster's item range is read together with the header (the grid
  // never has more clusters than the workspace's range table) and used
  // only if the plan matches.
  const int cs_lo = cstart[cluster_id], cs_hi = cstart[cluster_id + 1];
  const bool plan_ok = hd->planned == 1 && hd->batch == a.batch && hd->num_heads == a.num_heads &&
                       hd->q_len == a.q_len &&
                       hd->page_size == a.page_size && hd->window == a.window;
  int it_begin = 0, it_end = 0;
  if (plan_ok && cluster_id < hd->num_clusters) {
    it_begin = cs_lo;
    it_end = cs_hi;
  }
  if (!plan_ok && threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, MLA_STATUS_PLAN_MISMATCH);
  if (threadIdx.x == 0) MLA_TRACE_EVENT(trc5, 5, kEvSetupDone, it_end - it_begin);
  const int wide_x = 256 * static_cast<int>(rank);        // first c_kv dim of this rank
  const int narrow_x = 512 + 32 * static_cast<int>(rank);  // first rope dim of this rank

  // Ring slots: every item takes two slots for its q (wide chunks 0-1 and
  // 2-3, 16 KB each, on their way to TMEM), then one slot per 64-token tile.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if constexpr (kFp8) setmaxnreg_dec<C::kRegsIssue>();
    // The whole warp walks the tiles; lane 0 issues the copies. Page ids are
    // fetched 32 at a time by the warp (one coalesced load) and handed out
    // by shuffle, so a tile waits on no global load. bf16 pools: tiles go
    // straight into the ring. fp8 pools: a tile's codes go into the back
    // half of its ring slot and q into the ring unconverted; the converter
    // warps finish both.
    const uint64_t kv_policy = l2_policy_evict_first();
    const int64_t layer_row0 = static_cast<int64_t>(a.layer) * a.num_pages * ps;
    const int oob_row = a.num_layers * a.num_pages * ps;  // reads as zeros
    const int rows_per_box = ps < kTile ? ps : kTile;
    const int boxes = kTile / rows_per_box;
    const uint32_t row_bytes = kFp8 ? 256u + 32u : kWideChunks * 128u + 64u;
    uint32_t sl = 0;     // ring slot
    uint32_t raw_par = 0;   // fp8 pools: per slot, parity of its next raw phase (tile or q chunks)
    uint32_t raw_used = 0;  // fp8 pools: slots that have received a raw copy
    int last_qn_item = -1;
    uint32_t n_items = 0, gt = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it, ++n_items) {
      const WorkItem w = items[it];
      const int first_page = max(w.tok_lo, w.blk_begin * kTile) / ps;
      const int last_page = (min(w.tok_hi, w.blk_end * kTile) - 1) / ps;
      const int nb = a.page_indptr ? a.page_indptr[w.b + 1] - a.page_indptr[w.b] : a.max_blocks;
      const int32_t* ids = a.page_indptr ? a.page_ids + a.page_indptr[w.b]
                                         : a.page_ids + static_cast<int64_t>(w.b) * a.max_blocks;
      int batch0 = -64, my_id = -1;
      // q of this item: wide chunks through two ring slots, the rope part
      // into its own buffer once the previous item's copy into TMEM is done.
      for (int h = 0; h < 2 && ok; ++h, ++sl) {
        const uint32_t stage = sl % kStages, use = sl / kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarKvEmpty + stage), (use & 1u) ^ 1u, abort_flag));
        if (ok && lane == 0) {
          const uint32_t fb = kFp8 ? bar(kBarRawFull + stage) : bar(kBarKvFull + stage);
          mbar_arrive_expect_tx(fb, 2 * kQWideBytes);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(sbase + kOffKV + stage * kStageBytes + c * kQWideBytes, &p.q_wide, fb,
                        wide_x + 64 * (2 * h + c), w.b * a.rows + w.row0);
        }
        if (ok && kFp8) {
          raw_par ^= 1u << stage;
          raw_used |= 1u << stage;
        }
      }
      if (!ok) break;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarQnFree), (n_items & 1u) ^ 1u, abort_flag));
      if (!ok) break;
      if (lane == 0) {
        const uint32_t qb = bar(kFp8 ? kBarQnRaw : kBarQnFull);
        mbar_arrive_expect_tx(qb, kQNarrowBytes);
        tma_load_2d(sbase + kOffQn, &p.q_narrow, qb, narrow_x, w.b * a.rows + w.row0);
      }
      last_qn_item = static_cast<int>(n_items);
      for (int blk = w.blk_begin; blk < w.blk_end; ++blk) {
        int rows[4];
        int nbox = 0;
#pragma unroll
        for (int bx = 0; bx < 4; ++bx) {
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
            if (j - batch0 >= 32) {
              batch0 = j;
              const int jj = j + lane;
              my_id = (jj <= last_page && jj < nb) ? ids[jj] : -1;
            }
            const int pid = __shfl_sync(0xffffffffu, my_id, j - batch0);
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
        // Every ring slot is waited for here, in order, for both pool types:
        // a role that skipped slots could run two phases ahead of a slot's
        // barrier, where a parity wait cannot tell the phases apart. For
        // fp8 pools the raw tile lands in the slot's back half and the
        // converters widen it in place.
        const uint32_t stage = sl % kStages, use = sl / kStages;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarKvEmpty + stage), (use & 1u) ^ 1u, abort_flag));
        uint32_t full_bar, dst0;
        if constexpr (kFp8) {
          full_bar = bar(kBarRawFull + stage);
          dst0 = sbase + kOffKV + stage * kStageBytes + kRawOff;
        } else {
          full_bar = bar(kBarKvFull + stage);
          dst0 = sbase + kOffKV + stage * kStageBytes;
        }
        ++sl;
        if (!ok) break;
        if (kFp8) {
          raw_par ^= 1u << stage;
          raw_used |= 1u << stage;
        }
        if (lane == 0) {
          MLA_TRACE_EVENT(trc, 0, kEvSlotAcquired, gt);
          mbar_arrive_expect_tx(full_bar, static_cast<uint32_t>(nbox * rows_per_box) * row_bytes);
#pragma unroll
          for (int bx = 0; bx < 4; ++bx) {
            if (rows[bx] < 0) continue;
            if constexpr (kFp8) {
              tma_load_2d_hint(dst0 + bx * rows_per_box * 256, &p.kv_wide, full_bar, wide_x, rows[bx], kv_policy);
              tma_load_2d_hint(dst0 + kF8WideBytes + bx * rows_per_box * 32, &p.kv_narrow, full_bar, narrow_x,
                               rows[bx], kv_policy);
            } else if (rows_per_box == kTile) {
              // one copy for this rank's four 64-dim chunks, chunk-major as the MMAs read them
              tma_load_3d_hint(dst0, &p.kv_chunks, full_bar, 0, rows[bx], 4 * static_cast<int>(rank), kv_policy);
              tma_load_2d_hint(dst0 + kWideChunks * kWideBytes, &p.kv_narrow, full_bar, narrow_x, rows[bx],
                               kv_policy);
            } else {
              for (int c = 0; c < kWideChunks; ++c)
                tma_load_2d_hint(dst0 + c * kWideBytes + bx * rows_per_box * 128, &p.kv_wide, full_bar,
                                 wide_x + 64 * c, rows[bx], kv_policy);
              tma_load_2d_hint(dst0 + kWideChunks * kWideBytes + bx * rows_per_box * 64, &p.kv_narrow, full_bar,
                               narrow_x, rows[bx], kv_policy);
            }
          }
          MLA_TRACE_EVENT(trc, 0, kEvTileIssued, gt);
        }
        ++gt;
      }
    }
    if (lane == 0) {
      if (!ok) {
        *abort_flag = 1;
        flag_status(status, MLA_STATUS_TIMEOUT);
      }
      if (*abort_flag) {
        // Let every copy already issued land before the CTA can exit (bf16:
        // ring slots complete KvFull; fp8: tiles and q chunks complete
        // RawFull, the last phase of each slot). Each of these waits is itself
        // bounded.
        if (kFp8) {
          for (int st = 0; st < kStages; ++st)
            if (raw_used >> st & 1u) mbar_wait(bar(kBarRawFull + st), ((raw_par >> st) & 1u) ^ 1u, nullptr);
        } else {
          for (uint32_t k = (sl > kStages ? sl - kStages : 0); k < sl; ++k)
            mbar_wait(bar(kBarKvFull + k % kStages), (k / kStages) & 1u, nullptr);
        }
        if (last_qn_item >= 0) mbar_wait(bar(kFp8 ? kBarQnRaw : kBarQnFull), last_qn_item & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issuer
    if constexpr (kFp8) setmaxnreg_dec<C::kRegsIssue>();
    // Per item: once the previous item's QK is complete, copy q into TMEM
    // (tcgen05.cp, wide part 128 columns + rope part 16 columns); per tile:
    // S = q K^T with A read from TMEM (TS form), so shared memory streams
    // only the K tile through the tensor core.
    if (lane == 0) {
      const uint32_t idesc_qk = kIdescQk;
      const uint32_t tQ = tmem + kColQ;
      const uint32_t tS = tmem + kColS;
      uint32_t sl = 0, g = 0, n_items = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it, ++n_items) {
        const WorkItem w = items[it];
        const int nt = w.blk_end - w.blk_begin;
        const uint32_t s0 = sl % kStages, s1 = (sl + 1) % kStages;
        if (!mbar_wait(bar(kBarKvFull + s0), (sl / kStages) & 1u, abort_flag) ||
            !mbar_wait(bar(kBarKvFull + s1), ((sl + 1) / kStages) & 1u, abort_flag) ||
            !mbar_wait(bar(kBarQnFull), n_items & 1u, abort_flag) ||
            !mbar_wait(bar(kBarQDone), (n_items & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kWideChunks; ++c) {
          const uint32_t src = sbase + kOffKV + ((c < 2) ? s0 : s1) * kStageBytes + (c & 1) * kQWideBytes;
#pragma unroll
          for (int k = 0; k < 4; ++k) tmem_cp_128x256b(tQ + 8u * (4 * c + k), sdesc_sw128(src + k * 32, 16, 1024));
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) tmem_cp_128x256b(tQ + 128u + 8u * k, sdesc_sw64(sbase + kOffQn + k * 32, 512));
        mma_commit(bar(kBarKvEmpty + s0));
        mma_commit(bar(kBarKvEmpty + s1));
        mma_commit(bar(kBarQnFree));
        MLA_TRACE_EVENT(trc, 1, kEvQLoaded, g);
        sl += 2;
        for (int t = 0; t < nt; ++t, ++g, ++sl) {
          const uint32_t stage = sl % kStages, use = sl / kStages;
          if (!mbar_wait(bar(kBarKvFull + stage), use & 1u, abort_flag)) { ok = false; break; }
          MLA_TRACE_EVENT(trc, 1, kEvQkTileReady, g);
          if (!mbar_wait(bar(kBarSFree), (g & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          MLA_TRACE_EVENT(trc, 1, kEvQkSFree, g);
          tc_fence_after();
          const uint32_t kv = sbase + kOffKV + stage * kStageBytes;
          // Descriptors of the tile's first chunk; the others differ only in
          // the start address field (bytes / 16).
          const uint64_t dw = sdesc_sw128(kv, 16, 1024);
          const uint64_t dn = sdesc_sw64(kv + kWideChunks * kWideBytes, 512);
#pragma unroll
          for (int c = 0; c < kWideChunks; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16_ts(tS, tQ + 8u * (4 * c + k), dw + static_cast<uint64_t>((c * kWideBytes + k * 32) >> 4),
                          idesc_qk, (c | k) != 0);
#pragma unroll
          for (int k = 0; k < 2; ++k)
            mma_bf16_ts(tS, tQ + 128u + 8u * k, dn + static_cast<uint64_t>((k * 32) >> 4), idesc_qk, 1u);
          mma_commit(bar(kBarSFull));
          MLA_TRACE_EVENT(trc, 1, kEvQkIssued, g);
        }
        if (ok) mma_commit(bar(kBarQDone));  // every QK of this item complete: q may be replaced
      }
      if (!ok) {
        *abort_flag = 1;
        flag_status(status, MLA_STATUS_TIMEOUT);
      }
      mma_commit(bar(kBarDrain));
      mbar_wait(bar(kBarDrain), 0, nullptr);
    }
  } else if (warp == C::kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    if constexpr (kFp8) setmaxnreg_dec<C::kRegsIssue>();
    if (lane == 0) {
      const uint32_t idesc_pv = kIdescPv;
      const uint32_t tO = tmem + kColO;
      uint32_t sl = 0, g = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it) {
        const WorkItem w = items[it];
        const int nt = w.blk_end - w.blk_begin;
        sl += 2;
        for (int t = 0; t < nt; ++t, ++g, ++sl) {
          if (!mbar_wait(bar(kBarOFixed), g & 1u, abort_flag)) { ok = false; break; }
          MLA_TRACE_EVENT(trc, 2, kEvPvOFixed, g);
          tc_fence_after();
          fence_proxy_async_smem();
          const uint64_t dv = sdesc_sw128(sbase + kOffKV + (sl % kStages) * kStageBytes, kWideBytes, 1024);
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_bf16_ts(tO, tmem + kColP + 8u * k, dv + static_cast<uint64_t>((k * 16 * 128) >> 4), idesc_pv,
                        (t | k) != 0);
          mma_commit(bar(kBarKvEmpty + sl % kStages));
          mma_commit(bar(kBarPvDone));
          MLA_TRACE_EVENT(trc, 2, kEvPvIssued, g);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        flag_status(status, MLA_STATUS_TIMEOUT);
      }
      mma_commit(bar(kBarDrainPv));
      mbar_wait(bar(kBarDrainPv), 0, nullptr);
    }
  } else if (kFp8 && warp >= C::kCvtWarp0) {
    // ------------------------------------------------------------ converters (fp8 pools)
    if constexpr (kFp8) setmaxnreg_dec<C::kRegsCvt>();
    // Per item: q's bf16 chunks and rope part become f16 in place. Per tile:
    // the raw e4m3 codes become f16 (exact: every e4m3 value is an f16) in
    // the swizzled layout the tensor core reads, the one TMA writes for bf16
    // pools. kv_scale is applied to the scores and the output instead.
    const int ct = threadIdx.x - 32 * C::kCvtWarp0;  // 0..127
    auto q_to_f16 = [&](uint32_t base, int units) {
      for (int u = ct; u < units; u += 128) {
        uint32_t x[4];
        ld_shared_v4(base + u * 16, x[0], x[1], x[2], x[3]);
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = pack_f16x2(__uint_as_float(x[k] << 16), __uint_as_float(x[k] & 0xffff0000u));
        st_shared_v4(base + u * 16, x[0], x[1], x[2], x[3]);
      }
    };
    uint32_t sl = 0, n_items = 0, n_tiles = 0;
    uint32_t raw_par = 0;  // per slot, parity of its next raw phase (tile or q chunks)
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it, ++n_items) {
      const WorkItem w = items[it];
      for (int h = 0; h < 2; ++h, ++sl) {
        const uint32_t stage = sl % kStages;
        if (!mbar_wait(bar(kBarRawFull + stage), (raw_par >> stage) & 1u, abort_flag)) { ok = false; break; }
        raw_par ^= 1u << stage;
        q_to_f16(sbase + kOffKV + stage * kStageBytes, 2 * kQWideBytes / 16);
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarKvFull + stage));
      }
      if (!ok) break;
      if (!mbar_wait(bar(kBarQnRaw), n_items & 1u, abort_flag)) { ok = false; break; }
      q_to_f16(sbase + kOffQn, kQNarrowBytes / 16);
      fence_proxy_async_smem();
      mbar_arrive(bar(kBarQnFull));
      for (int blk = w.blk_begin; blk < w.blk_end; ++blk, ++sl, ++n_tiles) {
        // The producer waited for this slot's release before the raw copy
        // that completes RawFull was issued.
        const uint32_t stage = sl % kStages;
        if (!mbar_wait(bar(kBarRawFull + stage), (raw_par >> stage) & 1u, abort_flag)) { ok = false; break; }
        raw_par ^= 1u << stage;
        const uint32_t dst = sbase + kOffKV + stage * kStageBytes;
        const uint32_t src = dst + kRawOff;
        // 16 codes per unit: 64 rows x 16 units of c_kv, then 64 rows x 2 of
        // rope; 1152 units, nine per thread (units ct + 128 k: eight of
        // c_kv, one of rope). All nine are loaded first; once every
        // converter holds its codes the slot is overwritten with the
        // widened tile.
        static_assert(kTile * 18 == 9 * 128, "nine 16-code units per converter thread");
        uint32_t x[9][4];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int u = ct + 128 * k, r = u >> 4, c = u & 15;
          ld_shared_v4(src + r * 256 + c * 16, x[k][0], x[k][1], x[k][2], x[k][3]);
        }
        {
          const int r = ct >> 1, c = ct & 1;
          ld_shared_v4(src + kF8WideBytes + r * 32 + c * 16, x[8][0], x[8][1], x[8][2], x[8][3]);
        }
        mbar_arrive(bar(kBarCvtRead));
        if (!mbar_wait(bar(kBarCvtRead), n_tiles & 1u, abort_flag)) { ok = false; break; }
#pragma unroll
        for (int k = 0; k < 9; ++k) {
          uint32_t y[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            y[2 * j] = e4m3x2_to_f16x2(static_cast<uint16_t>(x[k][j] & 0xffffu));
            y[2 * j + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(x[k][j] >> 16));
          }
          if (k < 8) {
            // dims 16c .. 16c+15: 128-byte-swizzled chunk c / 4, 16-byte
            // pieces 2(c % 4) and +1. A warp's 16-byte stores are served
            // eight lanes at a time; lanes of odd chunks store their two
            // pieces in the other order, so that the eight lanes of a phase
            // (two chunks of one row) fill all eight bank groups.
            const int u = ct + 128 * k, r = u >> 4, c = u & 15;
            const uint32_t row_base = dst + (c >> 2) * kWideBytes + r * 128;
            const int odd = (c >> 2) & 1;
            const int pa = (c & 3) * 2 + odd, pb = pa ^ 1;
            st_shared_v4(row_base + ((pa ^ (r & 7)) << 4), odd ? y[4] : y[0], odd ? y[5] : y[1], odd ? y[6] : y[2],
                         odd ? y[7] : y[3]);
            st_shared_v4(row_base + ((pb ^ (r & 7)) << 4), odd ? y[0] : y[4], odd ? y[1] : y[5], odd ? y[2] : y[6],
                         odd ? y[3] : y[7]);
          } else {
            // rope dims 16c .. 16c+15: 64-byte-swizzled rows, pieces 2c and 2c+1
            const int r = ct >> 1, c = ct & 1;
            const uint32_t row_base = dst + kWideChunks * kWideBytes + r * 64;
            const int sw = (r >> 1) & 3;
            st_shared_v4(row_base + (((2 * c) ^ sw) << 4), y[0], y[1], y[2], y[3]);
            st_shared_v4(row_base + (((2 * c + 1) ^ sw) << 4), y[4], y[5], y[6], y[7]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarKvFull + stage));
      }
    }
    if (!ok) {
      *abort_flag = 1;
      flag_status(status, MLA_STATUS_TIMEOUT);
    }
  } else if (warp >= C::kSmWarp0 && warp < C::kSmWarp0 + 8) {
    // ------------------------------------------------------------ exchange, softmax, correction, epilogue
    if constexpr (kFp8) setmaxnreg_inc<C::kRegsSoftmax>();
    // Warp w works on 16 rows (heads) of TMEM lane quarter q4 = w & 3: the
    // first four softmax warps on its lanes 0-15, the next four on 16-31. A
    // row belongs to two threads: t and t + 16 hold its tokens [0, 32) and
    // [32, 64) of every tile (and value dims [0, 128) and [128, 256) of this
    // rank's O), so the row max and sum need one shuffle and no other warp.
    // Per tile g: this rank's partial scores, scaled to log2 units and
    // rounded to fp16, go to the peer (st.async) and the peer's arrive the
    // same way; both ranks form the same sum f16(S_0) + f16(S_1) in fp32
    // (addition commutes), run the same online softmax and keep the same P
    // in their own TMEM.
    const int q4 = warp & 3;
    const int half = (warp - C::kSmWarp0) >> 2;     // lane half of the quarter
    const int th = lane >> 4;                       // token half of a tile / value-dim half
    const int row = 32 * q4 + 16 * half + (lane & 15);
    // rows of a row group in use (heads, or query positions x heads)
    const int nrow = min(max(a.group_rows - 32 * q4 - 16 * half, 0), 16);  // valid rows of this warp
    const bool valid = (lane & 15) < nrow;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4 + 16 * half) << 16;
    const uint32_t tO = tmem + lane_base + kColO;   // this warp's 16 rows of O
    const uint32_t dim0 = 256u * rank + 128u * th;  // first value dim of this thread
    constexpr int kHalf = kTile / 2;
    const bool tracer = lane == 0 && (warp == C::kSmWarp0 || warp == C::kSmWarp0 + 7);
    auto tr = [&](uint32_t ev, uint32_t t) {
      if (tracer) MLA_TRACE_EVENT(trc, warp == C::kSmWarp0 ? 3 : 4, ev, t);
    };
    auto wwait = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, abort_flag));
    };
    auto wwait_cluster = [&](uint32_t b, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait<true>(b, parity, abort_flag));
    };
    // X[b]: the peer's partial rows; per warp 16 rows x 64 tokens as 16-byte
    // pieces, piece-major (lane-contiguous): piece j of thread t holds
    // tokens 32 th + 8 j .. + 8 of row t & 15.
    auto xq = [&](uint32_t b) { return sbase + kOffX + b * kXBytes + q4 * (32 * kTile * 2) + half * (16 * kTile * 2); };
    auto xfull = [&](uint32_t b) { return bar(kBarXFull + 8 * b + 2 * q4 + half); };
    auto xfree = [&](uint32_t b) { return bar(kBarXFree + 8 * b + 2 * q4 + half); };
    // The peer's copies of this warp's exchange buffers and barriers.
    const uint32_t peer_xq0 = mapa(xq(0), peer), peer_xq1 = mapa(xq(1), peer);
    const uint32_t peer_xfull0 = mapa(xfull(0), peer), peer_xfull1 = mapa(xfull(1), peer);
    const uint32_t peer_xfree0 = mapa(xfree(0), peer), peer_xfree1 = mapa(xfree(1), peer);
    // Epilogue of an item: wait for its last PV, normalise this thread's
    // 128 value dims, store. TMEM is read several 16-column chunks per wait.
    // A row with no attended token in an item (a query position whose range
    // ends before a split item of a later one) has l = 0: its partial is 0
    // with lse = -inf, which the merge weighs 0.
    auto store_item = [&](const WorkItem& w, uint32_t g_last, float m, float l) -> bool {
      tr(kEvSmItemStore, g_last);
      if (!wwait(bar(kBarPvDone), g_last & 1u)) return false;
      tc_fence_after();
      const bool keep = valid && w.row0 + row < a.rows;  // rows past the request's last row are not stored
      const size_t out_row = static_cast<size_t>(w.b) * a.rows + w.row0 + row;
      const size_t part_row = static_cast<size_t>(w.slot) * a.group_rows + row;
      if (rank == 0 && th == 0 && keep) {
        const float lse2 = l > 0.f ? m + log2f(l) : -CUDART_INF_F;
        if (w.slot < 0) {
          if (a.lse) a.lse[out_row] = lse2 * 0.69314718055994531f;
        } else {
          reinterpret_cast<float*>(ws + a.lay.partial_lse)[part_row] = lse2;
        }
      }
      if (nrow > 0) {
        const float inv_l = keep && l > 0.f ? a.out_scale / l : 0.f;  // out_scale: kv_scale for fp8 pools
        constexpr int kBatch = kFp8 ? 2 : 4;  // 16-column chunks per TMEM wait (registers)
#pragma unroll 1
        for (int c0 = 0; c0 < 128 / 16; c0 += kBatch) {
          uint32_t o[kBatch][16];
#pragma unroll
          for (int c = 0; c < kBatch; ++c) tmem_ld_h16<128>(tO + (c0 + c) * 16, o[c]);
          tmem_wait_ld();
          if (keep) {
#pragma unroll
            for (int c = 0; c < kBatch; ++c) {
              // Whole 32-byte sectors per store (16 bf16 or 8 fp32 dims).
              if (w.slot < 0) {
                __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + out_row * kDimCkv + dim0 + (c0 + c) * 16;
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  pk[i] = pack_bf16x2(__uint_as_float(o[c][2 * i]) * inv_l, __uint_as_float(o[c][2 * i + 1]) * inv_l);
                st_global_v8(dst, pk);
              } else {
                float* dst = reinterpret_cast<float*>(ws + a.lay.partial_o) + part_row * kDimCkv + dim0 + (c0 + c) * 16;
#pragma unroll
                for (int i = 0; i < 16; ++i) o[c][i] = __float_as_uint(__uint_as_float(o[c][i]) * inv_l);
                st_global_v8(dst, o[c]);
                st_global_v8(dst + 8, o[c] + 8);
              }
            }
          }
        }
      }
      tc_fence_before();
      tr(kEvSmItemStored, g_last);
      return true;
    };
    // Software pipeline: the partial scores of tile g+1 are fetched from TMEM
    // and shipped before the softmax of tile g, so the transfer to the peer
    // overlaps the exponentials instead of sitting in this loop.
    int total_tiles = 0;
    for (int it = it_begin; it < it_end; ++it) total_tiles += items[it].blk_end - items[it].blk_begin;
    // Wait for S(gg), keep this rank's partial (this thread's 32 tokens,
    // log2 units) as fp16 pairs in xp, release S, and send the pairs to the
    // peer once it has read that buffer's previous contents.
    auto fetch = [&](uint32_t gg, uint32_t* xp) -> bool {
      const uint32_t b = gg & 1u, u = gg >> 1;
      if (!wwait(bar(kBarSFull), gg & 1u)) return false;
      tr(kEvSmSFull, gg);
      tc_fence_after();
      if (nrow > 0) {
        uint32_t r[kHalf];
        tmem_ld_h16<kHalf>(tmem + lane_base + kColS, r);
        tmem_ld_h16<kHalf>(tmem + lane_base + kColS + 16, r + 16);
        tmem_wait_ld();
        const uint64_t sc2 = f2_make(a.scale_log2, a.scale_log2);
#pragma unroll
        for (int i = 0; i < kHalf / 2; ++i) {
          float s0, s1;
          f2_split(f2_mul(f2_make(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc2), s0, s1);
          xp[i] = pack_f16x2(s0, s1);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarSFree));
      if (nrow > 0) {
        if (!wwait(xfree(b), (u & 1u) ^ 1u)) return false;
        if (valid) {
          const uint32_t dst = b ? peer_xq1 : peer_xq0;
          const uint32_t fb = b ? peer_xfull1 : peer_xfull0;
#pragma unroll
          for (int j = 0; j < kHalf / 8; ++j)
            st_async_v4(dst + (j * 32 + lane) * 16, xp[4 * j], xp[4 * j + 1], xp[4 * j + 2], xp[4 * j + 3], fb);
        }
        if (lane == 0) mbar_arrive_expect_tx(xfull(b), static_cast<uint32_t>(2 * nrow * kHalf * 2));
      }
      tr(kEvSmSent, gg);
      return true;
    };
    // Fetching S(g+1) needs its ring slot, whose previous tile must have
    // finished PV. Across an item boundary (two q slots in between) that
    // tile is g itself unless the ring has at least 4 stages: there the
    // first tile of the next item is fetched in its own iteration.
    constexpr bool kEarlyAcrossItems = kStages >= 4;
    uint32_t g = 0, sl = 0;
    bool ok = true;
    uint32_t xp[kHalf / 2];
    bool have = false;  // xp holds this thread's partial of tile g
    if (total_tiles > 0) {
      ok = fetch(0, xp);
      have = true;
    }
    for (int it = it_begin; it < it_end && ok; ++it) {
      const WorkItem w = items[it];
      // Positions of the item: [lo, hi) for all of its rows; this row (query
      // position qi) attends [lo_r, hi_r) of them: positions up to L + qi.
      const int lo = max(w.blk_begin * kTile, w.tok_lo);
      const int hi = min(w.blk_end * kTile, w.tok_hi);
      const int qi = (w.row0 + row) / H;
      const int row_end = w.tok_hi - (a.q_len - 1 - qi);
      const int hi_r = min(hi, row_end);
      const int lo_r = a.window > 0 ? max(lo, row_end - a.window) : lo;
      float m = -CUDART_INF_F, l = 0.f;  // l: this thread's tokens only
      sl += 2;  // the item's q slots
      for (int blk = w.blk_begin; blk < w.blk_end; ++blk, ++g, ++sl) {
        const int base = blk * kTile + kHalf * th;  // first token of this thread
        const uint32_t b = g & 1u, u = g >> 1;
        const bool first_tile = blk == w.blk_begin;
        if (!have && !fetch(g, xp)) { ok = false; break; }
        uint32_t xp_next[kHalf / 2];
        const bool have_next =
            static_cast<int>(g) + 1 < total_tiles && (kEarlyAcrossItems || blk + 1 < w.blk_end);
        if (have_next && !fetch(g + 1, xp_next)) { ok = false; break; }
        float alpha = 1.f;
        uint32_t pk[kHalf / 2];
        if (nrow > 0) {
          if (!wwait_cluster(xfull(b), u & 1u)) { ok = false; break; }
          tr(kEvSmXFull, g);
          // Scores as packed fp32 pairs (tokens 2i, 2i+1): both ranks add the
          // same two fp16 partials.
          uint64_t s2[kHalf / 2];
          float mxa = -CUDART_INF_F, mxb = -CUDART_INF_F;
          if (valid) {
#pragma unroll
            for (int j = 0; j < kHalf / 8; ++j) {
              uint32_t x[4];
              ld_shared_v4(xq(b) + (j * 32 + lane) * 16, x[0], x[1], x[2], x[3]);
#pragma unroll
              for (int k = 0; k < 4; ++k) s2[4 * j + k] = f2_sum_f16x2(xp[4 * j + k], x[k]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_remote_relaxed(b ? peer_xfree1 : peer_xfree0);  // X[b] read
          if (valid) {
            if (lo_r > base || hi_r < base + kHalf) {
#pragma unroll
              for (int i = 0; i < kHalf / 2; ++i) {
                float s0, s1;
                f2_split(s2[i], s0, s1);
                const int pos = base + 2 * i;
                if (pos < lo_r || pos >= hi_r) s0 = -CUDART_INF_F;
                if (pos + 1 < lo_r || pos + 1 >= hi_r) s1 = -CUDART_INF_F;
                s2[i] = f2_make(s0, s1);
              }
            }
#pragma unroll
            for (int i = 0; i < kHalf / 2; i += 2) {
              float s0, s1, s2_, s3_;
              f2_split(s2[i], s0, s1);
              f2_split(s2[i + 1], s2_, s3_);
              mxa = fmax3(mxa, s0, s1);
              mxb = fmax3(mxb, s2_, s3_);
            }
          }
          // The row max over both token halves (the partials were scaled to
          // log2 units before the exchange).
          float mx = fmaxf(mxa, mxb);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          if (valid) {
            if (mx > m + kRescaleThreshold) {
              alpha = fast_exp2(m - mx);  // 0 on the first tile (m = -inf)
              l *= alpha;
              m = mx;
            }
            // (a row that has seen no attended token yet keeps m = -inf; its
            // masked scores then give P = 0, not 2^(-inf + inf))
            const float m_use = m == -CUDART_INF_F ? 0.f : m;
            const uint64_t nm2 = f2_make(-m_use, -m_use);
            uint64_t rs2[2] = {f2_make(0.f, 0.f), f2_make(0.f, 0.f)};
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) {
              float t0, t1;
              f2_split(f2_add(s2[i], nm2), t0, t1);
              const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
              rs2[i & 1] = f2_add(rs2[i & 1], f2_make(p0, p1));
              pk[i] = kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
            float r0, r1, r2, r3;
            f2_split(rs2[0], r0, r1);
            f2_split(rs2[1], r2, r3);
            l += (r0 + r1) + (r2 + r3);
            tr(kEvSmComputed, g);
          } else {
#pragma unroll
            for (int i = 0; i < kHalf / 2; ++i) pk[i] = 0;
          }
        }
#pragma unroll
        for (int i = 0; i < kHalf / 2; ++i) xp[i] = xp_next[i];
        have = have_next;
        // Value rows of this tile outside [lo, hi) may hold anything (stale
        // or unwritten slots): zero this rank's value dims there so that
        // 0 * garbage cannot reach O. QK of the tile is complete here.
        const int tbase = blk * kTile;
        if (lo > tbase || hi < tbase + kTile) {
          const uint32_t v0 = sbase + kOffKV + (sl % kStages) * kStageBytes;
          for (int e = threadIdx.x - 32 * C::kSmWarp0; e < kTile * kWideChunks * 8; e += 256) {
            const int rr = e >> 5, c = (e >> 3) & 3, piece = e & 7;
            const int pos = tbase + rr;
            if (pos < lo || pos >= hi) st_shared_v4(v0 + c * kWideBytes + rr * 128 + piece * 16, 0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        // TMEM P and O are free once PV(g-1) is done. Waiting here also keeps
        // a warp without heads from arriving twice in one phase of OFixed.
        if (!wwait(bar(kBarPvDone), (g & 1u) ^ 1u)) { ok = false; break; }
        tr(kEvSmPvDone, g);
        tc_fence_after();
        if (nrow > 0) {
          tmem_st_h16<kHalf / 2>(tmem + lane_base + kColP, pk);
          // Rescale this thread's half of the row's O before PV(g) when the
          // max moved (both threads of a row see the same alpha).
          if (!first_tile && __any_sync(0xffffffffu, valid && alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < 128 / 16; ++c) {
              uint32_t o[16];
              tmem_ld_h16<128>(tO + c * 16, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st_h16<128>(tO + c * 16, o);
            }
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(bar(kBarOFixed));
        tr(kEvSmOFixed, g);
      }
      if (!ok) break;
      // The row sum over both token halves.
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (!store_item(w, g - 1, m, l)) { ok = false; break; }
    }
    if (!ok) {
      *abort_flag = 1;
      flag_status(status, MLA_STATUS_TIMEOUT);
    }
  } else if (kFp8) {
    // fp8 pools: warp 3 has no role; it releases its registers with the rest
    // of its warpgroup.
    setmaxnreg_dec<C::kRegsIssue>();
  }

  if (threadIdx.x == 0) MLA_TRACE_EVENT(trc5, 5, kEvKernelEnd, 0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) MLA_TRACE_EVENT(trc5, 5, kEvGlobalEnd, 0);
  pdl_launch_dependents();  // the merge may be scheduled as CTAs finish
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();  // the peer may still address this CTA's shared memory
  if (threadIdx.x == 0) MLA_TRACE_EVENT(trc5, 5, kEvGlobalExit, 0);
}

template <bool kFp8>
int max_active_clusters_of() {
  using C = Cfg<kFp8>;
  if (cudaFuncSetAttribute(mla_decode_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
      cudaSuccess)
    return -1;
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
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<kFp8>, &cfg) != cudaSuccess || n <= 0) return -1;
  return n;
}

template <bool kFp8>
cudaError_t launch_variant(const CUtensorMap* maps, const DecodeArgs& a, int clusters, cudaStream_t stream) {
  using C = Cfg<kFp8>;
  static bool attr_set[kMaxDevices] = {};
  const cudaError_t e = set_smem_once(mla_decode_kernel<kFp8>, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  Params p;
  p.kv_wide = maps[0];
  p.kv_narrow = maps[1];
  p.q_wide = maps[2];
  p.q_narrow = maps[3];
  p.kv_chunks = maps[4];
  p.a = a;
  return launch_pdl(mla_decode_kernel<kFp8>, dim3(2 * clusters), dim3(C::kThreads), C::kSmemBytes, stream, p);
}

}  // namespace

// Co-resident clusters on the current device: the smaller of the two
// variants' counts, so that one plan serves either pool type (cached per
// device).
int decode_max_active_clusters() {
  static int cached[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return -1;
  if (cached[dev] > 0) return cached[dev];
  const int a = max_active_clusters_of<false>(), b = max_active_clusters_of<true>();
  if (a <= 0 || b <= 0) return -1;
  cached[dev] = a < b ? a : b;
  return cached[dev];
}

cudaError_t launch_decode(const CUtensorMap* maps, const DecodeArgs& a, int clusters, cudaStream_t stream) {
  return a.dtype == MLA_DTYPE_FP8_E4M3 ? launch_variant<true>(maps, a, clusters, stream)
                                       : launch_variant<false>(maps, a, clusters, stream);
}

}  // namespace mla

#ifdef MLA_TRACE
// Copies the trace buffer to the host ([ctas][roles][cap] records and
// [ctas][roles] counts) and clears the counts. Traced builds only.
extern "C" int mla_trace_read(void* records, void* counts) {
  if (cudaMemcpyFromSymbol(records, mla::g_trace, sizeof(mla::g_trace)) != cudaSuccess) return -4;
  if (cudaMemcpyFromSymbol(counts, mla::g_trace_n, sizeof(mla::g_trace_n)) != cudaSuccess) return -4;
  static uint32_t zero[mla::kTraceCtas][mla::kTraceRoles] = {};
  if (cudaMemcpyToSymbol(mla::g_trace_n, zero, sizeof(zero)) != cudaSuccess) return -4;
  return 0;
}
#endif
