// Split-KV schedule and partial-result merge.
//
// The plan runs on the device so that it can be captured with the decode
// and so that a replay reads exactly the buffer the last plan filled (the
// plan/run contract described in SGLang PR #32972 "Let Kimi-Linear use the
// paged MLA attention backends", Correction). It reads only the lengths:
// request b attends positions [s_b, L_b] (s_b = 0, or max(0, L_b + 1 - W)
// for a sliding window, FastDeploy PR #8049 "Support MLA_SWA
// functionality"), i.e. 64-token blocks s_b/64 .. L_b/64. The blocks of all
// requests, concatenated in request order, are cut into C equal contiguous
// ranges, one per cluster; a request crossing a range boundary becomes
// several items whose partial (O, lse) are merged afterwards. Batches of up
// to 1024 requests also get a packed schedule (only requests heavier than a
// cluster's share are split; pieces dealt largest-first) and keep whichever
// has the lower estimated cost. With several
// query positions per request (q_len > 1) request b attends [s_b, L_b +
// q_len - 1] over all its queries, and each of its row groups is scheduled
// like a request of its own (virtual request v = b * groups + group).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kPlanThreads = 1024;
// A work item costs about this many 64-token blocks beyond its blocks (its
// epilogue and the pipeline refill when the next item starts: in an event
// trace of the V3-shaped workload, clusters with one more item ended 4-5
// blocks' time later): small batches count it in the balance, so clusters
// that start more requests get fewer blocks.
constexpr int kItemCostBlocks = 4;
// Pieces (and clusters) the packed schedule handles in shared memory.
constexpr int kPackMax = 256;

// Block-wide exclusive scan of one int per thread; returns the prefix and
// writes the block total to *total. The plan runs once per step on one CTA
// whose time goes mostly to latency, so its helpers are called, not inlined:
// one copy of their code serves every call.
__device__ __noinline__ int block_excl_scan(int v, int* total, int* smem32) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem32[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? smem32[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    smem32[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int warp_prefix = warp ? smem32[warp - 1] : 0;
  *total = smem32[31];
  __syncthreads();
  return warp_prefix + x - v;
}

// The same for three counts at once, 21 bits each (every count and every sum
// stays below 2^21): one pass of 64-bit shuffles instead of three passes.
__device__ __noinline__ unsigned long long block_excl_scan3(unsigned long long v, unsigned long long* total,
                                               unsigned long long* smem64) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem64[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = lane < nwarps ? smem64[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    smem64[lane] = w;
  }
  __syncthreads();
  const unsigned long long warp_prefix = warp ? smem64[warp - 1] : 0;
  *total = smem64[31];
  __syncthreads();
  return warp_prefix + x - v;
}
constexpr unsigned long long kField = (1ull << 21) - 1;
// items, partial slots (items of a split request) and split requests
__device__ __forceinline__ unsigned long long counts3(int items) {
  const unsigned long long k = static_cast<unsigned>(items);
  return items > 1 ? k | (k << 21) | (1ull << 42) : k;
}

// The products below stay under 2^32 whenever T * C does (T blocks, C <= 1024
// clusters), which is then divided in 32 bits; 64-bit division is a long
// software routine.
__device__ __forceinline__ long long range_lo(long long c, long long T, long long C) {
  if (T * C < (1ll << 32)) return static_cast<unsigned>(c * T) / static_cast<unsigned>(C);
  return c * T / C;
}

// Cluster whose range [lo(c), lo(c+1)) holds block x (requires T >= C).
__device__ __forceinline__ int cluster_of(long long x, long long T, long long C) {
  if (T * C + T < (1ll << 32))
    return static_cast<int>((static_cast<unsigned>((x + 1) * C + T - 1)) / static_cast<unsigned>(T)) - 1;
  return static_cast<int>(((x + 1) * C + T - 1) / T - 1);
}

__global__ void __launch_bounds__(kPlanThreads)
    plan_kernel(const int32_t* __restrict__ lens, int B, int q_len, int G, int H, int ps, int window, int C_req,
                uint8_t* __restrict__ ws, WsLayout lay) {
  __shared__ int smem32[32];
  __shared__ int bad_len;
  WsHeader* hd = reinterpret_cast<WsHeader*>(ws);
  int* req = reinterpret_cast<int*>(ws + lay.req_scratch);  // [V][4]: first_blk, n_blk, off, start
  WorkItem* items = reinterpret_cast<WorkItem*>(ws + lay.items);
  int* cstart = reinterpret_cast<int*>(ws + lay.cluster_start);
  SplitRequest* split = reinterpret_cast<SplitRequest*>(ws + lay.split);
  const int tid = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  if (tid == 0) bad_len = 0;
  __syncthreads();
  const int V = B * G;  // scheduled (request, row group) pairs
  // Attended positions of request b over all its queries, [s, L + q_len).
  auto range_of = [&](int b, int& L, int& s, int& first, int& n) {
    L = lens[b];
    if (L < 0) {
      bad_len = 1;
      L = 0;
    }
    s = window > 0 ? max(0, L + 1 - window) : 0;
    first = s / kBlockTokens;
    n = (L + q_len - 1) / kBlockTokens - first + 1;
  };

  if (V <= static_cast<int>(blockDim.x)) {
    // One request per thread, everything in registers or shared memory: no
    // pass through global memory between the scans. Two schedules are
    // formed and the cheaper one is written:
    //  - cut: request b weighs its n_b blocks plus kItemCostBlocks; the
    //    weights are concatenated in request order and cut into C equal
    //    ranges (a request's blocks sit after its extra weight), so nearly
    //    every range boundary splits a request;
    //  - packed: a request heavier than a cluster's share of the weight is
    //    split into that many near-equal pieces, the pieces are ranked by
    //    size (largest first) and dealt in two rounds: rank r < C to
    //    cluster r, rank C + j to cluster C - 1 - j, the least loaded after
    //    the first round. Only the split requests leave partials.
    // Cost of a schedule, in sixteenths of a block: 16 x its largest cluster
    // load (blocks plus kItemCostBlocks per item) plus, per partial, its
    // rows / 128: writing a 128-row fp32 partial and reading it back in the
    // merge takes about a sixteenth of a block's time over the whole GPU.
    __shared__ int last_cluster[kPlanThreads];
    __shared__ unsigned long long smem64[32];
    __shared__ __align__(16) int piece_size[kPackMax + 4];
    __shared__ int piece_rank[kPackMax];
    __shared__ int by_rank[kPackMax];
    __shared__ int max_load_packed;
    if (tid == 0) max_load_packed = 0;  // published by the scans' barriers
    int L = 0, s = 0, first = 0, n = 0;
    const int vb = tid / G, vg = tid - (tid / G) * G;  // request and row group of this thread
    if (tid < V) range_of(vb, L, s, first, n);
    int T32;
    const int off = block_excl_scan(tid < V ? n + kItemCostBlocks : 0, &T32, smem32) + kItemCostBlocks;
    const long long T = T32;
    const long long C = T > 0 ? (T < C_req ? T : C_req) : 1;
    const int Ci = static_cast<int>(C);
    int cf = 0, cl = -1, ns = 0;
    if (tid < V) {
      cf = cluster_of(off, T, C);
      cl = cluster_of(static_cast<long long>(off) + n - 1, T, C);
      ns = cl - cf + 1;
    }
    last_cluster[tid] = cl;
    auto cut_range = [&](int k, long long& lo, long long& hi) {
      const int c = cf + k;
      lo = max(static_cast<long long>(off), range_lo(c, T, C));
      hi = min(static_cast<long long>(off) + n, range_lo(c + 1, T, C));
    };
    // Pieces of this request in the packed schedule: its weight over a
    // cluster's share, rounded up (at most one per block).
    int kv = 0;
    if (tid < V) {
      const long long num = static_cast<long long>(n + kItemCostBlocks) * C + T - 1;
      kv = num < (1ll << 32) ? static_cast<int>(static_cast<unsigned>(num) / static_cast<unsigned>(T))
                             : static_cast<int>(num / T);
      kv = min(max(kv, 1), n);
    }
    // Items, partial slots and split requests of both schedules: prefixes
    // (this request's first of each) and totals.
    unsigned long long tot_cut, tot_pk;
    const unsigned long long ex_cut = block_excl_scan3(counts3(ns), &tot_cut, smem64);
    const unsigned long long ex_pk = block_excl_scan3(counts3(kv), &tot_pk, smem64);
    const int item0 = static_cast<int>(ex_cut & kField), part0 = static_cast<int>((ex_cut >> 21) & kField),
              split0 = static_cast<int>(ex_cut >> 42);
    const int t_items = static_cast<int>(tot_cut & kField), t_part = static_cast<int>((tot_cut >> 21) & kField),
              t_split = static_cast<int>(tot_cut >> 42);
    const int pitem0 = static_cast<int>(ex_pk & kField), ppart0 = static_cast<int>((ex_pk >> 21) & kField),
              psplit0 = static_cast<int>(ex_pk >> 42);
    const int p_items = static_cast<int>(tot_pk & kField), p_part = static_cast<int>((tot_pk >> 21) & kField),
              p_split = static_cast<int>(tot_pk >> 42);
    // The packed schedule is formed only where it can pay: it fits (at most
    // two pieces per cluster) and the partials it saves are worth at least
    // half a block. The cut's largest load is its share rounded up plus one
    // item cost (a cluster starts inside one request).
    const long long rows = min(q_len * H, kGroupRows);
    bool packed = false;
    if (V > 0 && Ci <= kPackMax && p_items <= 2 * Ci && p_items <= kPackMax &&
        ((t_part - p_part) * rows >> 7) >= 8) {  // the same for every thread
      if (tid < V) {
        const int base = n / kv, rem = n - base * kv;
        for (int i = 0; i < kv; ++i) piece_size[pitem0 + i] = base + (i < rem ? 1 : 0);
      }
      if (tid < 3) piece_size[p_items + tid] = -1;  // pad to whole int4 (sizes are >= 1)
      __syncthreads();
      // Rank of each piece (larger first, then by index); sizes by rank.
      // Sizes are read four at a time and counted in two chains.
      for (int p = tid; p < p_items; p += blockDim.x) {
        const int sz = piece_size[p];
        int ra = 0, rb = 0;
        const int4* ps4 = reinterpret_cast<const int4*>(piece_size);
#pragma unroll 1
        for (int q4 = 0; q4 < (p_items + 3) >> 2; ++q4) {
          const int4 v = ps4[q4];
          const int q = 4 * q4;
          ra += (v.x > sz || (v.x == sz && q < p)) ? 1 : 0;
          rb += (v.y > sz || (v.y == sz && q + 1 < p)) ? 1 : 0;
          ra += (v.z > sz || (v.z == sz && q + 2 < p)) ? 1 : 0;
          rb += (v.w > sz || (v.w == sz && q + 3 < p)) ? 1 : 0;
        }
        const int rank = ra + rb;
        piece_rank[p] = rank;
        by_rank[rank] = sz;
      }
      __syncthreads();
      // Cluster c holds rank c and, for the last p_items - C clusters, rank
      // 2C - 1 - c.
      int mx = 0;
      for (int c = tid; c < min(p_items, Ci); c += blockDim.x) {
        const int r2 = 2 * Ci - 1 - c;
        mx = max(mx, by_rank[c] + kItemCostBlocks + (r2 < p_items ? by_rank[r2] + kItemCostBlocks : 0));
      }
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if ((tid & 31) == 0) atomicMax(&max_load_packed, mx);
      __syncthreads();
      const long long share = (T + C - 1) / C;
      const long long cost_cut = 16ll * (share + kItemCostBlocks) + ((t_part * rows) >> 7);
      const long long cost_packed = 16ll * max_load_packed + ((p_part * rows) >> 7);
      packed = cost_packed < cost_cut;
      if (packed) {
        // Cluster c holds its first-round piece, then its second-round one
        // (the last n2 clusters have one).
        const int n1 = min(p_items, Ci), n2 = p_items - n1;
        auto first_item = [&](int cc) { return min(cc, n1) + max(0, cc - (Ci - n2)); };
        if (tid < V) {
          const int base = n / kv, rem = n - base * kv;
          int b0 = first;
          for (int i = 0; i < kv; ++i) {
            const int size = base + (i < rem ? 1 : 0);
            const int rank = piece_rank[pitem0 + i];
            WorkItem w;
            w.b = vb;
            w.blk_begin = b0;
            w.blk_end = b0 + size;
            w.slot = kv > 1 ? ppart0 + i : -1;
            w.tok_lo = s;
            w.tok_hi = L + q_len;
            w.cluster = rank < Ci ? rank : 2 * Ci - 1 - rank;
            w.row0 = vg * kGroupRows;
            items[first_item(w.cluster) + (rank < Ci ? 0 : 1)] = w;
            b0 += size;
          }
          if (kv > 1) {
            SplitRequest r;
            r.b = vb;
            r.num_splits = kv;
            r.first_partial = ppart0;
            r.row0 = vg * kGroupRows;
            split[psplit0] = r;
          }
        }
        for (int cc = tid; cc <= C_req; cc += blockDim.x) cstart[cc] = cc <= Ci ? first_item(cc) : p_items;
      }
    }
    if (!packed) {
      if (tid < V) {
        for (int k = 0; k < ns; ++k) {
          long long lo, hi;
          cut_range(k, lo, hi);
          WorkItem w;
          w.b = vb;
          w.blk_begin = first + static_cast<int>(lo - off);
          w.blk_end = first + static_cast<int>(hi - off);
          w.slot = ns > 1 ? part0 + k : -1;
          w.tok_lo = s;
          w.tok_hi = L + q_len;
          w.cluster = cf + k;
          w.row0 = vg * kGroupRows;
          items[item0 + k] = w;
        }
        if (ns > 1) {
          SplitRequest r;
          r.b = vb;
          r.num_splits = ns;
          r.first_partial = part0;
          r.row0 = vg * kGroupRows;
          split[split0] = r;
        }
        // First item of each cluster after the previous request's last one
        // (clusters whose range holds no block of any request get an empty
        // range at this request's first item).
        const int prev = tid > 0 ? last_cluster[tid - 1] : -1;
        for (int c = prev + 1; c <= cl; ++c) cstart[c] = item0 + (c > cf ? c - cf : 0);
      }
      const int cl_last = V > 0 ? last_cluster[V - 1] : -1;
      for (int c = cl_last + 1 + tid; c <= C_req; c += blockDim.x) cstart[c] = t_items;
    }
    __syncthreads();
    if (tid == 0) {
      if (bad_len) atomicOr(&hd->status, MLA_STATUS_BAD_LENGTH);
      hd->batch = B;
      hd->num_heads = H;
      hd->q_len = q_len;
      hd->page_size = ps;
      hd->window = window;
      hd->num_clusters = Ci;
      hd->total_blocks = static_cast<int>(T);
      hd->num_items = packed ? p_items : t_items;
      hd->num_partials = packed ? p_part : t_part;
      hd->num_split = packed ? p_split : t_split;
      hd->schedule = packed ? kSchedulePacked : kScheduleCut;
      hd->planned = 1;
    }
    return;
  }

  // Larger batches: pass 1, blocks per request and their offsets in the
  // concatenated order.
  long long T = 0;
  for (int base = 0; base < V; base += kPlanThreads) {
    const int i = base + tid;
    int n = 0;
    if (i < V) {
      int L, s, first;
      range_of(i / G, L, s, first, n);
      req[4 * i + 0] = first;
      req[4 * i + 1] = n;
      req[4 * i + 3] = s;
    }
    int chunk_total;
    const int ex = block_excl_scan(n, &chunk_total, smem32);
    if (i < V) req[4 * i + 2] = static_cast<int>(T) + ex;
    T += chunk_total;
  }
  __syncthreads();
  const long long C = T > 0 ? (T < C_req ? T : C_req) : 1;

  // Pass 2: one item per (request, cluster range it meets), in request order,
  // which is also cluster order.
  int n_items = 0, n_part = 0, n_split = 0;
  for (int base = 0; base < V; base += kPlanThreads) {
    const int i = base + tid;
    int ns = 0, first = 0, n = 0, off = 0, s = 0, cf = 0;
    if (i < V) {
      first = req[4 * i + 0];
      n = req[4 * i + 1];
      off = req[4 * i + 2];
      s = req[4 * i + 3];
      cf = cluster_of(off, T, C);
      const int cl = cluster_of(static_cast<long long>(off) + n - 1, T, C);
      ns = cl - cf + 1;
    }
    int t_items, t_part, t_split;
    const int ex_items = block_excl_scan(ns, &t_items, smem32);
    const int ex_part = block_excl_scan(ns > 1 ? ns : 0, &t_part, smem32);
    const int ex_split = block_excl_scan(ns > 1 ? 1 : 0, &t_split, smem32);
    if (i < V) {
      const int rb = i / G, rg = i - (i / G) * G;
      int L = lens[rb];
      if (L < 0) L = 0;
      const int item0 = n_items + ex_items;
      const int part0 = n_part + ex_part;
      for (int k = 0; k < ns; ++k) {
        const int c = cf + k;
        const long long lo = max(static_cast<long long>(off), range_lo(c, T, C));
        const long long hi = min(static_cast<long long>(off) + n, range_lo(c + 1, T, C));
        WorkItem w;
        w.b = rb;
        w.blk_begin = first + static_cast<int>(lo - off);
        w.blk_end = first + static_cast<int>(hi - off);
        w.slot = ns > 1 ? part0 + k : -1;
        w.tok_lo = s;
        w.tok_hi = L + q_len;
        w.cluster = c;
        w.row0 = rg * kGroupRows;
        items[item0 + k] = w;
      }
      if (ns > 1) {
        SplitRequest r;
        r.b = rb;
        r.num_splits = ns;
        r.first_partial = part0;
        r.row0 = rg * kGroupRows;
        split[n_split + ex_split] = r;
      }
    }
    n_items += t_items;
    n_part += t_part;
    n_split += t_split;
  }
  __syncthreads();

  // Pass 3: first item of each cluster (items are sorted by cluster).
  for (int c = tid; c <= C_req; c += kPlanThreads) {
    int lo = 0, hi = n_items;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (items[mid].cluster < c) lo = mid + 1;
      else hi = mid;
    }
    cstart[c] = lo;
  }
  if (tid == 0) {
    if (bad_len) atomicOr(&hd->status, MLA_STATUS_BAD_LENGTH);
    hd->batch = B;
    hd->num_heads = H;
    hd->q_len = q_len;
    hd->page_size = ps;
    hd->window = window;
    hd->num_clusters = static_cast<int>(C);
    hd->total_blocks = static_cast<int>(T);
    hd->num_items = n_items;
    hd->num_partials = n_part;
    hd->num_split = n_split;
    hd->schedule = kScheduleCut;
    hd->planned = 1;
  }
}

constexpr int kMergeHeadsPerBlock = 4;
constexpr int kMergeBatch = 4;  // partials whose loads are issued together

// out[b,h] = sum_s 2^(lse_s - m) O_s / sum_s 2^(lse_s - m), O_s normalised
// per split, lse in log2 units; the natural-log lse is reported. The loads
// of the first kMergeBatch partials (lse and O) are issued together, so the
// chain of dependent global loads is short; the sums run in split order.
__global__ void __launch_bounds__(32 * kMergeHeadsPerBlock)
    merge_kernel(uint8_t* __restrict__ ws, WsLayout lay, int R, int RG,
                 __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  pdl_launch_dependents();
  pdl_wait();
  WsHeader* hd = reinterpret_cast<WsHeader*>(ws);
  // The grid covers at most min(batch, clusters) split requests; a schedule
  // with more would leave some unmerged, so it is reported. The split table
  // holds `batch` records, so the record of this row is read in the same
  // step as the count and used only when the row is in range.
  const int num_split = hd->num_split;
  const SplitRequest sr = reinterpret_cast<const SplitRequest*>(ws + lay.split)[blockIdx.x];
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && num_split > static_cast<int>(gridDim.x))
    atomicOr(&hd->status, MLA_STATUS_PLAN_MISMATCH);
  if (static_cast<int>(blockIdx.x) >= num_split) return;
  const int lane = threadIdx.x & 31;
  // row h of the split request's row group; R rows per request, RG per group
  const int h = blockIdx.y * kMergeHeadsPerBlock + (threadIdx.x >> 5);
  if (h >= RG || sr.row0 + h >= R) return;
  const int H = RG;  // partials are [slot][RG][512]
  const float* plse = reinterpret_cast<const float*>(ws + lay.partial_lse);
  const float* po = reinterpret_cast<const float*>(ws + lay.partial_o);
  const int ns = sr.num_splits;
  auto src = [&](int s) {
    return reinterpret_cast<const float4*>(po + (static_cast<size_t>(sr.first_partial + s) * H + h) * kDimCkv);
  };
  float lv[kMergeBatch];
  float4 v[kMergeBatch][4];
#pragma unroll
  for (int k = 0; k < kMergeBatch; ++k) {
    if (k < ns) {
      lv[k] = plse[(sr.first_partial + k) * H + h];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[k][j] = src(k)[lane + 32 * j];
    }
  }
  float m = -CUDART_INF_F;
#pragma unroll
  for (int k = 0; k < kMergeBatch; ++k)
    if (k < ns) m = fmaxf(m, lv[k]);
  for (int s = kMergeBatch; s < ns; ++s) m = fmaxf(m, plse[(sr.first_partial + s) * H + h]);
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  auto add = [&](float w, const float4* x) {
    wsum += w;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j].x += w * x[j].x;
      acc[j].y += w * x[j].y;
      acc[j].z += w * x[j].z;
      acc[j].w += w * x[j].w;
    }
  };
#pragma unroll
  for (int k = 0; k < kMergeBatch; ++k)
    if (k < ns) add(exp2f(lv[k] - m), v[k]);
  for (int s = kMergeBatch; s < ns; ++s) {
    float4 x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) x[j] = src(s)[lane + 32 * j];
    add(exp2f(plse[(sr.first_partial + s) * H + h] - m), x);
  }
  const float inv = 1.f / wsum;
  const size_t out_row = static_cast<size_t>(sr.b) * R + sr.row0 + h;
  __nv_bfloat16* dst = out + out_row * kDimCkv;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[j].x * inv, acc[j].y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[j].z * inv, acc[j].w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst + 4 * (lane + 32 * j)) = pk;
  }
  if (lse_out && lane == 0)
    lse_out[out_row] = (m + log2f(wsum)) * 0.69314718055994531f;
}

}  // namespace

cudaError_t launch_plan(const int32_t* context_lens, int batch, int q_len, int heads, int page_size,
                        int window, int clusters, uint8_t* ws, const WsLayout& lay,
                        cudaStream_t stream) {
  // Small batches: one thread per scheduled (request, row group) and at
  // least one per piece of the packed schedule (at most two per cluster),
  // whole warps; larger ones: 1024 threads looping.
  const int G = row_groups(q_len, heads);
  const int V = batch * G;
  int threads = kPlanThreads;
  if (V <= kPlanThreads) {
    const int pieces = 2 * clusters < kPackMax ? 2 * clusters : kPackMax;
    threads = (max(max(V, pieces), 1) + 31) / 32 * 32;
  }
  return launch_pdl(plan_kernel, dim3(1), dim3(threads), 0, stream, context_lens, batch, q_len, G, heads, page_size,
                    window, clusters, ws, lay);
}

cudaError_t launch_merge(const DecodeArgs& a, int clusters, cudaStream_t stream) {
  if (a.batch <= 0) return cudaSuccess;
  // A split (request, row group) holds one of the schedule's cluster
  // boundaries (fewer than `clusters`), so at most min(scheduled, clusters)
  // of them are split.
  const int V = a.batch * a.groups;
  const int rows = V < clusters ? V : clusters;
  const dim3 grid(rows, (a.group_rows + kMergeHeadsPerBlock - 1) / kMergeHeadsPerBlock);
  return launch_pdl(merge_kernel, grid, dim3(32 * kMergeHeadsPerBlock), 0, stream,
                    a.ws, a.lay, a.rows, a.group_rows, static_cast<__nv_bfloat16*>(a.out), a.lse);
}

}  // namespace mla
