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
// several items whose partial (O, lse) are merged afterwards. With several
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
// epilogue and the pipeline refill when the next item starts; a fit of
// per-cluster time against blocks and items on the V3-shaped workload gave
// 3.3): small batches count it in the balance, so clusters that start more
// requests get fewer blocks.
constexpr int kItemCostBlocks = 3;

// Block-wide exclusive scan of one int per thread; returns the prefix and
// writes the block total to *total.
__device__ int block_excl_scan(int v, int* total, int* smem32) {
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
    // One request per thread, everything in registers: no pass through
    // global memory between the scans. Request b weighs its n_b blocks plus
    // kItemCostBlocks; the weights are concatenated in request order and cut
    // into C equal ranges; a request's blocks sit after its extra weight.
    __shared__ int last_cluster[kPlanThreads];
    int L = 0, s = 0, first = 0, n = 0;
    const int vb = tid / G, vg = tid - (tid / G) * G;  // request and row group of this thread
    if (tid < V) range_of(vb, L, s, first, n);
    int T32;
    const int off = block_excl_scan(tid < V ? n + kItemCostBlocks : 0, &T32, smem32) + kItemCostBlocks;
    const long long T = T32;
    const long long C = T > 0 ? (T < C_req ? T : C_req) : 1;
    int cf = 0, cl = -1, ns = 0;
    if (tid < V) {
      cf = cluster_of(off, T, C);
      cl = cluster_of(static_cast<long long>(off) + n - 1, T, C);
      ns = cl - cf + 1;
    }
    last_cluster[tid] = cl;
    int t_items, t_part, t_split;
    const int item0 = block_excl_scan(ns, &t_items, smem32);
    const int part0 = block_excl_scan(ns > 1 ? ns : 0, &t_part, smem32);
    const int split0 = block_excl_scan(ns > 1 ? 1 : 0, &t_split, smem32);
    if (tid < V) {
      for (int k = 0; k < ns; ++k) {
        const int c = cf + k;
        const long long lo = max(static_cast<long long>(off), range_lo(c, T, C));
        const long long hi = min(static_cast<long long>(off) + n, range_lo(c + 1, T, C));
        WorkItem w;
        w.b = vb;
        w.blk_begin = first + static_cast<int>(lo - off);
        w.blk_end = first + static_cast<int>(hi - off);
        w.slot = ns > 1 ? part0 + k : -1;
        w.tok_lo = s;
        w.tok_hi = L + q_len;
        w.cluster = c;
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
    __syncthreads();
    if (tid == 0) {
      if (bad_len) atomicOr(&hd->status, MLA_STATUS_BAD_LENGTH);
      hd->batch = B;
      hd->num_heads = H;
      hd->q_len = q_len;
      hd->page_size = ps;
      hd->window = window;
      hd->num_clusters = static_cast<int>(C);
      hd->total_blocks = static_cast<int>(T);
      hd->num_items = t_items;
      hd->num_partials = t_part;
      hd->num_split = t_split;
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
  // Small batches: one thread per scheduled (request, row group), whole
  // warps, every step in registers; larger ones: 1024 threads looping.
  const int G = row_groups(q_len, heads);
  const int V = batch * G;
  const int threads = V <= kPlanThreads ? ((V + 31) / 32 * 32 > 32 ? (V + 31) / 32 * 32 : 32) : kPlanThreads;
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
