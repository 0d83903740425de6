// Internal layout shared by the host entry points and the kernels: the
// decode workspace, the work-item record the planner writes, and the
// launcher prototypes of each kernel file.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mla {

constexpr int kDimCkv = 512;
constexpr int kDimRope = 64;
constexpr int kDimRow = 576;
constexpr int kDimV = 128;
constexpr int kBlockTokens = 64;  // tokens per schedule block = per decode tile
constexpr int kGroupRows = 128;   // rows per row group (one M=128 tensor-core tile)

// Row groups and rows per group of a request with q_len x heads rows.
__host__ __device__ inline int row_groups(int q_len, int heads) {
  return (q_len * heads + kGroupRows - 1) / kGroupRows;
}
__host__ __device__ inline int group_rows(int q_len, int heads) {
  return q_len * heads < kGroupRows ? q_len * heads : kGroupRows;
}

// Rows of a request: q_len query positions x num_heads heads, row
// r = i * num_heads + h (q, out and lse are [batch][q_len][heads][...]).
// Query i attends positions [lo_i, L + i] with L = context_lens[b] and
// lo_i = 0, or max(0, L + i + 1 - window). A request's rows are cut into
// groups of at most 128 (one M=128 tile of the tensor core); each (request,
// row group) is scheduled like a request of its own.

// One contiguous run of 64-token blocks of one (request, row group),
// processed by one cluster. Attended positions of the item (over all its
// query positions) are [tok_lo, tok_hi).
struct WorkItem {
  int b;
  int blk_begin;
  int blk_end;   // exclusive
  int slot;      // -1: whole request, write the final output; else partial index
  int tok_lo;
  int tok_hi;
  int cluster;
  int row0;      // first row of the row group
};

struct SplitRequest {
  int b;
  int num_splits;
  int first_partial;
  int row0;
};

// How the plan cut the work (WsHeader::schedule).
constexpr int kScheduleCut = 0;     // blocks of all requests concatenated, cut into equal ranges
constexpr int kSchedulePacked = 1;  // long requests split, pieces paired largest with smallest

struct WsHeader {
  int status;  // sticky MLA_STATUS_* bits
  int batch;
  int num_heads;
  int page_size;
  int window;
  int num_clusters;   // clusters the plan spread work over (<= requested)
  int total_blocks;
  int num_items;
  int num_partials;
  int num_split;
  int planned;        // 1 after a successful plan
  int q_len;
  int schedule;       // kScheduleCut or kSchedulePacked
  int pad[3];
};

struct WsLayout {
  size_t items, cluster_start, split, req_scratch, partial_lse, partial_o, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte offsets of each region for (scheduled requests, rows per scheduled
// request, clusters): with q_len > 1, batch x row groups requests of at most
// 128 rows.
__host__ __device__ inline WsLayout ws_layout(int batch, int heads, int clusters) {
  WsLayout L;
  size_t off = align_up(sizeof(WsHeader), 256);
  L.items = off;
  off = align_up(off + sizeof(WorkItem) * static_cast<size_t>(batch + clusters), 256);
  L.cluster_start = off;
  off = align_up(off + sizeof(int) * static_cast<size_t>(clusters + 1), 256);
  L.split = off;
  off = align_up(off + sizeof(SplitRequest) * static_cast<size_t>(batch), 256);
  L.req_scratch = off;
  off = align_up(off + sizeof(int) * 4 * static_cast<size_t>(batch), 256);
  const size_t max_partials = 2 * static_cast<size_t>(clusters);
  L.partial_lse = off;
  off = align_up(off + sizeof(float) * max_partials * heads, 256);
  L.partial_o = off;
  off = align_up(off + sizeof(float) * max_partials * heads * kDimCkv, 256);
  L.total = off;
  return L;
}

struct DecodeArgs {
  const void* pool;  // pool base (bf16 rows), for L2 prefetch
  const int32_t* page_indptr;
  const int32_t* page_ids;
  const int32_t* context_lens;
  void* out;        // bf16 [B][H][512]
  float* lse;       // [B][H] or null
  uint8_t* ws;
  WsLayout lay;
  int max_blocks;
  int batch;
  int num_heads;
  int q_len;         // query positions per request
  int rows;          // rows per request: q_len * num_heads
  int group_rows;    // rows per row group: min(rows, 128)
  int groups;        // row groups per request
  int page_size;
  int window;
  int num_pages;
  int num_layers;
  int layer;
  int dtype;
  float kv_scale;
  float scale_log2;  // softmax_scale * log2(e) (* kv_scale for fp8 pools)
  float out_scale;   // 1, or kv_scale for fp8 pools (codes are dequantised by scaling O)
};

// Index of the current device for per-device caches (kMaxDevices entries),
// or -1.
constexpr int kMaxDevices = 64;
inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Sets the dynamic shared memory limit of `kernel` once per device (the
// attribute belongs to the device's context).
template <typename K>
inline cudaError_t set_smem_once(K kernel, int bytes, bool (&done)[kMaxDevices]) {
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (done[dev]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev] = true;
  return e;
}

// Launch `kernel` on `stream` with programmatic stream serialization (see
// pdl_wait in ptx.cuh): it may start while the previous kernel finishes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// kv_write.cu
cudaError_t launch_kv_write(void* pool, int dtype, int64_t layer_rows, int layer, float kv_scale,
                            const void* rows, const int64_t* slots, int n, int* status,
                            cudaStream_t stream);
// plan_merge.cu
cudaError_t launch_plan(const int32_t* context_lens, int batch, int q_len, int heads, int page_size,
                        int window, int clusters, uint8_t* ws, const WsLayout& lay,
                        cudaStream_t stream);
cudaError_t launch_merge(const DecodeArgs& a, int clusters, cudaStream_t stream);
// decode_sm103.cu
// maps: {kv 64-dim boxes (128B swizzle), kv 32-dim boxes (64B swizzle),
//        q 64-dim boxes, q 32-dim boxes, kv four-chunk boxes (bf16, page size >= 64)}
cudaError_t launch_decode(const CUtensorMap* maps, const DecodeArgs& a, int clusters, cudaStream_t stream);
int decode_max_active_clusters();
// uv_project.cu
cudaError_t launch_uv_project(const CUtensorMap& a_map, const CUtensorMap& w_map, void* y,
                              int batch, int heads, int* status, cudaStream_t stream);

}  // namespace mla
