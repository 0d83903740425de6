// Host side of the C ABI declared in include/mla_decode.h: argument checks,
// workspace layout, TMA tensor maps, kernel launches. No allocation, no
// stream synchronisation (except mla_get_error).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <string.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"

// Scratch of mla_decode_noalloc: schedule, status and split partials.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

namespace {

using mla::WsHeader;
using mla::WsLayout;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D row-major map: rows x cols elements, row pitch `pitch_bytes`, box
// {box_cols, box_rows}, zero fill out of bounds.
bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t rows, uint64_t cols,
                 uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows,
                 CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of a bf16 pool for one copy of a rank's four 64-dim chunks: dims
// {64 dims, rows, 8 chunks}, strides {row pitch, 128 bytes}, box {64, 64, 4}
// (written to shared memory chunk-major, 128-byte swizzled).
bool make_chunk_map(CUtensorMap* m, const void* base, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, 8};
  cuuint64_t strides[2] = {mla::kDimRow * 2ull, 128};
  cuuint32_t box[3] = {64, 64, 4};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_pool(const mla_kv_pool* pool) {
  if (!pool || !pool->data || pool->num_layers <= 0 || pool->num_pages <= 0) return false;
  if (pool->page_size != 16 && pool->page_size != 32 && pool->page_size != 64 && pool->page_size != 128)
    return false;
  if (pool->dtype != MLA_DTYPE_BF16 && pool->dtype != MLA_DTYPE_FP8_E4M3) return false;
  if (pool->dtype == MLA_DTYPE_FP8_E4M3 && !(pool->kv_scale > 0.f)) return false;
  return aligned(pool->data, 16);
}

int max_clusters() { return mla::decode_max_active_clusters(); }

bool valid_heads(int h) { return h == 16 || h == 32 || h == 64 || h == 128; }

// Scheduled requests and rows per scheduled request of (batch, q_len,
// heads): each request's q_len x heads rows in groups of at most 128.
mla::WsLayout layout_of(int batch, int q_len, int heads, int clusters) {
  return mla::ws_layout(batch * mla::row_groups(q_len, heads), mla::group_rows(q_len, heads), clusters);
}

// The host-visible checks of mla_decode_q (everything but the workspace), so
// that mla_decode_noalloc can run them before it touches its scratch.
int check_decode_args(const mla_kv_pool* pool, int layer, const void* q, const int32_t* page_indptr,
                      const int32_t* page_ids, int max_blocks, const int32_t* context_lens, int batch,
                      int q_len, int num_heads, float softmax_scale, int window, const void* out) {
  if (!valid_pool(pool) || layer < 0 || layer >= pool->num_layers || batch < 0 || window < 0) return MLA_ERR_ARG;
  if (!valid_heads(num_heads)) return MLA_ERR_UNSUPPORTED;
  if (q_len < 1 || static_cast<int64_t>(batch) * q_len * num_heads >= (1ll << 31)) return MLA_ERR_ARG;
  if (batch == 0) return MLA_OK;
  if (!q || !page_ids || !context_lens || !out || !aligned(q, 16) || !aligned(out, 32)) return MLA_ERR_ARG;
  if (!page_indptr && max_blocks <= 0) return MLA_ERR_ARG;
  if (!(softmax_scale > 0.f)) return MLA_ERR_ARG;
  const uint64_t total_rows = static_cast<uint64_t>(pool->num_layers) * pool->num_pages * pool->page_size;
  if (total_rows >= (1ull << 31)) return MLA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
  return MLA_OK;
}

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (the host-side symbol is only a stand-in for it).
void* noalloc_scratch() {
  constexpr int kMaxDevices = 64;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

int mla_kv_write(const mla_kv_pool* pool, int layer, const void* new_rows, const int64_t* slot_mapping,
                 int n, void* workspace, void* stream) {
  if (n < 0 || !valid_pool(pool) || layer < 0 || layer >= pool->num_layers) return MLA_ERR_ARG;
  if (n == 0) return MLA_OK;
  if (!new_rows || !slot_mapping || !aligned(new_rows, 16)) return MLA_ERR_ARG;
  int* status = workspace ? &reinterpret_cast<WsHeader*>(workspace)->status : nullptr;
  const int64_t layer_rows = static_cast<int64_t>(pool->num_pages) * pool->page_size;
  cudaError_t e = mla::launch_kv_write(pool->data, pool->dtype, layer_rows, layer, pool->kv_scale, new_rows,
                                       slot_mapping, n, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode_num_clusters(void) {
  const int c = max_clusters();
  return c > 0 ? c : MLA_ERR_CUDA;
}

size_t mla_decode_workspace_size_q(int batch, int q_len, int num_heads) {
  if (batch < 0 || q_len < 1 || !valid_heads(num_heads)) return 0;
  if (static_cast<int64_t>(batch) * q_len * num_heads >= (1ll << 31)) return 0;
  const int c = max_clusters();
  if (c <= 0) return 0;
  return layout_of(batch, q_len, num_heads, c).total;
}

size_t mla_decode_workspace_size(int batch, int num_heads) {
  if (batch < 0 || num_heads <= 0 || num_heads > 128) return 0;
  const int c = max_clusters();
  if (c <= 0) return 0;
  return mla::ws_layout(batch, num_heads, c).total;
}

int mla_decode_plan_q(const int32_t* context_lens, int batch, int q_len, int num_heads, int page_size, int window,
                      int num_clusters, void* workspace, size_t workspace_bytes, void* stream) {
  if (batch < 0 || q_len < 1 || window < 0 || num_clusters < 0 || !workspace) return MLA_ERR_ARG;
  if (batch > 0 && !context_lens) return MLA_ERR_ARG;
  if (!valid_heads(num_heads)) return MLA_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128) return MLA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(batch) * q_len * num_heads >= (1ll << 31)) return MLA_ERR_ARG;
  const int cmax = max_clusters();
  if (cmax <= 0) return MLA_ERR_CUDA;
  const WsLayout lay = layout_of(batch, q_len, num_heads, cmax);
  if (!aligned(workspace, 256) || workspace_bytes < lay.total) return MLA_ERR_WORKSPACE;
  const int c = (num_clusters == 0 || num_clusters > cmax) ? cmax : num_clusters;
  cudaError_t e = mla::launch_plan(context_lens, batch, q_len, num_heads, page_size, window, c,
                                   static_cast<uint8_t*>(workspace), lay, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode_plan(const int32_t* context_lens, int batch, int num_heads, int page_size, int window,
                    int num_clusters, void* workspace, size_t workspace_bytes, void* stream) {
  return mla_decode_plan_q(context_lens, batch, 1, num_heads, page_size, window, num_clusters, workspace,
                           workspace_bytes, stream);
}

int mla_decode_q(const mla_kv_pool* pool, int layer, const void* q, const int32_t* page_indptr,
                 const int32_t* page_ids, int max_blocks, const int32_t* context_lens, int batch, int q_len,
                 int num_heads, float softmax_scale, int window, void* workspace, void* out, float* lse,
                 void* stream) {
  if (!workspace) return MLA_ERR_ARG;
  const int rc = check_decode_args(pool, layer, q, page_indptr, page_ids, max_blocks, context_lens, batch,
                                   q_len, num_heads, softmax_scale, window, out);
  if (rc != MLA_OK || batch == 0) return rc;
  const int cmax = max_clusters();
  if (cmax <= 0) return MLA_ERR_CUDA;
  if (!aligned(workspace, 256)) return MLA_ERR_WORKSPACE;

  const int ps = pool->page_size;
  const uint64_t total_rows = static_cast<uint64_t>(pool->num_layers) * pool->num_pages * ps;
  // Each rank of the decode cluster reads its 256 c_kv dims and 32 rope
  // dims of every row: bf16 pools as 64-dim boxes (128-byte swizzle) and one
  // 32-dim box (64-byte swizzle), the layout the tensor core reads; fp8
  // pools as one 256-byte and one 32-byte box, unswizzled, which the kernel
  // widens to f16 in that same layout.
  CUtensorMap maps[5];
  memset(maps, 0, sizeof maps);
  const uint32_t box_rows = ps < mla::kBlockTokens ? ps : mla::kBlockTokens;
  const uint64_t q_rows = static_cast<uint64_t>(batch) * q_len * num_heads;
  const bool fp8 = pool->dtype == MLA_DTYPE_FP8_E4M3;
  const bool kv_ok =
      fp8 ? make_map_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, pool->data, total_rows, mla::kDimRow, mla::kDimRow,
                        256, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE) &&
                make_map_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, pool->data, total_rows, mla::kDimRow,
                            mla::kDimRow, 32, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE)
          : make_map_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pool->data, total_rows, mla::kDimRow,
                        mla::kDimRow * 2, 64, box_rows) &&
                make_map_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pool->data, total_rows, mla::kDimRow,
                            mla::kDimRow * 2, 32, box_rows, CU_TENSOR_MAP_SWIZZLE_64B);
  if (!kv_ok ||
      !make_map_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, q_rows, mla::kDimRow, mla::kDimRow * 2, 64,
                   128) ||
      !make_map_2d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, q_rows, mla::kDimRow, mla::kDimRow * 2, 32,
                   128, CU_TENSOR_MAP_SWIZZLE_64B))
    return MLA_ERR_CUDA;
  if (!fp8 && ps >= mla::kBlockTokens && !make_chunk_map(&maps[4], pool->data, total_rows)) return MLA_ERR_CUDA;

  mla::DecodeArgs a;
  memset(&a, 0, sizeof a);
  a.pool = pool->data;
  a.page_indptr = page_indptr;
  a.page_ids = page_ids;
  a.context_lens = context_lens;
  a.out = out;
  a.lse = lse;
  a.ws = static_cast<uint8_t*>(workspace);
  a.lay = layout_of(batch, q_len, num_heads, cmax);
  a.max_blocks = max_blocks;
  a.batch = batch;
  a.num_heads = num_heads;
  a.q_len = q_len;
  a.rows = q_len * num_heads;
  a.group_rows = mla::group_rows(q_len, num_heads);
  a.groups = mla::row_groups(q_len, num_heads);
  a.page_size = ps;
  a.window = window;
  a.num_pages = pool->num_pages;
  a.num_layers = pool->num_layers;
  a.layer = layer;
  a.dtype = pool->dtype;
  a.kv_scale = pool->kv_scale;
  // fp8 pools: scores and output are scaled by kv_scale instead of the
  // codes (the kernel computes on the exact codes).
  a.scale_log2 = softmax_scale * 1.4426950408889634f * (fp8 ? pool->kv_scale : 1.f);
  a.out_scale = fp8 ? pool->kv_scale : 1.f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = mla::launch_decode(maps, a, cmax, st);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  e = mla::launch_merge(a, cmax, st);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode(const mla_kv_pool* pool, int layer, const void* q, const int32_t* page_indptr,
               const int32_t* page_ids, int max_blocks, const int32_t* context_lens, int batch, int num_heads,
               float softmax_scale, int window, void* workspace, void* out, float* lse, void* stream) {
  return mla_decode_q(pool, layer, q, page_indptr, page_ids, max_blocks, context_lens, batch, 1, num_heads,
                      softmax_scale, window, workspace, out, lse, stream);
}

int mla_uv_project(const void* attn_out, const void* w_uv, void* y, int batch, int num_heads, void* workspace,
                   void* stream) {
  if (batch < 0 || num_heads <= 0) return MLA_ERR_ARG;
  if (batch == 0) return MLA_OK;
  if (!attn_out || !w_uv || !y || !aligned(attn_out, 16) || !aligned(w_uv, 16) || !aligned(y, 16))
    return MLA_ERR_ARG;
  if (workspace && !aligned(workspace, 256)) return MLA_ERR_WORKSPACE;
  int* status = workspace ? &reinterpret_cast<WsHeader*>(workspace)->status : nullptr;
  auto fn = encode_fn();
  if (!fn) return MLA_ERR_CUDA;
  CUtensorMap a_map, w_map;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(mla::kDimCkv), static_cast<cuuint64_t>(num_heads),
                          static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[2] = {mla::kDimCkv * 2ull, static_cast<cuuint64_t>(num_heads) * mla::kDimCkv * 2ull};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&a_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(attn_out), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_CUDA;
  }
  if (!make_map_2d(&w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_uv, static_cast<uint64_t>(num_heads) * mla::kDimCkv,
                   mla::kDimV, mla::kDimV * 2, 64, 64))
    return MLA_ERR_CUDA;
  cudaError_t e =
      mla::launch_uv_project(a_map, w_map, y, batch, num_heads, status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode_noalloc(const mla_kv_pool* pool, int layer, const void* q, const int32_t* page_indptr,
                       const int32_t* page_ids, int max_blocks, const int32_t* context_lens, int batch,
                       int num_heads, float softmax_scale, int window, int num_clusters, void* out, float* lse,
                       int32_t* status, void* stream) {
  if (num_clusters < 0) return MLA_ERR_ARG;
  // Every argument check runs before the scratch is touched: a rejected call
  // leaves the schedule of an earlier call that has not run yet intact.
  const int rc0 = check_decode_args(pool, layer, q, page_indptr, page_ids, max_blocks, context_lens, batch, 1,
                                    num_heads, softmax_scale, window, out);
  if (rc0 != MLA_OK) return rc0;
  const int cmax = max_clusters();
  if (cmax <= 0) return MLA_ERR_CUDA;
  const size_t need = mla::ws_layout(batch, num_heads, cmax).total;
  if (need > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  void* ws = noalloc_scratch();
  if (!ws) return MLA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The scratch keeps the previous call's bytes: start this call's status at 0.
  if (cudaMemsetAsync(ws, 0, sizeof(mla::WsHeader), st) != cudaSuccess) return MLA_ERR_CUDA;
  int rc = mla_decode_plan(context_lens, batch, num_heads, pool->page_size, window, num_clusters, ws, need,
                           stream);
  if (rc != MLA_OK) return rc;
  rc = mla_decode(pool, layer, q, page_indptr, page_ids, max_blocks, context_lens, batch, num_heads,
                  softmax_scale, window, ws, out, lse, stream);
  if (rc != MLA_OK) return rc;
  if (status && cudaMemcpyAsync(status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_get_error(void* workspace, int* code, int clear, void* stream) {
  if (!workspace || !code) return MLA_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  *code = v;
  if (clear) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // extern "C"
