// Latent-row write through slot_mapping (MoE-Infinity PR #195
// "DeepSeek-V2/V3 paged-attention shim (MLA)", Root causes 2 / Changes: the
// decode token's KV is persisted on every step; SGLang PR #32972, Cuda-graph
// safety: pad rows must not scatter, so a negative slot writes nothing).
//
// One warp per row: 576 bf16 = 72 16-byte vectors. bf16 pools copy the row;
// fp8 pools store e4m3(float(x) / kv_scale), round-to-nearest-even with
// saturation, 8 codes per 16-byte input vector.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kVecPerRow = kDimRow * 2 / 16;  // 72
constexpr int kWarpsPerBlock = 8;

template <int kDtype>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    kv_write_kernel(uint8_t* __restrict__ layer_base, int64_t layer_rows,
                    const uint4* __restrict__ rows, const int64_t* __restrict__ slots, int n,
                    float kv_scale, int* __restrict__ status) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= n) return;
  const int64_t s = slots[i];
  if (s < 0) return;  // pad row
  if (s >= layer_rows) {
    if (lane == 0 && status) atomicOr(status, MLA_STATUS_BAD_SLOT);
    return;
  }
  const uint4* src = rows + static_cast<int64_t>(i) * kVecPerRow;
  if (kDtype == MLA_DTYPE_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(layer_base) + s * kVecPerRow;
    for (int v = lane; v < kVecPerRow; v += 32) dst[v] = src[v];
  } else {
    uint2* dst = reinterpret_cast<uint2*>(layer_base + s * kDimRow);
    for (int v = lane; v < kVecPerRow; v += 32) {
      const uint4 x = src[v];
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t out[2] = {0, 0};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t bits = (w[k >> 1] >> ((k & 1) * 16)) & 0xFFFFu;
        const float f = __uint_as_float(bits << 16);
        const float t = __fdiv_rn(f, kv_scale);
        const uint32_t code =
            static_cast<uint32_t>(__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3));
        out[k >> 2] |= code << ((k & 3) * 8);
      }
      dst[v] = make_uint2(out[0], out[1]);
    }
  }
}

}  // namespace

cudaError_t launch_kv_write(void* pool, int dtype, int64_t layer_rows, int layer, float kv_scale,
                            const void* rows, const int64_t* slots, int n, int* status,
                            cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int elem = dtype == MLA_DTYPE_BF16 ? 2 : 1;
  uint8_t* base = static_cast<uint8_t*>(pool) + static_cast<int64_t>(layer) * layer_rows * kDimRow * elem;
  const dim3 grid((n + kWarpsPerBlock - 1) / kWarpsPerBlock);
  const dim3 block(32 * kWarpsPerBlock);
  if (dtype == MLA_DTYPE_BF16)
    return launch_pdl(kv_write_kernel<MLA_DTYPE_BF16>, grid, block, 0, stream, base, layer_rows,
                      static_cast<const uint4*>(rows), slots, n, kv_scale, status);
  return launch_pdl(kv_write_kernel<MLA_DTYPE_FP8_E4M3>, grid, block, 0, stream, base, layer_rows,
                    static_cast<const uint4*>(rows), slots, n, kv_scale, status);
}

}  // namespace mla
