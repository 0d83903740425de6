// W_UV projection after latent attention: y[b,h,:] = attn_out[b,h,:] W_UV[h]
// (v_head_dim 128 of MoE-Infinity PR #195 "DeepSeek-V2/V3 paged-attention
// shim (MLA)", Root causes 3). Per head a [B x 512] x [512 x 128] GEMM.
//
// One CTA per (head, 128 requests): TMA stages 64-wide K chunks of the
// attention output (K-major A) and of W_UV (N contiguous, MN-major B) in a
// 6-stage ring (the first six W chunks requested before the wait for the
// previous kernel); one thread issues tcgen05.mma M=128 N=128 K=16 into a
// 128-column TMEM accumulator; four warps read it back (one TMEM lane per
// request row) and store bf16.
#include <cuda_bf16.h>

#include "../../include/mla_decode.h"
#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kStages = 6;
constexpr int kKChunks = kDimCkv / 64;        // 8
constexpr int kABytes = 128 * 128;            // [128 rows][64 k] bf16
constexpr int kWBytes = 64 * 128;             // [64 k][64 n] bf16
constexpr int kStageBytes = kABytes + 2 * kWBytes;
constexpr int kOffBar = kStages * kStageBytes;
constexpr int kSmemBytes = kOffBar + 256 + 1024;
constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads, 1)
    uv_project_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap w_map,
                      __nv_bfloat16* __restrict__ y, int B, int H, int* __restrict__ status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto full = [&](int s) -> uint32_t { return bar0 + 8u * s; };
  auto empty = [&](int s) -> uint32_t { return bar0 + 8u * (kStages + s); };
  const uint32_t done = bar0 + 8u * (2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + 8 * (2 * kStages + 1));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int b0 = blockIdx.y * 128;
  pdl_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // W_UV does not come from the previous kernel: the first stages' W chunks
  // are requested before waiting for it, so they stream in while it ends.
  auto load_w = [&](int kc, int s) {
    const uint32_t dst = sbase + s * kStageBytes;
    tma_load_2d(dst + kABytes, &w_map, full(s), 0, h * kDimCkv + kc * 64);
    tma_load_2d(dst + kABytes + kWBytes, &w_map, full(s), 64, h * kDimCkv + kc * 64);
  };
  if (warp == 0 && lane == 0) {
    for (int kc = 0; kc < kStages; ++kc) {
      mbar_arrive_expect_tx(full(kc), kStageBytes);
      load_w(kc, kc);
    }
  }
  pdl_wait();  // the attention output is complete

  // A wait that runs out in the producer or the issuer stops its loop: the
  // accumulator's commit then never arrives and the epilogue's own bounded
  // wait reports it.
  if (warp == 0 && lane == 0) {
    for (int kc = 0; kc < kKChunks; ++kc) {
      const int s = kc % kStages, use = kc / kStages;
      if (kc >= kStages) {
        if (!mbar_wait(empty(s), (use & 1) ^ 1, nullptr)) break;
        mbar_arrive_expect_tx(full(s), kStageBytes);
        load_w(kc, s);
      }
      tma_load_3d(sbase + s * kStageBytes, &a_map, full(s), kc * 64, h, b0);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16(128, 128, false, true);
    for (int kc = 0; kc < kKChunks; ++kc) {
      const int s = kc % kStages, use = kc / kStages;
      if (!mbar_wait(full(s), use & 1, nullptr)) break;
      tc_fence_after();
      const uint32_t st = sbase + s * kStageBytes;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = sdesc_sw128(st + k * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(st + kABytes + k * 16 * 128, kWBytes, 1024);
        mma_bf16_ss(tmem, ad, bd, idesc, (kc | k) != 0);
      }
      mma_commit(empty(s));
      if (kc == kKChunks - 1) mma_commit(done);
    }
  }
  __syncwarp();
  // Every thread waits for the accumulator (bounded), then reads its row. If
  // a wait ran out (the producer's, the issuer's or this one), the rows of
  // this CTA are filled with NaN and the status word records the timeout, so
  // y is never left silently stale.
  const bool ready = __all_sync(0xffffffffu, mbar_wait(done, 0, nullptr));
  tc_fence_after();
  const int row = warp * 32 + lane;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  if (!ready) {
    if (status && threadIdx.x == 0) atomicOr(status, MLA_STATUS_TIMEOUT);
    if (b0 + row < B) {
      uint4* dst = reinterpret_cast<uint4*>(y + (static_cast<size_t>(b0 + row) * H + h) * kDimV);
      const uint4 nan4 = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
#pragma unroll 1
      for (int v = 0; v < kDimV * 2 / 16; ++v) dst[v] = nan4;
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < 128 / 32; ++c) {
      uint32_t r[32];
      tmem_ld16(taddr + c * 32, r);
      tmem_ld16(taddr + c * 32 + 16, r + 16);
      tmem_wait_ld();
      if (b0 + row < B) {
        __nv_bfloat16* dst = y + (static_cast<size_t>(b0 + row) * H + h) * kDimV + c * 32;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 pk;
          pk.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
          pk.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
          pk.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
          pk.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
          reinterpret_cast<uint4*>(dst)[v] = pk;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 128);
}

}  // namespace

cudaError_t launch_uv_project(const CUtensorMap& a_map, const CUtensorMap& w_map, void* y, int batch,
                              int heads, int* status, cudaStream_t stream) {
  static bool attr_set[kMaxDevices] = {};
  const cudaError_t e = set_smem_once(uv_project_kernel, kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(heads, (batch + 127) / 128);
  return launch_pdl(uv_project_kernel, grid, dim3(kThreads), kSmemBytes, stream, a_map, w_map,
                    static_cast<__nv_bfloat16*>(y), batch, heads, status);
}

}  // namespace mla
