// Self-test of the bounded wait that every kernel of the library uses for its
// mbarrier waits: one thread initialises an mbarrier and waits for its first
// phase with a short limit. When nothing arrives the wait runs out, the
// kernel records MLA_STATUS_TIMEOUT and returns, and the context stays
// usable; when the thread arrives first the wait returns at once.
#include "../../include/mla_decode.h"
#include "mla_internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(int arrive, unsigned long long limit_ns,
                                                          int32_t* status) {
  __shared__ __align__(8) uint64_t bar_storage;
  if (threadIdx.x != 0) return;
  const uint32_t bar = smem_addr(&bar_storage);
  mbar_init(bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (arrive) mbar_arrive(bar);
  if (!mbar_wait(bar, 0, nullptr, limit_ns)) atomicOr(status, MLA_STATUS_TIMEOUT);
}

}  // namespace
}  // namespace mla

extern "C" int mla_selftest_bounded_wait(int arrive, unsigned int limit_us, int32_t* status, void* stream) {
  if (!status || limit_us == 0 || limit_us > 1000000u) return MLA_ERR_ARG;
  mla::bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      arrive, static_cast<unsigned long long>(limit_us) * 1000ull, status);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
