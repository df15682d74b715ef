// Self-test of the bounded-wait failure path.  One thread initialises an
// mbarrier that nothing will ever arrive on and waits on it with the same
// bounded wait the prefill pipeline uses; when the limit runs out it records
// a status code in the library's status word and returns, exactly as a
// stalled pipeline would, without trapping or hanging the GPU.
#include <cuda_runtime.h>

#include "../../include/jetlong.h"
#include "internal.h"
#include "sm100.cuh"

namespace jl {
namespace {

constexpr int kSelftestCode = 99;

__global__ void bounded_wait_selftest_kernel(long long limit_cycles, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  const uint32_t b = sm100::smem_u32(&bar);
  abort_flag = 0;
  sm100::mbar_init(b, 1);
  sm100::fence_barrier_init();
  if (!sm100::mbar_wait(b, 0, &abort_flag, limit_cycles)) atomicCAS(status, 0, kSelftestCode);
}

}  // namespace
}  // namespace jl

extern "C" int jl_selftest_bounded_wait(long long limit_cycles, void* cuda_stream) {
  if (limit_cycles < 1 || limit_cycles > 4000000000LL)
    return jl::set_error(JL_ERR_INVALID, "selftest: limit_cycles must be in [1, 4e9]");
  int* status = jl::device_status_ptr();
  if (status == nullptr) return jl::set_error(JL_ERR_CUDA, "selftest: cannot resolve the status word");
  jl::bounded_wait_selftest_kernel<<<1, 1, 0, static_cast<cudaStream_t>(cuda_stream)>>>(limit_cycles, status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return jl::set_error(JL_ERR_CUDA, cudaGetErrorString(e));
  return JL_OK;
}
