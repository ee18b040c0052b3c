// Self-test of the failure path every tensor-core kernel of the library shares:
// a wait on an mbarrier that polls with try_wait and gives up after a time
// limit, recording MLA_ERR_DEVICE_TIMEOUT in the caller's status word instead
// of hanging or trapping.
#include "mla_internal.cuh"
#include "sm100_ptx.cuh"

namespace mla {
using namespace ptx;

// One block waits on a barrier that nothing ever arrives on.
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init_cluster();
  }
  __syncwarp();
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(b, 0)) return;  // cannot happen: no arrival is ever made
    if ((i & 63) == 0 && globaltimer() - t0 > limit_ns) {
      if (threadIdx.x == 0) set_status(status, MLA_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

}  // namespace mla

extern "C" {

int mla_selftest_bounded_wait(uint64_t limit_ns, int32_t* status, mla_stream_t stream) {
  if (status == nullptr || limit_ns > 2000000000ull) return MLA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_NO_DEVICE;
  mla::bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, status);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"
