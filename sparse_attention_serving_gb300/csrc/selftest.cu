// selftest.cu -- device-side failure path check: a bounded wait that nothing
// satisfies must give up, record DSA_ERR_DEVICE_TIMEOUT in the workspace status
// word and return, leaving the CUDA context usable.
#include "dsa_status.cuh"
#include "internal.h"
#include "sm103.cuh"

namespace dsa {

constexpr uint32_t SITE_SELFTEST = 0x500;

__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // no thread ever arrives on `bar`: the wait runs out after limit_ns
  mbar_wait(&bar, 0, status, limit_ns, SITE_SELFTEST);
}

}  // namespace dsa

extern "C" dsa_status_t dsa_selftest_wait_timeout(void* workspace, size_t ws_bytes,
                                                  uint64_t limit_ns, dsa_stream_t stream) {
  using namespace dsa;
  if (workspace == nullptr || ws_bytes < kWorkspaceHeader ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return DSA_ERR_INVALID_ARGUMENT;
  if (limit_ns == 0 || limit_ns > 200000000ull) return DSA_ERR_INVALID_ARGUMENT;  // <= 200 ms
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint32_t*>(workspace), limit_ns);
  return launch_status("selftest_wait_kernel");
}
