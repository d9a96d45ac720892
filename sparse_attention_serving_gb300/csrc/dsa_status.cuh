// dsa_status.cuh -- the sticky device status word kept at the head of every
// workspace: word 0 holds the first error code a kernel raised, word 1 a site
// tag (which wait or check), word 2 a detail value (e.g. the offending index).
#pragma once
#include <cstdint>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kStatusWords = 64;            // 256-byte header
constexpr size_t kWorkspaceHeader = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait: far above any legitimate wait

__device__ __forceinline__ void status_raise(uint32_t* status, uint32_t code, uint32_t where,
                                             uint32_t detail = 0) {
  if (status == nullptr) return;
  if (atomicCAS(status, 0u, code) == 0u) {
    status[1] = where;
    status[2] = detail;
  }
}

}  // namespace dsa
