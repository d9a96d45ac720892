// noalloc.cu -- sparse_mla_fwd_noalloc: sparse MLA forward without a caller
// workspace.  The split-K partial results (and, when the caller passes no
// status pointer, the device status word) live in one fixed array of device
// memory that belongs to this library.
//
// Some callers cannot allocate device memory at the point where they run this
// operation: an inference server that hands all device memory to its own
// fixed pool at start-up, or a plugin interface of a host framework that
// passes tensors in and out but has no way to request extra scratch.  This
// entry point serves them: it calls no cudaMalloc / cudaFree and no allocating
// library routine.
#include <cuda_runtime.h>

#include "dsa_status.cuh"
#include "internal.h"

namespace {

// 32 MiB of scratch, held by every GPU that loads the library until the
// process exits.  The split count keeps (queries x splits) at or below the SM
// count, and a (query, split) pair needs H x 512 BF16 outputs and H FP32
// log-sum-exps: with 96 heads at most SMs x 98,688 bytes, which fits for any
// part with up to about 340 SMs.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// In host code `g_noalloc_scratch` is only a host-side stand-in for the device
// array: passing it to a kernel would fault (or, where the GPU can reach host
// memory, silently use the wrong memory).  The device address is looked up on
// every call, with the caller's device current.  The lookup allocates nothing,
// and a fresh lookup stays right after cudaDeviceReset or when the caller
// switches contexts, where an address kept from an earlier call would point at
// memory that is no longer mapped.  The first lookup on a device also loads
// this library's device code there, which is why the first call should come
// before any stream capture.
dsa_status_t scratch_on_current_device(unsigned char** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();  // the failed lookup must not stick to later launches
    return DSA_ERR_CUDA;
  }
  *out = static_cast<unsigned char*>(p);
  return DSA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" dsa_status_t sparse_mla_fwd_noalloc(const uint16_t* q_lat, const dsa_rows_t* kv,
                                               const int32_t* idx, const int32_t* q_start,
                                               const int32_t* kv_len, int B, int Tq, int H,
                                               int topk, int max_kv_len, float scale,
                                               uint16_t* o_lat, float* lse,
                                               uint32_t* device_status, dsa_stream_t stream) {
  using namespace dsa;
  if (!q_lat || !idx || !q_start || !kv_len || !o_lat || kv == nullptr || kv->base == nullptr)
    return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_lat, 16) || !aligned(idx, 4) || !aligned(o_lat, 16) ||
      (lse != nullptr && !aligned(lse, 4)) || !aligned(q_start, 4) || !aligned(kv_len, 4) ||
      !aligned(kv->base, 16) || (device_status != nullptr && !aligned(device_status, 4)))
    return DSA_ERR_INVALID_ARGUMENT;
  if (B <= 0 || Tq <= 0 || max_kv_len <= 0 || topk <= 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!(scale > 0.f)) return DSA_ERR_INVALID_ARGUMENT;
  if (H != 96 && H != 8) return DSA_ERR_UNSUPPORTED;
  if (topk > 2048) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Tq * H >= (int64_t(1) << 31) ||
      static_cast<int64_t>(B) * Tq >= (int64_t(1) << 31) / 8)
    return DSA_ERR_UNSUPPORTED;

  SparseMlaArgs a{};
  RowStore& s = a.kv;
  s.base = static_cast<const uint16_t*>(kv->base);
  if (kv->block_table == nullptr) {
    if (kv->seq_stride < max_kv_len) return DSA_ERR_INVALID_ARGUMENT;
    s.seq_stride = kv->seq_stride;
    s.total_rows = static_cast<int64_t>(B) * kv->seq_stride;
  } else {
    if (kv->page_size != kPage) return DSA_ERR_UNSUPPORTED;
    if (kv->num_pages <= 0 || kv->max_pages <= 0 ||
        static_cast<int64_t>(kv->max_pages) * kPage < max_kv_len || !aligned(kv->block_table, 4))
      return DSA_ERR_INVALID_ARGUMENT;
    s.block_table = kv->block_table;
    s.max_pages = kv->max_pages;
    s.num_pages = kv->num_pages;
    s.total_rows = static_cast<int64_t>(kv->num_pages) * kPage;
  }
  if (s.total_rows >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;

  // the split-K partials must fit the fixed array (after its 256-byte status header)
  const size_t need = sparse_mla_scratch_bytes(B, Tq, H, topk);
  if (need > kNoAllocScratchBytes - kWorkspaceHeader) return DSA_ERR_WORKSPACE_TOO_SMALL;

  unsigned char* scratch = nullptr;
  dsa_status_t st = scratch_on_current_device(&scratch);
  if (st != DSA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the status header must start at zero
  // (the partials are written in full before they are read)
  if (device_status == nullptr &&
      cudaMemsetAsync(scratch, 0, kWorkspaceHeader, cs) != cudaSuccess)
    return DSA_ERR_CUDA;

  a.q_lat = q_lat;
  a.idx = idx;
  a.q_start = q_start;
  a.kv_len = kv_len;
  a.B = B;
  a.Tq = Tq;
  a.H = H;
  a.topk = topk;
  a.max_kv_len = max_kv_len;
  a.scale = scale;
  a.o_lat = o_lat;
  a.lse = lse;
  a.status = device_status != nullptr ? device_status : reinterpret_cast<uint32_t*>(scratch);
  a.scratch = scratch + kWorkspaceHeader;
  a.scratch_bytes = kNoAllocScratchBytes - kWorkspaceHeader;
  return sparse_mla_launch(a, cs);
}
