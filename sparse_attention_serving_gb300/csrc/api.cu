// api.cu -- the C ABI of libdsa.so (declared in include/dsa.h): host-side
// argument checks, workspace layout, tensor-map encoding and dispatch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "dsa_status.cuh"
#include "internal.h"

namespace dsa {

// ---------------------------------------------------------------------------
// tensor maps (driver entry point fetched through the runtime: no link-time
// dependency on libcuda, so the library loads on machines without a driver)
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

bool encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                    bool swizzle128) {
  auto enc = encoder();
  if (enc == nullptr || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUresult r =
      enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE,
          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

dsa_status_t launch_status(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) return DSA_OK;
  if (std::getenv("DSA_VERBOSE") != nullptr)
    std::fprintf(stderr, "libdsa: %s: %s\n", what, cudaGetErrorString(e));
  return DSA_ERR_CUDA;
}

int indexer_prefill_max_topk(int H_I, int D_I);
dsa_status_t indexer_prefill_launch(const IndexerArgs& a, cudaStream_t stream);
dsa_status_t indexer_decode_launch(const IndexerArgs& a, cudaStream_t stream);
size_t indexer_decode_scratch_bytes(int B, int max_kv_len);
size_t indexer_prefill_scratch_bytes(int B, int Tq, int H_I, int D_I);

// Tq == 1 (one new token per request) takes the split decode path, which keeps
// a linear FP32 score vector per request in the workspace; Tq > 1 takes the
// fused prefill kernel, which keeps the candidates above each query's running
// threshold in per-CTA buffers of the workspace.  The indexer head width is
// 128 with 64 heads and 64 with 4 heads, the two supported shapes.
size_t indexer_scratch_bytes(int B, int Tq, int max_kv_len, int H_I, int topk) {
  (void)topk;
  if (Tq == 1) return indexer_decode_scratch_bytes(B, max_kv_len);
  return indexer_prefill_scratch_bytes(B, Tq, H_I, H_I == 4 ? 64 : 128);
}

dsa_status_t indexer_launch(const IndexerArgs& a, cudaStream_t stream) {
  if (a.Tq == 1) return indexer_decode_launch(a, stream);
  return indexer_prefill_launch(a, stream);
}

}  // namespace dsa

using namespace dsa;

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Resolve and check a row store.  width = row width in elements.
dsa_status_t resolve_rows(const dsa_rows_t* r, int B, int max_kv_len, int width, RowStore* out) {
  if (r == nullptr || r->base == nullptr || !aligned(r->base, 16)) return DSA_ERR_INVALID_ARGUMENT;
  RowStore s{};
  s.base = static_cast<const uint16_t*>(r->base);
  if (r->block_table == nullptr) {
    if (r->seq_stride < max_kv_len) return DSA_ERR_INVALID_ARGUMENT;
    s.seq_stride = r->seq_stride;
    s.total_rows = static_cast<int64_t>(B) * r->seq_stride;
  } else {
    if (r->page_size != kPage) return DSA_ERR_UNSUPPORTED;
    if (r->num_pages <= 0 || r->max_pages <= 0) return DSA_ERR_INVALID_ARGUMENT;
    if (static_cast<int64_t>(r->max_pages) * kPage < max_kv_len) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(r->block_table, 4)) return DSA_ERR_INVALID_ARGUMENT;
    s.block_table = r->block_table;
    s.max_pages = r->max_pages;
    s.num_pages = r->num_pages;
    s.total_rows = static_cast<int64_t>(r->num_pages) * kPage;
  }
  if (s.total_rows >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
  (void)width;
  *out = s;
  return DSA_OK;
}

dsa_status_t check_ws(void* ws, size_t bytes, size_t need) {
  if (ws == nullptr || !aligned(ws, 256)) return DSA_ERR_INVALID_ARGUMENT;
  if (bytes < need) return DSA_ERR_WORKSPACE_TOO_SMALL;
  return DSA_OK;
}

}  // namespace

extern "C" {

int dsa_abi_version(void) { return 1; }

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case DSA_ERR_BAD_INDEX: return "index, page id or length out of range";
    case DSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
  }
  return "unknown status";
}

size_t dsa_workspace_bytes(dsa_op_t op, int B, int Tq, int max_kv_len, int heads, int topk) {
  size_t extra = 0;
  if (B > 0 && Tq > 0) {
    if (op == DSA_OP_INDEXER_TOPK) extra = indexer_scratch_bytes(B, Tq, max_kv_len, heads, topk);
    if (op == DSA_OP_SPARSE_MLA) extra = sparse_mla_scratch_bytes(B, Tq, heads, topk);
    if (op == DSA_OP_SPARSE_MLA_BWD && heads == 96 && topk > 0) {
      // P and dZ of up to 512 queries at a time for the tensor-core kernels
      const int64_t nq = static_cast<int64_t>(B) * Tq;
      extra = static_cast<size_t>(nq < 512 ? nq : 512) * sparse_mla_bwd_tc_query_bytes(topk);
    }
  }
  return kWorkspaceHeader + ((extra + 255) / 256) * 256;
}

dsa_status_t dsa_workspace_init(void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  if (workspace == nullptr || ws_bytes < kWorkspaceHeader || !aligned(workspace, 256))
    return DSA_ERR_INVALID_ARGUMENT;
  return cudaMemsetAsync(workspace, 0, kWorkspaceHeader, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}

dsa_status_t dsa_read_device_status(void* workspace, dsa_stream_t stream, uint32_t* where,
                                    uint32_t* detail) {
  if (workspace == nullptr || !aligned(workspace, 256)) return DSA_ERR_INVALID_ARGUMENT;
  uint32_t h[3] = {0, 0, 0};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(h, workspace, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof h, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (where) *where = h[1];
  if (detail) *detail = h[2];
  return static_cast<dsa_status_t>(h[0]);
}

static dsa_status_t indexer_topk(const void* q_idx, const float* q_scale, const uint16_t* w,
                                 const dsa_rows_t* k_idx, const float* k_scale,
                                 const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                                 int H_I, int D_I, int max_kv_len, int topk, int32_t* out_idx,
                                 void* workspace, size_t ws_bytes, dsa_stream_t stream, bool fp8) {
  if (!q_idx || !w || !q_start || !kv_len || !out_idx) return DSA_ERR_INVALID_ARGUMENT;
  if (fp8) {
    if (!q_scale || !k_scale || !aligned(q_scale, 4) || !aligned(k_scale, 16))
      return DSA_ERR_INVALID_ARGUMENT;
    if (!(H_I == 64 && D_I == 128)) return DSA_ERR_UNSUPPORTED;
    // contiguous keys: each tile's scales are copied in whole 16-byte units
    if (k_idx != nullptr && k_idx->block_table == nullptr && k_idx->seq_stride % 4 != 0)
      return DSA_ERR_UNSUPPORTED;
  }
  if (!aligned(q_idx, 16) || !aligned(w, 2) || !aligned(out_idx, 4) || !aligned(q_start, 4) ||
      !aligned(kv_len, 4))
    return DSA_ERR_INVALID_ARGUMENT;
  if (B <= 0 || Tq <= 0 || max_kv_len <= 0 || topk <= 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!((H_I == 64 && D_I == 128) || (H_I == 4 && D_I == 64))) return DSA_ERR_UNSUPPORTED;
  if (topk > 2048 || topk % 4 != 0 || topk > indexer_prefill_max_topk(H_I, D_I))
    return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Tq * H_I >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;
  IndexerArgs a{};
  dsa_status_t st = resolve_rows(k_idx, B, max_kv_len, D_I, &a.k);
  if (st != DSA_OK) return st;
  st = check_ws(workspace, ws_bytes,
                dsa_workspace_bytes(DSA_OP_INDEXER_TOPK, B, Tq, max_kv_len, H_I, topk));
  if (st != DSA_OK) return st;
  a.q_idx = static_cast<const uint16_t*>(q_idx);
  a.q_scale = q_scale;
  a.k_scale = k_scale;
  a.fp8 = fp8;
  a.w = w;
  a.q_start = q_start;
  a.kv_len = kv_len;
  a.B = B;
  a.Tq = Tq;
  a.H_I = H_I;
  a.D_I = D_I;
  a.max_kv_len = max_kv_len;
  a.topk = topk;
  a.out_idx = out_idx;
  a.status = static_cast<uint32_t*>(workspace);
  a.scratch = static_cast<uint8_t*>(workspace) + kWorkspaceHeader;
  a.scratch_bytes = ws_bytes - kWorkspaceHeader;
  return indexer_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_indexer_topk(const uint16_t* q_idx, const uint16_t* w, const dsa_rows_t* k_idx,
                              const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                              int H_I, int D_I, int max_kv_len, int topk, int32_t* out_idx,
                              void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  return indexer_topk(q_idx, nullptr, w, k_idx, nullptr, q_start, kv_len, B, Tq, H_I, D_I,
                      max_kv_len, topk, out_idx, workspace, ws_bytes, stream, false);
}

dsa_status_t dsa_indexer_topk_fp8(const uint8_t* q_codes, const float* q_scale, const uint16_t* w,
                                  const dsa_rows_t* k_codes, const float* k_scale,
                                  const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                                  int H_I, int D_I, int max_kv_len, int topk, int32_t* out_idx,
                                  void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  return indexer_topk(q_codes, q_scale, w, k_codes, k_scale, q_start, kv_len, B, Tq, H_I, D_I,
                      max_kv_len, topk, out_idx, workspace, ws_bytes, stream, true);
}

dsa_status_t dsa_quant_fp8(const uint16_t* x, int64_t n_rows, int D, uint8_t* codes, float* scale,
                           dsa_stream_t stream) {
  if (!x || !codes || !scale || n_rows < 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 8) || !aligned(codes, 4) || !aligned(scale, 4)) return DSA_ERR_INVALID_ARGUMENT;
  if (D != 64 && D != 128) return DSA_ERR_UNSUPPORTED;
  if (n_rows >= (int64_t(1) << 36)) return DSA_ERR_UNSUPPORTED;
  if (n_rows == 0) return DSA_OK;
  return quant_fp8_launch(x, n_rows, D, codes, scale, reinterpret_cast<cudaStream_t>(stream));
}

static dsa_status_t mla_fwd(const uint16_t* q_lat, const dsa_rows_t* kv, const int32_t* idx,
                            const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int H,
                            int topk, int max_kv_len, float scale, const float* sink,
                            uint16_t* o_lat, float* lse, void* workspace, size_t ws_bytes,
                            dsa_stream_t stream) {
  if (!q_lat || !idx || !q_start || !kv_len || !o_lat) return DSA_ERR_INVALID_ARGUMENT;
  if (sink != nullptr && !aligned(sink, 4)) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_lat, 16) || !aligned(idx, 4) || !aligned(o_lat, 16) ||
      (lse != nullptr && !aligned(lse, 4)) || !aligned(q_start, 4) || !aligned(kv_len, 4))
    return DSA_ERR_INVALID_ARGUMENT;
  if (B <= 0 || Tq <= 0 || max_kv_len <= 0 || topk <= 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!(scale > 0.f) || scale != scale) return DSA_ERR_INVALID_ARGUMENT;
  if (H != 96 && H != 8) return DSA_ERR_UNSUPPORTED;
  if (topk > 2048) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Tq * H >= (int64_t(1) << 31) ||
      static_cast<int64_t>(B) * Tq >= (int64_t(1) << 31) / 8)
    return DSA_ERR_UNSUPPORTED;
  SparseMlaArgs a{};
  dsa_status_t st = resolve_rows(kv, B, max_kv_len, kRlat, &a.kv);
  if (st != DSA_OK) return st;
  st = check_ws(workspace, ws_bytes, dsa_workspace_bytes(DSA_OP_SPARSE_MLA, B, Tq, max_kv_len, H, topk));
  if (st != DSA_OK) return st;
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
  a.sink = sink;
  a.status = static_cast<uint32_t*>(workspace);
  a.scratch = static_cast<uint8_t*>(workspace) + kWorkspaceHeader;
  a.scratch_bytes = ws_bytes - kWorkspaceHeader;
  return sparse_mla_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dsa_status_t sparse_mla_fwd(const uint16_t* q_lat, const dsa_rows_t* kv, const int32_t* idx,
                            const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int H,
                            int topk, int max_kv_len, float scale, uint16_t* o_lat, float* lse,
                            void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  return mla_fwd(q_lat, kv, idx, q_start, kv_len, B, Tq, H, topk, max_kv_len, scale, nullptr,
                 o_lat, lse, workspace, ws_bytes, stream);
}

dsa_status_t sparse_mla_fwd_sink(const uint16_t* q_lat, const dsa_rows_t* kv, const int32_t* idx,
                                 const int32_t* q_start, const int32_t* kv_len, int B, int Tq,
                                 int H, int topk, int max_kv_len, float scale, const float* sink,
                                 uint16_t* o_lat, float* lse, void* workspace, size_t ws_bytes,
                                 dsa_stream_t stream) {
  if (sink == nullptr) return DSA_ERR_INVALID_ARGUMENT;
  return mla_fwd(q_lat, kv, idx, q_start, kv_len, B, Tq, H, topk, max_kv_len, scale, sink, o_lat,
                 lse, workspace, ws_bytes, stream);
}

dsa_status_t sparse_mla_bwd(const uint16_t* q_lat, const dsa_rows_t* kv, const int32_t* idx,
                            const int32_t* q_start, const int32_t* kv_len, int B, int Tq, int H,
                            int topk, int max_kv_len, float scale, const uint16_t* o_lat,
                            const float* lse, const uint16_t* d_o, float* dq, float* dkv,
                            void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  if (!q_lat || !idx || !q_start || !kv_len || !o_lat || !lse || !d_o || !dq || !dkv)
    return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(q_lat, 16) || !aligned(idx, 4) || !aligned(q_start, 4) || !aligned(kv_len, 4) ||
      !aligned(o_lat, 4) || !aligned(lse, 4) || !aligned(d_o, 4) || !aligned(dq, 4) ||
      !aligned(dkv, 16))
    return DSA_ERR_INVALID_ARGUMENT;
  if (B <= 0 || Tq <= 0 || H <= 0 || topk <= 0 || max_kv_len <= 0) return DSA_ERR_INVALID_ARGUMENT;
  if (!(scale > 0.f) || scale != scale) return DSA_ERR_INVALID_ARGUMENT;
  if (H > 128 || topk > 2048) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Tq * ((H + 15) / 16) >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;
  SparseMlaBwdArgs a{};
  dsa_status_t st = resolve_rows(kv, B, max_kv_len, kRlat, &a.kv);
  if (st != DSA_OK) return st;
  // the status header is required; a workspace as large as dsa_workspace_bytes
  // reports (96 heads) selects the tensor-core kernels
  st = check_ws(workspace, ws_bytes, kWorkspaceHeader);
  if (st != DSA_OK) return st;
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
  a.d_o = d_o;
  a.dq = dq;
  a.dkv = dkv;
  a.status = static_cast<uint32_t*>(workspace);
  a.scratch = static_cast<uint8_t*>(workspace) + kWorkspaceHeader;
  a.scratch_bytes = ws_bytes - kWorkspaceHeader;
  return sparse_mla_bwd_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dsa_status_t mla_gate_apply(const uint16_t* x, const uint16_t* W_g, const uint16_t* o_lat,
                            const uint16_t* W_uv, int N, int hid, int H, int dv, uint16_t* out,
                            void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  if (!x || !W_g || !o_lat || !W_uv || !out) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(W_g, 16) || !aligned(o_lat, 16) || !aligned(W_uv, 16) ||
      !aligned(out, 16))
    return DSA_ERR_INVALID_ARGUMENT;
  if (N <= 0 || hid <= 0 || H <= 0 || dv <= 0) return DSA_ERR_INVALID_ARGUMENT;
  if (dv != 128 || hid % 64 != 0 || H % 2 != 0) return DSA_ERR_UNSUPPORTED;
  dsa_status_t st = check_ws(workspace, ws_bytes, dsa_workspace_bytes(DSA_OP_GATE, N, 1, 0, H, 0));
  if (st != DSA_OK) return st;
  GateArgs a{x, W_g, o_lat, W_uv, N, hid, H, dv, out, static_cast<uint32_t*>(workspace)};
  return gate_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

static dsa_status_t cache_append(const float* k_pre, const uint16_t* kv_new,
                                 const dsa_rows_t* k_cache, float* k_scale,
                                 const dsa_rows_t* kv_cache, const int32_t* q_start, int B,
                                 int Tq, int D_I, float eps, void* workspace, size_t ws_bytes,
                                 dsa_stream_t stream) {
  if (!k_pre || !kv_new || !q_start) return DSA_ERR_INVALID_ARGUMENT;
  if (k_scale != nullptr && !aligned(k_scale, 4)) return DSA_ERR_INVALID_ARGUMENT;
  if (!aligned(k_pre, 16) || !aligned(kv_new, 16) || !aligned(q_start, 4))
    return DSA_ERR_INVALID_ARGUMENT;
  if (B <= 0 || Tq <= 0 || !(eps >= 0.f) || !(eps < 3.0e38f)) return DSA_ERR_INVALID_ARGUMENT;
  if (D_I != 64 && D_I != 128) return DSA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * Tq >= (int64_t(1) << 31)) return DSA_ERR_UNSUPPORTED;
  AppendArgs a{};
  // positions live on the device: only the structure is checked here, each
  // row's existence on the device
  dsa_status_t st = resolve_rows(k_cache, B, 0, D_I, &a.k_cache);
  if (st != DSA_OK) return st;
  st = resolve_rows(kv_cache, B, 0, kRlat, &a.kv_cache);
  if (st != DSA_OK) return st;
  st = check_ws(workspace, ws_bytes, dsa_workspace_bytes(DSA_OP_CACHE_APPEND, B, Tq, 0, 0, 0));
  if (st != DSA_OK) return st;
  a.k_pre = k_pre;
  a.kv_new = kv_new;
  a.q_start = q_start;
  a.B = B;
  a.Tq = Tq;
  a.D_I = D_I;
  a.eps = eps;
  a.k_scale = k_scale;
  a.status = static_cast<uint32_t*>(workspace);
  return cache_append_launch(a, reinterpret_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_cache_append(const float* k_pre, const uint16_t* kv_new,
                              const dsa_rows_t* k_cache, const dsa_rows_t* kv_cache,
                              const int32_t* q_start, int B, int Tq, int D_I, float eps,
                              void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  return cache_append(k_pre, kv_new, k_cache, nullptr, kv_cache, q_start, B, Tq, D_I, eps,
                      workspace, ws_bytes, stream);
}

dsa_status_t dsa_cache_append_fp8(const float* k_pre, const uint16_t* kv_new,
                                  const dsa_rows_t* k_codes, float* k_scale,
                                  const dsa_rows_t* kv_cache, const int32_t* q_start, int B,
                                  int Tq, int D_I, float eps, void* workspace, size_t ws_bytes,
                                  dsa_stream_t stream) {
  if (k_scale == nullptr) return DSA_ERR_INVALID_ARGUMENT;
  return cache_append(k_pre, kv_new, k_codes, k_scale, kv_cache, q_start, B, Tq, D_I, eps,
                      workspace, ws_bytes, stream);
}

}  // extern "C"
