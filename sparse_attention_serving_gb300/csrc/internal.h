// internal.h -- host-side launch interfaces shared between the C ABI layer and
// the kernel files.  Everything here is C++ and not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kRlat = 576;  // latent row: 512 c_kv + 64 unrotated k_pe
constexpr int kVlat = 512;  // value width
constexpr int kPage = 64;   // tokens per cache page

// A resolved row store as the kernels see it (physical row r lives at
// base + r * width elements).
struct RowStore {
  const uint16_t* base;
  int64_t seq_stride;          // contiguous: rows per sequence
  const int32_t* block_table;  // paged when non-null
  int32_t max_pages;
  int32_t num_pages;
  int64_t total_rows;          // rows addressable through the tensor map
};

// Encode a 2D BF16 tensor map [rows, cols] with a {box_cols, box_rows} box and
// 128-byte swizzle.  Returns false on failure.
bool encode_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows,
                    bool swizzle128);

// --- sparse MLA ---------------------------------------------------------------
struct SparseMlaArgs {
  const uint16_t* q_lat;
  RowStore kv;
  const int32_t* idx;
  const int32_t* q_start;
  const int32_t* kv_len;
  int B, Tq, H, topk, max_kv_len;
  float scale;
  uint16_t* o_lat;
  float* lse;
  const float* sink;   // [H] learnable sink logits (natural log), or null
  uint32_t* status;
  void* scratch;       // split partials (decode); may be null when nsplit == 1
  size_t scratch_bytes;
};
size_t sparse_mla_scratch_bytes(int B, int Tq, int H, int topk);
dsa_status_t sparse_mla_launch(const SparseMlaArgs& a, cudaStream_t stream);

// --- sparse MLA backward ----------------------------------------------------------
struct SparseMlaBwdArgs {
  const uint16_t* q_lat;
  RowStore kv;
  const int32_t* idx;
  const int32_t* q_start;
  const int32_t* kv_len;
  int B, Tq, H, topk, max_kv_len;
  float scale;
  const uint16_t* o_lat;
  const float* lse;
  const uint16_t* d_o;
  float* dq;
  float* dkv;        // FP32 rows numbered like kv's rows (accumulated into)
  uint32_t* status;
  void* scratch;     // P and dZ of a chunk of queries (tensor-core path), or null
  size_t scratch_bytes;
};
dsa_status_t sparse_mla_bwd_launch(const SparseMlaBwdArgs& a, cudaStream_t stream);
// The tcgen05 path (H = 96): P and dZ scratch bytes per query, and the launch.
size_t sparse_mla_bwd_tc_query_bytes(int topk);
dsa_status_t sparse_mla_bwd_tc_launch(const SparseMlaBwdArgs& a, void* scratch, size_t scratch_bytes,
                                      cudaStream_t stream);

// --- indexer + top-k --------------------------------------------------------------
struct IndexerArgs {
  const uint16_t* q_idx;       // BF16 queries, or E4M3 codes when fp8
  const float* q_scale;        // fp8: [B, Tq, H_I]
  const float* k_scale;        // fp8: one per key row, numbered like k's rows
  bool fp8;
  const uint16_t* w;
  RowStore k;
  const int32_t* q_start;
  const int32_t* kv_len;
  int B, Tq, H_I, D_I, max_kv_len, topk;
  int32_t* out_idx;
  uint32_t* status;
  void* scratch;
  size_t scratch_bytes;
};
size_t indexer_scratch_bytes(int B, int Tq, int max_kv_len, int H_I, int topk);
dsa_status_t indexer_launch(const IndexerArgs& a, cudaStream_t stream);

// --- gate -------------------------------------------------------------------------
struct GateArgs {
  const uint16_t* x;
  const uint16_t* W_g;
  const uint16_t* o_lat;
  const uint16_t* W_uv;
  int N, hid, H, dv;
  uint16_t* out;
  uint32_t* status;
};
dsa_status_t gate_launch(const GateArgs& a, cudaStream_t stream);

// --- cache append (indexer-key LayerNorm + latent row copy) -----------------------
struct AppendArgs {
  const float* k_pre;
  const uint16_t* kv_new;
  RowStore k_cache;   // written through (base is cast to non-const)
  RowStore kv_cache;
  const int32_t* q_start;
  int B, Tq, D_I;
  float eps;
  float* k_scale;     // non-null: FP8 variant (k_cache holds E4M3 code rows)
  uint32_t* status;
};
dsa_status_t cache_append_launch(const AppendArgs& a, cudaStream_t stream);
// BF16 rows [n_rows, D] -> E4M3 codes + one FP32 scale per row (D in {64, 128}).
dsa_status_t quant_fp8_launch(const uint16_t* x, int64_t n_rows, int D, uint8_t* codes,
                              float* scale, cudaStream_t stream);

int num_sms();

// DSA_ERR_CUDA when the last launch failed (the CUDA error text goes to stderr
// when the environment variable DSA_VERBOSE is set), else DSA_OK.
dsa_status_t launch_status(const char* what);

}  // namespace dsa
