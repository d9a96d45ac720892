// cache_append.cu -- the step before the indexer on sm_103a: LayerNorm of the
// new tokens' indexer keys and their append, with the new latent rows, to the
// key and latent caches ("Kimi K3.1 Pro" archdiff blueprint: LayerNorm on the
// indexer key, unit gain and zero bias; eps = KimiK3TextConfig rms_norm_eps).
//
//   k_cache[row(b, q_start[b]+i)] = BF16((x - mean x) / sqrt(var x + eps)),  x = k_pre[b,i,:]
//   kv_cache[row(b, q_start[b]+i)] = kv_new[b,i,:]
//
// One warp per new token.  The key row (D_I FP32 values) is held in registers,
// 4 (D_I = 128) or 2 (D_I = 64) per lane; mean and population variance come
// from two warp reductions (variance of the centred values, so no cancellation
// between sum of squares and squared mean), FP32 throughout, then one
// round-to-nearest-even per element.  The 1,152-byte latent row is copied with
// 16-byte loads and stores.  HBM-bound: per token D_I*4 + 1152 bytes read and
// D_I*2 + 1152 written; no shared memory, no tensor work.
//
// FP8 variant ("Kimi-K3.1-Pro", NeMo AutoModel, Implementation Limits,
// bullet 2 sets the BF16 indexer against the FP8 indexer of some serving
// kernels): the key row is written as E4M3 codes plus one FP32 scale, the
// quantisation of exactly the BF16 row the BF16 variant writes:
//   scale = max(amax, 2^-100) / 448,  code = E4M3(x * (1 / scale))
// with the division, reciprocal and product each one IEEE float operation
// rounded to nearest (__fdiv_rn, __frcp_rn, __fmul_rn), and the E4M3 rounding
// to nearest even, saturating, done by the hardware conversion.  The same
// quantiser (quant_fp8_kernel) turns the BF16 indexer queries into codes.
#include <cuda_bf16.h>

#include "dsa_status.cuh"
#include "internal.h"
#include "sm103.cuh"

namespace dsa {
namespace app {

constexpr int WARPS = 8;
enum : uint32_t { SITE_KROW = 0x600, SITE_VROW = 0x601 };

struct Params {
  const float* k_pre;
  const uint16_t* kv_new;
  void* k_base;       // BF16 rows, or E4M3 code rows (FP8 variant)
  float* k_scale;     // FP8 variant: one scale per key row, same row numbering
  uint16_t* kv_base;
  const int32_t* k_bt;
  const int32_t* kv_bt;
  int64_t k_stride, kv_stride;  // contiguous rows per sequence
  int32_t k_max_pages, k_num_pages, kv_max_pages, kv_num_pages;
  const int32_t* q_start;
  int B, Tq;
  float eps;
  uint32_t* status;
};

// Physical row of position pos of sequence b, or -1 if the store has no such row.
__device__ __forceinline__ int64_t store_row(const int32_t* bt, int64_t stride, int32_t max_pages,
                                             int32_t num_pages, int b, int pos) {
  if (pos < 0) return -1;
  if (bt == nullptr) return pos < stride ? static_cast<int64_t>(b) * stride + pos : -1;
  const int pg = pos >> 6;
  if (pg >= max_pages) return -1;
  const int pid = __ldg(bt + static_cast<int64_t>(b) * max_pages + pg);
  if (pid < 0 || pid >= num_pages) return -1;
  return static_cast<int64_t>(pid) * kPage + (pos & (kPage - 1));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// E4M3 codes of one D = 32 * PER wide row whose lane l holds elements
// l*PER .. l*PER+PER-1 in x (the values of BF16 numbers).  Returns the row's
// scale; `packed` receives the lane's PER codes, element l*PER+e in byte e.
template <int PER>
__device__ __forceinline__ float quant_row_e4m3(const float (&x)[PER], uint32_t& packed) {
  float a = 0.f;
#pragma unroll
  for (int e = 0; e < PER; ++e) a = fmaxf(a, fabsf(x[e]));
  // non-negative floats order like their bit patterns
  const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(a)));
  const float scale = __fdiv_rn(fmaxf(amax, 0x1p-100f), 448.f);
  const float inv = __frcp_rn(scale);
  if constexpr (PER == 4) {
    packed = e4m3x2(__fmul_rn(x[1], inv), __fmul_rn(x[0], inv)) |
             (e4m3x2(__fmul_rn(x[3], inv), __fmul_rn(x[2], inv)) << 16);
  } else {
    packed = e4m3x2(__fmul_rn(x[1], inv), __fmul_rn(x[0], inv));
  }
  return scale;
}

// BF16 rows [n, D] -> E4M3 codes [n, D] and scales [n]; one warp per row.
template <int D>
__global__ void __launch_bounds__(WARPS * 32)
    quant_fp8_kernel(const uint16_t* __restrict__ x, int64_t n, uint8_t* __restrict__ codes,
                     float* __restrict__ scale) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  if (row >= n) return;
  float v[PER];
  const uint16_t* src = x + row * D + lane * PER;
  if constexpr (PER == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(src));
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(src));
    v[0] = __uint_as_float(u << 16);
    v[1] = __uint_as_float(u & 0xffff0000u);
  }
  uint32_t packed;
  const float sc = quant_row_e4m3<PER>(v, packed);
  if constexpr (PER == 4)
    *reinterpret_cast<uint32_t*>(codes + row * D + lane * PER) = packed;
  else
    *reinterpret_cast<uint16_t*>(codes + row * D + lane * PER) = static_cast<uint16_t>(packed);
  if (lane == 0) scale[row] = sc;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(WARPS * 32) cache_append_kernel(const Params p) {
  constexpr int PER = D / 32;  // key values per lane (4 or 2)
  const int lane = threadIdx.x & 31;
  const int64_t tok = static_cast<int64_t>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  if (tok >= static_cast<int64_t>(p.B) * p.Tq) return;
  const int b = static_cast<int>(tok / p.Tq), i = static_cast<int>(tok % p.Tq);
  const int pos = __ldg(p.q_start + b) + i;

  // ---- indexer key: LayerNorm, BF16 ----
  const int64_t krow = store_row(p.k_bt, p.k_stride, p.k_max_pages, p.k_num_pages, b, pos);
  if (krow < 0) {
    if (lane == 0) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_KROW, static_cast<uint32_t>(pos));
  } else {
    float x[PER];
    const float* src = p.k_pre + tok * D + lane * PER;
    if constexpr (PER == 4) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src));
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
      const float2 v = __ldg(reinterpret_cast<const float2*>(src));
      x[0] = v.x; x[1] = v.y;
    }
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) s += x[e];
    const float mean = warp_sum(s) / static_cast<float>(D);
    float q = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      x[e] -= mean;
      q = fmaf(x[e], x[e], q);
    }
    const float var = warp_sum(q) / static_cast<float>(D);
    const float inv = 1.f / sqrtf(var + p.eps);
    uint32_t w[PER / 2];
#pragma unroll
    for (int e = 0; e < PER / 2; ++e) {
      const __nv_bfloat16 lo = __float2bfloat16_rn(x[2 * e] * inv);
      const __nv_bfloat16 hi = __float2bfloat16_rn(x[2 * e + 1] * inv);
      w[e] = static_cast<uint32_t>(__bfloat16_as_ushort(lo)) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
    }
    if constexpr (FP8) {
      // quantise the BF16 row just formed
      float v[PER];
#pragma unroll
      for (int e = 0; e < PER / 2; ++e) {
        v[2 * e] = __uint_as_float(w[e] << 16);
        v[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
      }
      uint32_t packed;
      const float sc = quant_row_e4m3<PER>(v, packed);
      uint8_t* dst = static_cast<uint8_t*>(p.k_base) + krow * D + lane * PER;
      if constexpr (PER == 4)
        *reinterpret_cast<uint32_t*>(dst) = packed;
      else
        *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
      if (lane == 0) p.k_scale[krow] = sc;
    } else {
      uint16_t* dst = static_cast<uint16_t*>(p.k_base) + krow * D + lane * PER;
      if constexpr (PER == 4)
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
      else
        *reinterpret_cast<uint32_t*>(dst) = w[0];
    }
  }

  // ---- latent row: copied as is ----
  const int64_t vrow = store_row(p.kv_bt, p.kv_stride, p.kv_max_pages, p.kv_num_pages, b, pos);
  if (vrow < 0) {
    if (lane == 0) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_VROW, static_cast<uint32_t>(pos));
    return;
  }
  constexpr int UNITS = kRlat * 2 / 16;  // 72 x 16 bytes
  const uint4* vs = reinterpret_cast<const uint4*>(p.kv_new + tok * kRlat);
  uint4* vd = reinterpret_cast<uint4*>(p.kv_base + vrow * kRlat);
#pragma unroll
  for (int u = lane; u < UNITS; u += 32) vd[u] = __ldg(vs + u);
}

}  // namespace app

dsa_status_t cache_append_launch(const AppendArgs& a, cudaStream_t stream) {
  app::Params p{};
  p.k_pre = a.k_pre;
  p.kv_new = a.kv_new;
  p.k_base = const_cast<uint16_t*>(a.k_cache.base);
  p.k_scale = a.k_scale;
  p.kv_base = const_cast<uint16_t*>(a.kv_cache.base);
  p.k_bt = a.k_cache.block_table;
  p.kv_bt = a.kv_cache.block_table;
  p.k_stride = a.k_cache.seq_stride;
  p.kv_stride = a.kv_cache.seq_stride;
  p.k_max_pages = a.k_cache.max_pages;
  p.k_num_pages = a.k_cache.num_pages;
  p.kv_max_pages = a.kv_cache.max_pages;
  p.kv_num_pages = a.kv_cache.num_pages;
  p.q_start = a.q_start;
  p.B = a.B;
  p.Tq = a.Tq;
  p.eps = a.eps;
  p.status = a.status;
  const int64_t tokens = static_cast<int64_t>(a.B) * a.Tq;
  const unsigned grid = static_cast<unsigned>((tokens + app::WARPS - 1) / app::WARPS);
  const bool fp8 = a.k_scale != nullptr;
  if (a.D_I == 128) {
    if (fp8)
      app::cache_append_kernel<128, true><<<grid, app::WARPS * 32, 0, stream>>>(p);
    else
      app::cache_append_kernel<128, false><<<grid, app::WARPS * 32, 0, stream>>>(p);
  } else {
    if (fp8)
      app::cache_append_kernel<64, true><<<grid, app::WARPS * 32, 0, stream>>>(p);
    else
      app::cache_append_kernel<64, false><<<grid, app::WARPS * 32, 0, stream>>>(p);
  }
  return launch_status("cache_append_kernel");
}

dsa_status_t quant_fp8_launch(const uint16_t* x, int64_t n_rows, int D, uint8_t* codes,
                              float* scale, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>((n_rows + app::WARPS - 1) / app::WARPS);
  if (D == 128)
    app::quant_fp8_kernel<128><<<grid, app::WARPS * 32, 0, stream>>>(x, n_rows, codes, scale);
  else
    app::quant_fp8_kernel<64><<<grid, app::WARPS * 32, 0, stream>>>(x, n_rows, codes, scale);
  return launch_status("quant_fp8_kernel");
}

}  // namespace dsa
