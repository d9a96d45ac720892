// sparse_mla_bwd.cu -- backward of the latent-space sparse MLA on sm_103a
// ("Kimi-K3.1-Pro", NeMo AutoModel, Implementation Limits: attention over the
// selected rows only (bullets 1-2), a native 96-head backward (the paragraph
// after bullet 4), and no gradient into the indexer (bullet 3): the index set
// is a constant here).
//
// Per query row and head, over the selected positions s_j (the forward's
// lse and o_lat are inputs, as in training):
//   p_j  = exp(scale * q . kv[s_j] - lse)
//   dp_j = dO . kv[s_j, 0:512],   D = dO . o_lat
//   dz_j = p_j (dp_j - D)
//   dq   = scale * sum_j dz_j kv[s_j, 0:576]
//   dkv[s_j, 0:576] += scale * dz_j q,   dkv[s_j, 0:512] += p_j dO
//
// First version, on the CUDA cores in FP32 (not the tensor cores), in two
// kernels that walk the selected keys in blocks of 32 rows gathered into
// shared memory:
//   bwd_dq_kernel   one CTA per (query row, group of 16 heads): the group's q,
//                   dO and dq rows live in shared memory; dq is written once.
//   bwd_dkv_kernel  one CTA per query row: for each key block the gradient of
//                   the 32 rows is summed over all heads (groups of 16 in
//                   turn) in registers, then added to the FP32 dkv rows with
//                   16-byte vector atomics (rows are shared by the many queries
//                   that selected them, so the order of the additions, and the
//                   FP32 rounding of dkv, vary from run to run).
// Shared-memory rows use a stride of 289 words, so 32 lanes reading the same
// dim of 32 different rows hit 32 different banks.
#include <cuda_bf16.h>

#include "dsa_status.cuh"
#include "internal.h"

namespace dsa {
namespace mlab {

constexpr int KB = 32;         // keys per block
constexpr int HG = 16;         // heads per group
constexpr int NT = 256;        // threads per CTA
constexpr int KW = 289;        // shared-memory words per gathered row (576 BF16 + 2 pad)
constexpr int QW = kRlat + 4;  // floats per staged q row (pad: keeps float4 alignment)

enum : uint32_t { SITE_IDX = 0x700, SITE_PAGE = 0x701, SITE_QPOS = 0x702 };

struct Params {
  const uint16_t* q;      // [nq, H, 576]
  const uint16_t* kv;     // rows of 576
  const int32_t* idx;     // [nq, topk]
  const int32_t* q_start;
  const int32_t* kv_len;
  const int32_t* block_table;
  int64_t seq_stride;
  int32_t max_pages, num_pages;
  int paged;
  int Tq, H, topk, max_kv_len;
  float scale, scale_log2;
  const uint16_t* o;      // [nq, H, 512]
  const float* lse;       // [nq, H] natural log
  const uint16_t* dO;     // [nq, H, 512]
  float* dq;              // [nq, H, 576]
  float* dkv;             // rows of 576 (FP32), numbered like kv's rows
  uint32_t* status;
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Physical row of the key at position s of sequence b, or -1 (recorded once,
// by the lane that reads the entry, when it is neither -1 nor valid).
__device__ __forceinline__ int64_t key_row(const Params& p, int b, int t, int L, int s, bool report) {
  if (s < 0) return -1;
  if (s > t || s >= L) {
    if (report) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_IDX, static_cast<uint32_t>(s));
    return -1;
  }
  if (!p.paged) return static_cast<int64_t>(b) * p.seq_stride + s;
  const int pg = s >> 6;
  const int pid = pg < p.max_pages ? __ldg(p.block_table + static_cast<int64_t>(b) * p.max_pages + pg) : -1;
  if (pid < 0 || pid >= p.num_pages) {
    if (report) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_PAGE, static_cast<uint32_t>(pid));
    return -1;
  }
  return static_cast<int64_t>(pid) * kPage + (s & (kPage - 1));
}

// The query position of flat row qf, or -1 when q_start / kv_len are inconsistent.
__device__ __forceinline__ int query_pos(const Params& p, int64_t qf, int& b, int& L) {
  b = static_cast<int>(qf / p.Tq);
  const int i = static_cast<int>(qf % p.Tq);
  const int t = __ldg(p.q_start + b) + i;
  L = __ldg(p.kv_len + b);
  if (t < 0 || t >= L || L > p.max_kv_len) return -1;
  return t;
}

// Gather key block kb of query row qf: rows[] (physical row or -1) and the
// 576 BF16 values of each valid row into ks (stride KW words; zeros for the
// rest).
__device__ __forceinline__ void gather_block(const Params& p, int64_t qf, int b, int t, int L,
                                             int kb, int64_t* rows, uint32_t* ks, bool report) {
  const int tid = threadIdx.x;
  if (tid < KB) {
    const int j = kb * KB + tid;
    const int s = j < p.topk ? __ldg(p.idx + qf * p.topk + j) : -1;
    rows[tid] = key_row(p, b, t, L, s, report);
  }
  __syncthreads();
  // 32 rows x 72 16-byte units, stored as 32-bit words at the padded stride
  for (int e = tid; e < KB * 72; e += NT) {
    const int j = e / 72, u = e % 72;
    const int64_t r = rows[j];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r >= 0) v = __ldg(reinterpret_cast<const uint4*>(p.kv + r * kRlat) + u);
    uint32_t* d = ks + j * KW + u * 4;
    d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
  }
  __syncthreads();
}

// Stage the q and dO rows of heads h0 .. h0+HG-1 of query row qf as FP32
// (heads past H are zero).
__device__ __forceinline__ void stage_group(const Params& p, int64_t qf, int h0, float* qs,
                                            float* ds) {
  for (int e = threadIdx.x; e < HG * (kRlat / 2); e += NT) {
    const int h = e / (kRlat / 2), w = e % (kRlat / 2);
    uint32_t v = 0u;
    if (h0 + h < p.H)
      v = __ldg(reinterpret_cast<const uint32_t*>(p.q + (qf * p.H + h0 + h) * kRlat) + w);
    qs[h * QW + 2 * w] = bf_lo(v);
    qs[h * QW + 2 * w + 1] = bf_hi(v);
  }
  for (int e = threadIdx.x; e < HG * (kVlat / 2); e += NT) {
    const int h = e / (kVlat / 2), w = e % (kVlat / 2);
    uint32_t v = 0u;
    if (h0 + h < p.H)
      v = __ldg(reinterpret_cast<const uint32_t*>(p.dO + (qf * p.H + h0 + h) * kVlat) + w);
    ds[h * kVlat + 2 * w] = bf_lo(v);
    ds[h * kVlat + 2 * w + 1] = bf_hi(v);
  }
}

// D = dO . o_lat and lse in log2 units for heads h0 .. h0+n-1: one warp per head.
__device__ __forceinline__ void head_stats(const Params& p, int64_t qf, int h0, int n, float* Dh,
                                           float* lse2) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int h = warp; h < n; h += NT / 32) {
    const uint32_t* g = reinterpret_cast<const uint32_t*>(p.dO + (qf * p.H + h0 + h) * kVlat);
    const uint32_t* o = reinterpret_cast<const uint32_t*>(p.o + (qf * p.H + h0 + h) * kVlat);
    float acc = 0.f;
    for (int w = lane; w < kVlat / 2; w += 32) {
      const uint32_t a = __ldg(g + w), c = __ldg(o + w);
      acc = fmaf(bf_lo(a), bf_lo(c), acc);
      acc = fmaf(bf_hi(a), bf_hi(c), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      Dh[h] = acc;
      lse2[h] = __ldg(p.lse + qf * p.H + h0 + h) * 1.4426950408889634f;
    }
  }
}

// Probabilities and scaled logit gradients of the block for the staged head
// group: pz[0][h][j] = p, pz[1][h][j] = scale * dz (0 for invalid keys and
// heads past H).  Thread = (key j = lane, heads warp and warp + 8).
__device__ __forceinline__ void block_grads(const Params& p, const uint32_t* ks, const float* qs,
                                            const float* ds, const float* Dh, const float* lse2,
                                            const int64_t* rows, int h0, float* pz) {
  const int warp = threadIdx.x >> 5, j = threadIdx.x & 31;
  const uint32_t* kr = ks + j * KW;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int h = warp + 8 * hh;
    const float* qh = qs + h * QW;
    const float* dh = ds + h * kVlat;
    float z0 = 0.f, z1 = 0.f, d0 = 0.f, d1 = 0.f;
#pragma unroll 4
    for (int w = 0; w < kVlat / 2; ++w) {
      const uint32_t kw = kr[w];
      const float k0 = bf_lo(kw), k1 = bf_hi(kw);
      z0 = fmaf(qh[2 * w], k0, z0);
      z1 = fmaf(qh[2 * w + 1], k1, z1);
      d0 = fmaf(dh[2 * w], k0, d0);
      d1 = fmaf(dh[2 * w + 1], k1, d1);
    }
#pragma unroll 4
    for (int w = kVlat / 2; w < kRlat / 2; ++w) {
      const uint32_t kw = kr[w];
      z0 = fmaf(qh[2 * w], bf_lo(kw), z0);
      z1 = fmaf(qh[2 * w + 1], bf_hi(kw), z1);
    }
    float pr = 0.f, dz = 0.f;
    if (rows[j] >= 0 && h0 + h < p.H) {
      pr = exp2f((z0 + z1) * p.scale_log2 - lse2[h]);
      dz = pr * ((d0 + d1) - Dh[h]) * p.scale;
    }
    pz[h * KB + j] = pr;
    pz[HG * KB + h * KB + j] = dz;
  }
}

// ---------------------------------------------------------------------------
// dq: one CTA per (query row, head group)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 1) bwd_dq_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t sm[];
  uint32_t* ks = reinterpret_cast<uint32_t*>(sm);                  // [KB][KW]
  float* qs = reinterpret_cast<float*>(ks + KB * KW);               // [HG][QW]
  float* ds = qs + HG * QW;                                         // [HG][512]
  float* dqs = ds + HG * kVlat;                                     // [HG][QW]
  float* pz = dqs + HG * QW;                                        // [2][HG][KB]
  float* Dh = pz + 2 * HG * KB;                                     // [HG]
  float* lse2 = Dh + HG;                                            // [HG]
  int64_t* rows = reinterpret_cast<int64_t*>(lse2 + HG);            // [KB]

  const int ngrp = (p.H + HG - 1) / HG;
  const int64_t qf = blockIdx.x / ngrp;
  const int h0 = static_cast<int>(blockIdx.x % ngrp) * HG;
  const int nh = min(HG, p.H - h0);
  const int tid = threadIdx.x;
  int b, L;
  const int t = query_pos(p, qf, b, L);
  if (t < 0) {
    if (tid == 0 && h0 == 0) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_QPOS, static_cast<uint32_t>(qf));
    for (int e = tid; e < nh * kRlat; e += NT) p.dq[(qf * p.H + h0) * kRlat + e] = 0.f;
    return;
  }
  stage_group(p, qf, h0, qs, ds);
  for (int e = tid; e < HG * QW; e += NT) dqs[e] = 0.f;
  if (tid < HG) { Dh[tid] = 0.f; lse2[tid] = 0.f; }
  __syncthreads();
  head_stats(p, qf, h0, nh, Dh, lse2);
  // thread -> (head h = tid / 16, 36 consecutive dims from (tid % 16) * 36)
  const int hq = tid >> 4, d0 = (tid & 15) * 36;
  const int nkb = (p.topk + KB - 1) / KB;
  for (int kb = 0; kb < nkb; ++kb) {
    gather_block(p, qf, b, t, L, kb, rows, ks, h0 == 0);
    block_grads(p, ks, qs, ds, Dh, lse2, rows, h0, pz);
    __syncthreads();
    float acc[36];
#pragma unroll
    for (int e = 0; e < 36; ++e) acc[e] = 0.f;
    const float* dzh = pz + HG * KB + hq * KB;
#pragma unroll 2
    for (int j = 0; j < KB; ++j) {
      const float w = dzh[j];
      const uint32_t* kr = ks + j * KW + d0 / 2;
#pragma unroll
      for (int e = 0; e < 18; ++e) {
        const uint32_t kw = kr[e];
        acc[2 * e] = fmaf(w, bf_lo(kw), acc[2 * e]);
        acc[2 * e + 1] = fmaf(w, bf_hi(kw), acc[2 * e + 1]);
      }
    }
#pragma unroll
    for (int e = 0; e < 36; ++e) dqs[hq * QW + d0 + e] += acc[e];
    __syncthreads();
  }
  for (int e = tid; e < nh * kRlat; e += NT) {
    const int h = e / kRlat, d = e % kRlat;
    p.dq[(qf * p.H + h0 + h) * kRlat + d] = dqs[h * QW + d];
  }
}

// ---------------------------------------------------------------------------
// dkv: one CTA per query row, every head group in turn per key block
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 1) bwd_dkv_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t sm[];
  uint32_t* ks = reinterpret_cast<uint32_t*>(sm);                  // [KB][KW]
  float* qs = reinterpret_cast<float*>(ks + KB * KW);               // [HG][QW]
  float* ds = qs + HG * QW;                                         // [HG][512]
  float* pz = ds + HG * kVlat;                                      // [2][HG][KB]
  float* Dh = pz + 2 * HG * KB;                                     // [H rounded up to HG]
  float* lse2 = Dh + 128;                                           // [128]
  int64_t* rows = reinterpret_cast<int64_t*>(lse2 + 128);           // [KB]

  const int64_t qf = blockIdx.x;
  const int tid = threadIdx.x;
  int b, L;
  const int t = query_pos(p, qf, b, L);
  if (t < 0) return;  // flagged by bwd_dq_kernel
  const int ngrp = (p.H + HG - 1) / HG;
  for (int e = tid; e < ngrp * HG; e += NT) { Dh[e] = 0.f; lse2[e] = 0.f; }
  __syncthreads();
  head_stats(p, qf, 0, p.H, Dh, lse2);
  __syncthreads();
  // thread -> (key j = tid / 8, 72 consecutive dims from (tid % 8) * 72)
  const int jk = tid >> 3, d0 = (tid & 7) * 72;
  const int nkb = (p.topk + KB - 1) / KB;
  for (int kb = 0; kb < nkb; ++kb) {
    gather_block(p, qf, b, t, L, kb, rows, ks, false);
    float acc[72];
#pragma unroll
    for (int e = 0; e < 72; ++e) acc[e] = 0.f;
    for (int g = 0; g < ngrp; ++g) {
      stage_group(p, qf, g * HG, qs, ds);
      __syncthreads();
      block_grads(p, ks, qs, ds, Dh + g * HG, lse2 + g * HG, rows, g * HG, pz);
      __syncthreads();
#pragma unroll 1
      for (int h = 0; h < HG; ++h) {
        const float pr = pz[h * KB + jk], dz = pz[HG * KB + h * KB + jk];
        const float* qh = qs + h * QW + d0;
        const float* dh = ds + h * kVlat + d0;
#pragma unroll
        for (int e = 0; e < 72; ++e) {
          float a = fmaf(dz, qh[e], acc[e]);
          if (d0 + e < kVlat) a = fmaf(pr, dh[e], a);
          acc[e] = a;
        }
      }
      __syncthreads();
    }
    // the block's rows: 16-byte vector atomics into the FP32 gradient rows
    const int64_t r = rows[jk];
    if (r >= 0) {
      float4* dst = reinterpret_cast<float4*>(p.dkv + r * kRlat + d0);
#pragma unroll
      for (int e = 0; e < 18; ++e)
        atomicAdd(dst + e, make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]));
    }
    __syncthreads();
  }
}

}  // namespace mlab

dsa_status_t sparse_mla_bwd_launch(const SparseMlaBwdArgs& a, cudaStream_t stream) {
  using namespace mlab;
  Params p{};
  p.q = a.q_lat;
  p.kv = a.kv.base;
  p.idx = a.idx;
  p.q_start = a.q_start;
  p.kv_len = a.kv_len;
  p.block_table = a.kv.block_table;
  p.seq_stride = a.kv.seq_stride;
  p.max_pages = a.kv.max_pages;
  p.num_pages = a.kv.num_pages;
  p.paged = a.kv.block_table != nullptr;
  p.Tq = a.Tq;
  p.H = a.H;
  p.topk = a.topk;
  p.max_kv_len = a.max_kv_len;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.o = a.o_lat;
  p.lse = a.lse;
  p.dO = a.d_o;
  p.dq = a.dq;
  p.dkv = a.dkv;
  p.status = a.status;
  const int64_t nq = static_cast<int64_t>(a.B) * a.Tq;
  const int ngrp = (a.H + HG - 1) / HG;
  const size_t smem_q = KB * KW * 4 + (HG * QW + HG * kVlat + HG * QW + 2 * HG * KB + 2 * HG) * 4 +
                        KB * 8;
  const size_t smem_kv = KB * KW * 4 + (HG * QW + HG * kVlat + 2 * HG * KB + 256) * 4 + KB * 8;
  if (cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_q)) != cudaSuccess ||
      cudaFuncSetAttribute(bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_kv)) != cudaSuccess)
    return launch_status("cudaFuncSetAttribute");
  bwd_dq_kernel<<<static_cast<unsigned>(nq * ngrp), NT, smem_q, stream>>>(p);
  if (launch_status("bwd_dq_kernel") != DSA_OK) return DSA_ERR_CUDA;
  bwd_dkv_kernel<<<static_cast<unsigned>(nq), NT, smem_kv, stream>>>(p);
  return launch_status("bwd_dkv_kernel");
}

}  // namespace dsa
