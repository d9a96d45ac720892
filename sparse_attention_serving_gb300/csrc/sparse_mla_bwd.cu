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
// Two kernels walk each query's selected keys in blocks of 32 rows gathered
// into shared memory and work on 16 heads at a time, so that every operand
// of a head group is small: q 18 KB, dO 16 KB, a key block 36 KB (BF16).
// The five contractions run on the warp-level tensor-core MMA (m16n8k16,
// BF16 in, FP32 accumulate; the fragments are loaded with ldmatrix from rows
// padded by 16 bytes, so eight consecutive rows fall in eight different bank
// groups):
//   S  = q_g . K^T, dP = dO_g . V^T        [16 heads x 32 keys]
//   dq_g += dZ . K                          [16 x 576], in registers
//   dK += dZ^T . q_g, dV += P^T . dO_g      [32 keys x 576], in registers
// with P = exp2(S*scale*log2e - lse2) and dZ = scale * P * (dP - D) formed
// in FP32 and rounded to BF16 for the products (as the forward rounds P).
//   bwd_dq_kernel   one CTA per (query row, head group); dq is written once.
//   bwd_dkv_kernel  one CTA per query row; each key block's gradient is summed
//                   over all head groups in registers and added to the FP32
//                   dkv rows with 8-byte vector atomics (rows are shared by the
//                   many queries that selected them, so the order of the
//                   additions, and the FP32 rounding of dkv, vary run to run).
// The latent rows dims (576) split into 72 tiles of 8; warp w owns tiles
// 9w .. 9w+8 in both accumulation products.
#include <cuda_bf16.h>

#include "dsa_status.cuh"
#include "internal.h"
#include "sm103.cuh"

namespace dsa {
namespace mlab {

constexpr int KB = 32;           // keys per block
constexpr int HG = 16;           // heads per group (the MMA's M)
constexpr int NT = 256;          // threads per CTA (8 warps)
constexpr int KS = kRlat + 8;    // BF16 per staged key / q row (1,168 bytes)
constexpr int DS = kVlat + 8;    // BF16 per staged dO row (1,040 bytes)
constexpr int ZS = KB + 8;       // BF16 per row of P / dZ ([head][key], 80 bytes)
constexpr int SF = KB + 1;       // floats per row of the S / dP scratch

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

// Shared memory of both kernels (bytes are rounded to 16).
struct Smem {
  uint16_t ks[KB * KS];       // gathered key rows
  uint16_t qs[HG * KS];       // the head group's q rows
  uint16_t dsg[HG * DS];      // the head group's dO rows
  uint16_t zs[HG * ZS];       // scale * dz, BF16 [head][key]
  uint16_t ps[HG * ZS];       // p, BF16 [head][key]
  float sf[HG * SF];          // S (then P) scratch
  float df[HG * SF];          // dP scratch
  float Dh[128];              // D = dO . o_lat per head
  float lse2[128];            // lse in log2 units per head
  int64_t rows[KB];           // physical key rows (-1: skipped)
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
// D[16x8] += A[16x16] . B[16x8], BF16 in, FP32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Physical row of the key at position s of sequence b, or -1 (recorded when it
// is neither -1 nor valid and `report` is set).
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

// Gather key block kb of query row qf into sm.ks (zeros for skipped entries).
__device__ __forceinline__ void gather_block(const Params& p, int64_t qf, int b, int t, int L,
                                             int kb, Smem& sm, bool report) {
  const int tid = threadIdx.x;
  if (tid < KB) {
    const int j = kb * KB + tid;
    const int s = j < p.topk ? __ldg(p.idx + qf * p.topk + j) : -1;
    sm.rows[tid] = key_row(p, b, t, L, s, report);
  }
  __syncthreads();
  for (int e = tid; e < KB * 72; e += NT) {
    const int j = e / 72, u = e % 72;
    const int64_t r = sm.rows[j];
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r >= 0) v = __ldg(reinterpret_cast<const uint4*>(p.kv + r * kRlat) + u);
    *reinterpret_cast<uint4*>(sm.ks + j * KS + u * 8) = v;
  }
  __syncthreads();
}

// Stage the q and dO rows of heads h0 .. h0+15 of query row qf (zeros past H).
__device__ __forceinline__ void stage_group(const Params& p, int64_t qf, int h0, Smem& sm) {
  for (int e = threadIdx.x; e < HG * 72; e += NT) {
    const int h = e / 72, u = e % 72;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (h0 + h < p.H) v = __ldg(reinterpret_cast<const uint4*>(p.q + (qf * p.H + h0 + h) * kRlat) + u);
    *reinterpret_cast<uint4*>(sm.qs + h * KS + u * 8) = v;
  }
  for (int e = threadIdx.x; e < HG * 64; e += NT) {
    const int h = e / 64, u = e % 64;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (h0 + h < p.H) v = __ldg(reinterpret_cast<const uint4*>(p.dO + (qf * p.H + h0 + h) * kVlat) + u);
    *reinterpret_cast<uint4*>(sm.dsg + h * DS + u * 8) = v;
  }
}

// D = dO . o_lat and lse in log2 units for heads h0 .. h0+n-1 (into Dh[h0 + h]).
__device__ __forceinline__ void head_stats(const Params& p, int64_t qf, int h0, int n, Smem& sm) {
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
      sm.Dh[h0 + h] = acc;
      sm.lse2[h0 + h] = __ldg(p.lse + qf * p.H + h0 + h) * 1.4426950408889634f;
    }
  }
}

// S = q_g . K^T and dP = dO_g . V^T for the staged head group and key block
// (warps 0-3: S, key tile w; warps 4-7: dP, key tile w-4), then P and
// scale * dZ in FP32, stored as BF16 [head][key] (0 for skipped keys and heads
// past H).  Ends with the block synchronised.
__device__ __forceinline__ void block_pz(const Params& p, Smem& sm, int h0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  {
    const bool is_s = warp < 4;
    const int n0 = 8 * (warp & 3);                 // key tile
    const uint16_t* A = is_s ? sm.qs : sm.dsg;
    const int astride = is_s ? KS : DS;
    const int nk = is_s ? kRlat / 16 : kVlat / 16;  // K-steps: 36 (576 dims) or 32 (512)
    const uint32_t a_base = smem_u32(A + (lane & 15) * astride + 8 * (lane >> 4));
    const uint32_t b_base = smem_u32(sm.ks + (n0 + (lane & 7)) * KS + 8 * ((lane >> 3) & 1));
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int kk = 0; kk < nk; ++kk) {
      uint32_t a0, a1, a2, a3, b0, b1;
      ldsm_x4(a_base + kk * 32, a0, a1, a2, a3);
      ldsm_x2(b_base + kk * 32, b0, b1);
      mma_bf16(d, a0, a1, a2, a3, b0, b1);
    }
    float* out = is_s ? sm.sf : sm.df;
    out[g * SF + n0 + 2 * c] = d[0];
    out[g * SF + n0 + 2 * c + 1] = d[1];
    out[(g + 8) * SF + n0 + 2 * c] = d[2];
    out[(g + 8) * SF + n0 + 2 * c + 1] = d[3];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < HG * KB; e += NT) {
    const int h = e / KB, j = e % KB;
    float pr = 0.f, dz = 0.f;
    if (sm.rows[j] >= 0 && h0 + h < p.H) {
      pr = exp2f(sm.sf[h * SF + j] * p.scale_log2 - sm.lse2[h0 + h]);
      dz = pr * (sm.df[h * SF + j] - sm.Dh[h0 + h]) * p.scale;
    }
    sm.ps[h * ZS + j] = __bfloat16_as_ushort(__float2bfloat16_rn(pr));
    sm.zs[h * ZS + j] = __bfloat16_as_ushort(__float2bfloat16_rn(dz));
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// dq: one CTA per (query row, head group)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 2) bwd_dq_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int ngrp = (p.H + HG - 1) / HG;
  const int64_t qf = blockIdx.x / ngrp;
  const int h0 = static_cast<int>(blockIdx.x % ngrp) * HG;
  const int nh = min(HG, p.H - h0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  int b, L;
  const int t = query_pos(p, qf, b, L);
  if (t < 0) {
    if (tid == 0 && h0 == 0) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_QPOS, static_cast<uint32_t>(qf));
    for (int e = tid; e < nh * kRlat; e += NT) p.dq[(qf * p.H + h0) * kRlat + e] = 0.f;
    return;
  }
  stage_group(p, qf, h0, sm);
  for (int e = tid; e < 128; e += NT) { sm.Dh[e] = 0.f; sm.lse2[e] = 0.f; }
  __syncthreads();
  head_stats(p, qf, h0, nh, sm);
  // dq tiles: warp w owns dims 72w .. 72w+71 (nine tiles of 8) of the 16 heads
  float acc[9][4];
#pragma unroll
  for (int i = 0; i < 9; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const uint32_t za = smem_u32(sm.zs + (lane & 15) * ZS + 8 * (lane >> 4));
  const uint32_t kb_base = smem_u32(sm.ks + (lane & 15) * KS + 72 * warp);
  const int nkb = (p.topk + KB - 1) / KB;
  for (int kb = 0; kb < nkb; ++kb) {
    gather_block(p, qf, b, t, L, kb, sm, h0 == 0);
    block_pz(p, sm, h0);
    // dq_g += dZ[16 x 32] . K[32 x 576]: two K-steps of 16 keys
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(za + ks * 32, a0, a1, a2, a3);
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        uint32_t b0, b1;
        ldsm_x2_t(kb_base + ks * 16 * KS * 2 + i * 16, b0, b1);
        mma_bf16(acc[i], a0, a1, a2, a3, b0, b1);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 9; ++i) {
    const int d = 72 * warp + 8 * i + 2 * c;
    if (g < nh) {
      float* o = p.dq + (qf * p.H + h0 + g) * kRlat + d;
      o[0] = acc[i][0];
      o[1] = acc[i][1];
    }
    if (g + 8 < nh) {
      float* o = p.dq + (qf * p.H + h0 + g + 8) * kRlat + d;
      o[0] = acc[i][2];
      o[1] = acc[i][3];
    }
  }
}

// ---------------------------------------------------------------------------
// dkv: one CTA per query row, every head group in turn per key block
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(NT, 2) bwd_dkv_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int64_t qf = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  int b, L;
  const int t = query_pos(p, qf, b, L);
  if (t < 0) return;  // flagged by bwd_dq_kernel
  const int ngrp = (p.H + HG - 1) / HG;
  for (int e = tid; e < 128; e += NT) { sm.Dh[e] = 0.f; sm.lse2[e] = 0.f; }
  __syncthreads();
  head_stats(p, qf, 0, p.H, sm);
  // A = dZ^T / P^T [keys x heads] from the [head][key] tiles (transposed loads):
  // lane l addresses row (head) (l & 7) + 8 * (l >> 4), key 8 * ((l >> 3) & 1)
  const int a_row = (lane & 7) + 8 * (lane >> 4), a_col = 8 * ((lane >> 3) & 1);
  const uint32_t za = smem_u32(sm.zs + a_row * ZS + a_col);
  const uint32_t pa = smem_u32(sm.ps + a_row * ZS + a_col);
  // B = q_g / dO_g [heads x dims] (transposed loads): lane l < 16 addresses head l
  const uint32_t qb = smem_u32(sm.qs + (lane & 15) * KS + 72 * warp);
  const uint32_t db = smem_u32(sm.dsg + (lane & 15) * DS + 72 * warp);
  const int nkb = (p.topk + KB - 1) / KB;
  for (int kb = 0; kb < nkb; ++kb) {
    gather_block(p, qf, b, t, L, kb, sm, false);
    float acc[2][9][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 9; ++i) acc[m][i][0] = acc[m][i][1] = acc[m][i][2] = acc[m][i][3] = 0.f;
    for (int gr = 0; gr < ngrp; ++gr) {
      stage_group(p, qf, gr * HG, sm);
      __syncthreads();
      block_pz(p, sm, gr * HG);
      // dK[32 x 576] += dZ^T . q_g and dV[32 x 512] += P^T . dO_g (one K-step of 16 heads)
      uint32_t az[2][4], ap[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        ldsm_x4_t(za + m * 32, az[m][0], az[m][1], az[m][2], az[m][3]);
        ldsm_x4_t(pa + m * 32, ap[m][0], ap[m][1], ap[m][2], ap[m][3]);
      }
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        uint32_t b0, b1;
        ldsm_x2_t(qb + i * 16, b0, b1);
#pragma unroll
        for (int m = 0; m < 2; ++m) mma_bf16(acc[m][i], az[m][0], az[m][1], az[m][2], az[m][3], b0, b1);
        if (72 * warp + 8 * i < kVlat) {
          ldsm_x2_t(db + i * 16, b0, b1);
#pragma unroll
          for (int m = 0; m < 2; ++m)
            mma_bf16(acc[m][i], ap[m][0], ap[m][1], ap[m][2], ap[m][3], b0, b1);
        }
      }
      __syncthreads();
    }
    // the block's rows: 8-byte vector atomics into the FP32 gradient rows
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const int64_t r0 = sm.rows[16 * m + g], r1 = sm.rows[16 * m + g + 8];
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        const int d = 72 * warp + 8 * i + 2 * c;
        if (r0 >= 0)
          atomicAdd(reinterpret_cast<float2*>(p.dkv + r0 * kRlat + d), make_float2(acc[m][i][0], acc[m][i][1]));
        if (r1 >= 0)
          atomicAdd(reinterpret_cast<float2*>(p.dkv + r1 * kRlat + d), make_float2(acc[m][i][2], acc[m][i][3]));
      }
    }
    __syncthreads();
  }
}

}  // namespace mlab

dsa_status_t sparse_mla_bwd_launch(const SparseMlaBwdArgs& a, cudaStream_t stream) {
  using namespace mlab;
  // 96 heads with room for at least one query's P and dZ: the tcgen05 kernels
  const auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  if (a.H == 96 && a.scratch != nullptr &&
      a.scratch_bytes >= sparse_mla_bwd_tc_query_bytes(a.topk) && al16(a.d_o) && al16(a.o_lat) &&
      al16(a.dq))
    return sparse_mla_bwd_tc_launch(a, a.scratch, a.scratch_bytes, stream);
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
  const int smem = static_cast<int>(sizeof(Smem));
  if (cudaFuncSetAttribute(bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(bwd_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess)
    return launch_status("cudaFuncSetAttribute");
  bwd_dq_kernel<<<static_cast<unsigned>(nq * ngrp), NT, smem, stream>>>(p);
  if (launch_status("bwd_dq_kernel") != DSA_OK) return DSA_ERR_CUDA;
  bwd_dkv_kernel<<<static_cast<unsigned>(nq), NT, smem, stream>>>(p);
  return launch_status("bwd_dkv_kernel");
}

}  // namespace dsa
