// sparse_mla_bwd_tc.cu -- backward of the latent-space sparse MLA on the 5th-gen
// tensor cores (tcgen05, TMEM accumulators) for the model's 96 heads
// ("Kimi-K3.1-Pro", NeMo AutoModel, Implementation Limits: attention over the
// selected rows only (bullets 1-2), a native 96-head backward (the paragraph
// after bullet 4), no gradient into the indexer (bullet 3)).
//
// The same quantities as the warp-level path (per query row t, head h, list
// entry j with row s_j; the forward's lse and o_lat are inputs):
//   p_j  = exp(scale * q . kv[s_j] - lse),   dp_j = dO . kv[s_j, 0:512]
//   dz_j = scale * p_j (dp_j - D),           D = dO . o_lat
//   dq   = sum_j dz_j kv[s_j, 0:576]
//   dkv[s_j, 0:576] += dz_j q,   dkv[s_j, 0:512] += p_j dO
// One query's operands do not fit one SM together (q 108 KB, dO 96 KB, a block
// of rows, and a [96 x 576] FP32 dq accumulator that alone exceeds TMEM), so
// the work is three CTA kinds over a chunk of queries, with P and dZ (BF16,
// the precision the products take them in) passed through the workspace as
// [query][head][list entry].  K1 is one launch; K2 and K3 read only its output
// and share the next (bwd_dq_dkv_kernel: the chunk's K2 CTAs, then its K3 CTAs):
//   K1 bwd_pz   grid (2 head groups of 48; queries).  Rows of 128 list entries
//               are gathered one 64-dim chunk (16 KB) at a time into a ring;
//                 [S^T | dP^T] [128 x 96] += rows_c . [q_g,c ; dO_g,c]^T   (c < 8)
//                 S^T [128 x 48]          += rows_c . q_g,c^T              (c = 8)
//               (M=128 entries; q and dO of a chunk stored as one 96-row
//               operand, so the gathered rows are read once per chunk) and
//               each TMEM lane (one entry) forms p and dz for its 48 heads.
//   K2 dq       one CTA per query.  Rows of 64 entries gathered as in the
//               forward (four 64-key pairs of two 64-dim chunks, and the rope
//               chunk) and the entries' dz (TMA, [96 heads x 64 entries]):
//                 dq^T[512 x 96] += rows^T . dz^T        (4 x M=128 dims, N=96)
//                 dq_rope[96 x 64] += dz . rows_rope     (M=128 heads, N=64)
//   K3 dkv      one CTA per (dim range 0-255, 256-511, 512-575; query).  q and
//               dO of the range (TMA, dims contiguous) against dz and p of 128
//               entries (TMA, entries contiguous), both MN-major:
//                 dKV^T[128 dims x 128] = q_r^T . dz + dO_r^T . p   (M=128, N=128)
//               then each lane (one dim) adds its value for each entry into
//               the FP32 dkv row with atomics, a warp covering 32 consecutive
//               dims of one row (rows are shared by the queries that selected
//               them, so the order of the additions, and the FP32 rounding of
//               dkv, vary run to run).
// Every wait is bounded (an abort flag per CTA stops the other roles).
#include <cuda_bf16.h>

#include "dsa_status.cuh"
#include "internal.h"
#include "sm103.cuh"

namespace dsa {
namespace mlbt {

constexpr int H = 96;
constexpr int HG = 48;          // heads per K1 CTA
constexpr int CH = 64 * 128;    // one 64-key x 64-dim chunk (8 KB)

enum : uint32_t {
  SITE_IDX = 0x900, SITE_PAGE = 0x901,
  SITE_W1_Q = 0x910, SITE_W1_F = 0x911, SITE_W1_E = 0x912, SITE_W1_SF = 0x913, SITE_W1_SE = 0x914,
  SITE_W2_F = 0x920, SITE_W2_E = 0x921, SITE_W2_D = 0x922,
  SITE_W3_B = 0x930, SITE_W3_F = 0x931, SITE_W3_E = 0x932, SITE_W3_DF = 0x933, SITE_W3_DE = 0x934,
  SITE_DRAIN = 0x93f
};

struct Params {
  const uint16_t* kv;       // rows of 576 BF16
  const int32_t* idx;       // [nq_total, topk]
  const int32_t* q_start;
  const int32_t* kv_len;
  const int32_t* block_table;
  int64_t seq_stride;
  int32_t max_pages, num_pages;
  int paged;
  int Tq, topk, max_kv_len, tpad;  // tpad: topk rounded up to 128
  int64_t q0;                      // first query row (b * Tq + i) of this chunk
  float scale, c1;                 // c1 = scale * log2(e)
  const uint16_t* o;               // [nq_total, 96, 512]
  const float* lse;                // [nq_total, 96], natural log
  const uint16_t* dO;              // [nq_total, 96, 512]
  float* dq;                       // [nq_total, 96, 576]
  float* dkv;                      // FP32 rows of 576
  uint16_t* pbuf;                  // [chunk queries, 96, tpad] BF16
  uint16_t* zbuf;                  // [chunk queries, 96, tpad] BF16
  uint32_t* status;
};

__device__ __forceinline__ bool vflag(const volatile int* f) { return *f != 0; }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The query row's sequence, position and key count.
struct QInfo {
  int b, t, L;
  bool ok;
};
__device__ __forceinline__ QInfo qinfo(const Params& p, int64_t qg) {
  QInfo r;
  r.b = static_cast<int>(qg / p.Tq);
  const int i = static_cast<int>(qg % p.Tq);
  const int qs = __ldg(p.q_start + r.b);
  r.L = __ldg(p.kv_len + r.b);
  r.t = qs + i;
  r.ok = qs >= 0 && r.t < r.L && r.L <= p.max_kv_len;
  return r;
}

// List entry e of query qg as stored (-1 past topk or for an invalid query);
// loaded one block ahead of its use, so that its latency overlaps work.
__device__ __forceinline__ int entry_raw(const Params& p, int64_t qg, const QInfo& Q, int e) {
  return (Q.ok && e < p.topk) ? __ldg(p.idx + qg * p.topk + e) : -1;
}

// Physical row of list entry s, or -1 (unused or invalid; an invalid entry is
// recorded when `report` is set).
__device__ __forceinline__ int64_t raw_row(const Params& p, const QInfo& Q, int s, bool report) {
  if (s < 0) return -1;
  if (s > Q.t || s >= Q.L) {
    if (report) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_IDX, static_cast<uint32_t>(s));
    return -1;
  }
  if (!p.paged) return static_cast<int64_t>(Q.b) * p.seq_stride + s;
  const int pg = s >> 6;
  const int pid = pg < p.max_pages ? __ldg(p.block_table + static_cast<int64_t>(Q.b) * p.max_pages + pg) : -1;
  if (pid < 0 || pid >= p.num_pages) {
    if (report) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_PAGE, static_cast<uint32_t>(pid));
    return -1;
  }
  return static_cast<int64_t>(pid) * kPage + (s & (kPage - 1));
}

// =============================================================================
// K1: p and dz.  Threads: warps 0-7 gather, warps 8-11 epilogue (one TMEM lane
// quarter each), warp 12 MMA issuer and TMEM owner.
// =============================================================================
namespace k1 {
constexpr int NT = 416;
constexpr int QCH = HG * 128;          // one 64-dim chunk of the group's 48 q (or dO) rows
constexpr int SLOT = 128 * 128;        // 128 entries x one 64-dim chunk
constexpr int NR = 7;                  // ring slots
constexpr int KB = 3;                  // chunks per wait of the MMA issuer (one wait and fence per three chunks)
// chunk c < 8: q rows at OFF_QD + 2c QCH, dO rows right after (one 96-row
// operand); the rope chunk of q at OFF_QD + 16 QCH
constexpr int OFF_QD = 0;
constexpr int OFF_RING = OFF_QD + 17 * QCH;
constexpr int OFF_MISC = OFF_RING + NR * SLOT;
// barriers: Q/dO loaded, ring full [NR], ring empty [NR], S full [2], S empty [2], drain
constexpr int B_Q = 0, B_F = 1, B_E = B_F + NR, B_SF = B_E + NR, B_SE = B_SF + 2, B_DRAIN = B_SE + 2,
              NBAR = B_DRAIN + 1;
constexpr int SMEM = OFF_MISC + 1024 + 1024;
static_assert(NBAR * 8 + 8 + 2 * HG * 4 <= 1024, "misc block");
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(OFF_RING % 1024 == 0 && QCH % 1024 == 0, "swizzle atoms");
}  // namespace k1

__global__ void __launch_bounds__(k1::NT, 1)
    bwd_pz_kernel(const __grid_constant__ CUtensorMap tm_q48, const __grid_constant__ CUtensorMap tm_do48,
                  const Params p) {
  using namespace k1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_MISC);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  float* s_D = reinterpret_cast<float*>(sm + OFF_MISC + NBAR * 8 + 8);
  float* s_l2 = s_D + HG;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ql = blockIdx.y, g = blockIdx.x;  // the two head groups of a query adjacent
  const int64_t qg = p.q0 + ql;
  const QInfo Q = qinfo(p, qg);
  const int nblk = p.tpad / 128;
  constexpr uint32_t IDESC_SD = idesc_bf16(128, 2 * HG, false, false);  // S and dP together
  constexpr uint32_t IDESC_S = idesc_bf16(128, HG, false, false);       // rope chunk: S only

  if (tid == 0) {
    mbar_init(&bars[B_Q], 1);
    for (int i = 0; i < NR; ++i) {
      mbar_init(&bars[B_F + i], 256);
      mbar_init(&bars[B_E + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_SF + i], 1);
      mbar_init(&bars[B_SE + i], 4);
    }
    mbar_init(&bars[B_DRAIN], 1);
    s_abort[0] = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp < 8) {
    // ============ gather (8 warps): eight consecutive lanes copy the eight
    // 16-byte units of one entry's 128-byte piece (whole 128-byte lines per
    // request); thread t covers unit t % 8 of entries t / 8 + 32 i, i = 0..3 ============
    if (tid == 0) {
      mbar_expect_tx(&bars[B_Q], (9 + 8) * QCH);
      const int row = static_cast<int>(qg * H + g * HG);
      for (int c = 0; c < 9; ++c) tma_load_2d(sm + OFF_QD + 2 * c * QCH, &tm_q48, &bars[B_Q], 64 * c, row);
      for (int c = 0; c < 8; ++c)
        tma_load_2d(sm + OFF_QD + (2 * c + 1) * QCH, &tm_do48, &bars[B_Q], 64 * c, row);
    }
    const int64_t dummy = p.paged ? 0 : static_cast<int64_t>(Q.b) * p.seq_stride;
    const int u8 = tid & 7, e0 = tid >> 3;
    uint32_t doff[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) doff[i] = sw128_unit(e0 + 32 * i, u8);
    int nxt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) nxt[i] = entry_raw(p, qg, Q, e0 + 32 * i);
    for (int j = 0; j < nblk; ++j) {
      const uint16_t* src[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t r = raw_row(p, Q, nxt[i], false);
        src[i] = p.kv + (r >= 0 ? r : dummy) * kRlat + u8 * 8;
        nxt[i] = entry_raw(p, qg, Q, 128 * (j + 1) + e0 + 32 * i);
      }
      bool stop = false;
      for (int c = 0; c < 9; ++c) {
        const int gc = 9 * j + c, slot = gc % NR, use = gc / NR;
        if (use > 0 && !mbar_wait(&bars[B_E + slot], (use - 1) & 1, p.status, kWaitLimitNs, SITE_W1_E))
          s_abort[0] = 1;
        if (vflag(s_abort)) { stop = true; break; }
        const uint32_t dst = smem_u32(sm + OFF_RING + slot * SLOT);
#pragma unroll
        for (int i = 0; i < 4; ++i) cp_async_16(dst + doff[i], src[i] + c * 64);
        cp_async_arrive(&bars[B_F + slot]);
      }
      if (stop) break;
    }
    cp_async_wait_all();
  } else if (warp < 12) {
    // ============ epilogue: lane = list entry of the block ============
    const int ew = warp - 8, sub = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    const int el = sub * 32 + lane;  // entry within the block (TMEM lane)
    // D = dO . o and lse (log2) of the group's heads: a warp takes heads
    // ew + 4i, four at a time with all their loads issued first
    for (int h0 = ew; h0 < HG; h0 += 16) {
      uint4 x[4][2], y[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t row = qg * H + g * HG + h0 + 4 * i;
        const uint4* a = reinterpret_cast<const uint4*>(p.dO + row * kVlat) + lane * 2;
        const uint4* b = reinterpret_cast<const uint4*>(p.o + row * kVlat) + lane * 2;
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          x[i][v] = __ldg(a + v);
          y[i][v] = __ldg(b + v);
        }
      }
      const float l = lane < 4 ? __ldg(p.lse + qg * H + g * HG + h0 + 4 * lane) : 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const uint32_t xs[4] = {x[i][v].x, x[i][v].y, x[i][v].z, x[i][v].w};
          const uint32_t ys[4] = {y[i][v].x, y[i][v].y, y[i][v].z, y[i][v].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc = fmaf(__uint_as_float(xs[k] << 16), __uint_as_float(ys[k] << 16), acc);
            acc = fmaf(__uint_as_float(xs[k] & 0xffff0000u), __uint_as_float(ys[k] & 0xffff0000u), acc);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) s_D[h0 + 4 * i] = acc;
      }
      if (lane < 4) s_l2[h0 + 4 * lane] = l * 1.4426950408889634f;
    }
    named_bar_sync(1, 128);
    uint16_t* pz = p.pbuf + (static_cast<int64_t>(ql) * H + g * HG) * p.tpad;
    uint16_t* zz = p.zbuf + (static_cast<int64_t>(ql) * H + g * HG) * p.tpad;
    int nxt = entry_raw(p, qg, Q, el);
    for (int j = 0; j < nblk; ++j) {
      const int buf = j & 1;
      const int cur = nxt;
      nxt = entry_raw(p, qg, Q, 128 * (j + 1) + el);
      bool ok = !vflag(s_abort) &&
                mbar_wait(&bars[B_SF + buf], (j >> 1) & 1, p.status, kWaitLimitNs, SITE_W1_SF);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) { s_abort[0] = 1; break; }
      tc_fence_after();
      const int e = 128 * j + el;
      const bool valid = raw_row(p, Q, cur, g == 0) >= 0;
      uint32_t sv[HG], dv[HG];
      {
        uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(sv);
        uint32_t (&s1)[16] = *reinterpret_cast<uint32_t(*)[16]>(sv + 32);
        uint32_t (&d0)[32] = *reinterpret_cast<uint32_t(*)[32]>(dv);
        uint32_t (&d1)[16] = *reinterpret_cast<uint32_t(*)[16]>(dv + 32);
        const uint32_t col = lane_base + buf * 96;
        tmem_ld32(tmem + col, s0);
        tmem_ld16(tmem + col + 32, s1);
        tmem_ld32(tmem + col + HG, d0);
        tmem_ld16(tmem + col + HG + 32, d1);
        tmem_ld_wait();
      }
      tc_fence_before();
      mbar_arrive_warp(&bars[B_SE + buf]);
#pragma unroll
      for (int hh = 0; hh < HG; ++hh) {
        float pr = 0.f, z = 0.f;
        if (valid) {
          pr = ex2(fmaf(__uint_as_float(sv[hh]), p.c1, -s_l2[hh]));
          z = p.scale * pr * (__uint_as_float(dv[hh]) - s_D[hh]);
        }
        pz[static_cast<int64_t>(hh) * p.tpad + e] = __bfloat16_as_ushort(__float2bfloat16_rn(pr));
        zz[static_cast<int64_t>(hh) * p.tpad + e] = __bfloat16_as_ushort(__float2bfloat16_rn(z));
      }
    }
  } else if (warp == 12) {
    // ============ MMA issuer ============
    if (lane == 0) {
      bool ok = mbar_wait(&bars[B_Q], 0, p.status, kWaitLimitNs, SITE_W1_Q);
      const uint64_t qd = smem_desc(smem_u32(sm + OFF_QD), 16, 1024);
      const uint64_t rd = smem_desc(smem_u32(sm + OFF_RING), 16, 1024);
      int slot = 0;       // ring slot of the next chunk (chunk counter modulo NR) ...
      uint32_t ph = 0;    // ... and the parity of its use
      for (int j = 0; j < nblk && ok; ++j) {
        const int buf = j & 1;
        if (vflag(s_abort) || (j >= 2 && !mbar_wait(&bars[B_SE + buf], ((j >> 1) - 1) & 1, p.status,
                                                     kWaitLimitNs, SITE_W1_SE))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ds = tmem + buf * 96;  // S^T in columns 0-47, dP^T in 48-95
        // chunks taken KB at a time: one wait and one fence for KB chunks
        for (int c = 0; c < 9 && ok; c += KB) {
          const int nc = c + KB <= 9 ? KB : 9 - c;
          int sl[KB];
#pragma unroll
          for (int i = 0; i < KB; ++i) {
            if (i < nc) {
              sl[i] = slot;
              if (ok && !mbar_wait(&bars[B_F + slot], ph, p.status, kWaitLimitNs, SITE_W1_F)) ok = false;
              if (++slot == NR) { slot = 0; ph ^= 1; }
            }
          }
          if (!ok) break;
          fence_proxy_async_smem();  // cp.async (generic proxy) writes -> tensor core reads
          tc_fence_after();
#pragma unroll
          for (int i = 0; i < KB; ++i) {
            if (i < nc) {
              const int cc = c + i;
              const uint64_t ad = desc_add(rd, sl[i] * SLOT);
              if (cc < 8) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  umma_bf16(ds, desc_add(ad, kk * 32), desc_add(qd, 2 * cc * QCH + kk * 32), IDESC_SD,
                            (cc | kk) ? 1u : 0u);
              } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  umma_bf16(ds, desc_add(ad, kk * 32), desc_add(qd, 16 * QCH + kk * 32), IDESC_S, 1u);
              }
              umma_commit(&bars[B_E + sl[i]]);
            }
          }
        }
        if (!ok) break;
        umma_commit(&bars[B_SF + buf]);
      }
      if (!ok) s_abort[0] = 1;
      umma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, p.status, kWaitLimitNs, SITE_DRAIN);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// =============================================================================
// K2: dq.  Threads: warps 0-7 gather (+ the dz TMA), warps 8-11 epilogue,
// warp 12 MMA issuer and TMEM owner.  The rows of a 64-entry block move
// through rings finer than a block, so that a slot is gathered again as soon
// as the MMAs that read it are done: a ring of eight 16 KB pair slots (64
// entries x 128 dims, the A operand of one 128-dim tile of dq^T) and a ring of
// three (rope chunk, dz tile) slots per block.
// =============================================================================
namespace k2 {
constexpr int NT = 416;
constexpr int PAIR = 2 * CH;                 // 64 entries x 128 dims
constexpr int ZT = 128 * 128;                // dz tile: 96 head rows (+32 spare) x 64 entries
constexpr int NP = 8;                        // pair slots (two blocks)
constexpr int NX = 3;                        // rope + dz slots
constexpr int OFF_P = 0;
constexpr int OFF_R = OFF_P + NP * PAIR;
constexpr int OFF_Z = OFF_R + NX * CH;
constexpr int OFF_MISC = OFF_Z + NX * ZT;
// barriers: pair full / empty [NP], dz full, rope full, rope+dz empty [NX], done
constexpr int B_PF = 0, B_PE = B_PF + NP, B_ZF = B_PE + NP, B_RF = B_ZF + NX, B_XE = B_RF + NX,
              B_D = B_XE + NX, NBAR = B_D + 1;
constexpr int MISC = 256 + 2 * 64 * 8;       // barriers, then the row table [2][64]
constexpr int SMEM = OFF_MISC + MISC + 1024;
static_assert(NBAR * 8 + 8 <= 256, "barriers before the row table");
static_assert(SMEM <= 232448, "shared memory budget");
static_assert((NP & (NP - 1)) == 0, "pair slot index by mask");
}  // namespace k2

// K2's CTA body (query ql of the chunk); threads past k2::NT wait at the
// CTA-wide barriers only.
__device__ __forceinline__ void bwd_dq_body(const CUtensorMap& tm_z, const Params& p, int ql) {
  using namespace k2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_MISC);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  int64_t* s_row = reinterpret_cast<int64_t*>(sm + OFF_MISC + 256);  // [2][64]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t qg = p.q0 + ql;
  const QInfo Q = qinfo(p, qg);
  const int nblk = p.tpad / 64;
  constexpr uint32_t IDESC_T = idesc_bf16(128, H, true, false);   // rows^T (MN-major) . dz^T
  constexpr uint32_t IDESC_R = idesc_bf16(128, 64, false, true);  // dz . rope rows (MN-major B)

  if (tid == 0) {
    for (int i = 0; i < NP; ++i) {
      mbar_init(&bars[B_PF + i], 256);  // the 256 gathering threads
      mbar_init(&bars[B_PE + i], 1);
    }
    for (int i = 0; i < NX; ++i) {
      mbar_init(&bars[B_ZF + i], 1);    // the dz copy
      mbar_init(&bars[B_RF + i], 256);
      mbar_init(&bars[B_XE + i], 1);
    }
    mbar_init(&bars[B_D], 1);
    s_abort[0] = 0;
    fence_mbar_init();
  }
  // the spare dz rows 96..127 feed only accumulator lanes nobody reads; zero
  // them once so that they hold finite values
  for (int i = tid; i < NX * 32 * 128 / 16; i += blockDim.x) {
    const int x = i / (32 * 8), r = i % (32 * 8);
    *reinterpret_cast<uint4*>(sm + OFF_Z + x * ZT + 96 * 128 + r * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  if (warp == 12) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp < 8) {
    // ============ gather.  Pair i of a block: its 64 rows x 16 units (dims
    // 128 i .. 128 i + 127), unit U = tid + 256 m, m = 0..3 (sixteen consecutive
    // lanes per row: whole 128-byte lines per request); the rope chunk: 64 rows
    // x 8 units, U = tid + 256 m, m = 0..1.  The entries' rows are looked up
    // once per block into shared memory ============
    const int64_t dummy = p.paged ? 0 : static_cast<int64_t>(Q.b) * p.seq_stride;
    int nxt = tid < 64 ? entry_raw(p, qg, Q, tid) : -1;
    for (int j = 0; j < nblk; ++j) {
      if (tid < 64) {
        const int64_t r = raw_row(p, Q, nxt, false);
        s_row[(j & 1) * 64 + tid] = r >= 0 ? r : dummy;
        nxt = entry_raw(p, qg, Q, 64 * (j + 1) + tid);
      }
      // the rows are visible to all 256 threads after this barrier, and the stop
      // decision is the same for all of them
      if (named_bar_or(2, 256, vflag(s_abort))) break;
      const int64_t* rows = s_row + (j & 1) * 64;
      const int x = j % NX, xu = j / NX;
      bool fail = xu > 0 && !mbar_wait(&bars[B_XE + x], (xu - 1) & 1, p.status, kWaitLimitNs, SITE_W2_E);
      if (!fail && tid == 0) {
        mbar_expect_tx(&bars[B_ZF + x], 96 * 128);
        tma_load_2d(sm + OFF_Z + x * ZT, &tm_z, &bars[B_ZF + x], 64 * j, ql * H);
      }
      for (int i = 0; i < 4 && !fail; ++i) {
        const int gp = 4 * j + i, slot = gp & (NP - 1), pu = gp / NP;
        if (pu > 0 && !mbar_wait(&bars[B_PE + slot], (pu - 1) & 1, p.status, kWaitLimitNs, SITE_W2_E)) {
          fail = true;
          break;
        }
        const uint32_t b32 = smem_u32(sm + OFF_P + slot * PAIR);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int U = tid + 256 * m, key = U >> 4, w = U & 15;
          cp_async_16(b32 + (w >> 3) * CH + sw128_unit(key, w & 7), p.kv + rows[key] * kRlat + (16 * i + w) * 8);
        }
        cp_async_arrive(&bars[B_PF + slot]);
      }
      if (!fail) {
        const uint32_t r32 = smem_u32(sm + OFF_R + x * CH);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const int U = tid + 256 * m, key = U >> 3, uu = U & 7;
          cp_async_16(r32 + sw128_unit(key, uu), p.kv + rows[key] * kRlat + (64 + uu) * 8);
        }
        cp_async_arrive(&bars[B_RF + x]);
      }
      if (fail) s_abort[0] = 1;  // everyone stops at the next block's barrier
    }
    cp_async_wait_all();
  } else if (warp < 12) {
    // ============ epilogue: dq written once ============
    const int sub = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    bool ok = mbar_wait(&bars[B_D], 0, p.status, kWaitLimitNs, SITE_W2_D) && !vflag(s_abort);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    float* dqq = p.dq + qg * H * kRlat;
    // dq^T tiles: lane = dim 128 i + sub*32 + lane, columns = heads
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
#pragma unroll 1
      for (int v = 0; v < 3; ++v) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + i * H + 32 * v, rr);
        tmem_ld_wait();
        const int d = 128 * i + sub * 32 + lane;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          dqq[static_cast<int64_t>(32 * v + c) * kRlat + d] = ok ? __uint_as_float(rr[c]) : 0.f;
      }
    }
    // dq rope: lane = head, 64 columns = dims 512..575
    const int h = sub * 32 + lane;
#pragma unroll 1
    for (int v = 0; v < 2; ++v) {
      uint32_t rr[32];
      tmem_ld32(tmem + lane_base + 4 * H + 32 * v, rr);
      tmem_ld_wait();
      if (h < H) {
        float4* dst = reinterpret_cast<float4*>(dqq + static_cast<int64_t>(h) * kRlat + kVlat + 32 * v);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c] = ok ? make_float4(__uint_as_float(rr[4 * c]), __uint_as_float(rr[4 * c + 1]),
                                    __uint_as_float(rr[4 * c + 2]), __uint_as_float(rr[4 * c + 3]))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  } else if (warp == 12) {
    // ============ MMA issuer: per block, the dz tile, then two pairs per wait,
    // then the rope chunk ============
    if (lane == 0) {
      bool ok = true;
      int pslot = 0;      // pair slot of the next pair ...
      uint32_t pph = 0;   // ... and the parity of its use
      for (int j = 0; j < nblk && ok; ++j) {
        const int x = j % NX;
        const uint32_t xph = (j / NX) & 1;
        if (vflag(s_abort) || !mbar_wait(&bars[B_ZF + x], xph, p.status, kWaitLimitNs, SITE_W2_F)) {
          ok = false;
          break;
        }
        const uint64_t zd = smem_desc(smem_u32(sm + OFF_Z + x * ZT), 16, 1024);  // dz, K-major rows = heads
        for (int i0 = 0; i0 < 4 && ok; i0 += 2) {
          int sl[2];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            sl[t] = pslot;
            if (ok && !mbar_wait(&bars[B_PF + pslot], pph, p.status, kWaitLimitNs, SITE_W2_F)) ok = false;
            if (++pslot == NP) { pslot = 0; pph ^= 1; }
          }
          if (!ok) break;
          fence_proxy_async_smem();  // cp.async (generic proxy) writes -> tensor core reads
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint64_t vd = smem_desc(smem_u32(sm + OFF_P + sl[t] * PAIR), CH, 1024);  // 128 dims x 64 entries, MN-major
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tmem + (i0 + t) * H, desc_add(vd, kk * 2048), desc_add(zd, kk * 32), IDESC_T,
                        (j | kk) ? 1u : 0u);
            umma_commit(&bars[B_PE + sl[t]]);
          }
        }
        if (!ok || !mbar_wait(&bars[B_RF + x], xph, p.status, kWaitLimitNs, SITE_W2_F)) {
          ok = false;
          break;
        }
        fence_proxy_async_smem();
        tc_fence_after();
        const uint64_t rd = smem_desc(smem_u32(sm + OFF_R + x * CH), CH, 1024);  // rope rows, MN-major
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + 4 * H, desc_add(zd, kk * 32), desc_add(rd, kk * 2048), IDESC_R,
                    (j | kk) ? 1u : 0u);
        umma_commit(&bars[B_XE + x]);
      }
      if (!ok) s_abort[0] = 1;
      umma_commit(&bars[B_D]);
      // drain: every MMA complete before TMEM is released
      mbar_wait(&bars[B_D], 0, p.status, kWaitLimitNs, SITE_DRAIN);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================================
// K3: dkv, computed transposed so that a TMEM lane is one dim and a column one
// list entry: each warp's atomic then covers 32 consecutive dims of one dkv
// row (one 128-byte line) instead of 32 different rows.
//   dKV^T[dims x 128 entries] = q_r^T . dz + dO_r^T . p    (M=128 dims, N=128)
// A = q^T / dO^T of the range ([96 heads x 64 dims] boxes, dims contiguous:
// MN-major), B = dz / p of 128 entries ([96 heads x 64 entries] boxes, entries
// contiguous: MN-major).  Threads: warp 0 TMA producer, warp 1 MMA issuer and
// TMEM owner, warps 2-17 epilogue.  A warp's reductions into global memory
// issue at a fixed rate whatever the other warps do, so every warp that can
// reach a tile's TMEM lanes takes a share of its columns: in the two 128-dim
// tiles, one warp per (tile, lane quarter, half of the 128 entries); in the
// rope tile (64 live lanes), four warps per live lane quarter, 32 entries each.
// =============================================================================
namespace k3 {
constexpr int NT = 576;
constexpr int QB = H * 128;                // [96 heads x 64] box (12 KB)
constexpr int OFF_QR = 0;                  // q^T of the range: 4 boxes (the rope range: 2, one past the end)
constexpr int OFF_DR = OFF_QR + 4 * QB;    // dO^T of the range: 4 boxes
constexpr int STAGE = 4 * QB;              // dz (2 boxes) + p (2 boxes) of 128 entries
constexpr int OFF_ST = OFF_DR + 4 * QB;
constexpr int NS = 2;
constexpr int OFF_MISC = OFF_ST + NS * STAGE;
constexpr int B_B = 0, B_F = 1, B_E = B_F + NS, B_DF = B_E + NS, B_DE = B_DF + 2, B_DRAIN = B_DE + 2,
              NBAR = B_DRAIN + 1;
constexpr int MISC = 256 + 2 * 128 * 8;    // barriers, then the entries' rows [2][128]
constexpr int SMEM = OFF_MISC + MISC + 1024;
static_assert(NBAR * 8 + 8 <= 256, "barriers before the row table");
static_assert(SMEM <= 232448, "shared memory budget");
}  // namespace k3

// K3's CTA body: `lin` numbers the chunk's 3 n dKV CTAs in launch order.
__device__ __forceinline__ void bwd_dkv_body(const CUtensorMap& tm_q96, const CUtensorMap& tm_do96,
                                             const CUtensorMap& tm_z, const CUtensorMap& tm_p,
                                             const Params& p, int lin, int n) {
  using namespace k3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_MISC);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + NBAR);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  int64_t* s_row = reinterpret_cast<int64_t*>(sm + OFF_MISC + 256);  // [2][128]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // launch order: the two 256-dim CTAs of each query next to each other (the
  // second reads the query's p and dz from L2), then every query's rope CTA,
  // which has a quarter of the work and so evens out the last wave
  const int n2 = 2 * n;
  const int ql = lin < n2 ? (lin >> 1) : lin - n2;
  const int rg = lin < n2 ? (lin & 1) : 2;  // dims [256 rg, 256 rg + 256) (rope: 512..575)
  const int64_t qg = p.q0 + ql;
  const QInfo Q = qinfo(p, qg);
  const int nblk = p.tpad / 128;
  const bool rope = rg == 2;
  const int ntile = rope ? 1 : 2;             // 128-dim M tiles of the range
  constexpr uint32_t IDESC = idesc_bf16(128, 128, true, true);

  if (tid == 0) {
    mbar_init(&bars[B_B], 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars[B_F + i], 1);
      mbar_init(&bars[B_E + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_DF + i], 1);
      mbar_init(&bars[B_DE + i], 16);
    }
    mbar_init(&bars[B_DRAIN], 1);
    s_abort[0] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      // q (and dO) of the range: [96 heads x 64 dims] boxes; the rope range's
      // second box lies past dim 575 and is filled with zeros by the copy
      mbar_expect_tx(&bars[B_B], (rope ? 2 : 8) * QB);
      for (int c = 0; c < 2 * ntile; ++c)
        tma_load_2d(sm + OFF_QR + c * QB, &tm_q96, &bars[B_B], 256 * rg + 64 * c, static_cast<int>(qg * H));
      if (!rope)
        for (int c = 0; c < 4; ++c)
          tma_load_2d(sm + OFF_DR + c * QB, &tm_do96, &bars[B_B], 256 * rg + 64 * c, static_cast<int>(qg * H));
      int last[NS] = {-1, -1};
      for (int j = 0; j < nblk; ++j) {
        const int st = j % NS, use = j / NS;
        if (use > 0 && !mbar_wait(&bars[B_E + st], (use - 1) & 1, p.status, kWaitLimitNs, SITE_W3_E))
          s_abort[0] = 1;
        if (vflag(s_abort)) break;
        uint8_t* base = sm + OFF_ST + st * STAGE;
        mbar_expect_tx(&bars[B_F + st], (rope ? 2 : 4) * QB);
        for (int h = 0; h < 2; ++h)
          tma_load_2d(base + h * QB, &tm_z, &bars[B_F + st], 128 * j + 64 * h, ql * H);
        if (!rope)
          for (int h = 0; h < 2; ++h)
            tma_load_2d(base + (2 + h) * QB, &tm_p, &bars[B_F + st], 128 * j + 64 * h, ql * H);
        last[st] = use;
      }
      // every copy issued has landed before the CTA may exit
      for (int st = 0; st < NS; ++st)
        if (last[st] >= 0) mbar_wait(&bars[B_F + st], last[st] & 1, p.status, kWaitLimitNs, SITE_W3_F);
      mbar_wait(&bars[B_B], 0, p.status, kWaitLimitNs, SITE_W3_B);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = mbar_wait(&bars[B_B], 0, p.status, kWaitLimitNs, SITE_W3_B);
      const uint64_t qd = smem_desc(smem_u32(sm + OFF_QR), QB, 1024);  // [K=heads][M=dims], MN-major
      const uint64_t dd = smem_desc(smem_u32(sm + OFF_DR), QB, 1024);
      for (int j = 0; j < nblk && ok; ++j) {
        const int st = j % NS, buf = j & 1;
        if (j >= 2 && !mbar_wait(&bars[B_DE + buf], ((j >> 1) - 1) & 1, p.status, kWaitLimitNs, SITE_W3_DE)) {
          ok = false;
          break;
        }
        if (vflag(s_abort) ||
            !mbar_wait(&bars[B_F + st], (j / NS) & 1, p.status, kWaitLimitNs, SITE_W3_F)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(sm + OFF_ST + st * STAGE);
        const uint64_t zd = smem_desc(base, QB, 1024);           // [K=heads][N=entries], MN-major
        const uint64_t pd = smem_desc(base + 2 * QB, QB, 1024);
        for (int mt = 0; mt < ntile; ++mt) {
          const uint32_t d = tmem + buf * 256 + mt * 128;
#pragma unroll
          for (int kk = 0; kk < 6; ++kk)
            umma_bf16(d, desc_add(qd, mt * 2 * QB + kk * 2048), desc_add(zd, kk * 2048), IDESC,
                      kk ? 1u : 0u);
          if (!rope) {
#pragma unroll
            for (int kk = 0; kk < 6; ++kk)
              umma_bf16(d, desc_add(dd, mt * 2 * QB + kk * 2048), desc_add(pd, kk * 2048), IDESC, 1u);
          }
        }
        umma_commit(&bars[B_E + st]);
        umma_commit(&bars[B_DF + buf]);
      }
      if (!ok) s_abort[0] = 1;
      // drain: every MMA complete before TMEM is released
      umma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, p.status, kWaitLimitNs, SITE_DRAIN);
    }
    __syncwarp();
  } else {
    // ============ epilogue: lane = dim, columns = entries ============
    const int et = tid - 64;                       // 0..511
    const int sub = warp & 3, grp = (warp - 2) >> 2;  // lane quarter; each group of four has every quarter
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    // tile, first column and number of 32-column loads of this warp
    const int mt = rope ? 0 : (grp & 1);
    const int col0 = rope ? 32 * grp : 64 * (grp >> 1);
    const int nld = rope ? 1 : 2;
    const int dim = 256 * rg + 128 * mt + sub * 32 + lane;
    const bool act = !rope || sub < 2;             // the rope tile's lanes 64..127 are past dim 575
    const bool dim_ok = dim < kRlat;
    // the entries' rows, double-buffered by block parity: block j+1's are
    // looked up while block j's are added (its readers of that half passed the
    // barrier of block j first)
    if (et < 128) s_row[et] = raw_row(p, Q, entry_raw(p, qg, Q, et), false);
    int nxt = et < 128 ? entry_raw(p, qg, Q, 128 + et) : -1;
    for (int j = 0; j < nblk; ++j) {
      const int buf = j & 1;
      bool ok = !vflag(s_abort) &&
                mbar_wait(&bars[B_DF + buf], (j >> 1) & 1, p.status, kWaitLimitNs, SITE_W3_DF);
      // one decision for all epilogue warps; the rows are visible after it
      if (named_bar_or(1, 512, !ok)) { s_abort[0] = 1; break; }
      tc_fence_after();
      if (act) {
        const int64_t* rows = s_row + buf * 128 + col0;
#pragma unroll 1
        for (int v = 0; v < nld; ++v) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + buf * 256 + mt * 128 + col0 + 32 * v, rr);
          tmem_ld_wait();
          if (dim_ok) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int64_t r = rows[32 * v + c];
              if (r >= 0) atomicAdd(p.dkv + r * kRlat + dim, __uint_as_float(rr[c]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&bars[B_DE + buf]);
      if (et < 128) {
        s_row[(buf ^ 1) * 128 + et] = raw_row(p, Q, nxt, false);
        nxt = entry_raw(p, qg, Q, 128 * (j + 2) + et);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// K2 and K3 of a chunk in one launch: both read only K1's p and dz, so the
// dKV CTAs (launched after the chunk's n dq CTAs) fill the SMs the last wave
// of dq CTAs leaves idle.
static_assert(k3::NT >= k2::NT, "one block size for both bodies");
constexpr int KDQ_SMEM = k2::SMEM > k3::SMEM ? k2::SMEM : k3::SMEM;
__global__ void __launch_bounds__(k3::NT, 1)
    bwd_dq_dkv_kernel(const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_q96,
                      const __grid_constant__ CUtensorMap tm_do96, const __grid_constant__ CUtensorMap tm_p,
                      const Params p, int n) {
  const int b = static_cast<int>(blockIdx.x);
  if (b < n)
    bwd_dq_body(tm_z, p, b);
  else
    bwd_dkv_body(tm_q96, tm_do96, tm_z, tm_p, p, b - n, n);
}

}  // namespace mlbt

// Bytes of P and dZ scratch per query (BF16, both matrices).
size_t sparse_mla_bwd_tc_query_bytes(int topk) {
  const size_t tpad = static_cast<size_t>((topk + 127) / 128) * 128;
  return 2 * static_cast<size_t>(mlbt::H) * tpad * 2;
}

dsa_status_t sparse_mla_bwd_tc_launch(const SparseMlaBwdArgs& a, void* scratch, size_t scratch_bytes,
                                      cudaStream_t stream) {
  using namespace mlbt;
  if (a.H != H) return DSA_ERR_UNSUPPORTED;
  const int64_t nq = static_cast<int64_t>(a.B) * a.Tq;
  const size_t per_q = sparse_mla_bwd_tc_query_bytes(a.topk);
  const int64_t qc_max = static_cast<int64_t>(scratch_bytes / per_q);
  if (scratch == nullptr || qc_max < 1) return DSA_ERR_WORKSPACE_TOO_SMALL;
  const int64_t qc = qc_max < nq ? qc_max : nq;
  Params p{};
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
  p.topk = a.topk;
  p.max_kv_len = a.max_kv_len;
  p.tpad = (a.topk + 127) / 128 * 128;
  p.scale = a.scale;
  p.c1 = a.scale * 1.4426950408889634f;
  p.o = a.o_lat;
  p.lse = a.lse;
  p.dO = a.d_o;
  p.dq = a.dq;
  p.dkv = a.dkv;
  p.status = a.status;
  p.pbuf = static_cast<uint16_t*>(scratch);
  p.zbuf = p.pbuf + static_cast<size_t>(qc) * H * p.tpad;
  const uint64_t qrows = static_cast<uint64_t>(nq) * H;
  CUtensorMap tq48, tdo48, tq96, tdo96, tz, tp;
  if (!encode_tmap_2d(&tq48, a.q_lat, qrows, kRlat, kRlat * 2, 64, HG, true) ||
      !encode_tmap_2d(&tdo48, a.d_o, qrows, kVlat, kVlat * 2, 64, HG, true) ||
      !encode_tmap_2d(&tq96, a.q_lat, qrows, kRlat, kRlat * 2, 64, H, true) ||
      !encode_tmap_2d(&tdo96, a.d_o, qrows, kVlat, kVlat * 2, 64, H, true) ||
      !encode_tmap_2d(&tz, p.zbuf, static_cast<uint64_t>(qc) * H, p.tpad, p.tpad * 2ull, 64, H, true) ||
      !encode_tmap_2d(&tp, p.pbuf, static_cast<uint64_t>(qc) * H, p.tpad, p.tpad * 2ull, 64, H, true))
    return DSA_ERR_CUDA;
  if (cudaFuncSetAttribute(bwd_pz_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, k1::SMEM) != cudaSuccess ||
      cudaFuncSetAttribute(bwd_dq_dkv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KDQ_SMEM) != cudaSuccess)
    return launch_status("cudaFuncSetAttribute");
  for (int64_t q0 = 0; q0 < nq; q0 += qc) {
    const unsigned n = static_cast<unsigned>(nq - q0 < qc ? nq - q0 : qc);
    p.q0 = q0;
    bwd_pz_kernel<<<dim3(2, n), k1::NT, k1::SMEM, stream>>>(tq48, tdo48, p);
    if (launch_status("bwd_pz_kernel") != DSA_OK) return DSA_ERR_CUDA;
    bwd_dq_dkv_kernel<<<4 * n, k3::NT, KDQ_SMEM, stream>>>(tz, tq96, tdo96, tp, p, n);
    if (launch_status("bwd_dq_dkv_kernel") != DSA_OK) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // namespace dsa
