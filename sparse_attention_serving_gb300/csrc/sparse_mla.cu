// sparse_mla.cu -- sparse MLA forward in latent space on sm_103a.
//
// Computes, per query t and head h (the absorbed form of "Kimi-K3.1-Pro",
// NeMo AutoModel, Implementation Limits, bullets 1-2: attend directly to the
// selected latent KV, never expanding per-head K/V; dims from KimiK3TextConfig):
//   z_s  = scale * q_lat[t,h,:] . KV[s,:]          over the 576-wide rows s in idx[t]
//   o    = sum_s softmax(z)_s * KV[s, 0:512],       lse = log sum_s exp(z_s)
//
// One CTA per query (or per query x key-split for small batches):
//   warps 0-3   producer: TMA load of the query's 96x576 q_lat block; 16-byte
//               cp.async gather of the selected rows, 64 keys per block, into a
//               ring of 16 KB "pair" slots (two 64-dim chunks, dims 0..511) and
//               8 KB "rope" slots (dims 512..575), 128-byte swizzled.  (TMA
//               tile::gather4 moves these 1,152-byte rows about 4x slower.)
//   warp 4      tcgen05 issuer (one lane):
//                 S  [128 x 64]  = Q [128(96 heads) x 576] . KV_blk^T   (M=128, N=64)
//                 O^T[512 x 96] += V_blk^T [512 x 64] . P^T [64 x 96]   (4 x M=128, N=96)
//               S double-buffered in TMEM columns 384..511, O^T in 0..383.
//   warps 5-8   softmax (one lane per head; the row max and sum stay in the
//               thread), write P^T as BF16 into shared memory, then the
//               epilogue (O^T / l -> BF16 o_lat, lse).
// Q rows 96..127 of the M=128 operand alias the next 64-dim chunk of Q (or the
// P^T buffer after the last chunk): they only feed accumulator rows no thread
// reads, so 96 heads cost 108 KB of shared memory instead of 144 KB.
#include <cmath>

#include <cuda_bf16.h>

#include "internal.h"
#include "sm103.cuh"

namespace dsa {
namespace mla {

constexpr int BK = 64;                    // keys per block
constexpr int CHUNK = BK * 128;           // 64 keys x 64 dims x 2 B
constexpr int PAIR = 2 * CHUNK;
constexpr int NPAIR = 5;                  // pair slots (a block uses 4)
constexpr int NROPE = 2;                  // rope slots (a block uses 1)
constexpr int MAX_TOPK = 2048;
constexpr int OFF_Q = 0;
constexpr int Q_BYTES = 9 * 96 * 128;     // 110592
constexpr int OFF_P = OFF_Q + Q_BYTES;    // P^T, up to 96 rows x 128 B
constexpr int P_BYTES = 96 * 128;
constexpr int OFF_PAIR = OFF_P + P_BYTES;
constexpr int OFF_ROPE = OFF_PAIR + NPAIR * PAIR;
constexpr int OFF_ROWS = OFF_ROPE + NROPE * CHUNK;
constexpr int OFF_MISC = OFF_ROWS + MAX_TOPK * 4;
constexpr int MISC_BYTES = 2048;
constexpr int SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr int NPROD = 128;                 // producer threads (warps 0-3)
constexpr int MMA_WARP = NPROD / 32;       // warp 4
constexpr int NTHREADS = NPROD + 32 + 128; // + MMA warp + 4 softmax warps
constexpr uint32_t S_COL = 384;

// barrier indices
enum {
  B_Q = 0,
  B_PF = 1,   // pair full [5]
  B_PE = 6,   // pair empty [5]
  B_RF = 11,  // rope full [2]
  B_RE = 13,  // rope empty [2]
  B_SF = 15,  // S full [2]
  B_SE = 17,  // S empty [2]
  B_P = 19,   // P^T written (and O^T rescaled)
  B_O = 20,   // O^T accumulated for a block
  B_DRAIN = 21,
  NBAR = 22
};

// status site tags
enum : uint32_t {
  SITE_QPOS = 0x100, SITE_IDX = 0x101, SITE_PAGE = 0x102,
  SITE_W_Q = 0x110, SITE_W_PE = 0x111, SITE_W_RE = 0x112, SITE_W_PF = 0x113,
  SITE_W_RF = 0x114, SITE_W_SE = 0x115, SITE_W_P = 0x116, SITE_W_SF = 0x117,
  SITE_W_O = 0x118, SITE_W_DRAIN = 0x119
};

struct Params {
  const uint16_t* kv;  // row store base (contiguous or page pool)
  const int32_t* idx;
  const int32_t* q_start;
  const int32_t* kv_len;
  const int32_t* block_table;
  int64_t seq_stride;
  int32_t max_pages, num_pages;
  int paged;
  int Tq, topk, max_kv_len, nsplit;
  float scale_log2;  // scale * log2(e)
  uint16_t* o_lat;
  float* lse;
  float* part_o;     // [q, split, H, 512] normalised partial outputs (nsplit > 1)
  float* part_lse;   // [q, split, H] partial log2-sum-exp
  uint32_t* status;
};

__device__ __forceinline__ bool vload(const volatile int* p) { return *p != 0; }

template <int H>
__global__ void __launch_bounds__(NTHREADS, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const Params p) {
  constexpr int HN = (H + 15) / 16 * 16;  // N of the PV product
  constexpr int QRS = H * 128;            // bytes of one 64-dim chunk of Q
  constexpr uint32_t IDESC_S = idesc_bf16(128, BK, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16(128, HN, true, false);
  static_assert(HN * 4 <= (int)S_COL, "O^T columns");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_MISC);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 24);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* g_abort = s_abort + 1;      // [4] softmax-group abort, by iteration parity x checkpoint
  volatile int* s_resc = s_abort + 5;       // [2] any head needs O^T rescale, by parity
  int* s_nvalid = const_cast<int*>(s_abort + 7);
  int* s_wsum = s_nvalid + 1;               // [16]
  float* s_alpha = reinterpret_cast<float*>(s_wsum + 16);  // [128]
  float* s_invl = s_alpha + 128;                          // [128]
  int32_t* rows = reinterpret_cast<int32_t*>(sm + OFF_ROWS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qflat = blockIdx.x / p.nsplit, sp = blockIdx.x % p.nsplit;
  const int b = qflat / p.Tq, qi = qflat % p.Tq;

  if (tid == 0) {
    for (int k = 0; k < NBAR; ++k) {
      uint32_t cnt = 1;
      if (k == B_SE || k == B_SE + 1 || k == B_P) cnt = 128;
      if ((k >= B_PF && k < B_PF + NPAIR) || (k >= B_RF && k < B_RF + NROPE)) cnt = NPROD;
      mbar_init(&bars[k], cnt);
    }
    s_abort[0] = 0;
    for (int k = 0; k < 4; ++k) g_abort[k] = 0;
    s_resc[0] = 0; s_resc[1] = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }

  // ---- validate and compact the query's index list (stable order) ----------
  const int t = __ldg(p.q_start + b) + qi;
  const int L = __ldg(p.kv_len + b);
  const bool q_ok = t >= 0 && t < L && L <= p.max_kv_len;
  if (!q_ok && tid == 0) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_QPOS, (uint32_t)t);
  constexpr int MAXPER = (MAX_TOPK + NTHREADS - 1) / NTHREADS;
  const int per = (p.topk + NTHREADS - 1) / NTHREADS;
  const int32_t* ix = p.idx + static_cast<int64_t>(qflat) * p.topk;
  int loc[MAXPER];
  int cnt = 0;
#pragma unroll
  for (int u = 0; u < MAXPER; ++u) {
    loc[u] = -1;
    const int e = tid * per + u;
    if (u < per && e < p.topk && q_ok) {
      const int s = __ldg(ix + e);
      if (s >= 0) {
        if (s > t) {
          status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_IDX, (uint32_t)s);
        } else if (p.paged) {
          const int pg = s >> 6;
          const int pid = pg < p.max_pages
                              ? __ldg(p.block_table + static_cast<int64_t>(b) * p.max_pages + pg)
                              : -1;
          if (pid < 0 || pid >= p.num_pages)
            status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_PAGE, (uint32_t)pid);
          else
            loc[u] = pid * kPage + (s & (kPage - 1));
        } else {
          loc[u] = static_cast<int>(static_cast<int64_t>(b) * p.seq_stride + s);
        }
      }
    }
    cnt += loc[u] >= 0 ? 1 : 0;
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_wsum[warp] = incl;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  int off = incl - cnt;
  int n_valid = 0;
  for (int w = 0; w < NTHREADS / 32; ++w) {
    if (w < warp) off += s_wsum[w];
    n_valid += s_wsum[w];
  }
#pragma unroll
  for (int u = 0; u < MAXPER; ++u)
    if (loc[u] >= 0) rows[off++] = loc[u];
  __syncthreads();
  const int nb_total = (n_valid + BK - 1) / BK;
  for (int e = n_valid + tid; e < nb_total * BK; e += NTHREADS) rows[e] = rows[0];
  const int bps = (nb_total + p.nsplit - 1) / p.nsplit;
  const int blk0 = min(sp * bps, nb_total);
  const int nb = min(nb_total, blk0 + bps) - blk0;
  __syncthreads();
  const uint32_t tmem = *tslot;

  if (warp < NPROD / 32) {
    // ====================== producer (4 warps, cp.async) ======================
    // Each 16-byte unit of a selected row is copied by one thread straight into
    // its 128-byte-swizzled place; a warp covers 4 keys x 8 units of one 64-dim
    // chunk (4 x 128 contiguous bytes of global memory).
    const int ptid = tid;  // 0..127
    if (nb > 0) {
      if (ptid == 0) {
        tma_prefetch_desc(&tm_q);
        mbar_expect_tx(&bars[B_Q], 9u * H * 128u);
#pragma unroll 1
        for (int c = 0; c < 9; ++c)
          tma_load_2d(sm + OFF_Q + c * QRS, &tm_q, &bars[B_Q], 64 * c, qflat * H);
      }
      bool ok = true;
      for (int jj = 0; jj < nb && ok; ++jj) {
        const int kb = (blk0 + jj) * BK;  // first list entry of the block
        // parts in the order the MMA consumes them: pair 0, rope, pair 1..3
        for (int part = 0; part < 5; ++part) {
          const bool rope = part == 1;
          const int pr = part == 0 ? 0 : part - 1;  // pair index 0..3
          uint64_t *full, *empty;
          uint32_t use;
          uint8_t* dst;
          if (rope) {
            const int slot = jj % NROPE;
            use = jj / NROPE;
            full = &bars[B_RF + slot];
            empty = &bars[B_RE + slot];
            dst = sm + OFF_ROPE + slot * CHUNK;
          } else {
            const uint32_t g = 4u * jj + pr;
            const int slot = g % NPAIR;
            use = g / NPAIR;
            full = &bars[B_PF + slot];
            empty = &bars[B_PE + slot];
            dst = sm + OFF_PAIR + slot * PAIR;
          }
          if (use > 0 && !mbar_wait(empty, (use - 1) & 1, p.status, kWaitLimitNs,
                                    rope ? SITE_W_RE : SITE_W_PE))
            s_abort[0] = 1;
          if (vload(s_abort)) { ok = false; break; }
          const uint32_t dbase = smem_u32(dst);
          const int nunits = rope ? 4 : 8;  // per thread
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (i < nunits) {
              const int u = ptid + NPROD * i;
              const int ln = u & 31, grp = u >> 5;
              const int h2 = grp >> 4, kg = grp & 15;
              const int key = kg * 4 + (ln >> 3), unit = ln & 7;
              const int c = rope ? 8 : 2 * pr + h2;
              const uint16_t* src =
                  p.kv + static_cast<int64_t>(rows[kb + key]) * kRlat + c * 64 + unit * 8;
              cp_async_16(dbase + h2 * CHUNK + sw128_unit(key, unit), src);
            }
          }
          cp_async_arrive(full);
        }
      }
      // every copy this thread issued has landed before the CTA may exit
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (warp == MMA_WARP) {
    // ============================ MMA issuer =================================
    if (nb > 0 && lane == 0) {
      const uint32_t q_base = smem_u32(sm + OFF_Q);
      const uint32_t p_base = smem_u32(sm + OFF_P);
      bool ok = mbar_wait(&bars[B_Q], 0, p.status, kWaitLimitNs, SITE_W_Q);
      if (!ok) s_abort[0] = 1;
      tc_fence_after();
      auto s_pair = [&](int jj, int pr, uint32_t d, bool& first) -> bool {
        const uint32_t g = 4u * jj + pr;
        const int slot = g % NPAIR;
        if (!mbar_wait(&bars[B_PF + slot], (g / NPAIR) & 1, p.status, kWaitLimitNs, SITE_W_PF))
          return false;
        fence_proxy_async_smem();  // cp.async (generic proxy) writes -> tensor core reads
        tc_fence_after();
        const uint32_t sb = smem_u32(sm + OFF_PAIR + slot * PAIR);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int c = 2 * pr + h2;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            umma_bf16(d, smem_desc(q_base + c * QRS + kk * 32, 16, 1024),
                      smem_desc(sb + h2 * CHUNK + kk * 32, 16, 1024), IDESC_S, first ? 0u : 1u);
            first = false;
          }
        }
        return true;
      };
      auto pv = [&](int jj) -> bool {
        if (!mbar_wait(&bars[B_P], jj & 1, p.status, kWaitLimitNs, SITE_W_P)) return false;
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t g = 4u * jj + i;
          const int slot = g % NPAIR;
          const uint32_t vb = smem_u32(sm + OFF_PAIR + slot * PAIR);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + i * HN, smem_desc(vb + kk * 2048, CHUNK, 1024),
                      smem_desc(p_base + kk * 32, 16, 1024), IDESC_O,
                      (jj > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars[B_PE + slot]);
        }
        umma_commit(&bars[B_O]);
        return true;
      };
      for (int jj = 0; jj < nb && ok; ++jj) {
        if (vload(s_abort)) { ok = false; break; }
        const int sbuf = jj & 1;
        const uint32_t d = tmem + S_COL + BK * sbuf;
        if (jj >= 2 &&
            !mbar_wait(&bars[B_SE + sbuf], ((jj >> 1) - 1) & 1, p.status, kWaitLimitNs,
                       SITE_W_SE)) { ok = false; break; }
        tc_fence_after();
        bool first = true;
        if (!s_pair(jj, 0, d, first)) { ok = false; break; }
        {  // rope chunk
          const int rs = jj % NROPE;
          if (!mbar_wait(&bars[B_RF + rs], (jj / NROPE) & 1, p.status, kWaitLimitNs,
                         SITE_W_RF)) { ok = false; break; }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t rb = smem_u32(sm + OFF_ROPE + rs * CHUNK);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, smem_desc(q_base + 8 * QRS + kk * 32, 16, 1024),
                      smem_desc(rb + kk * 32, 16, 1024), IDESC_S, 1u);
          umma_commit(&bars[B_RE + rs]);
        }
        if (jj >= 1 && !pv(jj - 1)) { ok = false; break; }
        if (!s_pair(jj, 1, d, first) || !s_pair(jj, 2, d, first) || !s_pair(jj, 3, d, first)) {
          ok = false;
          break;
        }
        umma_commit(&bars[B_SF + sbuf]);
      }
      if (ok && !vload(s_abort)) ok = pv(nb - 1);
      if (!ok) s_abort[0] = 1;
      // drain: all issued MMAs complete before TMEM is released
      umma_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, p.status, kWaitLimitNs, SITE_W_DRAIN);
    }
    __syncwarp();
  } else {
    // ====================== softmax + epilogue (warps 5..8) ====================
    const int sub = warp & 3;             // TMEM lane quarter this warp may access
    const int h = sub * 32 + lane;        // head owned in the softmax
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    // l_sum: sum of the BF16-rounded P fed to the PV product (normalises O);
    // l_exact: the unrounded sum (log-sum-exp)
    float m_ref = -INFINITY, l_sum = 0.f, l_exact = 0.f;
    bool ok = true;
    uint8_t* prow = sm + OFF_P;
    for (int jj = 0; jj < nb; ++jj) {
      const int sbuf = jj & 1;
      bool w_ok = mbar_wait(&bars[B_SF + sbuf], (jj >> 1) & 1, p.status, kWaitLimitNs, SITE_W_SF);
      if (!w_ok || vload(s_abort)) { g_abort[(jj & 1) * 2] = 1; }
      named_bar_sync(1, 128);
      if (vload(&g_abort[(jj & 1) * 2])) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[64];
      {
        uint32_t(&a)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
        uint32_t(&c)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
        tmem_ld32(tmem + lane_base + S_COL + BK * sbuf, a);
        tmem_ld32(tmem + lane_base + S_COL + BK * sbuf + 32, c);
      }
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&bars[B_SE + sbuf]);
      const int kb = (blk0 + jj) * BK;
      const int nvk = min(BK, n_valid - kb);
      float z[64];
      float mb = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        z[c] = c < nvk ? __uint_as_float(sr[c]) * p.scale_log2 : -INFINITY;
        mb = fmaxf(mb, z[c]);
      }
      // lazy reference max: keep the current one unless this block exceeds it by
      // more than 2^64; P = 2^(z - m_ref) then stays far inside the FP32/BF16 range
      float m_new = m_ref;
      if (mb > m_ref + 64.f) m_new = mb;
      const float alpha = (m_new == m_ref) ? 1.f : exp2f(m_ref - m_new);
      l_sum *= alpha;
      l_exact *= alpha;
      uint32_t pk[32];
      float lsum_blk = 0.f, lex_blk = 0.f;
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float p0 = exp2f(z[c] - m_new), p1 = exp2f(z[c + 1] - m_new);
        const uint32_t v = pack_bf16x2(p0, p1);
        pk[c >> 1] = v;
        lsum_blk += __uint_as_float(v << 16) + __uint_as_float(v & 0xffff0000u);
        lex_blk += p0 + p1;
      }
      l_sum += lsum_blk;
      l_exact += lex_blk;
      m_ref = m_new;
      // P^T buffer and O^T are free once the previous block's PV product is done
      if (jj >= 1) {
        w_ok = mbar_wait(&bars[B_O], (jj - 1) & 1, p.status, kWaitLimitNs, SITE_W_O);
        if (!w_ok || vload(s_abort)) g_abort[(jj & 1) * 2 + 1] = 1;
      }
      s_alpha[h] = alpha;
      if (jj >= 1 && h < H && alpha != 1.f) s_resc[jj & 1] = 1;
      named_bar_sync(1, 128);
      if (vload(&g_abort[(jj & 1) * 2 + 1])) { ok = false; break; }
      tc_fence_after();
      if (vload(&s_resc[jj & 1])) {
        // rare: rescale every O^T column by its head's alpha
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
#pragma unroll 1
          for (int c0 = 0; c0 < HN; c0 += 16) {
            uint32_t r[16];
            const uint32_t ta = tmem + lane_base + i * HN + c0;
            tmem_ld16(ta, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e)
              r[e] = __float_as_uint(__uint_as_float(r[e]) * s_alpha[c0 + e]);
            tmem_st16(ta, r);
          }
        }
        tmem_st_wait();
      }
      // write this head's row of P^T (K-major: row = head, 64 keys = 128 B)
      if (h < HN) {
        uint8_t* row = prow + (h >> 3) * 1024 + (h & 7) * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint4 v;
          if (h < H)
            v = make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          else
            v = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(row + (((u ^ h) & 7) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 128);
      if (warp == MMA_WARP + 1 && lane == 0) s_resc[jj & 1] = 0;  // reused two blocks later, after two barriers
      mbar_arrive(&bars[B_P]);
    }
    // ------------------------------ epilogue ---------------------------------
    if (h < H) s_invl[h] = l_sum > 0.f ? 1.f / l_sum : 0.f;
    float lse2 = (l_exact > 0.f) ? m_ref + log2f(l_exact) : -INFINITY;
    bool have_o = ok && nb > 0;
    if (have_o) {
      const bool w_ok = mbar_wait(&bars[B_O], (nb - 1) & 1, p.status, kWaitLimitNs, SITE_W_O);
      if (!w_ok) have_o = false;
    }
    named_bar_sync(1, 128);
    tc_fence_after();
    if (p.nsplit == 1) {
      if (h < H && p.lse != nullptr)
        p.lse[static_cast<int64_t>(qflat) * H + h] = have_o ? lse2 * 0.6931471805599453f : -INFINITY;
      uint16_t* ob = p.o_lat + static_cast<int64_t>(qflat) * H * kVlat;
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        const int dim = 128 * i + 32 * sub + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < HN; c0 += 16) {
          uint32_t r[16];
          if (have_o) {
            tmem_ld16(tmem + lane_base + i * HN + c0, r);
            tmem_ld_wait();
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int hh = c0 + e;
            if (hh < H) {
              const float v = have_o ? __uint_as_float(r[e]) * s_invl[hh] : 0.f;
              ob[static_cast<int64_t>(hh) * kVlat + dim] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
            }
          }
        }
      }
    } else {
      const int64_t pq = static_cast<int64_t>(qflat) * p.nsplit + sp;
      if (h < H) p.part_lse[pq * H + h] = have_o ? lse2 : -INFINITY;
      float* ob = p.part_o + pq * H * kVlat;
#pragma unroll 1
      for (int i = 0; i < 4; ++i) {
        const int dim = 128 * i + 32 * sub + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < HN; c0 += 16) {
          uint32_t r[16];
          if (have_o) {
            tmem_ld16(tmem + lane_base + i * HN + c0, r);
            tmem_ld_wait();
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int hh = c0 + e;
            if (hh < H)
              ob[static_cast<int64_t>(hh) * kVlat + dim] =
                  have_o ? __uint_as_float(r[e]) * s_invl[hh] : 0.f;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the per-split partial results: lse = log2 sum_p 2^lse_p,
// o = sum_p 2^(lse_p - lse) o_p.  One thread per (query, head, 4 dims).
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      int nq, int H, int nsplit,
                                                      uint16_t* __restrict__ o_lat,
                                                      float* __restrict__ lse) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_qh = kVlat / 4;
  if (gid >= static_cast<int64_t>(nq) * H * per_qh) return;
  const int64_t qh = gid / per_qh;
  const int d4 = static_cast<int>(gid % per_qh) * 4;
  const int64_t q = qh / H, h = qh % H;
  float mx = -INFINITY;
  for (int s = 0; s < nsplit; ++s) mx = fmaxf(mx, part_lse[(q * nsplit + s) * H + h]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float ls = part_lse[(q * nsplit + s) * H + h];
      if (ls == -INFINITY) continue;
      const float wgt = exp2f(ls - mx);
      wsum += wgt;
      const float4 v =
          *reinterpret_cast<const float4*>(part_o + ((q * nsplit + s) * H + h) * kVlat + d4);
      acc[0] += wgt * v.x; acc[1] += wgt * v.y; acc[2] += wgt * v.z; acc[3] += wgt * v.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint16_t* o = o_lat + qh * kVlat + d4;
  const uint32_t lo = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  const uint32_t hi = pack_bf16x2(acc[2] * inv, acc[3] * inv);
  *reinterpret_cast<uint2*>(o) = make_uint2(lo, hi);
  if (d4 == 0 && lse != nullptr)
    lse[qh] = wsum > 0.f ? (mx + log2f(wsum)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace mla

static int mla_nsplit(int B, int Tq) {
  const int nq = B * Tq;
  const int sms = num_sms();
  if (nq >= sms) return 1;
  int ns = sms / nq;
  return ns < 1 ? 1 : (ns > 8 ? 8 : ns);
}

size_t sparse_mla_scratch_bytes(int B, int Tq, int H, int topk) {
  (void)topk;
  const int ns = mla_nsplit(B, Tq);
  if (ns <= 1) return 0;
  const size_t nq = static_cast<size_t>(B) * Tq;
  return nq * ns * H * (kVlat + 1) * sizeof(float) + 256;
}

template <int H>
static dsa_status_t launch_h(const SparseMlaArgs& a, cudaStream_t stream) {
  using namespace mla;
  CUtensorMap tq;
  const uint64_t qrows = static_cast<uint64_t>(a.B) * a.Tq * H;
  if (!encode_tmap_2d(&tq, a.q_lat, qrows, kRlat, kRlat * 2, 64, H, true))
    return DSA_ERR_CUDA;
  const int ns = mla_nsplit(a.B, a.Tq);
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
  p.nsplit = ns;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.o_lat = a.o_lat;
  p.lse = a.lse;
  p.status = a.status;
  if (ns > 1) {
    const size_t nq = static_cast<size_t>(a.B) * a.Tq;
    if (a.scratch == nullptr || a.scratch_bytes < sparse_mla_scratch_bytes(a.B, a.Tq, H, a.topk))
      return DSA_ERR_WORKSPACE_TOO_SMALL;
    p.part_o = static_cast<float*>(a.scratch);
    p.part_lse = p.part_o + nq * ns * H * kVlat;
  }
  auto kern = sparse_mla_kernel<H>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(a.B) * a.Tq * ns);
  kern<<<grid, NTHREADS, SMEM_BYTES, stream>>>(tq, p);
  if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  if (ns > 1) {
    const int64_t nq = static_cast<int64_t>(a.B) * a.Tq;
    const int64_t threads = nq * H * (kVlat / 4);
    combine_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
        p.part_o, p.part_lse, static_cast<int>(nq), H, ns, a.o_lat, a.lse);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

dsa_status_t sparse_mla_launch(const SparseMlaArgs& a, cudaStream_t stream) {
  if (a.H == 96) return launch_h<96>(a, stream);
  if (a.H == 8) return launch_h<8>(a, stream);
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
