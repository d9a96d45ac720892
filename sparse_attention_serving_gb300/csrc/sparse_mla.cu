// sparse_mla.cu -- sparse MLA forward in latent space on sm_103a.
//
// Computes, per query t and head h (the absorbed form of "Kimi-K3.1-Pro",
// NeMo AutoModel, Implementation Limits, bullets 1-2: attend directly to the
// selected latent KV, never expanding per-head K/V; dims from KimiK3TextConfig):
//   z_s  = scale * q_lat[t,h,:] . KV[s,:]          over the 576-wide rows s in idx[t]
//   o    = sum_s softmax(z)_s * KV[s, 0:512],       lse = log sum_s exp(z_s)
//
// Persistent CTAs, one per SM, walk units -- a query, or a query x key split
// for small batches -- round robin; each unit is processed in blocks of 64
// list entries, and the next unit's index scan, query load, first gathers and
// first score products overlap the current unit's last blocks and epilogue
// (barrier phases run off a per-CTA block counter that continues across
// units).  Roles:
//   warps 0-5   producer: per unit, the index scan (last valid entry, bad
//               entries flagged) published to the other roles; TMA load of
//               the query's 96x576 q_lat block once the previous unit's score
//               products are done with it; 16-byte
//               cp.async gather of the selected rows into a ring of six 16 KB
//               "pair" slots (two 64-dim chunks, dims 0..511) and one 8 KB
//               "rope" slot (dims 512..575), 128-byte swizzled.  Each thread
//               copies one 16-byte unit of up to three fixed keys, so its
//               shared and global addresses are computed once per block.
//               (TMA tile::gather4 moves these 1,152-byte rows about 4x slower;
//               six gathering warps instead of four keep the 512-thread CTA
//               at 128 registers and shorten the decode gathers from DRAM.)
//   warps 6-13  softmax (two warps per TMEM lane quarter: a thread owns one
//               head and 32 of the block's 64 keys; P = 2^(z - m_ref) against
//               a lazy reference max, which only moves -- through a rarer,
//               synchronised path that rescales O^T -- when an exponent would
//               exceed 64), P^T written as BF16, then the unit's epilogue
//               (O^T / l written straight from registers, 32 consecutive dims
//               per warp and head, and lse).
//   warp 14     tcgen05 issuer of the scores (one lane), TMEM owner:
//                 S  [128 x 64]  = Q [128(96 heads) x 576] . KV_blk^T   (M=128, N=64)
//   warp 15     tcgen05 issuer of the value product (one lane):
//                 O^T[512 x 96] += V_blk^T [512 x 64] . P^T [64 x 96]   (4 x M=128, N=96)
//               S double-buffered in TMEM columns 384..511, O^T in 0..383.
//               With six pair slots, the first two pairs and the rope chunk of
//               block j+1 are multiplied while the softmax of block j runs; two
//               issuers let the value product of block j start the moment P^T
//               is written, whatever loads the score issuer is waiting on, so
//               the slots it frees reach the producer sooner.
// Per 64-key block the tensor core reads about 328 KB of operands from shared
// memory (Q alone is 144 KB of it) and the gather writes 72 KB, so the shared
// memory port (128 B/clk) rather than the gather or the tensor pipe sets the
// floor; more producer warps only contend for it.
// Q rows 96..127 of the M=128 operand alias the next 64-dim chunk of Q (or the
// P^T buffer after the last chunk): they only feed accumulator rows no thread
// reads, so 96 heads cost 108 KB of shared memory instead of 144 KB.
//
// The index list is not compacted: a block covers 64 consecutive list entries
// and entries that are -1 (or invalid, which is also flagged) are masked out
// of the softmax.  Blocks run up to the last valid entry, so a list with its
// valid entries first (as dsa_indexer_topk writes it) wastes no work.
#include <cmath>

#include <cuda_bf16.h>

#include "internal.h"
#include "sm103.cuh"

namespace dsa {
namespace mla {

constexpr int BK = 64;                    // list entries (keys) per block
constexpr int CHUNK = BK * 128;           // 64 keys x 64 dims x 2 B
constexpr int PAIR = 2 * CHUNK;
constexpr int NPAIR = 6;                  // pair slots (a block uses 4)
constexpr int MAX_TOPK = 2048;
constexpr int OFF_Q = 0;
constexpr int Q_BYTES = 9 * 96 * 128;     // 110592
constexpr int OFF_P = OFF_Q + Q_BYTES;    // P^T, up to 96 rows x 128 B
constexpr int P_BYTES = 96 * 128;
constexpr int OFF_PAIR = OFF_P + P_BYTES;
constexpr int OFF_ROPE = OFF_PAIR + NPAIR * PAIR;
constexpr int OFF_MISC = OFF_ROPE + CHUNK;
constexpr int MISC_BYTES = 2048;
constexpr int SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Roles: warps 0-5 producer, 6-13 softmax, 14 score issuer, 15 value issuer.
constexpr int NPROD = 192;                        // producer threads (warps 0-5)
constexpr int NPW = NPROD / 32;
constexpr int KROW = 4 * NPW;                     // keys one pass of the producers covers
constexpr int KPT = (BK + KROW - 1) / KROW;       // keys per producer thread (the last partly)
constexpr int SMX_WARP0 = NPW;                    // warps 6-13
constexpr int NSMX = 256;                         // softmax / epilogue threads
constexpr int MMA_WARP = SMX_WARP0 + NSMX / 32;   // warp 14: scores, TMEM owner
constexpr int PV_WARP = MMA_WARP + 1;             // warp 15: value product
constexpr int NTHREADS = NPROD + NSMX + 64;
static_assert(KPT * KROW >= BK && (KPT - 1) * KROW < BK, "producer key split");
// 16 warps at 128 registers: the 4 warps that share an SM sub-partition
// exactly fill its 16K-register file.
static_assert(NTHREADS <= 512, "register budget of the 128-register build");
constexpr uint32_t S_COL = 384;

// barrier indices
enum {
  B_Q = 0,              // query block landed
  B_QE = 1,             // query block free: the unit's last score MMA is done
  B_PF = 2,             // pair full [6]
  B_PE = B_PF + NPAIR,  // pair empty [6]
  B_RF = B_PE + NPAIR,  // rope full
  B_RE = B_RF + 1,      // rope empty
  B_SF = B_RE + 1,      // S full [2]
  B_SE = B_SF + 2,      // S empty [2]
  B_P = B_SE + 2,       // P^T written (common path)
  B_RARE = B_P + 1,     // rare path done: P^T rewritten, O^T rescaled
  B_O = B_RARE + 1,     // O^T accumulated for a block
  B_OE = B_O + 1,       // O^T read out by the unit's epilogue
  B_INFO_F = B_OE + 1,  // unit info published [2]
  B_INFO_E = B_INFO_F + 2,  // unit info read by the three consumer roles [2]
  B_DRAIN = B_INFO_E + 2,
  NBAR = B_DRAIN + 1
};
static_assert(NBAR * 8 <= 232, "barriers overlap the unit-info ring");

// status site tags
enum : uint32_t {
  SITE_QPOS = 0x100, SITE_IDX = 0x101, SITE_PAGE = 0x102,
  SITE_W_Q = 0x110, SITE_W_PE = 0x111, SITE_W_RE = 0x112, SITE_W_PF = 0x113,
  SITE_W_RF = 0x114, SITE_W_SE = 0x115, SITE_W_P = 0x116, SITE_W_SF = 0x117,
  SITE_W_O = 0x118, SITE_W_DRAIN = 0x119, SITE_W_QE = 0x11a, SITE_W_OE = 0x11b,
  SITE_W_INFO = 0x11c
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
  int B, Tq, topk, max_kv_len, nsplit;
  float scale_log2;  // scale * log2(e)
  uint16_t* o_lat;
  float* lse;
  const float* sink;  // [H] learnable sink logits (natural log), or null
  uint16_t* part_o;  // [q, split, H, 512] normalised partial outputs, BF16 (nsplit > 1)
  float* part_lse;   // [q, split, H] partial log2-sum-exp
  uint32_t* status;
};

__device__ __forceinline__ bool vload(const volatile int* p) { return *p != 0; }

// mbar_wait that gives up quietly (no status) once another role has aborted.
__device__ __forceinline__ bool mbar_wait_unless(uint64_t* bar, uint32_t parity,
                                                 const volatile int* abort_flag,
                                                 uint32_t* status, uint32_t where) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_test(bar, parity)) return true;
    if (vload(abort_flag)) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      status_raise(status, DSA_ERR_DEVICE_TIMEOUT, where);
      return false;
    }
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Physical row of list entry s for the query at position t of sequence b, or
// -1 when the entry is unused (-1) or invalid (not causal, page outside the pool).
__device__ __forceinline__ int entry_row(const Params& p, int b, int t, int s) {
  if (s < 0 || s > t) return -1;
  if (p.paged) {
    const int pg = s >> 6;
    const int pid =
        pg < p.max_pages ? __ldg(p.block_table + static_cast<int64_t>(b) * p.max_pages + pg) : -1;
    if (pid < 0 || pid >= p.num_pages) return -1;
    return pid * kPage + (s & (kPage - 1));
  }
  return static_cast<int>(static_cast<int64_t>(b) * p.seq_stride + s);
}

// One unit of work: a query, or a query x key split.  Rows are resolved the
// same way by every role.
struct Unit {
  int qflat, sp, b, t;
  bool q_ok;
  const int32_t* ix;
};
__device__ __forceinline__ Unit unit_of(const Params& p, int u) {
  Unit w;
  w.qflat = u / p.nsplit;
  w.sp = u % p.nsplit;
  w.b = w.qflat / p.Tq;
  const int qi = w.qflat % p.Tq;
  w.t = __ldg(p.q_start + w.b) + qi;
  const int L = __ldg(p.kv_len + w.b);
  w.q_ok = w.t >= 0 && w.t < L && L <= p.max_kv_len;
  w.ix = p.idx + static_cast<int64_t>(w.qflat) * p.topk;
  return w;
}

// Persistent: CTA c takes units c, c + gridDim.x, ...  Every per-block barrier
// phase runs off a per-CTA block counter that continues across units, so the
// next unit's index scan, query load, first gathers and first score products
// overlap the current unit's last blocks and epilogue.
template <int H>
__global__ void __launch_bounds__(NTHREADS, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q, const Params p) {
  constexpr int HN = (H + 15) / 16 * 16;  // N of the PV product
  constexpr int QRS = H * 128;            // bytes of one 64-dim chunk of Q
  constexpr uint32_t IDESC_S = idesc_bf16(128, BK, false, false);
  constexpr uint32_t IDESC_O = idesc_bf16(128, HN, true, false);
  static_assert(HN * 4 <= (int)S_COL, "O^T columns");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_MISC);           // NBAR (<= 29)
  int* s_info = reinterpret_cast<int*>(sm + OFF_MISC + 232);             // [2][3] unit info ring
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_MISC + 256);
  volatile int* s_abort = reinterpret_cast<volatile int*>(sm + OFF_MISC + 260);
  volatile int* g_abort = s_abort + 1;  // [3] softmax-group abort, by block mod 3
  volatile int* s_resc = s_abort + 4;   // [3] some head needs an O^T rescale, by block mod 3
  int* s_red = reinterpret_cast<int*>(sm + OFF_MISC + 288);              // [2][8] producer scan
  float* s_cmax = reinterpret_cast<float*>(sm + OFF_MISC + 352);         // [2][128] rare path
  float* s_alpha = s_cmax + 256;                                         // [128] rare path
  volatile uint8_t* s_hover = reinterpret_cast<volatile uint8_t*>(s_alpha + 128);  // [128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nunits = p.B * p.Tq * p.nsplit;

  if (tid == 0) {
    for (int k = 0; k < NBAR; ++k) {
      uint32_t cnt = 1;
      if (k == B_SE || k == B_SE + 1 || k == B_P || k == B_RARE || k == B_OE) cnt = NSMX;
      if (k == B_DRAIN) cnt = 2;  // both issuers
      if (k == B_INFO_E || k == B_INFO_E + 1) cnt = 3;  // score issuer, value issuer, softmax
      if ((k >= B_PF && k < B_PF + NPAIR) || k == B_RF) cnt = NPROD;
      mbar_init(&bars[k], cnt);
    }
    s_abort[0] = 0;
    for (int k = 0; k < 3; ++k) { g_abort[k] = 0; s_resc[k] = 0; }
    for (int k = 0; k < 128; ++k) s_hover[k] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    // the first unit's query block does not depend on its index list: start it
    // now (a unit loads its query block iff it has blocks or is the first one)
    if (blockIdx.x < nunits) {
      mbar_expect_tx(&bars[B_Q], 9u * H * 128u);
#pragma unroll 1
      for (int c = 0; c < 9; ++c)
        tma_load_2d(sm + OFF_Q + c * QRS, &tm_q, &bars[B_Q], 64 * c,
                    (static_cast<int>(blockIdx.x) / p.nsplit) * H);
    }
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp < SMX_WARP0) {
    // ====================== producer (6 warps, cp.async) ======================
    // Per unit: validate the index list (one batched load round trip) and
    // publish (n_list, nb, blk0); load the query block once the previous
    // unit's score products are done with it; gather the unit's blocks.
    // thread: 16-byte unit u = lane & 7 of keys 4w + (lane >> 3) + 24i, i = 0..2
    // (the last pass covers keys 48..63 only: warps 0-3)
    const int w = warp, unit = lane & 7;
    int key[KPT];
    uint32_t doff[KPT];
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      key[i] = 4 * w + (lane >> 3) + KROW * i;  // >= BK: no key (the last pass is partial)
      doff[i] = sw128_unit(key[i] < BK ? key[i] : 0, unit);
    }
    bool ok = true;
    int gb = 0, qcnt = 0, it = 0;
    for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++it) {
      const Unit U = unit_of(p, u);
      if (!U.q_ok && tid == 0) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_QPOS, (uint32_t)U.t);
      // ---- scan: last valid entry (topk <= MAX_TOPK is checked on the host) ----
      constexpr int SCAN = (MAX_TOPK + NPROD - 1) / NPROD;
      int sv[SCAN];
#pragma unroll
      for (int i = 0; i < SCAN; ++i) {
        const int e = tid + i * NPROD;
        sv[i] = (U.q_ok && e < p.topk) ? __ldg(U.ix + e) : -1;
      }
      // paged: the block-table entries of all of them in a second batch (the
      // same checks as entry_row, without one dependent load per entry)
      int pid[SCAN];
#pragma unroll
      for (int i = 0; i < SCAN; ++i) {
        const int s = sv[i], pg = s >> 6;
        pid[i] = (p.paged && s >= 0 && s <= U.t && pg < p.max_pages)
                     ? __ldg(p.block_table + static_cast<int64_t>(U.b) * p.max_pages + pg)
                     : 0;
      }
      int last = -1;
#pragma unroll
      for (int i = 0; i < SCAN; ++i) {
        const int s = sv[i];
        if (s < 0) continue;
        const bool valid = s <= U.t && (!p.paged || ((s >> 6) < p.max_pages && pid[i] >= 0 &&
                                                     pid[i] < p.num_pages));
        if (valid) {
          last = tid + i * NPROD;
        } else if (U.sp == 0) {
          status_raise(p.status, DSA_ERR_BAD_INDEX, s > U.t ? SITE_IDX : SITE_PAGE, (uint32_t)s);
        }
      }
      last = __reduce_max_sync(0xffffffffu, last);
      int* red = s_red + (it & 1) * 8;
      if (lane == 0) red[w] = last;
      named_bar_sync(2, NPROD);
      int n_list = -1;
#pragma unroll
      for (int k = 0; k < NPW; ++k) n_list = max(n_list, red[k]);
      n_list += 1;  // entries [0, n_list) hold every valid key
      const int nb_total = (n_list + BK - 1) / BK;
      const int bps = (nb_total + p.nsplit - 1) / p.nsplit;
      const int blk0 = min(U.sp * bps, nb_total);
      const int nb = min(nb_total, blk0 + bps) - blk0;
      if (tid == 0) {
        const int slot = it & 1;
        if (it >= 2 &&
            !mbar_wait(&bars[B_INFO_E + slot], ((it >> 1) - 1) & 1, p.status, kWaitLimitNs,
                       SITE_W_INFO))
          s_abort[0] = 1;
        s_info[slot * 3 + 0] = n_list;
        s_info[slot * 3 + 1] = nb;
        s_info[slot * 3 + 2] = blk0;
        mbar_arrive(&bars[B_INFO_F + slot]);  // release: the info is visible to the waiters
        if (it > 0 && nb > 0 && !vload(s_abort)) {
          // the query block: once the previous unit's score products have read it
          if (qcnt >= 1 && !mbar_wait(&bars[B_QE], (qcnt - 1) & 1, p.status, kWaitLimitNs, SITE_W_QE))
            s_abort[0] = 1;
          mbar_expect_tx(&bars[B_Q], 9u * H * 128u);
#pragma unroll 1
          for (int c = 0; c < 9; ++c)
            tma_load_2d(sm + OFF_Q + c * QRS, &tm_q, &bars[B_Q], 64 * c, U.qflat * H);
        }
      }
      if (nb > 0 || it == 0) ++qcnt;
      // a valid physical row to read in place of unused entries (masked later)
      const int dummy_row =
          p.paged ? 0 : static_cast<int>(static_cast<int64_t>(U.b) * p.seq_stride);
      // raw list entries of the next block, fetched one block ahead
      int s_next[KPT];
#pragma unroll
      for (int i = 0; i < KPT; ++i) {
        const int e = blk0 * BK + key[i];
        s_next[i] = (nb > 0 && key[i] < BK && e < n_list) ? __ldg(U.ix + e) : -1;
      }
      for (int jj = 0; jj < nb && ok; ++jj) {
        const int gbj = gb + jj;
        const uint16_t* src[KPT];
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
          const int r = entry_row(p, U.b, U.t, s_next[i]);
          src[i] = p.kv + static_cast<int64_t>(r >= 0 ? r : dummy_row) * kRlat + unit * 8;
        }
#pragma unroll
        for (int i = 0; i < KPT; ++i) {
          const int e = (blk0 + jj + 1) * BK + key[i];
          s_next[i] = (jj + 1 < nb && key[i] < BK && e < n_list) ? __ldg(U.ix + e) : -1;
        }
        if (p.nsplit > 1) {
          // split units (decode): the rows come from HBM, not L2.  Ask L2 for
          // the next block's rows now (the 8 threads of a key take one
          // 128-byte chunk each, the first also the ninth), so their gather
          // one block later finds them there.
#pragma unroll
          for (int i = 0; i < KPT; ++i) {
            const int r = entry_row(p, U.b, U.t, s_next[i]);
            if (r >= 0) {
              const uint16_t* row = p.kv + static_cast<int64_t>(r) * kRlat;
              prefetch_l2(row + unit * 64);
              if (unit == 0) prefetch_l2(row + 8 * 64);
            }
          }
        }
        // parts in the order the MMA consumes them: pair 0, pair 1, rope, pair 2, pair 3
        for (int part = 0; part < 5; ++part) {
          const bool rope = part == 2;
          const int pr = part < 2 ? part : part - 1;  // pair index 0..3
          uint64_t *full, *empty;
          uint32_t use;
          uint32_t dbase;
          if (rope) {
            use = gbj;
            full = &bars[B_RF];
            empty = &bars[B_RE];
            dbase = smem_u32(sm + OFF_ROPE);
          } else {
            const uint32_t g = 4u * gbj + pr;
            const int slot = g % NPAIR;
            use = g / NPAIR;
            full = &bars[B_PF + slot];
            empty = &bars[B_PE + slot];
            dbase = smem_u32(sm + OFF_PAIR + slot * PAIR);
          }
          if (use > 0 && !mbar_wait(empty, (use - 1) & 1, p.status, kWaitLimitNs,
                                    rope ? SITE_W_RE : SITE_W_PE))
            s_abort[0] = 1;
          if (vload(s_abort)) { ok = false; break; }
          if (rope) {
#pragma unroll
            for (int i = 0; i < KPT; ++i)
              if (key[i] < BK) cp_async_16(dbase + doff[i], src[i] + 8 * 64);
          } else {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
              for (int i = 0; i < KPT; ++i)
                if (key[i] < BK) cp_async_16(dbase + h2 * CHUNK + doff[i], src[i] + (2 * pr + h2) * 64);
          }
          cp_async_arrive(full);
        }
      }
      gb += nb;
      // one decision for all producer threads (they meet at a named barrier in
      // the next unit's scan, so none may leave the loop alone)
      ok = !named_bar_or(2, NPROD, !ok || vload(s_abort));
    }
    // every copy this thread issued has landed before the CTA may exit
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp >= MMA_WARP) {
    if (warp == MMA_WARP) {
      // ========================== score issuer ================================
      if (lane == 0) {
        const uint64_t qd0 = smem_desc(smem_u32(sm + OFF_Q), 16, 1024);
        const uint64_t rd0 = smem_desc(smem_u32(sm + OFF_ROPE), 16, 1024);
        bool ok = true;
        int gb = 0, qcnt = 0, it = 0;
        auto s_pair = [&](int gbj, int pr, uint32_t d, bool& first) -> bool {
          const uint32_t g = 4u * gbj + pr;
          const int slot = g % NPAIR;
          if (!mbar_wait(&bars[B_PF + slot], (g / NPAIR) & 1, p.status, kWaitLimitNs, SITE_W_PF))
            return false;
          fence_proxy_async_smem();  // cp.async (generic proxy) writes -> tensor core reads
          tc_fence_after();
          const uint64_t sd = smem_desc(smem_u32(sm + OFF_PAIR + slot * PAIR), 16, 1024);
          const uint64_t qd = desc_add(qd0, 2 * pr * QRS);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              umma_bf16(d, desc_add(qd, h2 * QRS + kk * 32), desc_add(sd, h2 * CHUNK + kk * 32),
                        IDESC_S, first ? 0u : 1u);
              first = false;
            }
          }
          return true;
        };
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++it) {
          const int slot = it & 1;
          if (!mbar_wait_unless(&bars[B_INFO_F + slot], (it >> 1) & 1, s_abort, p.status,
                                SITE_W_INFO)) { ok = false; break; }
          const int nb = s_info[slot * 3 + 1];
          mbar_arrive(&bars[B_INFO_E + slot]);
          if (nb == 0 && it > 0) continue;
          if (!mbar_wait_unless(&bars[B_Q], qcnt & 1, s_abort, p.status, SITE_W_Q)) {
            ok = false;
            break;
          }
          if (nb == 0) {  // the first unit's query block, loaded before its scan
            umma_commit(&bars[B_QE]);
            ++qcnt;
            continue;
          }
          tc_fence_after();
          for (int jj = 0; jj < nb && ok; ++jj) {
            if (vload(s_abort)) { ok = false; break; }
            const int gbj = gb + jj;
            const int sbuf = gbj & 1;
            const uint32_t d = tmem + S_COL + BK * sbuf;
            if (gbj >= 2 &&
                !mbar_wait(&bars[B_SE + sbuf], ((gbj >> 1) - 1) & 1, p.status, kWaitLimitNs,
                           SITE_W_SE)) { ok = false; break; }
            tc_fence_after();
            bool first = true;
            if (!s_pair(gbj, 0, d, first) || !s_pair(gbj, 1, d, first)) { ok = false; break; }
            {  // rope chunk
              if (!mbar_wait(&bars[B_RF], gbj & 1, p.status, kWaitLimitNs, SITE_W_RF)) {
                ok = false;
                break;
              }
              fence_proxy_async_smem();
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_bf16(d, desc_add(qd0, 8 * QRS + kk * 32), desc_add(rd0, kk * 32), IDESC_S, 1u);
              umma_commit(&bars[B_RE]);
            }
            if (!s_pair(gbj, 2, d, first) || !s_pair(gbj, 3, d, first)) { ok = false; break; }
            umma_commit(&bars[B_SF + sbuf]);
          }
          // the query block is free once these score products are done
          umma_commit(&bars[B_QE]);
          ++qcnt;
          gb += nb;
        }
        if (!ok) s_abort[0] = 1;
        // drain: all issued MMAs complete before TMEM is released
        umma_commit(&bars[B_DRAIN]);
        mbar_wait(&bars[B_DRAIN], 0, p.status, kWaitLimitNs, SITE_W_DRAIN);
      }
      __syncwarp();
    } else if (warp == PV_WARP) {
      // ======================= value-product issuer ===========================
      if (lane == 0) {
        const uint64_t pd0 = smem_desc(smem_u32(sm + OFF_P), 16, 1024);
        bool ok = true;
        uint32_t nrare = 0;
        int gb = 0, qcnt = 0, it = 0;
        auto pv = [&](int gbj, bool first_blk) -> bool {
          if (!mbar_wait_unless(&bars[B_P], gbj & 1, s_abort, p.status, SITE_W_P)) return false;
          if (vload(&s_resc[gbj % 3])) {
            if (!mbar_wait_unless(&bars[B_RARE], nrare & 1, s_abort, p.status, SITE_W_P))
              return false;
            ++nrare;
          }
          fence_proxy_async_smem();
          tc_fence_after();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t g = 4u * gbj + i;
            const int slot = g % NPAIR;
            const uint64_t vd = smem_desc(smem_u32(sm + OFF_PAIR + slot * PAIR), CHUNK, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16(tmem + i * HN, desc_add(vd, kk * 2048), desc_add(pd0, kk * 32), IDESC_O,
                        (!first_blk || kk > 0) ? 1u : 0u);
            umma_commit(&bars[B_PE + slot]);
          }
          umma_commit(&bars[B_O]);
          return true;
        };
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x, ++it) {
          const int slot = it & 1;
          if (!mbar_wait_unless(&bars[B_INFO_F + slot], (it >> 1) & 1, s_abort, p.status,
                                SITE_W_INFO)) { ok = false; break; }
          const int nb = s_info[slot * 3 + 1];
          mbar_arrive(&bars[B_INFO_E + slot]);
          if (nb == 0) continue;
          // O^T is free once the previous unit's epilogue has read it out
          if (qcnt >= 1 && !mbar_wait_unless(&bars[B_OE], (qcnt - 1) & 1, s_abort, p.status,
                                              SITE_W_OE)) { ok = false; break; }
          tc_fence_after();
          for (int jj = 0; jj < nb && ok; ++jj) ok = pv(gb + jj, jj == 0);
          ++qcnt;
          gb += nb;
        }
        if (!ok) s_abort[0] = 1;
        umma_commit(&bars[B_DRAIN]);
        mbar_wait(&bars[B_DRAIN], 0, p.status, kWaitLimitNs, SITE_W_DRAIN);
      }
      __syncwarp();
    }
  } else {
    // ================ softmax + epilogue (warps 4..11, 8 warps) ================
    // Two warps per TMEM lane quarter: thread (half, h) owns head h and the
    // keys 32*half .. 32*half+31 of each block.  Both halves of a head move the
    // reference max together (through s_cmax, on the rare path only).
    const int sub = warp & 3;                         // TMEM lane quarter
    const int half = (warp - SMX_WARP0) >> 2;         // 0: keys 0-31, 1: keys 32-63
    const int h = sub * 32 + lane;                    // head owned in the softmax
    const int gt = tid - SMX_WARP0 * 32;              // 0..255 within the group
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    uint8_t* prow = sm + OFF_P + (h >> 3) * 1024 + (h & 7) * 128;
    const float c2 = p.scale_log2;
    bool ok = true;
    int gb = 0, it = 0;
    for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++it) {
      // ---- unit info from the producer; one decision for the whole group ----
      const int islot = it & 1;
      const bool got = mbar_wait_unless(&bars[B_INFO_F + islot], (it >> 1) & 1, s_abort,
                                        p.status, SITE_W_INFO);
      const int n_list = s_info[islot * 3 + 0];
      const int nb = s_info[islot * 3 + 1];
      const int blk0 = s_info[islot * 3 + 2];
      if (named_bar_or(1, NSMX, !got || !ok || vload(s_abort))) {
        ok = false;
        break;
      }
      if (gt == 0) mbar_arrive(&bars[B_INFO_E + islot]);
      const Unit U = unit_of(p, u);
      // l_sum: this thread's share (its 32 keys) of sum_s 2^(z_s - m_ref)
      float m_ref = -INFINITY, l_sum = 0.f;
      // list entries kb + lane and kb + 32 + lane, fetched one block ahead
      int e_lo = -1, e_hi = -1;
      if (nb > 0) {
        const int kb = blk0 * BK;
        e_lo = kb + lane < n_list ? __ldg(U.ix + kb + lane) : -1;
        e_hi = kb + 32 + lane < n_list ? __ldg(U.ix + kb + 32 + lane) : -1;
      }
      for (int jj = 0; jj < nb; ++jj) {
        const int gbj = gb + jj;
        const int sbuf = gbj & 1, k3 = gbj % 3;
        const uint32_t m_lo = __ballot_sync(0xffffffffu, entry_row(p, U.b, U.t, e_lo) >= 0);
        const uint32_t m_hi = __ballot_sync(0xffffffffu, entry_row(p, U.b, U.t, e_hi) >= 0);
        const uint32_t mine = half ? m_hi : m_lo;
        if (jj + 1 < nb) {
          const int kb = (blk0 + jj + 1) * BK;
          e_lo = kb + lane < n_list ? __ldg(U.ix + kb + lane) : -1;
          e_hi = kb + 32 + lane < n_list ? __ldg(U.ix + kb + 32 + lane) : -1;
        }
        bool w_ok = mbar_wait(&bars[B_SF + sbuf], (gbj >> 1) & 1, p.status, kWaitLimitNs, SITE_W_SF);
        tc_fence_after();
        uint32_t own[32];
        if (w_ok) {
          tmem_ld32(tmem + lane_base + S_COL + BK * sbuf + 32 * half, own);
          tmem_ld_wait();
        }
        tc_fence_before();
        mbar_arrive(&bars[B_SE + sbuf]);
        // Common path: P = 2^(z - m_ref) against the running reference max.  Any
        // exponent above 64 (or no reference yet) sends the whole group through
        // the rare path below, which moves the reference and rescales O^T.
        const float neg_m = -m_ref;
        bool over = (m_ref == -INFINITY);
        uint32_t pk[16];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
        if (mine == 0xffffffffu) {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float a0 = fmaf(__uint_as_float(own[c]), c2, neg_m);
            const float a1 = fmaf(__uint_as_float(own[c + 1]), c2, neg_m);
            over |= fmaxf(a0, a1) > 64.f;
            const float p0 = ex2(a0), p1 = ex2(a1);
            pk[c >> 1] = pack_bf16x2(p0, p1);
            ls[(c >> 1) & 3] += p0 + p1;
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const bool v0 = ((mine >> c) & 1u) != 0, v1 = ((mine >> (c + 1)) & 1u) != 0;
            const float a0 = v0 ? fmaf(__uint_as_float(own[c]), c2, neg_m) : -INFINITY;
            const float a1 = v1 ? fmaf(__uint_as_float(own[c + 1]), c2, neg_m) : -INFINITY;
            over |= fmaxf(a0, a1) > 64.f;
            const float p0 = ex2(a0), p1 = ex2(a1);
            pk[c >> 1] = pack_bf16x2(p0, p1);
            ls[(c >> 1) & 3] += p0 + p1;
          }
        }
        float blk_sum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // P^T buffer and O^T are free once the previous block's PV product is done
        if (gbj >= 1 && w_ok)
          w_ok = mbar_wait(&bars[B_O], (gbj - 1) & 1, p.status, kWaitLimitNs, SITE_W_O);
        // this thread's half of its head's row of P^T (K-major: row = head, 64 keys = 128 B)
        if (h < HN) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            if (h < H)
              v = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            else
              v = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(prow + ((((4 * half + q) ^ h) & 7) << 4)) = v;
          }
        }
        fence_proxy_async_smem();
        if (over && h < H) {
          s_hover[h] = 1;
          s_resc[k3] = 1;
        }
        if (!w_ok || vload(s_abort)) g_abort[k3] = 1;
        // P^T is complete for the common path: the value product may start now;
        // a block that takes the rare path holds it back (s_resc, B_RARE)
        mbar_arrive(&bars[B_P]);
        named_bar_sync(1, NSMX);
        if (vload(&g_abort[k3])) {
          s_abort[0] = 1;
          ok = false;
          break;
        }
        // slot (gbj-1) mod 3 is free again: the softmax threads read it before this
        // barrier and the value-product issuer before it committed B_O(gbj-1)
        if (gt == 0) s_resc[(gbj + 2) % 3] = 0;
        if (!vload(&s_resc[k3])) {
          l_sum += blk_sum;
        } else {
          // ---- rare path (first block, or an exponent above 64): uniform ----
          float cm = -INFINITY;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if ((mine >> c) & 1u) cm = fmaxf(cm, __uint_as_float(own[c]));
          s_cmax[half * 128 + h] = cm;
          named_bar_sync(1, NSMX);
          const bool hov = h < H && s_hover[h] != 0;
          float alpha = 1.f;
          if (hov) {
            const float mb2 = fmaxf(s_cmax[h], s_cmax[128 + h]) * c2;
            if (mb2 != -INFINITY) {
              alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - mb2);
              m_ref = mb2;
              const float nm = -mb2;
              float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int c = 0; c < 32; c += 2) {
                const bool v0 = ((mine >> c) & 1u) != 0, v1 = ((mine >> (c + 1)) & 1u) != 0;
                const float p0 = v0 ? ex2(fmaf(__uint_as_float(own[c]), c2, nm)) : 0.f;
                const float p1 = v1 ? ex2(fmaf(__uint_as_float(own[c + 1]), c2, nm)) : 0.f;
                pk[c >> 1] = pack_bf16x2(p0, p1);
                rs[(c >> 1) & 3] += p0 + p1;
              }
              blk_sum = (rs[0] + rs[1]) + (rs[2] + rs[3]);
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(prow + ((((4 * half + q) ^ h) & 7) << 4)) =
                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            } else {
              // no valid key seen yet for this head: nothing to weigh
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(prow + ((((4 * half + q) ^ h) & 7) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
              blk_sum = 0.f;
            }
          }
          l_sum = l_sum * alpha + blk_sum;
          if (half == 0) s_alpha[h] = alpha;
          fence_proxy_async_smem();
          named_bar_sync(1, NSMX);
          if (half == 0) s_hover[h] = 0;  // read by both halves before the barrier above
          tc_fence_after();
          if (jj >= 1) {
            // rescale every O^T column by its head's alpha (half 0: tiles 0-1, half 1: 2-3)
#pragma unroll 1
            for (int i = 2 * half; i < 2 * half + 2; ++i) {
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
          tc_fence_before();
          mbar_arrive(&bars[B_RARE]);
        }
      }
      if (!ok) break;  // uniform: taken from g_abort after a group barrier
      // ------------------------------ epilogue ---------------------------------
      bool o_ok = true;
      if (nb > 0)
        o_ok = mbar_wait(&bars[B_O], (gb + nb - 1) & 1, p.status, kWaitLimitNs, SITE_W_O);
      // one decision for the group: O^T holds this unit's result (or nothing failed
      // and the unit had no valid entry)
      const bool failed = named_bar_or(1, NSMX, !o_ok || vload(s_abort));
      const bool have_o = nb > 0 && !failed;
      const bool empty_ok = nb == 0 && !failed;
      // the two halves' sums, through the rare-path buffers (idle until the next unit)
      float* s_l = s_cmax;     // [2 halves][128]
      float* s_invl = s_alpha;  // [128]
      s_l[half * 128 + h] = l_sum;
      named_bar_sync(1, NSMX);
      tc_fence_after();
      if (half == 0) {
        const float lx = s_l[h] + s_l[128 + h];
        float inv = lx > 0.f ? 1.f / lx : 0.f;
        float lse2 = (lx > 0.f) ? m_ref + log2f(lx) : -INFINITY;
        if (p.sink != nullptr && p.nsplit == 1 && (have_o || empty_ok)) {
          // learnable sink: one more term 2^(s2 - M) in the denominator, no value;
          // O^T was accumulated against m_ref, so it is rescaled by 2^(m_ref - M)
          const float s2 = h < H ? __ldg(p.sink + h) * 1.4426950408889634f : -INFINITY;
          const float mr = have_o ? m_ref : -INFINITY;
          const float M = fmaxf(mr, s2);
          if (M == -INFINITY) {
            inv = 0.f;
            lse2 = -INFINITY;
          } else {
            const float f = ex2(mr - M);
            const float lt = (have_o ? lx : 0.f) * f + ex2(s2 - M);
            inv = lt > 0.f ? f / lt : 0.f;
            lse2 = M + log2f(lt);
          }
        }
        s_invl[h] = have_o ? inv : 0.f;
        const int64_t pq = static_cast<int64_t>(U.qflat) * p.nsplit + U.sp;
        if (h < H) {
          if (p.nsplit == 1) {
            if (p.lse != nullptr)
              p.lse[static_cast<int64_t>(U.qflat) * H + h] =
                  (have_o || (empty_ok && p.sink != nullptr)) ? lse2 * 0.6931471805599453f
                                                              : -INFINITY;
          } else {
            p.part_lse[pq * H + h] = have_o ? lse2 : -INFINITY;
          }
        }
      }
      named_bar_sync(1, NSMX);
      // O^T tile i (128 dims x H heads): each thread owns one dim of the two tiles
      // of its half (0: tiles 0-1, 1: tiles 2-3) and writes that dim of every
      // head straight to global memory as BF16 (a warp covers 32 consecutive
      // dims: 64 contiguous bytes per head).  No shared-memory
      // staging: the pair slots already hold the next unit's rows.
      const int64_t pq = static_cast<int64_t>(U.qflat) * p.nsplit + U.sp;
      const int dloc = 32 * sub + lane;
#pragma unroll 1
      for (int ti = 0; ti < 2; ++ti) {
        const int i = 2 * half + ti;
        // 16 heads per TMEM load keeps the live state small
#pragma unroll 1
        for (int c0 = 0; c0 < HN; c0 += 16) {
          uint32_t r[16];
          if (have_o) {
            tmem_ld16(tmem + lane_base + i * HN + c0, r);
            tmem_ld_wait();
          }
          float iv[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(s_invl + c0 + 4 * q);
            iv[4 * q] = v.x; iv[4 * q + 1] = v.y; iv[4 * q + 2] = v.z; iv[4 * q + 3] = v.w;
          }
          if (p.nsplit == 1) {
            uint16_t* ob = p.o_lat + (static_cast<int64_t>(U.qflat) * H + c0) * kVlat + 128 * i + dloc;
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (c0 + e < H)
                ob[e * kVlat] = __bfloat16_as_ushort(
                    __float2bfloat16_rn(have_o ? __uint_as_float(r[e]) * iv[e] : 0.f));
          } else {
            uint16_t* ob = p.part_o + (pq * H + c0) * kVlat + 128 * i + dloc;
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (c0 + e < H)
                ob[e * kVlat] = __bfloat16_as_ushort(
                    __float2bfloat16_rn(have_o ? __uint_as_float(r[e]) * iv[e] : 0.f));
          }
        }
      }
      // O^T has been read: the next unit's value product may overwrite it
      if (nb > 0) {
        tc_fence_before();
        mbar_arrive(&bars[B_OE]);
      }
      // the next unit's rare path reuses s_l / s_invl
      named_bar_sync(1, NSMX);
      gb += nb;
      if (failed) {
        ok = false;
        break;
      }
    }
    if (!ok) s_abort[0] = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the per-split partial results (o_p normalised and stored as BF16, lse_p
// FP32): lse = log2 (sum_p 2^lse_p [+ 2^sink]), o = sum_p 2^(lse_p - lse) o_p,
// summed in FP32; a learnable sink (no value row) enters here once, not in
// every split.  One thread per (query, head, 4 dims).
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ part_o,
                                                      const float* __restrict__ part_lse,
                                                      int nq, int H, int nsplit,
                                                      const float* __restrict__ sink,
                                                      uint16_t* __restrict__ o_lat,
                                                      float* __restrict__ lse) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t per_qh = kVlat / 4;
  if (gid >= static_cast<int64_t>(nq) * H * per_qh) return;
  const int64_t qh = gid / per_qh;
  const int d4 = static_cast<int>(gid % per_qh) * 4;
  const int64_t q = qh / H, h = qh % H;
  const float s2 = sink != nullptr ? __ldg(sink + h) * 1.4426950408889634f : -INFINITY;
  float mx = s2;
  for (int s = 0; s < nsplit; ++s) mx = fmaxf(mx, part_lse[(q * nsplit + s) * H + h]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float ls = part_lse[(q * nsplit + s) * H + h];
      if (ls == -INFINITY) continue;
      const float wgt = exp2f(ls - mx);
      wsum += wgt;
      const uint2 v =
          *reinterpret_cast<const uint2*>(part_o + ((q * nsplit + s) * H + h) * kVlat + d4);
      acc[0] += wgt * __uint_as_float(v.x << 16);
      acc[1] += wgt * __uint_as_float(v.x & 0xffff0000u);
      acc[2] += wgt * __uint_as_float(v.y << 16);
      acc[3] += wgt * __uint_as_float(v.y & 0xffff0000u);
    }
    if (s2 != -INFINITY) wsum += exp2f(s2 - mx);
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
  // per (query, split): H x 512 BF16 outputs and H FP32 log-sum-exps
  const size_t nq = static_cast<size_t>(B) * Tq;
  return nq * ns * H * (kVlat * sizeof(uint16_t) + sizeof(float)) + 256;
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
  p.B = a.B;
  p.Tq = a.Tq;
  p.topk = a.topk;
  p.max_kv_len = a.max_kv_len;
  p.nsplit = ns;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.o_lat = a.o_lat;
  p.lse = a.lse;
  p.sink = a.sink;
  p.status = a.status;
  if (ns > 1) {
    const size_t nq = static_cast<size_t>(a.B) * a.Tq;
    if (a.scratch == nullptr || a.scratch_bytes < sparse_mla_scratch_bytes(a.B, a.Tq, H, a.topk))
      return DSA_ERR_WORKSPACE_TOO_SMALL;
    p.part_o = static_cast<uint16_t*>(a.scratch);
    p.part_lse = reinterpret_cast<float*>(p.part_o + nq * ns * H * kVlat);
  }
  auto kern = sparse_mla_kernel<H>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess)
    return launch_status("cudaFuncSetAttribute");
  // persistent: one CTA per SM (shared memory allows no more), each walking
  // units blockIdx.x, blockIdx.x + grid, ...
  const int64_t units = static_cast<int64_t>(a.B) * a.Tq * ns;
  const unsigned grid = static_cast<unsigned>(units < num_sms() ? units : num_sms());
  kern<<<grid, NTHREADS, SMEM_BYTES, stream>>>(tq, p);
  if (launch_status("sparse_mla_kernel") != DSA_OK) return DSA_ERR_CUDA;
  if (ns > 1) {
    const int64_t nq = static_cast<int64_t>(a.B) * a.Tq;
    const int64_t threads = nq * H * (kVlat / 4);
    combine_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(
        p.part_o, p.part_lse, static_cast<int>(nq), H, ns, a.sink, a.o_lat, a.lse);
    if (launch_status("combine_kernel") != DSA_OK) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

dsa_status_t sparse_mla_launch(const SparseMlaArgs& a, cudaStream_t stream) {
  if (a.H == 96) return launch_h<96>(a, stream);
  if (a.H == 8) return launch_h<8>(a, stream);
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
