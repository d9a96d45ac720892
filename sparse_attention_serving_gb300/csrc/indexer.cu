// indexer.cu -- lightning indexer + top-k on sm_103a.
//
// Score of key s for query t (the head-weighted ReLU form adopted for the
// indexer; BF16 inputs with FP32 accumulation and every causal key scanned,
// "Kimi-K3.1-Pro", NeMo AutoModel, Implementation Limits, bullet 2):
//   I[t,s] = sum_j w[t,j] * max(0, q[t,j,:] . k[s,:]),   s <= t
// The top-k keys per query are kept ("Kimi K3.1 Pro" archdiff summary: top-2,048;
// a query with at most k causal keys keeps all of them, Implementation Limits,
// bullet 4).
//
// Prefill (Tq > 1): one fused, persistent kernel, no score buffer in global
// memory.  One CTA per SM walks work items -- tiles of QT consecutive queries
// of one sequence (QT * H_I = 256 accumulator columns at 64 heads, 64 at 4),
// heaviest first -- and streams every causal key tile of 128 keys of each item:
//     D^T[128 keys x QT*H_I] = K_tile[128 x D_I] . Q^T[D_I x QT*H_I]   (tcgen05, M=128)
//   with two TMEM accumulator buffers at N = 256 (four at N = 64), so the head
//   reductions of one tile overlap the MMAs of the next; the barrier phases run
//   off per-CTA tile counters, so the next item's query load and first MMAs
//   overlap the current item's final selections.  Each epilogue thread owns
//   one key (a TMEM lane) and reduces over heads without any cross-lane
//   traffic; scores above the query's running threshold are appended to the
//   query's candidate buffer (CAP entries in this CTA's slice of the
//   workspace, L2-resident).  When a buffer nears capacity a radix select
//   (11-bit digits over order-preserving keys, candidates held in registers)
//   keeps the top k and raises the threshold to the k-th score.  The final
//   select writes the indices.
//
// FP8 variant (E4M3 code rows with one FP32 scale per key and per query head;
// "Kimi-K3.1-Pro", Implementation Limits, bullet 2 contrasts the BF16 indexer
// with the FP8 one of some serving kernels): the same kernel with one
// kind::f8f6f4 chunk per row (half the operand bytes through shared memory),
// the query scales folded into the head weights and each key's scale streamed
// into a ring of its own and applied to the head sum before the threshold test:
//   I[t,s] = k_scale[s] * sum_j (w[t,j] q_scale[t,j]) max(0, c_q[t,j] . c_k[s]).
#include <cmath>

#include <cuda_bf16.h>

#include "internal.h"
#include "sm103.cuh"

namespace dsa {
namespace idx {

constexpr int BKEY = 128;  // keys per tile (MMA M)
constexpr int NEPI = 16;   // epilogue warps: four query groups x four TMEM lane quarters
constexpr int NGRP = NEPI / 4;
constexpr int NTHREADS = 64 + NEPI * 32;

enum : uint32_t {
  SITE_QPOS = 0x200, SITE_PAGE = 0x201, SITE_W_Q = 0x210, SITE_W_KE = 0x211, SITE_W_KF = 0x212,
  SITE_W_DE = 0x213, SITE_W_DF = 0x214, SITE_W_DRAIN = 0x215, SITE_W_SE = 0x216, SITE_W_SF = 0x217
};

template <int H_I, int D_I, bool FP8>
struct Cfg {
  // Four queries per CTA at 64 heads (N = 256, two TMEM accumulator buffers):
  // each key tile copied into shared memory feeds the MMAs of four queries.
  // The candidate buffers are in global memory (a per-CTA slice of the
  // workspace, L2-resident), CAP per query, so shared memory holds only the
  // operands and a query up to CAP causal keys needs no selection before its
  // final one.
  static constexpr int QT = (H_I >= 64) ? 256 / H_I : 16;  // queries per CTA
  static constexpr int N = QT * H_I;                          // MMA N
  static constexpr int NBUF = 512 / N > 4 ? 4 : 512 / N;      // TMEM accumulator buffers
  static constexpr int ROWB = FP8 ? D_I : 2 * D_I;            // bytes per key / query-head row
  static constexpr int NCH = ROWB / 128;                      // 128-byte column chunks
  static constexpr int NST = FP8 ? 8 : 4;                     // key-tile stages
  static constexpr int NSC = FP8 ? 8 : 0;                     // key-scale slots (FP8)
  static constexpr int Q_BYTES = NCH * N * 128;
  static constexpr int K_STAGE = NCH * BKEY * 128;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_SC = OFF_K + NST * K_STAGE;
  static constexpr int OFF_W = OFF_SC + NSC * BKEY * 4;
  // barriers: Q full, Q empty, K full [NST], K empty [NST], D full [4], D empty
  // [4], drain, scale full [NSC], scale empty [NSC]
  static constexpr int BQ = 0, BQE = 1, BKF = 2, BKE = BKF + NST, BDF = BKE + NST,
                       BDE = BDF + 4, BDRAIN = BDE + 4, BSF = BDRAIN + 1, BSE = BSF + NSC,
                       NBARS = BSE + NSC;
  static_assert(NBARS <= 48, "barrier block");
  static_assert(NBUF * N <= 512, "accumulator buffers in TMEM");
  static constexpr int OFF_MISC = OFF_W + QT * H_I * 4;
  // barriers (48 x 8 B), flags, per-query counts and thresholds, then the
  // selection scratch (RBINS histogram bins and 16 counters)
  static constexpr int MISC_HDR = 1024;
  static constexpr int MISC_BYTES = MISC_HDR + (2048 + 16 + NEPI) * 4;
  // per query, a histogram of the QHB top bits of the order keys of its
  // candidates: it raises the append threshold while the keys stream and
  // seeds the final selection
  static constexpr int QHB = 10;
  static constexpr int OFF_QH = OFF_MISC + MISC_BYTES;
  static constexpr int SMEM_BYTES = OFF_QH + QT * (1 << QHB) * 4 + 1024;
  static constexpr int CAP = (H_I >= 64) ? 8192 : 1536;  // candidates per query
  // key tiles between the epilogue's group barriers (a candidate buffer keeps
  // room for GT tiles of appends between two checks)
  static constexpr int GT = (H_I >= 64) ? 8 : 4;
  static constexpr int CTA_SCRATCH = QT * CAP * 8;        // scores, then key indices
  static constexpr int EPT = (CAP + NEPI * 32 - 1) / (NEPI * 32);  // candidates per thread in a select
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(N % 16 == 0 && N <= 256, "MMA N");
  static_assert(H_I % 4 == 0, "four head columns per weight load");
};

struct Params {
  const uint16_t* w;
  const float* q_scale;  // FP8: [B, Tq, H_I]
  const float* k_scale;  // FP8: one per key row, numbered like the key rows
  const int32_t* q_start;
  const int32_t* kv_len;
  const int32_t* block_table;
  int64_t seq_stride;
  int32_t max_pages, num_pages;
  int paged;
  int B, Tq, topk, max_kv_len, ntq;  // ntq = query tiles per sequence
  int32_t* out_idx;
  uint8_t* cand;  // [gridDim.x][CTA_SCRATCH] candidate buffers
  uint32_t* status;
};

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ bool vflag(const volatile int* p) { return *p != 0; }

// ---------------------------------------------------------------------------
// Radix selection of the k largest candidates of one query, by all NEPI*32
// epilogue threads together (named barrier 1).  Scores are compared as
// order-preserving 32-bit keys.  The digits start at the highest bit where the
// smallest and the largest key differ and are RBITS wide, so the first
// histogram already spreads the candidates; the descent stops as soon as the
// bin holding the k-th key is kept whole (typically after one or two passes).
// Ties at the cut are broken arbitrarily.
//
// Scratch (shared memory): hist[RBINS] and ctr[16 + NEPI]:
//   ctr[0] smallest key, ctr[1] largest key, ctr[2] chosen bin, ctr[3] count
//   above it, ctr[4] count in it, ctr[15] smallest kept key, ctr[16 + w] the
//   total of warp w in a prefix sum.
// ---------------------------------------------------------------------------
constexpr int RBITS = 11;
constexpr int RBINS = 1 << RBITS;
constexpr int SEL_G = NEPI * 32;           // selecting threads
constexpr int SEL_CTR = 16 + NEPI;          // counters, then one total per selecting warp

// Bin of the need-th largest element (bins ordered by value, counted from the
// top) of an NB-bin histogram: ctr[2] = bin, ctr[3] = elements in higher bins,
// ctr[4] = elements in it.  Thread t owns the PER = NB / SEL_G contiguous bins
// NB-1-PER*t down to NB-PER*(t+1), read as vector loads.
template <int NB>
__device__ __forceinline__ void find_bin(const int* hist, int need, int gtid, int* ctr) {
  constexpr int PER = NB / SEL_G;
  static_assert((PER % 4 == 0 || PER == 2) && PER * SEL_G == NB, "whole vector loads of bins per thread");
  const int lane = gtid & 31, w = gtid >> 5;
  int c[PER];  // c[e] = bin NB-1-PER*gtid-e
  if constexpr (PER == 2) {
    const int2 x = *reinterpret_cast<const int2*>(hist + NB - PER * (gtid + 1));
    c[0] = x.y;
    c[1] = x.x;
  } else {
    const int4* hb = reinterpret_cast<const int4*>(hist + NB - PER * (gtid + 1));
#pragma unroll
    for (int v = 0; v < PER / 4; ++v) {
      const int4 x = hb[v];
      c[PER - 1 - 4 * v] = x.x;
      c[PER - 2 - 4 * v] = x.y;
      c[PER - 3 - 4 * v] = x.z;
      c[PER - 4 - 4 * v] = x.w;
    }
  }
  int tot = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) tot += c[e];
  int incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) ctr[16 + w] = incl;
  named_bar_sync(1, SEL_G);
#pragma unroll
  for (int ww = 0; ww < NEPI; ++ww)
    if (ww < w) incl += ctr[16 + ww];
  int run = incl - tot;
  if (run < need && need <= incl) {
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      if (run < need && need <= run + c[e]) {
        ctr[2] = NB - 1 - PER * gtid - e;
        ctr[3] = run;
        ctr[4] = c[e];
      }
      run += c[e];
    }
  }
  named_bar_sync(1, SEL_G);
}

// Radix refinement over keys delivered by `each(f)`, which calls f(key, valid)
// for this thread's elements (the same elements on every call).  On entry the
// need-th largest key is known to match `prefix` on the bits of `pmask`
// (= the bits [low, 32)); each pass histograms the next RBITS bits of the
// elements that match and narrows the prefix, until the bin holding the
// need-th key is kept whole or every bit is fixed.  On return every element
// with (key & pmask) > prefix is kept, and `need` of those equal to it.
template <class Each>
__device__ __forceinline__ void radix_refine(Each each, int gtid, int* hist, int* ctr,
                                             uint32_t& prefix, uint32_t& pmask, int& need,
                                             int low) {
  while (low > 0) {
    const int sh = low > RBITS ? low - RBITS : 0;
    const uint32_t dm = (1u << (low - sh)) - 1u;
#pragma unroll
    for (int e = 0; e < RBINS / SEL_G; ++e) hist[gtid + e * SEL_G] = 0;
    named_bar_sync(1, SEL_G);
    const uint32_t pm = pmask, pf = prefix;
    each([&](uint32_t key, bool valid) {
      if (valid && (key & pm) == pf) atomicAdd(&hist[(key >> sh) & dm], 1);
    });
    named_bar_sync(1, SEL_G);
    find_bin<RBINS>(hist, need, gtid, ctr);
    const uint32_t bin = static_cast<uint32_t>(ctr[2]);
    const int above = ctr[3], inbin = ctr[4];
    prefix |= bin << sh;
    pmask |= dm << sh;
    need -= above;
    low = sh;
    if (inbin == need) return;  // bin kept whole
  }
}

// The full descent: the digits start at the highest bit where the smallest
// and the largest key differ, so the first histogram already spreads the
// candidates.
template <class Each>
__device__ __forceinline__ void radix_descent(Each each, int k, int gtid, int* hist, int* ctr,
                                              uint32_t& prefix, uint32_t& pmask, int& need) {
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  each([&](uint32_t key, bool valid) {
    if (valid) {
      kmin = min(kmin, key);
      kmax = max(kmax, key);
    }
  });
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if ((gtid & 31) == 0) {
    atomicMin(reinterpret_cast<unsigned*>(&ctr[0]), kmin);
    atomicMax(reinterpret_cast<unsigned*>(&ctr[1]), kmax);
  }
  named_bar_sync(1, SEL_G);
  const uint32_t lo = static_cast<uint32_t>(ctr[0]), hi = static_cast<uint32_t>(ctr[1]);
  need = k;
  if (lo == hi) {  // every key equal: any k of them
    prefix = hi;
    pmask = 0xffffffffu;
    return;
  }
  const int top = 31 - __clz(lo ^ hi);
  pmask = top >= 31 ? 0u : ~((2u << top) - 1u);
  prefix = hi & pmask;
  radix_refine(each, gtid, hist, ctr, prefix, pmask, need, top + 1);
}

__device__ __forceinline__ void sel_reset(int* ctr, int gtid) {
  if (gtid == 0) {
    ctr[0] = static_cast<int>(0xffffffffu);
    ctr[1] = 0;
    ctr[15] = static_cast<int>(0xffffffffu);
  }
  named_bar_sync(1, SEL_G);
}

// The n candidates of one query into registers: element e = gtid + u*SEL_G
// sits in slot u (the buffer is in global memory: only the n filled entries
// are read).
template <int EPT>
__device__ __forceinline__ void sel_load(const float* cs, const int32_t* ci, int n, int gtid,
                                         uint32_t (&key)[EPT], int32_t (&id)[EPT]) {
#pragma unroll
  for (int u = 0; u < EPT; ++u) {
    const int e = gtid + u * SEL_G;
    key[u] = 0u;
    id[u] = -1;
    if (e < n) {
      key[u] = order_key(cs[e]);
      id[u] = ci[e];
    }
  }
}

// Output positions of the kept elements once the cut is known (every element
// with (key & pmask) > prefix, and the first `need` equal to it in thread
// order): per-thread counts above / equal (16 + 16 bits), one prefix sum; keys
// above the cut go to [0, above), the `need` equal ones right after them.
//   FINAL: the indices go to out[0..k) (in no particular order); returns 0.
//   else:  the kept candidates are compacted to the front of the buffer and
//          the smallest kept score (the query's new threshold) is returned.
template <int EPT, bool FINAL>
__device__ __forceinline__ float sel_emit(const uint32_t (&key)[EPT], const int32_t (&id)[EPT],
                                          uint32_t prefix, uint32_t pmask, int need, int gtid,
                                          int* ctr, float* cs, int32_t* ci, int32_t* out) {
  const int lane = gtid & 31, w = gtid >> 5;
  int n_hi = 0, n_eq = 0;
#pragma unroll
  for (int u = 0; u < EPT; ++u) {
    if (id[u] < 0) continue;
    const uint32_t m = key[u] & pmask;
    n_hi += m > prefix;
    n_eq += m == prefix;
  }
  const int packed = n_hi | (n_eq << 16);
  int incl = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) ctr[16 + w] = incl;
  named_bar_sync(1, SEL_G);
  int before = 0, total = 0;
#pragma unroll
  for (int ww = 0; ww < NEPI; ++ww) {
    const int t = ctr[16 + ww];
    if (ww < w) before += t;
    total += t;
  }
  const int excl = before + incl - packed;
  const int total_hi = total & 0xffff;
  int pos_hi = excl & 0xffff, pos_eq = excl >> 16;
  uint32_t kept_min = 0xffffffffu;
#pragma unroll
  for (int u = 0; u < EPT; ++u) {
    if (id[u] < 0) continue;
    const uint32_t m = key[u] & pmask;
    int pos = -1;
    if (m > prefix) {
      pos = pos_hi++;
    } else if (m == prefix) {
      if (pos_eq < need) pos = total_hi + pos_eq;
      ++pos_eq;
    }
    if (pos >= 0) {
      if (FINAL) {
        out[pos] = id[u];
      } else {
        cs[pos] = key_to_float(key[u]);
        ci[pos] = id[u];
        kept_min = min(kept_min, key[u]);
      }
    }
  }
  if (FINAL) {
    named_bar_sync(1, SEL_G);  // ctr / hist are reused by the next selection
    return 0.f;
  }
  kept_min = __reduce_min_sync(0xffffffffu, kept_min);
  if (lane == 0) atomicMin(reinterpret_cast<unsigned*>(&ctr[15]), kept_min);
  named_bar_sync(1, SEL_G);
  const float kth = key_to_float(static_cast<uint32_t>(ctr[15]));
  named_bar_sync(1, SEL_G);
  return kth;
}

// Keep the k largest of the n candidates of one query (a full radix descent)
// and compact them to the front of the buffer; returns the k-th score.
template <int EPT>
__device__ float select_keep(float* cs, int32_t* ci, int n, int k, int gtid, int* hist, int* ctr) {
  uint32_t key[EPT];
  int32_t id[EPT];
  sel_load<EPT>(cs, ci, n, gtid, key, id);
  sel_reset(ctr, gtid);
  uint32_t prefix, pmask;
  int need;
  auto each = [&](auto f) {
#pragma unroll
    for (int u = 0; u < EPT; ++u) f(key[u], id[u] >= 0);
  };
  radix_descent(each, k, gtid, hist, ctr, prefix, pmask, need);
  return sel_emit<EPT, false>(key, id, prefix, pmask, need, gtid, ctr, cs, ci, nullptr);
}

// Final selection of one query: the indices of its k largest candidates go to
// out[0..k) (in no particular order), -1 padded when n <= k.  qh is the
// query's histogram of the QHB top bits of every candidate's order key, kept
// up to date by the appends, so the first digit needs no pass over the
// candidates: the descent starts from the bin holding the k-th key.
template <int EPT, int QHB>
__device__ void select_final(const float* cs, const int32_t* ci, int n, int k, const int* qh,
                             int gtid, int* hist, int* ctr, int32_t* out) {
  if (n <= k) {
    for (int e = gtid; e < k; e += SEL_G) out[e] = e < n ? ci[e] : -1;
    return;
  }
  uint32_t key[EPT];
  int32_t id[EPT];
  sel_load<EPT>(cs, ci, n, gtid, key, id);
  find_bin<(1 << QHB)>(qh, k, gtid, ctr);
  uint32_t prefix = static_cast<uint32_t>(ctr[2]) << (32 - QHB);
  uint32_t pmask = ~((1u << (32 - QHB)) - 1u);
  int need = k - ctr[3];
  const int inbin = ctr[4];
  auto each = [&](auto f) {
#pragma unroll
    for (int u = 0; u < EPT; ++u) f(key[u], id[u] >= 0);
  };
  if (inbin != need) radix_refine(each, gtid, hist, ctr, prefix, pmask, need, 32 - QHB);
  sel_emit<EPT, true>(key, id, prefix, pmask, need, gtid, ctr, nullptr, nullptr, out);
}

// Raise a query's append threshold from its histogram (one warp): the lower
// edge of the bin where the count of candidates from the top first reaches k.
// At least k candidates lie at or above that edge, so the k-th largest score
// of the query does too and no key below it can be in the top k.  The
// histogram may be growing meanwhile (appends of other warps); a snapshot
// only undercounts, which lowers the edge found, so the bound stays valid.
// The 1024 bins are read as 32 rows of 32 (lane l reads bin 32r + l: no bank
// conflicts); a recursive-halving exchange leaves lane l with the total of
// row l, then suffix sums over the rows and over the bins of the row that
// holds the k-th pick the edge.
template <int QHB>
__device__ __forceinline__ void raise_threshold(const int* qh, int k, int lane, uint32_t* tkey) {
  constexpr int NR = (1 << QHB) / 32;
  static_assert(NR == 32, "one row per lane");
  int v[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) v[r] = qh[32 * r + lane];
  // after the step of width w, v[i] (i < w) is a partial total of row
  // (lane & ~(w-1) & 31) + i over the lanes that differ in bit w; the last step
  // leaves v[0] = the total of row `lane`
#pragma unroll
  for (int w = NR / 2; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const int send = upper ? v[i] : v[i + w];
      const int keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  // suffix sums over the rows from the top (row 31 = the largest keys)
  int cum = v[0];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_down_sync(0xffffffffu, cum, o);
    if (lane + o < 32) cum += t;
  }
  const uint32_t hit = __ballot_sync(0xffffffffu, cum >= k);
  if (hit == 0u) return;  // fewer than k candidates counted
  const int row = 31 - __clz(hit);
  const int above = __shfl_sync(0xffffffffu, cum - v[0], row);
  // within the row, from its top bin (lane 31) down: inclusive suffix sums
  int suf = qh[32 * row + lane];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += t;
  }
  // the highest bin with at least k counted at or above it (lane 0 always
  // qualifies: its suffix is the whole row, read after the row totals)
  const uint32_t hit2 = __ballot_sync(0xffffffffu, k <= above + suf);
  if (hit2 == 0u) return;
  const uint32_t edge = static_cast<uint32_t>(32 * row + 31 - __clz(hit2)) << (32 - QHB);
  if (lane == 0 && edge > *tkey) *tkey = edge;
}

// One work item: a tile of QT consecutive queries of one sequence.  Items are
// numbered heaviest first (w -> query tile ntq-1 - w/B of sequence w%B) and
// dealt to the persistent CTAs in snake order: in round r, CTA c takes item
// r*P + c (r even) or r*P + P-1-c (r odd), so that every CTA gets a similar mix.
struct Item {
  int b, qi0, nq, t0, t_last, L, ntiles;
  bool ok, stream;  // ok: positions valid; stream: some query has more than k keys
  int32_t* out;
};

template <int QT>
__device__ __forceinline__ bool item_at(const Params& p, int r, Item& I) {
  const int P = gridDim.x, c = blockIdx.x;
  const int64_t w = static_cast<int64_t>(r) * P + ((r & 1) ? P - 1 - c : c);
  if (w >= static_cast<int64_t>(p.B) * p.ntq) return false;
  I.b = static_cast<int>(w % p.B);
  const int qt = p.ntq - 1 - static_cast<int>(w / p.B);
  I.qi0 = qt * QT;
  I.nq = min(QT, p.Tq - I.qi0);
  const int q_start = __ldg(p.q_start + I.b);
  I.L = __ldg(p.kv_len + I.b);
  I.t0 = q_start + I.qi0;
  I.t_last = I.t0 + I.nq - 1;
  I.ok = q_start >= 0 && I.t_last < I.L && I.L <= p.max_kv_len;
  I.stream = I.ok && I.t_last + 1 > p.topk;
  I.ntiles = (I.t_last + BKEY) / BKEY;
  I.out = p.out_idx + (static_cast<int64_t>(I.b) * p.Tq + I.qi0) * p.topk;
  return true;
}

// Persistent: one CTA per SM walks its work items.  The barrier phases of the
// key stages, the TMEM accumulator buffers and (FP8) the key-scale slots run
// off per-CTA tile counters that continue across items, and the query block
// has its own full / empty pair, so the next item's query load and first MMAs
// overlap the current item's final selections.
template <int H_I, int D_I, bool FP8>
__global__ void __launch_bounds__(NTHREADS, 1)
    indexer_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k, const Params p) {
  using C = Cfg<H_I, D_I, FP8>;
  constexpr int QT = C::QT, N = C::N, NCH = C::NCH, CAP = C::CAP, NST = C::NST, NSC = C::NSC;
  constexpr int NBUF = C::NBUF;
  constexpr int NSC1 = NSC > 0 ? NSC : 1;
  constexpr uint32_t IDESC = FP8 ? idesc_e4m3(128, N) : idesc_bf16(128, N, false, false);
  constexpr int G = NEPI * 32;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  float* w_s = reinterpret_cast<float*>(sm + C::OFF_W);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_MISC);  // 48 barrier slots
  float* s_scale = reinterpret_cast<float*>(sm + C::OFF_SC);         // FP8: [NSC][128]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 48);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* g_abort = s_abort + 1;   // [4]
  int* cnt = const_cast<int*>(s_abort) + 8;  // [QT] candidates per query
  uint32_t* tkey = reinterpret_cast<uint32_t*>(cnt + 64);  // [QT] smallest order key still taken
  constexpr int QHB = C::QHB, QHN = 1 << QHB;
  int* qhist = reinterpret_cast<int*>(sm + C::OFF_QH);  // [QT][QHN]
  int* hist = reinterpret_cast<int*>(sm + C::OFF_MISC + C::MISC_HDR);  // [RBINS]
  int* ctr = hist + RBINS;                                              // [SEL_CTR]
  static_assert(48 * 8 + 4 + 4 * 8 + 64 * 4 + 64 * 4 <= C::MISC_HDR, "misc header");
  static_assert(RBINS == 2048 && SEL_CTR == 16 + NEPI, "selection scratch size");
  float* cand_s = reinterpret_cast<float*>(p.cand + static_cast<int64_t>(blockIdx.x) * C::CTA_SCRATCH);
  int32_t* cand_i = reinterpret_cast<int32_t*>(cand_s + QT * CAP);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int k = 0; k < C::NBARS; ++k)
      mbar_init(&bars[k], ((k >= C::BDE && k < C::BDE + 4) || k >= C::BSE) ? NEPI : 1);  // warps
    s_abort[0] = 0;
    for (int k = 0; k < 4; ++k) g_abort[k] = 0;
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
    // ============================ producer ===================================
    if (lane == 0) {
      int last_use[NST];
      for (int k = 0; k < NST; ++k) last_use[k] = -1;
      int last_s[NSC1];
      for (int k = 0; k < NSC1; ++k) last_s[k] = -1;
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      int g = 0, nit = 0;  // tiles and streaming items so far
      Item I;
      for (int r = 0; item_at<QT>(p, r, I) && !vflag(s_abort); ++r) {
        if (!I.stream) continue;
        // the query block, once the previous item's MMAs are done with it
        if (nit > 0 &&
            !mbar_wait(&bars[C::BQE], (nit - 1) & 1, p.status, kWaitLimitNs, SITE_W_Q)) {
          s_abort[0] = 1;
          break;
        }
        mbar_expect_tx(&bars[C::BQ], C::Q_BYTES);
        const int qrow = (I.b * p.Tq + I.qi0) * H_I;
#pragma unroll
        for (int c = 0; c < NCH; ++c)
          tma_load_2d(sm + C::OFF_Q + c * N * 128, &tm_q, &bars[C::BQ], 64 * c, qrow);
        ++nit;
        for (int kt = 0; kt < I.ntiles; ++kt, ++g) {
          const int st = g % NST, use = g / NST;
          if (use > 0 && !mbar_wait(&bars[C::BKE + st], (use - 1) & 1, p.status, kWaitLimitNs, SITE_W_KE)) {
            s_abort[0] = 1;
            break;
          }
          if (vflag(s_abort)) break;
          mbar_expect_tx(&bars[C::BKF + st], C::K_STAGE);
          last_use[st] = use;
          uint8_t* dst = sm + C::OFF_K + st * C::K_STAGE;
          int pids[2] = {0, 0};
          if (!p.paged) {
            const int row = static_cast<int>(static_cast<int64_t>(I.b) * p.seq_stride + kt * BKEY);
#pragma unroll
            for (int c = 0; c < NCH; ++c) tma_load_2d(dst + c * BKEY * 128, &tm_k, &bars[C::BKF + st], 64 * c, row);
          } else {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int pg = kt * 2 + hf;
              int pid = 0;
              if (pg * kPage < I.L) {
                pid = pg < p.max_pages ? __ldg(p.block_table + static_cast<int64_t>(I.b) * p.max_pages + pg) : -1;
                if (pid < 0 || pid >= p.num_pages) {
                  status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_PAGE, (uint32_t)pid);
                  pid = 0;  // read a valid page; its keys are never selected (flagged above)
                }
              }
              pids[hf] = pid;
#pragma unroll
              for (int c = 0; c < NCH; ++c)
                tma_load_2d(dst + c * BKEY * 128 + hf * 64 * 128, &tm_k, &bars[C::BKF + st], 64 * c, pid * kPage);
            }
          }
          if constexpr (FP8) {
            // the tile's key scales, into a slot of their own
            const int sc = g % NSC, suse = g / NSC;
            if (suse > 0 &&
                !mbar_wait(&bars[C::BSE + sc], (suse - 1) & 1, p.status, kWaitLimitNs, SITE_W_SE)) {
              s_abort[0] = 1;
              break;
            }
            last_s[sc] = suse;
            float* sdst = s_scale + sc * BKEY;
            if (!p.paged) {
              // rows of this sequence only (seq_stride is a multiple of 4: whole
              // 16-byte units, never past the array)
              const int64_t r0 = static_cast<int64_t>(I.b) * p.seq_stride + static_cast<int64_t>(kt) * BKEY;
              const int64_t left = p.seq_stride - static_cast<int64_t>(kt) * BKEY;
              const uint32_t bytes = static_cast<uint32_t>(left < BKEY ? left : BKEY) * 4u;
              mbar_expect_tx(&bars[C::BSF + sc], bytes);
              bulk_load(sdst, p.k_scale + r0, bytes, &bars[C::BSF + sc]);
            } else {
              mbar_expect_tx(&bars[C::BSF + sc], 2 * kPage * 4);
#pragma unroll
              for (int hf = 0; hf < 2; ++hf)
                bulk_load(sdst + hf * kPage, p.k_scale + static_cast<int64_t>(pids[hf]) * kPage,
                          kPage * 4, &bars[C::BSF + sc]);
            }
          }
        }
      }
      // every copy issued has landed before the CTA may exit
      for (int k = 0; k < NSC; ++k)
        if (last_s[k] >= 0) mbar_wait(&bars[C::BSF + k], last_s[k] & 1, p.status, kWaitLimitNs, SITE_W_SF);
      for (int st = 0; st < NST; ++st)
        if (last_use[st] >= 0) mbar_wait(&bars[C::BKF + st], last_use[st] & 1, p.status, kWaitLimitNs, SITE_W_KF);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ============================ MMA issuer ==================================
    if (lane == 0) {
      bool ok = true;
      const uint64_t qd0 = smem_desc(smem_u32(sm + C::OFF_Q), 16, 1024);
      int g = 0, nit = 0;
      Item I;
      for (int r = 0; ok && item_at<QT>(p, r, I); ++r) {
        if (!I.stream) continue;
        if (!mbar_wait(&bars[C::BQ], nit & 1, p.status, kWaitLimitNs, SITE_W_Q)) { ok = false; break; }
        ++nit;
        for (int kt = 0; kt < I.ntiles; ++kt, ++g) {
          if (vflag(s_abort)) { ok = false; break; }
          const int st = g % NST, buf = g % NBUF;
          if (g >= NBUF && !mbar_wait(&bars[C::BDE + buf], ((g / NBUF) - 1) & 1, p.status, kWaitLimitNs, SITE_W_DE)) { ok = false; break; }
          if (!mbar_wait(&bars[C::BKF + st], (g / NST) & 1, p.status, kWaitLimitNs, SITE_W_KF)) { ok = false; break; }
          tc_fence_after();
          const uint64_t kd = smem_desc(smem_u32(sm + C::OFF_K + st * C::K_STAGE), 16, 1024);
#pragma unroll
          for (int c = 0; c < NCH; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              if constexpr (FP8)
                umma_e4m3(tmem + buf * N, desc_add(kd, c * BKEY * 128 + kk * 32),
                          desc_add(qd0, c * N * 128 + kk * 32), IDESC, (c | kk) ? 1u : 0u);
              else
                umma_bf16(tmem + buf * N, desc_add(kd, c * BKEY * 128 + kk * 32),
                          desc_add(qd0, c * N * 128 + kk * 32), IDESC, (c | kk) ? 1u : 0u);
          umma_commit(&bars[C::BKE + st]);
          umma_commit(&bars[C::BDF + buf]);
        }
        // the query block is free once this item's MMAs are done
        umma_commit(&bars[C::BQE]);
      }
      if (!ok) s_abort[0] = 1;
      umma_commit(&bars[C::BDRAIN]);
      mbar_wait(&bars[C::BDRAIN], 0, p.status, kWaitLimitNs, SITE_W_DRAIN);
    }
    __syncwarp();
  } else {
    // ========================== epilogue (8 warps) ============================
    const int gtid = tid - 64;
    const int sub = warp & 3;
    const int half = (warp - 2) >> 2;  // query group of this warp
    constexpr int QH = QT / NGRP;      // queries per group
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    const int key_lane = sub * 32 + lane;
    int g = 0;  // tiles of the streaming items so far
    Item I;
    for (int r = 0; item_at<QT>(p, r, I); ++r) {
      const int nq = I.nq, t0 = I.t0;
      int32_t* out = I.out;
      if (!I.ok) {
        if (gtid == 0) status_raise(p.status, DSA_ERR_BAD_INDEX, SITE_QPOS, (uint32_t)I.t_last);
        for (int e = gtid; e < nq * p.topk; e += G) out[e] = -1;
        continue;
      }
      if (!I.stream) {
        // every query of the tile keeps all of its causal keys
        for (int e = gtid; e < nq * p.topk; e += G) {
          const int q = e / p.topk, j = e % p.topk;
          out[e] = j <= t0 + q ? j : -1;
        }
        continue;
      }
      if (vflag(&g_abort[1])) {  // an earlier item gave up: no more tiles will come
        for (int e = gtid; e < nq * p.topk; e += G) out[e] = -1;
        continue;
      }
      // this item's head weights and empty candidate buffers (the previous
      // item's readers of w_s, cnt and thr are past the barrier)
      named_bar_sync(1, G);
      for (int e = gtid; e < QT * H_I; e += G) {
        const int q = e / H_I;
        float wq = q < nq ? __bfloat162float(__ushort_as_bfloat16(
                                p.w[(static_cast<int64_t>(I.b) * p.Tq + I.qi0) * H_I + e]))
                          : 0.f;
        if constexpr (FP8) {
          if (q < nq) wq *= p.q_scale[(static_cast<int64_t>(I.b) * p.Tq + I.qi0) * H_I + e];
        }
        w_s[e] = 0.5f * wq;  // the head reduction takes (x + |x|) = 2 max(x, 0)
      }
      for (int q = gtid; q < QT; q += G) {
        cnt[q] = 0;
        tkey[q] = 0u;
      }
      for (int e = gtid; e < QT * QHN; e += G) qhist[e] = 0;
      named_bar_sync(1, G);
      const int ntiles = I.ntiles;
      int kt = 0;
      bool stop = false;
      while (kt < ntiles && !stop) {
        // this group's head weights, read from shared memory (four per 16-byte
        // broadcast load) as the columns come out of TMEM
        const float* wh = w_s + half * QH * H_I;
        bool want_sel = false;
        // Tiles in groups of C::GT with one group barrier per group: a candidate
        // buffer keeps room for GT tiles' appends between checks, and the MMA runs
        // up to NBUF tiles ahead (TMEM accumulator buffers).
        for (; kt < ntiles; kt += C::GT) {
          const int n2 = ntiles - kt < C::GT ? ntiles - kt : C::GT;
          bool w_ok = !vflag(s_abort);
          {
            // each tile as soon as its accumulator is complete (with two TMEM
            // buffers the MMA of the next tile overlaps this one's
            // reduction)
            for (int u = 0; u < n2; ++u) {
              const int k = kt + u, gk = g + k, buf = gk % NBUF;
              if (w_ok)
                w_ok = mbar_wait(&bars[C::BDF + buf], (gk / NBUF) & 1, p.status, kWaitLimitNs, SITE_W_DF) &&
                       (!FP8 || mbar_wait(&bars[C::BSF + gk % NSC1], (gk / NSC1) & 1, p.status,
                                          kWaitLimitNs, SITE_W_SF));
              // the TMEM loads and ballots below are warp-collective: one decision per warp
              w_ok = __all_sync(0xffffffffu, w_ok);
              if (!w_ok) {
                g_abort[0] = 1;
                break;
              }
              tc_fence_after();
              // head reduction: 4 independent FMA chains per query (the MMA's FP32
              // accumulators are summed in a fixed order: chain c takes heads c, c+4, ...),
              // issued as 2-wide FP32 FMAs on the chain pairs (0,1) and (2,3), each
              // lane an ordinary round-to-nearest FMA.  The ReLU runs on the FMA pipe
              // as x + |x| against halved weights: (x + |x|) (w/2) is max(x, 0) w
              // exactly (doubling and halving are exact in FP32), so every product
              // and sum is the one of w * max(x, 0)
              constexpr int COLS = QH * H_I;  // this group's accumulator columns
              constexpr int NCHAIN = 4;
              float acc[QH][NCHAIN];
#pragma unroll
              for (int q = 0; q < QH; ++q)
#pragma unroll
                for (int c = 0; c < NCHAIN; ++c) acc[q][c] = 0.f;
              const uint32_t col0 = buf * N + half * COLS;
              // four columns (one query's heads c..c+3) into the FMA chains
              auto reduce4 = [&](int col, const uint32_t* r) {
                const int q = col / H_I;  // columns col..col+3 belong to one query
                const float4 wv = *reinterpret_cast<const float4*>(wh + col);
                float x[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  x[j] = __uint_as_float(r[j]);
                  x[j] = __fadd_rn(x[j], fabsf(x[j]));
                }
                fma2_rn(acc[q][0], acc[q][1], wv.x, wv.y, x[0], x[1]);
                fma2_rn(acc[q][2], acc[q][3], wv.z, wv.w, x[2], x[3]);
              };
              if constexpr (COLS >= 32) {
                // 32 columns per TMEM load; the next load is in flight while the
                // current columns are reduced
                uint32_t rb[2][32];
                tmem_ld32(tmem + lane_base + col0, rb[0]);
#pragma unroll
                for (int v = 0; v < COLS / 32; ++v) {
                  uint32_t(&rr)[32] = rb[v & 1];
                  tmem_ld_wait_regs(rr);
                  if (v + 1 < COLS / 32) tmem_ld32(tmem + lane_base + col0 + (v + 1) * 32, rb[(v + 1) & 1]);
#pragma unroll
                  for (int e = 0; e < 32; e += 4) reduce4(v * 32 + e, rr + e);
                }
              } else {
                static_assert(COLS == 16, "a group's columns: a multiple of 32, or 16");
                uint32_t rr[16];
                tmem_ld16(tmem + lane_base + col0, rr);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; e += 4) reduce4(e, rr + e);
              }
              float score[QH];
#pragma unroll
              for (int q = 0; q < QH; ++q) score[q] = (acc[q][0] + acc[q][1]) + (acc[q][2] + acc[q][3]);
              tc_fence_before();
              mbar_arrive_warp(&bars[C::BDE + buf]);
              if constexpr (FP8) {
                const int sc = gk % NSC1;
                const float ks = s_scale[sc * BKEY + key_lane];
#pragma unroll
                for (int q = 0; q < QH; ++q) score[q] *= ks;
                mbar_arrive_warp(&bars[C::BSE + sc]);
              }
              // append candidates above each query's threshold (the queries'
              // slot reservations are issued back to back by lane 0)
              const int s = k * BKEY + key_lane;
              bool take[QH];
              uint32_t bal[QH];
              int base[QH];
              uint32_t okey[QH];
#pragma unroll
              for (int q = 0; q < QH; ++q) {
                const int qq = half * QH + q;
                okey[q] = order_key(score[q]);
                take[q] = qq < nq && s <= t0 + qq && okey[q] >= tkey[qq];
                bal[q] = __ballot_sync(0xffffffffu, take[q]);
                base[q] = 0;
              }
              if (lane == 0) {
#pragma unroll
                for (int q = 0; q < QH; ++q)
                  if (bal[q]) base[q] = atomicAdd(&cnt[half * QH + q], __popc(bal[q]));
              }
#pragma unroll
              for (int q = 0; q < QH; ++q) {
                const int qq = half * QH + q;
                const int pos = __shfl_sync(0xffffffffu, base[q], 0) +
                                __popc(bal[q] & ((1u << lane) - 1u));
                if (take[q]) {
                  cand_s[qq * CAP + pos] = score[q];
                  cand_i[qq * CAP + pos] = s;
                  atomicAdd(&qhist[qq * QHN + (okey[q] >> (32 - QHB))], 1);
                }
              }
            }
          }
          // The group's appends and abort flags are final after this barrier;
          // every warp reads them before the second barrier, so that no warp's
          // appends of the next group can change what another warp decides here.
          named_bar_sync(1, G);
          const bool abort_now = vflag(&g_abort[0]);
          // a buffer that could overflow on the next group is shrunk outside this loop
          for (int qq = 0; qq < nq; ++qq) want_sel |= cnt[qq] > CAP - C::GT * BKEY;
          named_bar_sync(1, G);
          if (abort_now) {
            if (gtid == 0) s_abort[0] = 1;  // no role waits for this item's tiles any more
            stop = true;
            break;
          }
          // warp q raises query q's threshold (no barrier: appends may read the
          // old or the new value, both valid)
          if (gtid / 32 < nq && cnt[gtid / 32] >= p.topk)
            raise_threshold<QHB>(qhist + (gtid / 32) * QHN, p.topk, lane, &tkey[gtid / 32]);
          if (want_sel) {
            kt += n2;
            break;
          }
        }
        if (want_sel) {
          for (int qq = 0; qq < nq; ++qq) {
            if (cnt[qq] > CAP - C::GT * BKEY) {
              const float kth = select_keep<C::EPT>(cand_s + qq * CAP, cand_i + qq * CAP, cnt[qq],
                                                    p.topk, gtid, hist, ctr);
              if (gtid == 0) {
                cnt[qq] = p.topk;
                tkey[qq] = order_key(kth);
              }
              // the histogram now describes the k kept candidates only
              for (int e = gtid; e < QHN; e += G) qhist[qq * QHN + e] = 0;
              named_bar_sync(1, G);
              for (int e = gtid; e < p.topk; e += G)
                atomicAdd(&qhist[qq * QHN + (order_key(cand_s[qq * CAP + e]) >> (32 - QHB))], 1);
              named_bar_sync(1, G);
            }
          }
        }
      }
      g += ntiles;
      // final selection and output (the abort decision is made uniform by one
      // writer before a group barrier)
      if (gtid == 0) g_abort[1] = vflag(s_abort) ? 1 : 0;
      named_bar_sync(1, G);
      const bool aborted = vflag(&g_abort[1]);
      // the queries one after another, each by all epilogue threads
      for (int qq = 0; qq < nq; ++qq) {
        int32_t* o = out + static_cast<int64_t>(qq) * p.topk;
        if (aborted) {
          for (int e = gtid; e < p.topk; e += G) o[e] = -1;
          continue;
        }
        select_final<C::EPT, QHB>(cand_s + qq * CAP, cand_i + qq * CAP, cnt[qq], p.topk,
                                  qhist + qq * QHN, gtid, hist, ctr, o);
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

}  // namespace idx

// Persistent grid: one CTA per SM, or one per work item when there are fewer.
template <int H_I, int D_I, bool FP8>
static int64_t prefill_grid(int B, int Tq) {
  using C = idx::Cfg<H_I, D_I, FP8>;
  const int64_t items = static_cast<int64_t>(B) * ((Tq + C::QT - 1) / C::QT);
  return items < num_sms() ? items : num_sms();
}

template <int H_I, int D_I, bool FP8>
static dsa_status_t prefill_launch(const IndexerArgs& a, cudaStream_t stream) {
  using C = idx::Cfg<H_I, D_I, FP8>;
  if (a.topk > C::CAP - C::GT * idx::BKEY) return DSA_ERR_UNSUPPORTED;
  const int64_t grid = prefill_grid<H_I, D_I, FP8>(a.B, a.Tq);
  if (a.scratch == nullptr ||
      a.scratch_bytes < static_cast<size_t>(grid) * C::CTA_SCRATCH)
    return DSA_ERR_WORKSPACE_TOO_SMALL;
  CUtensorMap tq, tk;
  const uint64_t qrows = static_cast<uint64_t>(a.B) * a.Tq * H_I;
  // (FP8 code rows are described as BF16 pairs: the copy moves bytes only)
  if (!encode_tmap_2d(&tq, a.q_idx, qrows, C::ROWB / 2, C::ROWB, 64, C::N, true))
    return DSA_ERR_CUDA;
  const bool paged = a.k.block_table != nullptr;
  if (!encode_tmap_2d(&tk, a.k.base, a.k.total_rows, C::ROWB / 2, C::ROWB, 64, paged ? 64 : 128,
                      true))
    return DSA_ERR_CUDA;
  idx::Params p{};
  p.w = a.w;
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.q_start = a.q_start;
  p.kv_len = a.kv_len;
  p.block_table = a.k.block_table;
  p.seq_stride = a.k.seq_stride;
  p.max_pages = a.k.max_pages;
  p.num_pages = a.k.num_pages;
  p.paged = paged;
  p.Tq = a.Tq;
  p.topk = a.topk;
  p.max_kv_len = a.max_kv_len;
  p.B = a.B;
  p.ntq = (a.Tq + C::QT - 1) / C::QT;
  p.out_idx = a.out_idx;
  p.cand = static_cast<uint8_t*>(a.scratch);
  p.status = a.status;
  auto kern = idx::indexer_prefill_kernel<H_I, D_I, FP8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
      cudaSuccess)
    return launch_status("cudaFuncSetAttribute");
  // persistent: one CTA per SM (shared memory allows no more)
  kern<<<static_cast<unsigned>(grid), idx::NTHREADS, C::SMEM_BYTES, stream>>>(tq, tk, p);
  return launch_status("indexer_prefill");
}

// The candidate buffers of the persistent grid (the same for BF16 and FP8).
size_t indexer_prefill_scratch_bytes(int B, int Tq, int H_I, int D_I) {
  if (H_I == 64 && D_I == 128)
    return static_cast<size_t>(prefill_grid<64, 128, false>(B, Tq)) * idx::Cfg<64, 128, false>::CTA_SCRATCH;
  if (H_I == 4 && D_I == 64)
    return static_cast<size_t>(prefill_grid<4, 64, false>(B, Tq)) * idx::Cfg<4, 64, false>::CTA_SCRATCH;
  return 0;
}
static_assert(idx::Cfg<64, 128, false>::CTA_SCRATCH == idx::Cfg<64, 128, true>::CTA_SCRATCH &&
                  idx::Cfg<64, 128, false>::QT == idx::Cfg<64, 128, true>::QT,
              "BF16 and FP8 share the workspace size");

int indexer_prefill_max_topk(int H_I, int D_I) {
  using C64 = idx::Cfg<64, 128, false>;
  using C4 = idx::Cfg<4, 64, false>;
  if (H_I == 64 && D_I == 128) return C64::CAP - C64::GT * idx::BKEY;
  if (H_I == 4 && D_I == 64) return C4::CAP - C4::GT * idx::BKEY;
  return 0;
}

dsa_status_t indexer_prefill_launch(const IndexerArgs& a, cudaStream_t stream) {
  if (a.fp8) {
    if (a.H_I == 64 && a.D_I == 128) return prefill_launch<64, 128, true>(a, stream);
    return DSA_ERR_UNSUPPORTED;
  }
  if (a.H_I == 64 && a.D_I == 128) return prefill_launch<64, 128, false>(a, stream);
  if (a.H_I == 4 && a.D_I == 64) return prefill_launch<4, 64, false>(a, stream);
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
