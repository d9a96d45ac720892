// gate.cu -- output gate on sm_103a:
//   out[n, h*dv+e] = sigmoid(x[n,:] . W_g[h*dv+e, :]) * (W_uv[h,e,:] . o_lat[n,h,:])
// ("Kimi K3.1 Pro" archdiff blueprint: the output gate sigma(x W_g) (.) o;
// "Kimi-K3.1-Pro", NeMo AutoModel, Implementation Limits, closing paragraph:
// the gate is kept; KimiK3TextConfig: mla_use_output_gate, v_head_dim 128).
//
// One CTA per (128 tokens, pair of heads): two tcgen05 accumulators in TMEM,
//   G[128 x 256] = x_tile . W_g[pair rows]^T          (K = hid, M=128, N=256)
//   U_h[128 x 128] = o_lat[tile, h, :] . W_uv[h]^T    (K = 512, M=128, N=128, per head)
// fed by a 4-stage TMA ring of 128-byte-swizzled K-chunks of 64; the epilogue
// applies the sigmoid in FP32 and writes BF16.
#include <cmath>

#include <cuda_bf16.h>

#include "internal.h"
#include "sm103.cuh"

namespace dsa {
namespace gate {

constexpr int NST = 4;
constexpr int STAGE = 48 * 1024;  // A 16 KB + B up to 32 KB
constexpr int OFF_MISC = NST * STAGE;
constexpr int SMEM_BYTES = OFF_MISC + 1024 + 1024;
constexpr int NTHREADS = 192;

enum : uint32_t { SITE_W_E = 0x300, SITE_W_F = 0x301, SITE_W_ACC = 0x302, SITE_W_DRAIN = 0x303 };

struct Params {
  int N, hid, H;
  uint16_t* out;
  uint32_t* status;
};

// sigma(g) = 1 / (1 + 2^(-g log2 e)) with the hardware approximations of 2^x and
// 1/x (relative error near 2^-22 each, far below the BF16 output's 2^-9).  An
// IEEE division here made the epilogue a quarter of the kernel.  Large |g|:
// 2^(-g log2 e) overflows to +inf for g << 0 (rcp gives 0) and underflows to 0
// for g >> 0 (rcp gives 1), the limits of sigma.
__device__ __forceinline__ float sigmoid_fast(float g) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(g * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
  return r;
}

__global__ void __launch_bounds__(NTHREADS, 1)
    gate_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_wg,
                const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_wu,
                const Params p) {
  constexpr uint32_t IDESC_G = idesc_bf16(128, 256, false, false);
  constexpr uint32_t IDESC_U = idesc_bf16(128, 128, false, false);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_MISC);  // full[4], empty[4], acc, drain
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* s_abort = reinterpret_cast<volatile int*>(tslot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Rasterise in groups of GT token tiles: a group's x tiles stay in L2 while
  // the CTAs sweep every head pair, so W_g (176 MB at 96 heads x hidden 7168,
  // larger than L2) is streamed from DRAM once per group instead of once per
  // token tile.
  constexpr int GT = 16;
  const int npair = p.H / 2;
  const int ntt = (p.N + 127) / 128;
  const int grp = blockIdx.x / (GT * npair);
  const int rem = blockIdx.x - grp * GT * npair;
  const int gt = min(GT, ntt - grp * GT);
  const int hp = rem / gt;                 // head pair
  const int n0 = (grp * GT + rem % gt) * 128;
  const int kg = p.hid / 64;               // G stages
  const int nstage = kg + 16;              // + 8 U stages per head

  if (tid == 0) {
    for (int k = 0; k < 2 * NST + 2; ++k) mbar_init(&bars[k], 1);
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
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_wg);
      tma_prefetch_desc(&tm_o);
      tma_prefetch_desc(&tm_wu);
      int last_use[NST] = {-1, -1, -1, -1};
      for (int s = 0; s < nstage; ++s) {
        const int st = s % NST, use = s / NST;
        if (use > 0 && !mbar_wait(&bars[NST + st], (use - 1) & 1, p.status, kWaitLimitNs, SITE_W_E)) {
          s_abort[0] = 1;
          break;
        }
        if (s_abort[0]) break;
        uint8_t* a = sm + st * STAGE;
        uint8_t* bb = a + 16 * 1024;
        last_use[st] = use;
        if (s < kg) {
          mbar_expect_tx(&bars[st], 48 * 1024);
          tma_load_2d(a, &tm_x, &bars[st], 64 * s, n0);
          tma_load_2d(bb, &tm_wg, &bars[st], 64 * s, hp * 256);
        } else {
          const int u = s - kg, hh = u >> 3, kc = u & 7, h = 2 * hp + hh;
          mbar_expect_tx(&bars[st], 32 * 1024);
          tma_load_2d(a, &tm_o, &bars[st], h * kVlat + 64 * kc, n0);
          tma_load_2d(bb, &tm_wu, &bars[st], 64 * kc, h * 128);
        }
      }
      for (int st = 0; st < NST; ++st)
        if (last_use[st] >= 0) mbar_wait(&bars[st], last_use[st] & 1, p.status, kWaitLimitNs, SITE_W_F);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      for (int s = 0; s < nstage; ++s) {
        const int st = s % NST;
        if (!mbar_wait(&bars[st], (s / NST) & 1, p.status, kWaitLimitNs, SITE_W_F)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ad = smem_desc(smem_u32(sm + st * STAGE), 16, 1024);
        const uint64_t bd = desc_add(ad, 16 * 1024);
        if (s < kg) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem, desc_add(ad, kk * 32), desc_add(bd, kk * 32), IDESC_G,
                      (s | kk) ? 1u : 0u);
        } else {
          const int u = s - kg, hh = u >> 3, kc = u & 7;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + 256 + hh * 128, desc_add(ad, kk * 32), desc_add(bd, kk * 32),
                      IDESC_U, (kc | kk) ? 1u : 0u);
        }
        umma_commit(&bars[NST + st]);
      }
      if (!ok) s_abort[0] = 1;
      umma_commit(&bars[2 * NST]);      // accumulators ready (or drained on abort)
      mbar_wait(&bars[2 * NST], 0, p.status, kWaitLimitNs, SITE_W_DRAIN);
    }
    __syncwarp();
  } else {
    // epilogue: thread = token row of the tile
    const int sub = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(sub * 32) << 16;
    const int n = n0 + sub * 32 + lane;
    const bool ok = mbar_wait(&bars[2 * NST], 0, p.status, kWaitLimitNs, SITE_W_ACC) && !s_abort[0];
    tc_fence_after();
    if (ok) {
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(tmem + lane_base + hh * 128 + c0, g);
          tmem_ld32(tmem + lane_base + 256 + hh * 128 + c0, u);
          tmem_ld_wait();
          if (n < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(n) * p.H * 128 +
                                                  (2 * hp + hh) * 128 + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i0 = 8 * v + 2 * e;
                const float s0 = sigmoid_fast(__uint_as_float(g[i0]));
                const float s1 = sigmoid_fast(__uint_as_float(g[i0 + 1]));
                w4[e] = pack_bf16x2(s0 * __uint_as_float(u[i0]), s1 * __uint_as_float(u[i0 + 1]));
              }
              dst[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
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

}  // namespace gate

dsa_status_t gate_launch(const GateArgs& a, cudaStream_t stream) {
  using namespace gate;
  CUtensorMap tx, twg, to, twu;
  if (!encode_tmap_2d(&tx, a.x, a.N, a.hid, static_cast<uint64_t>(a.hid) * 2, 64, 128, true) ||
      !encode_tmap_2d(&twg, a.W_g, static_cast<uint64_t>(a.H) * a.dv, a.hid,
                      static_cast<uint64_t>(a.hid) * 2, 64, 256, true) ||
      !encode_tmap_2d(&to, a.o_lat, a.N, static_cast<uint64_t>(a.H) * kVlat,
                      static_cast<uint64_t>(a.H) * kVlat * 2, 64, 128, true) ||
      !encode_tmap_2d(&twu, a.W_uv, static_cast<uint64_t>(a.H) * a.dv, kVlat, kVlat * 2, 64, 128,
                      true))
    return DSA_ERR_CUDA;
  Params p{a.N, a.hid, a.H, a.out, a.status};
  if (cudaFuncSetAttribute(gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess)
    return launch_status("cudaFuncSetAttribute");
  const unsigned grid = static_cast<unsigned>(((a.N + 127) / 128) * (a.H / 2));
  gate_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(tx, twg, to, twu, p);
  return launch_status("gate");
}

}  // namespace dsa
