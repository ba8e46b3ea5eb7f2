// attn_fwd.cu -- masked attention forward on sm_103a consuming a MaskPlan.
//
// Consumption protocol of "Flex Attention Mask Plan Design" §6.1: for one
// (sample, Q head, Q tile) task, the partial K tiles are processed with the
// packed predicate (§5: bit 1 keeps the score, bit 0 makes it -inf), then
// the full K tiles without it; empty tiles are never visited.  A row without
// any visible key ends with O = 0 and LSE = -inf.  The math is FlexAttention
// Eq. 1, softmax(mod(Q K^T * scale)) V, with an online softmax: the score
// matrix is never stored.
//
// Persistent CTAs (one per SM) walk the plan's work_desc with a static
// stride.  320 threads, warp-specialised:
//   warp 8     TMA producer: Q tiles into a 2-deep ring, K and V tiles into
//              their own rings, issued in the order the MMAs consume them
//              (K of tile g+1 before V of tile g).
//   warp 9     TMEM allocator and MMA issuer (one thread): S(g) = Q K^T into
//              one of three TMEM score buffers, then O += P(g-1) V with P read
//              from TMEM (it overwrites its score buffer in bf16).
//   warps 0-7  two softmax warpgroups; thread r of warpgroup w owns score row
//              r, columns 64w..64w+63 (TMEM lane r).  Per tile they exchange
//              the row max through shared memory, write P to TMEM, rescale
//              their half of O when the max moves, and store their half of
//              the output at the end of the task.
// Every mbarrier wait is bounded (global-timer limit).  After a timeout the
// CTA records an error bit and runs its loops to the end without waiting,
// so that every thread still reaches every named barrier; then it drains
// copies and MMAs in flight, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace bsm {

__device__ uint32_t g_fwd_err = 0;

namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;          // 64-column (128-byte) swizzle chunks
  static constexpr int kTileBytes = 128 * D * 2;  // Q, K or V tile, bf16
  static constexpr int kQStages = 2;
  static constexpr int kKStages = (D == 128) ? 2 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffSmall = kOffV + kVStages * kTileBytes;
  static constexpr int kSmallBytes = 512 + 2 * 2 * 128 * 4 + 2 * 128 * 4;  // barriers, max and sum exchange
  static constexpr int kSmem = kOffSmall + kSmallBytes + 1024;            // + slack for 1 KB alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 384;  // S buffers at 0, 128, 256; O after them
  static_assert(kColO + D <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

constexpr int kThreads = 320;
constexpr int kSoftmaxThreads = 256;
constexpr uint32_t kBarSoftmax = 1;  // named barrier id of the two softmax warpgroups

struct FwdParams {
  const int32_t* work;
  const int32_t* seq;
  const int32_t* p_off;
  const int32_t* f_off;
  const int32_t* p_idx;
  const int32_t* f_idx;
  const uint32_t* payload;
  __nv_bfloat16* o;
  float* lse;
  int Hq, Hk, Hmask, rows, total_q, ntasks;
  int flags;
  float scale;       // multiplies Q K^T
  float scale_log2;  // scale * log2(e)
  float softcap, inv_softcap;
  float slopes[kMaxHeads];
};

// Per-task view of the plan shared by every role.
struct Task {
  int m_block, h, b, qv, q_off, k_off, hk, p0, np, f0, n;
};

__device__ __forceinline__ Task load_task(const FwdParams& p, int t) {
  Task k;
  const int* wd = p.work + 4LL * t;
  k.m_block = wd[0];
  k.h = wd[1];
  k.b = wd[2];
  k.qv = wd[3];
  const int* sq = p.seq + 8 * k.b;
  k.q_off = sq[0];
  k.k_off = sq[1];
  const int row_begin = sq[4];
  const int hm = (p.Hmask == 1) ? 0 : k.h;
  k.hk = k.h / (p.Hq / p.Hk);
  const long long flat = static_cast<long long>(hm) * p.rows + row_begin + k.m_block;
  k.p0 = p.p_off[flat];
  k.np = p.p_off[flat + 1] - k.p0;
  k.f0 = p.f_off[flat];
  k.n = k.np + (p.f_off[flat + 1] - k.f0);
  return k;
}

__device__ __forceinline__ int tile_index(const FwdParams& p, const Task& k, int j) {
  return (j < k.np) ? __ldg(p.p_idx + k.p0 + j) : __ldg(p.f_idx + k.f0 + (j - k.np));
}

// cap * tanh(x / cap) for |x / cap| < 0.5: Maclaurin series of tanh through
// y^13 (truncation error below 1e-6 relative at |y| = 0.5, far less below).
__device__ __forceinline__ float softcap_series(float x, float cap, float inv_cap) {
  const float y = x * inv_cap;
  const float y2 = y * y;
  float s = 21844.0f / 6081075.0f;
  s = fmaf(s, y2, -1382.0f / 155925.0f);
  s = fmaf(s, y2, 62.0f / 2835.0f);
  s = fmaf(s, y2, -17.0f / 315.0f);
  s = fmaf(s, y2, 2.0f / 15.0f);
  s = fmaf(s, y2, -1.0f / 3.0f);
  return cap * fmaf(s * y2, y, y);
}
// cap * tanh(x / cap) for any x, from tanh(y) = 1 - 2 / (exp(2y) + 1).
__device__ __forceinline__ float softcap_exp(float x, float cap, float inv_cap) {
  const float e = ex2_approx(2.0f * kLog2e * (x * inv_cap));
  return cap * (1.0f - __fdividef(2.0f, e + 1.0f));
}

template <int D, bool MODS>
__global__ void __launch_bounds__(kThreads, 1)
    k_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kOffQ;
  const uint32_t sK = base + C::kOffK;
  const uint32_t sV = base + C::kOffV;
  // barrier slots (8 bytes each)
  const uint32_t bar0 = base + C::kOffSmall;
  const uint32_t b_qfull = bar0;                 // [2]
  const uint32_t b_qempty = b_qfull + 16;        // [2]
  const uint32_t b_kfull = b_qempty + 16;        // [KS]
  const uint32_t b_kempty = b_kfull + 8 * KS;    // [KS]
  const uint32_t b_vfull = b_kempty + 8 * KS;    // [VS]
  const uint32_t b_vempty = b_vfull + 8 * VS;    // [VS]
  const uint32_t b_sfull = b_vempty + 8 * VS;    // [3]
  const uint32_t b_pfull = b_sfull + 24;         // [3]
  const uint32_t b_pvdone = b_pfull + 24;        // [3]
  const uint32_t b_odone = b_pvdone + 24;
  const uint32_t b_drain = b_odone + 8;
  uint8_t* small = gbase + C::kOffSmall;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(small + 400);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(small + 408);
  float* xmax = reinterpret_cast<float*>(small + 512);                 // [2 parity][2 wg][128]
  float* xsum = reinterpret_cast<float*>(small + 512 + 2 * 2 * 128 * 4);  // [2 wg][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_qfull + 8 * i, 1);
      mbar_init(b_qempty + 8 * i, 1);
    }
    for (int s = 0; s < KS; ++s) {
      mbar_init(b_kfull + 8 * s, 1);
      mbar_init(b_kempty + 8 * s, 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(b_vfull + 8 * s, 1);
      mbar_init(b_vempty + 8 * s, 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_pfull + 8 * i, kSoftmaxThreads);
      mbar_init(b_pvdone + 8 * i, 1);
    }
    mbar_init(b_odone, 1);
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int g = 0, tq = 0;
      int q_issued = 0, k_issued = 0, v_issued = 0;  // loads actually started (for the abort drain)
      bool pend = false;
      int pv_g = 0, pv_row = 0, pv_hk = 0;
      auto load_v = [&](int gv, int krow, int hk) {
        const int vs = gv % VS;
        if (gv >= VS) mbar_wait(b_vempty + 8 * vs, ((gv / VS) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        if (*abort_flag) return;
        v_issued = gv + 1;
        mbar_arrive_expect_tx(b_vfull + 8 * vs, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_2d(sV + vs * C::kTileBytes + c * 16384, &tmV, b_vfull + 8 * vs, hk * D + c * 64, krow);
      };
      for (int t = blockIdx.x; t < p.ntasks; t += gridDim.x) {
        const Task k = load_task(p, t);
        if (k.n == 0) continue;
        const int qb = tq & 1;
        if (tq >= 2) mbar_wait(b_qempty + 8 * qb, ((tq >> 1) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        if (!*abort_flag) {
          q_issued = tq + 1;
          mbar_arrive_expect_tx(b_qfull + 8 * qb, C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_2d(sQ + qb * C::kTileBytes + c * 16384, &tmQ, b_qfull + 8 * qb, k.h * D + c * 64,
                        k.q_off + k.m_block * kTile);
        }
        for (int j = 0; j < k.n; ++j) {
          const int gi = g + j;
          const int krow = k.k_off + tile_index(p, k, j) * kTile;
          const int ks = gi % KS;
          if (gi >= KS) mbar_wait(b_kempty + 8 * ks, ((gi / KS) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
          if (!*abort_flag) {
            k_issued = gi + 1;
            mbar_arrive_expect_tx(b_kfull + 8 * ks, C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_2d(sK + ks * C::kTileBytes + c * 16384, &tmK, b_kfull + 8 * ks, k.hk * D + c * 64, krow);
          }
          if (pend) load_v(pv_g, pv_row, pv_hk);
          pend = true;
          pv_g = gi;
          pv_row = krow;
          pv_hk = k.hk;
        }
        g += k.n;
        ++tq;
      }
      if (pend) load_v(pv_g, pv_row, pv_hk);
      if (*abort_flag) {
        // let the copies already started land before the CTA exits (the last
        // load of each ring slot is the only one that can still be in flight)
        for (int u = (q_issued > 2 ? q_issued - 2 : 0); u < q_issued; ++u)
          mbar_wait_drain(b_qfull + 8 * (u & 1), (u >> 1) & 1, kWaitTimeoutNs);
        for (int u = (k_issued > KS ? k_issued - KS : 0); u < k_issued; ++u)
          mbar_wait_drain(b_kfull + 8 * (u % KS), (u / KS) & 1, kWaitTimeoutNs);
        for (int u = (v_issued > VS ? v_issued - VS : 0); u < v_issued; ++u)
          mbar_wait_drain(b_vfull + 8 * (u % VS), (u / VS) & 1, kWaitTimeoutNs);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, 1);
      int g = 0, tq = 0;
      bool pend = false;
      int pg = 0;
      bool pacc = false;
      auto issue_pv = [&](int gp, bool acc) {
        const int sb = gp % 3, vs = gp % VS;
        mbar_wait(b_pfull + 8 * sb, (gp / 3) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        mbar_wait(b_vfull + 8 * vs, (gp / VS) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        if (*abort_flag) return;
        tc_fence_after();
        const uint32_t pcol = tmem + 128u * sb;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16_ts(tmem + C::kColO, pcol + 8u * kk,
                       sdesc_sw128(sV + vs * C::kTileBytes + kk * 2048, 16384, 1024), idO,
                       (acc || kk > 0) ? 1u : 0u);
        umma_commit(b_vempty + 8 * vs);
        umma_commit(b_pvdone + 8 * sb);
        umma_commit(b_odone);
      };
      for (int t = blockIdx.x; t < p.ntasks; t += gridDim.x) {
        const Task k = load_task(p, t);
        if (k.n == 0) continue;
        const int qb = tq & 1;
        mbar_wait(b_qfull + 8 * qb, (tq >> 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        for (int j = 0; j < k.n; ++j) {
          const int gi = g + j;
          const int ks = gi % KS, sb = gi % 3;
          mbar_wait(b_kfull + 8 * ks, (gi / KS) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
          if (gi >= 3) mbar_wait(b_pvdone + 8 * sb, ((gi / 3) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
          if (!*abort_flag) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              umma_bf16_ss(tmem + 128u * sb, sdesc_sw128(sQ + qb * C::kTileBytes + off, 16, 1024),
                           sdesc_sw128(sK + ks * C::kTileBytes + off, 16, 1024), idS, kk > 0);
            }
            umma_commit(b_sfull + 8 * sb);
            umma_commit(b_kempty + 8 * ks);
            if (j == k.n - 1) umma_commit(b_qempty + 8 * qb);
          }
          if (pend) issue_pv(pg, pacc);
          pend = true;
          pg = gi;
          pacc = j > 0;
        }
        g += k.n;
        ++tq;
      }
      if (pend) issue_pv(pg, pacc);
      // every MMA issued above completes before TMEM is released
      umma_commit(b_drain);
      mbar_wait_drain(b_drain, 0, kWaitTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wg = warp >> 2;               // column half: 64*wg .. 64*wg+63
    const int r = threadIdx.x & 127;         // score row, TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
    int g = 0;
    for (int t = blockIdx.x; t < p.ntasks; t += gridDim.x) {
      const Task k = load_task(p, t);
      const bool row_ok = r < k.qv;
      const long long grow = static_cast<long long>(k.q_off) + k.m_block * kTile + r;
      __nv_bfloat16* orow = p.o + (grow * p.Hq + k.h) * D + wg * (D / 2);
      if (k.n == 0) {
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int i = 0; i < D / 16; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          if (wg == 0 && p.lse != nullptr) p.lse[static_cast<long long>(k.h) * p.total_q + grow] = -INFINITY;
        }
        continue;
      }
      float slope = 0.0f;
      if (MODS && (p.flags & FA_MOD_ALIBI)) slope = p.slopes[k.h];
      const int q_local = k.m_block * kTile + r;
      float m_run = -INFINITY, l_half = 0.0f;
      for (int j = 0; j < k.n; ++j) {
        const int gi = g + j;
        const int sb = gi % 3;
        const bool partial = j < k.np;
        uint2 pm = make_uint2(0xffffffffu, 0xffffffffu);
        if (partial)
          pm = __ldg(reinterpret_cast<const uint2*>(p.payload) + (static_cast<long long>(k.p0 + j) * kTile + r) * 2 + wg);
        int kt = 0;
        if (MODS) kt = tile_index(p, k, j);
        mbar_wait(b_sfull + 8 * sb, (gi / 3) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        tc_fence_after();
        float s[64];
        tmem_ld64(lane_addr + 128u * sb + 64u * wg, s);
        if (MODS) {
          // natural units: scale, softcap, ALiBi, predicate
          float amax = 0.0f;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            s[c] *= p.scale;
            amax = fmaxf(amax, fabsf(s[c]));
          }
          if (p.flags & FA_MOD_SOFTCAP) {
            if (__any_sync(0xffffffffu, amax >= 0.5f * p.softcap)) {
#pragma unroll
              for (int c = 0; c < 64; ++c) s[c] = softcap_exp(s[c], p.softcap, p.inv_softcap);
            } else {
#pragma unroll
              for (int c = 0; c < 64; ++c) s[c] = softcap_series(s[c], p.softcap, p.inv_softcap);
            }
          }
          const float fd0 = static_cast<float>(kt * kTile + wg * 64 - q_local);  // k - q at column 0
#pragma unroll
          for (int c = 0; c < 64; ++c) s[c] = fmaf(slope, fd0 + static_cast<float>(c), s[c]);
        }
        if (partial) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const uint32_t w = (c < 32) ? pm.x : pm.y;
            if (!((w >> (c & 31)) & 1u)) s[c] = -INFINITY;
          }
        }
        // row max of this half (four independent chains), then of the row
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          m0 = max3f(m0, s[c], s[c + 1]);
          m1 = max3f(m1, s[c + 2], s[c + 3]);
          m2 = max3f(m2, s[c + 4], s[c + 5]);
          m3 = max3f(m3, s[c + 6], s[c + 7]);
        }
        const float mhalf = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        float* xm = xmax + (gi & 1) * 256;
        xm[wg * 128 + r] = mhalf;
        tc_fence_before();
        named_bar_sync(kBarSoftmax, kSoftmaxThreads);
        tc_fence_after();
        const float mrow = fmaxf(mhalf, xm[(wg ^ 1) * 128 + r]);
        // running max in the exponent's units (scaled log2 units without mods)
        const float m_tile = MODS ? mrow : mrow * p.scale_log2;
        const float m_new = fmaxf(m_run, m_tile);
        const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
        const float alpha = MODS ? ex2_approx((m_run - m_use) * kLog2e) : ex2_approx(m_run - m_use);
        m_run = m_new;
        uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;  // packed partial sums
        uint32_t pk[32];
        const uint64_t negm = f2_pack(-m_use, -m_use);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          uint64_t x = f2_pack(s[c], s[c + 1]);
          x = MODS ? f2_mul(f2_add(x, negm), l2e2) : f2_fma(x, sc2, negm);
          float x0, x1;
          f2_unpack(x, x0, x1);
          const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
          const uint64_t e = f2_pack(e0, e1);
          switch ((c >> 1) & 3) {
            case 0: acc0 = f2_add(acc0, e); break;
            case 1: acc1 = f2_add(acc1, e); break;
            case 2: acc2 = f2_add(acc2, e); break;
            default: acc3 = f2_add(acc3, e); break;
          }
          pk[c >> 1] = pack_bf16x2(e0, e1);
        }
        float a0, a1;
        f2_unpack(f2_add(f2_add(acc0, acc1), f2_add(acc2, acc3)), a0, a1);
        l_half = l_half * alpha + (a0 + a1);
        // P (bf16 pairs) over this half's 32 columns of the score buffer
        tmem_st32(lane_addr + 128u * sb + 32u * wg, pk);
        if (j > 0) {
          mbar_wait(b_odone, (gi - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
              uint32_t v[32];
              const uint32_t oa = lane_addr + C::kColO + wg * (D / 2) + 32u * c;
              tmem_ld32(oa, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
              tmem_st32(oa, v);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_pfull + 8 * sb);
      }
      g += k.n;
      // ---------------------------------------------------------- epilogue
      mbar_wait(b_odone, (g - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
      tc_fence_after();
      xsum[wg * 128 + r] = l_half;
      named_bar_sync(kBarSoftmax, kSoftmaxThreads);
      const float l = l_half + xsum[(wg ^ 1) * 128 + r];
      const bool have = l > 0.0f;
      const float inv_l = have ? 1.0f / l : 0.0f;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_addr + C::kColO + wg * (D / 2) + 32u * c, v);
        if (row_ok) {
          uint32_t pkd[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pkd[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
        }
      }
      if (wg == 0 && row_ok && p.lse != nullptr) {
        float lse = -INFINITY;
        if (have) lse = MODS ? (m_run + __logf(l)) : (m_run + __log2f(l)) * kLn2;
        p.lse[static_cast<long long>(k.h) * p.total_q + grow] = lse;
      }
      // the sum exchange slots are rewritten at the next task's epilogue only
      // after at least one more softmax barrier, so no extra barrier is needed
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D view [rows, heads*D] of a bf16 tensor, box 64 x 128, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t heads, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * D * 2)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool MODS>
cudaError_t launch_impl(const FwdLaunch& a, cudaStream_t st, const char** why) {
  const fa_plan* pl = a.plan;
  const Geometry& g = pl->geom;
  const int64_t rows_q = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_q : g.total_q;
  const int64_t rows_k = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_k : g.total_k;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, rows_q, g.heads_q, D) || !make_map(&mk, a.k, rows_k, g.heads_k, D) ||
      !make_map(&mv, a.v, rows_k, g.heads_k, D)) {
    *why = "cuTensorMapEncodeTiled failed (pointer alignment or driver entry point)";
    return cudaErrorInvalidValue;
  }
  FwdParams p{};
  p.ntasks = static_cast<int>(pl->tasks);
  p.work = pl->work_desc;
  p.seq = pl->seq_desc;
  p.p_off = pl->p_off;
  p.f_off = pl->f_off;
  p.p_idx = pl->p_idx;
  p.f_idx = pl->f_idx;
  p.payload = pl->payload;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.Hq = g.heads_q;
  p.Hk = g.heads_k;
  p.Hmask = pl->Hmask;
  p.rows = static_cast<int>(pl->rows);
  p.total_q = static_cast<int>(rows_q);
  p.flags = a.flags;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.softcap = a.softcap;
  p.inv_softcap = (a.softcap > 0.0f) ? 1.0f / a.softcap : 0.0f;
  if (a.flags & FA_MOD_ALIBI)
    for (int h = 0; h < g.heads_q; ++h) p.slopes[h] = a.slopes[h];
  auto kern = k_fwd<D, MODS>;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem);
  if (e != cudaSuccess) {
    *why = "device attribute / cudaFuncSetAttribute failed";
    return e;
  }
  // persistent: one CTA per SM (shared memory keeps it to one), tasks by static stride
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(pl->tasks, sms));
  kern<<<grid, kThreads, Cfg<D>::kSmem, st>>>(mq, mk, mv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) *why = "forward kernel launch failed";
  return e;
}

}  // namespace

cudaError_t launch_fwd_d64(const FwdLaunch& a, cudaStream_t st, const char** why) {
  return (a.flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI)) ? launch_impl<64, true>(a, st, why)
                                                     : launch_impl<64, false>(a, st, why);
}
cudaError_t launch_fwd_d128(const FwdLaunch& a, cudaStream_t st, const char** why) {
  return (a.flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI)) ? launch_impl<128, true>(a, st, why)
                                                     : launch_impl<128, false>(a, st, why);
}

uint32_t* fwd_error_word() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_fwd_err) != cudaSuccess) return nullptr;
  return static_cast<uint32_t*>(ptr);
}

}  // namespace bsm
