// attn_bwd.cu -- masked attention backward on sm_103a consuming a MaskPlan
// built with FA_PLAN_BACKWARD.
//
// "Flex Attention Mask Plan Design" §6.3: each backward consumer uses the
// traversal that matches its output.  Here:
//   k_bwd_delta  Delta = rowsum(dO * O) per (query row, Q head).
//   k_bwd_dq     Q-major, one CTA per forward task (work_desc entry): walks
//                the forward Q2K view (the backward consumers use the
//                forward's tile geometry), partial tiles with their packed
//                predicate, full tiles without; dQ accumulates in TMEM.
//   k_bwd_dkdv   K-major, one CTA per (K plan row, K/V head): walks the K2Q
//                view of every Q head of the K/V head's group (partial
//                entries with the key-major predicate, full entries
//                without); dK and dV accumulate in TMEM over the group.
// Gradients of FlexAttention Eq. 1 with the score mods of the forward
// (scale, tanh softcap, ALiBi): with z = mod(scale * QK^T) and the
// forward's LSE, P = exp(z - LSE), dP = dO V^T, dZ = P * (dP - Delta),
// dS = dZ * dz/ds (1 - tanh^2 under softcap, 1 otherwise; ALiBi adds a
// constant), dQ = scale * dS K, dK = scale * dS^T Q, dV = P^T dO.  Masked
// pairs have P = 0.  Scores are recomputed from Q and K.
//
// Both gradient kernels: warps 0-7 two compute warpgroups (each owns 64 of
// the 128 score columns of a tile pair), warp 8 the TMA producer, warp 9
// TMEM allocation and the single MMA-issuing thread.  S and dP land in
// TMEM; the compute threads read them, write P (dK/dV) and dS back into
// TMEM as bf16, and those are the A operand of the accumulating MMAs.
// Every wait is an mbarrier wait with a global-timer limit; after a timeout
// the CTA records an error bit and ends without hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace bsm {
namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr int D = 128;
constexpr int kTileBytes = 128 * D * 2;  // one 128-row bf16 tile: 32 KB
constexpr int kThreads = 320;
constexpr int kWarpProducer = 8, kWarpMma = 9;

struct BwdParams {
  // forward Q2K view
  const int32_t* work;
  const int32_t* seq;
  const int32_t* p_off;
  const int32_t* f_off;
  const int32_t* p_idx;
  const int32_t* f_idx;
  const uint32_t* payload;
  // backward K2Q view
  const int32_t* cu_krows;
  const int32_t* krow_batch;
  const int32_t* kp_off;
  const int32_t* kf_off;
  const int32_t* kp_idx;
  const int32_t* kf_idx;
  const uint32_t* kpayload;
  // per-row statistics [Hq, total_q]
  const float* lse;    // natural log, from the forward
  const float* delta;  // rowsum(dO * O)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  uint32_t* err;
  int Hq, Hk, Hmask, rows, k_rows, total_q, ntasks;
  int B, total_k;                  // samples, K rows of the tensors
  long long nP, nF, kP, kF;        // Q2K and K2Q entries (bounds of the checked build)
  int flags;
  float scale, scale_log2;
  float y_scale, cap;  // softcap: z = cap * tanh(y_scale * s)
  float slopes[kMaxHeads];
};

// One score element of the backward, from the raw q.k product s and dP:
// returns p (bf16-ready) in `pv` and dS (before the final scale) in `dsv`.
template <bool MODS>
__device__ __forceinline__ void grad_elem(const BwdParams& p, float s, float dp, float lse_l2, float delta,
                                          float alibi_l2, bool vis, float& pv, float& dsv) {
  float z_l2, dzds = 1.0f;
  if (MODS) {
    float z;
    if (p.flags & FA_MOD_SOFTCAP) {
      const float y = s * p.y_scale;
      const float e = ex2_approx(2.0f * kLog2e * y);
      const float th = 1.0f - __fdividef(2.0f, e + 1.0f);
      z = p.cap * th;
      dzds = 1.0f - th * th;
    } else {
      z = s * p.scale;
    }
    z_l2 = z * kLog2e + alibi_l2;
  } else {
    z_l2 = s * p.scale_log2;
  }
  const float pr = vis ? ex2_approx(z_l2 - lse_l2) : 0.0f;
  pv = pr;
  dsv = pr * (dp - delta) * dzds;
}

// ============================================================ Delta
__global__ void __launch_bounds__(256) k_bwd_delta(const __nv_bfloat16* __restrict__ o,
                                                   const __nv_bfloat16* __restrict__ dout,
                                                   float* __restrict__ delta, long long n_rows, int Hq) {
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;  // (row, head)
  const int lane = threadIdx.x & 31;
  if (w >= n_rows * Hq) return;
  const long long row = w / Hq;
  const int h = static_cast<int>(w % Hq);
  const uint2 a = __ldg(reinterpret_cast<const uint2*>(o + w * D) + lane);
  const uint2 b = __ldg(reinterpret_cast<const uint2*>(dout + w * D) + lane);
  auto dot2 = [](uint32_t x, uint32_t y) {
    const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x));
    const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&y));
    return fx.x * fy.x + fx.y * fy.y;
  };
  float acc = dot2(a.x, b.x) + dot2(a.y, b.y);
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
  if (lane == 0) delta[static_cast<long long>(h) * n_rows + row] = acc;
}

// ============================================================ dQ (Q-major)
struct DqTask {
  int m_block, h, b, qv, q_off, k_off, hk, p0, np, f0, n, pad;
};

__device__ __forceinline__ DqTask dq_task(const BwdParams& p, int t) {
  DqTask k;
  const int* wd = p.work + 4LL * t;
  k.m_block = __ldg(wd + 0);
  k.h = static_cast<int>(bsm_idx(__ldg(wd + 1), p.Hq, p.err));
  k.b = static_cast<int>(bsm_idx(__ldg(wd + 2), p.B, p.err));
  k.qv = __ldg(wd + 3);
  const int* sq = p.seq + 8 * k.b;
  k.q_off = __ldg(sq + 0);
  k.k_off = __ldg(sq + 1);
  const int row_begin = __ldg(sq + 4);
  const int hm = (p.Hmask == 1) ? 0 : k.h;
  k.hk = k.h / (p.Hq / p.Hk);
  const long long flat = bsm_idx(static_cast<long long>(hm) * p.rows + row_begin + k.m_block,
                                 static_cast<long long>(p.Hmask) * p.rows, p.err);
  k.p0 = __ldg(p.p_off + flat);
  k.np = __ldg(p.p_off + flat + 1) - k.p0;
  k.f0 = __ldg(p.f_off + flat);
  k.n = k.np + (__ldg(p.f_off + flat + 1) - k.f0);
  return k;
}

// Shared memory of the dQ kernel: Q and dO tiles of the task, a two-stage
// ring of (K, V) tiles, then barriers and a task broadcast slot.
constexpr int kDqOffQ = 0, kDqOffDO = kTileBytes, kDqOffKV = 2 * kTileBytes;
constexpr int kDqStages = 2;
constexpr int kDqOffSmall = kDqOffKV + kDqStages * 2 * kTileBytes;
constexpr int kDqSmall = 512;
constexpr int kDqSmem = kDqOffSmall + kDqSmall + 1024;
static_assert(kDqSmem <= 232448, "shared memory budget");
// TMEM columns: S of tile j at 128 (j % 2), dP at 256, dQ at 384.
constexpr uint32_t kColDP = 256, kColDQ = 384;

template <bool MODS>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_dq(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
             const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  if ((base - raw) + kDqOffSmall + kDqSmall > static_cast<uint32_t>(kDqSmem)) {
    if (threadIdx.x == 0) atomicOr(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  const uint32_t sQ = base + kDqOffQ, sDO = base + kDqOffDO, sKV = base + kDqOffKV;
  uint8_t* small = gbase + kDqOffSmall;
  const uint32_t bars = base + kDqOffSmall;
  const uint32_t b_qfull = bars, b_qempty = bars + 8;
  const uint32_t b_kvfull = bars + 16, b_kvempty = b_kvfull + 8 * kDqStages;
  const uint32_t b_sfull = b_kvempty + 8 * kDqStages;   // [2] per S buffer
  const uint32_t b_dpfree = b_sfull + 16;               // compute has read S and dP of a tile
  const uint32_t b_dsfull = b_dpfree + 8;               // [2] dS written into S buffer
  const uint32_t b_dqdone = b_dsfull + 16;              // [2] the dQ MMA of a tile has completed
  const uint32_t b_dqfree = b_dqdone + 16;              // epilogue has read dQ
  const uint32_t b_tfull = b_dqfree + 8, b_tempty = b_tfull + 16;  // [2] task ring
  const uint32_t b_clc = b_tempty + 16, b_drain = b_clc + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(small + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(small + 260);
  const uint32_t clc_resp = smem_u32(small + 272);
  DqTask* tring = reinterpret_cast<DqTask*>(small + 320);  // [2]
  DqTask* tdec = reinterpret_cast<DqTask*>(small + 416);   // broadcast to the compute warps
  static_assert(8 * 22 <= 256 && 416 + sizeof(DqTask) <= kDqSmall, "small area");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    for (int i = 0; i < kDqStages; ++i) {
      mbar_init(b_kvfull + 8 * i, 1);
      mbar_init(b_kvempty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_dsfull + 8 * i, 256);
      mbar_init(b_dqdone + 8 * i, 1);
      mbar_init(b_tfull + 8 * i, 1);
      mbar_init(b_tempty + 8 * i, 2);  // MMA issuer and compute thread 0
    }
    mbar_init(b_dpfree, 256);
    mbar_init(b_dqfree, 256);
    mbar_init(b_clc, 1);
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    const bool leader = lane == 0;
    int tq = 0, c = 0, ti = 0, q_issued = 0, c_issued = 0;
    ClcTasks tasks{clc_resp, b_clc};
    for (;;) {
      int t = -1;
      if (leader) t = tasks.next(abort_flag, p.err, kWaitTimeoutNs);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0 || t >= p.ntasks || *abort_flag) break;
      const DqTask k = dq_task(p, t);
      if (leader) {
        const int slot = ti & 1;
        if (ti >= 2) mbar_wait(b_tempty + 8 * slot, ((ti >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        tring[slot] = k;
        mbar_arrive(b_tfull + 8 * slot);
      }
      __syncwarp();
      ++ti;
      if (k.n == 0) continue;
      const int row = k.q_off + k.m_block * 128;
      if (leader) {
        if (tq >= 1) mbar_wait(b_qempty, (tq - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (!*abort_flag) {
          q_issued = tq + 1;
          mbar_arrive_expect_tx(b_qfull, 2 * kTileBytes);
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            tma_load_2d(sQ + ch * 16384, &tmQ, b_qfull, k.h * D + ch * 64, row);
            tma_load_2d(sDO + ch * 16384, &tmDO, b_qfull, k.h * D + ch * 64, row);
          }
        }
      }
      __syncwarp();
      ++tq;
      for (int j0 = 0; j0 < k.n; j0 += 32) {
        int my_kt = 0;
        if (j0 + lane < k.n)
          my_kt = (j0 + lane < k.np) ? __ldg(p.p_idx + bsm_idx(k.p0 + j0 + lane, p.nP, p.err))
                                     : __ldg(p.f_idx + bsm_idx(k.f0 + j0 + lane - k.np, p.nF, p.err));
        const int cnt = min(32, k.n - j0);
        for (int jj = 0; jj < cnt; ++jj) {
          const int kt = __shfl_sync(0xffffffffu, my_kt, jj);
          if (leader) {
            const int slot = c % kDqStages;
            if (c >= kDqStages)
              mbar_wait(b_kvempty + 8 * slot, ((c / kDqStages) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
            if (!*abort_flag) {
              c_issued = c + 1;
              const uint32_t dst = sKV + slot * 2 * kTileBytes;
              mbar_arrive_expect_tx(b_kvfull + 8 * slot, 2 * kTileBytes);
#pragma unroll
              for (int ch = 0; ch < 2; ++ch) {
                tma_load_2d(dst + ch * 16384, &tmK, b_kvfull + 8 * slot, k.hk * D + ch * 64, k.k_off + kt * 128);
                tma_load_2d(dst + kTileBytes + ch * 16384, &tmV, b_kvfull + 8 * slot, k.hk * D + ch * 64,
                            k.k_off + kt * 128);
              }
            }
          }
          __syncwarp();
          ++c;
        }
      }
    }
    if (leader) {
      const int slot = ti & 1;
      if (ti >= 2) mbar_wait(b_tempty + 8 * slot, ((ti >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
      DqTask end{};
      end.n = -1;
      tring[slot] = end;
      mbar_arrive(b_tfull + 8 * slot);
      if (*abort_flag) {
        if (q_issued > 0) mbar_wait_drain(b_qfull, (q_issued - 1) & 1, kWaitTimeoutNs);
        for (int u = (c_issued > kDqStages ? c_issued - kDqStages : 0); u < c_issued; ++u)
          mbar_wait_drain(b_kvfull + 8 * (u % kDqStages), (u / kDqStages) & 1, kWaitTimeoutNs);
        tasks.drain(kWaitTimeoutNs);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0);  // both K-major
      constexpr uint32_t idQ = idesc_bf16_f32(128, D, 1);    // dS (TMEM) x K (MN-major)
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024), dDO0 = sdesc_sw128(sDO, 16, 1024);
      const uint64_t dKV0 = sdesc_sw128(sKV, 16, 1024);
      const uint64_t dKmn0 = sdesc_sw128(sKV, 16384, 1024);
      int g = 0, c = 0, tq = 0;
      bool pend = false;
      int pg = 0, pslot = 0;
      bool pfirst = false;
      int ntask_dq = 0;  // tasks whose dQ has been accumulated (for the dQ buffer hand-back)
      auto issue_dq = [&]() {
        const int sb = pg & 1;
        mbar_wait(b_dsfull + 8 * sb, (pg >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (pfirst && ntask_dq >= 1) mbar_wait(b_dqfree, (ntask_dq - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (pfirst) ++ntask_dq;
        if (*abort_flag) return;
        tc_fence_after();
        const uint64_t dK = dKmn0 + static_cast<uint64_t>((pslot * 2 * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // dS of keys 16kk..16kk+15: compute warpgroup kk/4 packed them at
          // the start of its own 64-column half of the S buffer
          const uint32_t acol = 128u * sb + 64u * (kk >> 2) + 8u * (kk & 3);
          umma_bf16_ts(tmem + kColDQ, tmem + acol, dK + static_cast<uint64_t>((kk * 2048) >> 4), idQ,
                       (!pfirst || kk > 0) ? 1u : 0u);
        }
        umma_commit(b_kvempty + 8 * pslot);
        umma_commit(b_dqdone + 8 * sb);
      };
      for (int ti = 0;; ++ti) {
        const int tslot = ti & 1;
        mbar_wait(b_tfull + 8 * tslot, (ti >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        const DqTask k = tring[tslot];
        mbar_arrive(b_tempty + 8 * tslot);
        if (k.n < 0 || *abort_flag) break;
        if (k.n == 0) continue;
        mbar_wait(b_qfull, tq & 1, abort_flag, p.err, kWaitTimeoutNs);
        for (int j = 0; j < k.n; ++j, ++g) {
          const int slot = c % kDqStages, sb = g & 1;
          mbar_wait(b_kvfull + 8 * slot, (c / kDqStages) & 1, abort_flag, p.err, kWaitTimeoutNs);
          ++c;
          // S buffer sb: the dQ MMA that read dS from it two tiles ago is done;
          // dP: the compute threads have read the previous tile's
          if (g >= 2) mbar_wait(b_dqdone + 8 * sb, ((g >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (g >= 1) mbar_wait(b_dpfree, (g - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (*abort_flag) break;
          tc_fence_after();
          const uint64_t dK = dKV0 + static_cast<uint64_t>((slot * 2 * kTileBytes) >> 4);
          const uint64_t dV = dK + static_cast<uint64_t>(kTileBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tmem + 128u * sb, dQ0 + off, dK + off, idS, kk > 0);
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tmem + kColDP, dDO0 + off, dV + off, idS, kk > 0);
          }
          umma_commit(b_sfull + 8 * sb);
          if (pend) issue_dq();
          pend = true;
          pg = g;
          pslot = slot;
          pfirst = (j == 0);
        }
        // the task's last dQ MMA now (its epilogue waits for it), then Q/dO are free
        if (pend) issue_dq();
        pend = false;
        umma_commit(b_qempty);
        ++tq;
      }
      umma_commit(b_drain);
      mbar_wait_drain(b_drain, 0, kWaitTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2, r = threadIdx.x & 127;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    int g = 0;
    for (int ti = 0;; ++ti) {
      if (threadIdx.x == 0) {
        const int tslot = ti & 1;
        mbar_wait(b_tfull + 8 * tslot, (ti >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        DqTask kk = tring[tslot];
        mbar_arrive(b_tempty + 8 * tslot);
        if (*abort_flag) kk.n = -1;
        *tdec = kk;
      }
      named_bar_sync(1, 256);
      const DqTask k = *tdec;
      named_bar_sync(1, 256);
      if (k.n < 0) break;
      const long long grow = static_cast<long long>(k.q_off) + k.m_block * 128 + r;
      const bool row_ok = r < k.qv && bsm_ok(grow, p.total_q, p.err);
      __nv_bfloat16* dqrow = p.dq + (grow * p.Hq + k.h) * D + wg * 64;
      if (k.n == 0) {
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(dqrow);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const long long srow = static_cast<long long>(k.h) * p.total_q + grow;
      const float lse_l2 = row_ok ? __ldg(p.lse + srow) * kLog2e : 0.0f;
      const float dl = row_ok ? __ldg(p.delta + srow) : 0.0f;
      const float slope_l2 = (MODS && (p.flags & FA_MOD_ALIBI)) ? p.slopes[k.h] * kLog2e : 0.0f;
      const int q_local = k.m_block * 128 + r;
      for (int j = 0; j < k.n; ++j, ++g) {
        const int sb = g & 1;
        const bool partial = j < k.np;
        uint2 pw = make_uint2(~0u, ~0u);
        if (partial)
          pw = __ldg(reinterpret_cast<const uint2*>(p.payload + bsm_idx(k.p0 + j, p.nP, p.err) * 512 + r * 4) + wg);
        const int kt = (MODS && (p.flags & FA_MOD_ALIBI))
                           ? (partial ? __ldg(p.p_idx + bsm_idx(k.p0 + j, p.nP, p.err))
                                      : __ldg(p.f_idx + bsm_idx(k.f0 + j - k.np, p.nF, p.err)))
                           : 0;
        mbar_wait(b_sfull + 8 * sb, (g >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        tc_fence_after();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float s[32], dp[32];
          const uint32_t col = 64u * wg + 32u * h2;
          tmem_ld32f(lane_addr + 128u * sb + col, s);
          tmem_ld32f(lane_addr + kColDP + col, dp);
          if (h2 == 1) {
            tc_fence_before();
            mbar_arrive(b_dpfree);  // S and dP of this tile are in registers
          }
          const uint32_t bits = h2 ? pw.y : pw.x;
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float pv0, pv1, ds0, ds1;
            const float al0 = slope_l2 * static_cast<float>(kt * 128 + static_cast<int>(col) + c - q_local);
            grad_elem<MODS>(p, s[c], dp[c], lse_l2, dl, al0, (bits >> c) & 1u, pv0, ds0);
            grad_elem<MODS>(p, s[c + 1], dp[c + 1], lse_l2, dl, al0 + slope_l2, (bits >> (c + 1)) & 1u, pv1, ds1);
            pk[c / 2] = pack_bf16x2(ds0, ds1);
          }
          // dS of these 32 keys, packed, at the start of this group's half
          tmem_st16(lane_addr + 128u * sb + 64u * wg + 16u * h2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_dsfull + 8 * sb);
      }
      // ---------------------------------------------------------- epilogue
      mbar_wait(b_dqdone + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
      tc_fence_after();
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float v[32];
        tmem_ld32f(lane_addr + kColDQ + 64u * wg + 32u * h2, v);
        if (row_ok) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(v[2 * c] * p.scale, v[2 * c + 1] * p.scale);
          uint4* dst = reinterpret_cast<uint4*>(dqrow + 32 * h2);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(b_dqfree);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================ dK, dV (K-major)
// Shared memory: K and V tiles of the task, a two-stage ring of (Q, dO)
// tiles with the LSE (log2 units) and Delta of their 128 rows.
constexpr int kKvOffK = 0, kKvOffV = kTileBytes, kKvOffRing = 2 * kTileBytes;
constexpr int kKvStageBytes = 2 * kTileBytes + 1024;  // Q, dO, lse[128], delta[128]
constexpr int kKvStages = 2;
constexpr int kKvOffSmall = kKvOffRing + kKvStages * kKvStageBytes;
constexpr int kKvSmall = 256;
constexpr int kKvSmem = kKvOffSmall + kKvSmall + 1024;
static_assert(kKvSmem <= 232448, "shared memory budget");
// TMEM columns: dV at 0, dK at 128, S^T at 256, dP^T at 384.
constexpr uint32_t kColDV = 0, kColDK = 128, kColST = 256, kColDPT = 384;

// The step sequence of a K/V task: the K2Q entries of every Q head of the
// group, partial entries before full ones, heads in order.
struct KvWalk {
  int g = 0, e = 0, n_g = 0, np_g = 0, p0 = 0, f0 = 0;  // group member, entry within it
  __device__ __forceinline__ void load(const BwdParams& p, int hk, int krow) {
    const int h = hk * (p.Hq / p.Hk) + g;
    const int hm = (p.Hmask == 1) ? 0 : h;
    const long long flat = bsm_idx(static_cast<long long>(hm) * p.k_rows + krow,
                                   static_cast<long long>(p.Hmask) * p.k_rows, p.err);
    p0 = __ldg(p.kp_off + flat);
    np_g = __ldg(p.kp_off + flat + 1) - p0;
    f0 = __ldg(p.kf_off + flat);
    n_g = np_g + (__ldg(p.kf_off + flat + 1) - f0);
  }
  // advance to the next entry; false at the end of the group
  __device__ __forceinline__ bool next(const BwdParams& p, int hk, int krow) {
    const int G = p.Hq / p.Hk;
    ++e;
    while (e >= n_g) {
      if (++g >= G) return false;
      e = 0;
      load(p, hk, krow);
    }
    return true;
  }
  __device__ __forceinline__ bool start(const BwdParams& p, int hk, int krow) {
    g = 0;
    e = -1;
    n_g = 0;
    load(p, hk, krow);
    return next(p, hk, krow);
  }
  __device__ __forceinline__ int head(const BwdParams& p, int hk) const { return hk * (p.Hq / p.Hk) + g; }
  __device__ __forceinline__ bool partial() const { return e < np_g; }
  __device__ __forceinline__ int qtile(const BwdParams& p) const {
    return partial() ? __ldg(p.kp_idx + bsm_idx(p0 + e, p.kP, p.err))
                     : __ldg(p.kf_idx + bsm_idx(f0 + e - np_g, p.kF, p.err));
  }
  __device__ __forceinline__ long long entry(const BwdParams& p) const {
    return bsm_idx(static_cast<long long>(p0) + e, p.kP, p.err);
  }
};

template <bool MODS>
__global__ void __launch_bounds__(kThreads, 1)
    k_bwd_dkdv(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
               const __grid_constant__ BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  if ((base - raw) + kKvOffSmall + kKvSmall > static_cast<uint32_t>(kKvSmem)) {
    if (threadIdx.x == 0) atomicOr(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  const uint32_t sK = base + kKvOffK, sV = base + kKvOffV, sRing = base + kKvOffRing;
  uint8_t* small = gbase + kKvOffSmall;
  const uint32_t bars = base + kKvOffSmall;
  const uint32_t b_kvfull = bars;
  const uint32_t b_full = bars + 8, b_empty = b_full + 8 * kKvStages;  // ring stages
  const uint32_t b_sfull = b_empty + 8 * kKvStages;  // S^T and dP^T of a step are in TMEM
  const uint32_t b_pdsfull = b_sfull + 8;            // P^T and dS^T written back
  const uint32_t b_accdone = b_pdsfull + 8;          // the step's dV/dK MMAs completed
  const uint32_t b_drain = b_accdone + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(small + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(small + 132);
  static_assert(8 * (1 + 2 * kKvStages + 4) <= 128, "small area");

  // task: (K/V head, K plan row), heads outermost so that neighbouring CTAs
  // read the same heads' Q and dO
  const int hk = static_cast<int>(blockIdx.x / p.k_rows);
  const int krow = static_cast<int>(blockIdx.x % p.k_rows);
  const int b = static_cast<int>(bsm_idx(__ldg(p.krow_batch + krow), p.B, p.err));
  const int kt = krow - __ldg(p.cu_krows + b);
  const int* sq = p.seq + 8 * b;
  const int q_off = __ldg(sq + 0), k_off = __ldg(sq + 1), q_len = __ldg(sq + 2), k_len = __ldg(sq + 3);
  const int kv = min(128, k_len - kt * 128);  // valid keys of the tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(b_kvfull, 1);
    for (int i = 0; i < kKvStages; ++i) {
      mbar_init(b_full + 8 * i, 1);
      mbar_init(b_empty + 8 * i, 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_pdsfull, 256);
    mbar_init(b_accdone, 1);
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    const bool leader = lane == 0;
    int s = 0, issued = 0;
    KvWalk wk;
    bool more = wk.start(p, hk, krow);
    if (leader && more) {
      mbar_arrive_expect_tx(b_kvfull, 2 * kTileBytes);
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        tma_load_2d(sK + ch * 16384, &tmK, b_kvfull, hk * D + ch * 64, k_off + kt * 128);
        tma_load_2d(sV + ch * 16384, &tmV, b_kvfull, hk * D + ch * 64, k_off + kt * 128);
      }
    }
    for (; more && !*abort_flag; more = wk.next(p, hk, krow), ++s) {
      const int st = s % kKvStages;
      const int h = wk.head(p, hk);
      const int qt = wk.qtile(p);
      const int q0 = q_off + qt * 128, qv = min(128, q_len - qt * 128);
      if (leader && s >= kKvStages) mbar_wait(b_empty + 8 * st, ((s / kKvStages) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
      __syncwarp();
      // the rows' LSE (log2 units; +inf past the sample, where nothing is visible) and Delta
      float* lse_s = reinterpret_cast<float*>(gbase + kKvOffRing + st * kKvStageBytes + 2 * kTileBytes);
      float* del_s = lse_s + 128;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = lane + 32 * i;
        const long long idx = static_cast<long long>(h) * p.total_q + q0 + rr;
        const bool in = rr < qv && bsm_ok(q0 + rr, p.total_q, p.err);
        lse_s[rr] = in ? __ldg(p.lse + idx) * kLog2e : INFINITY;
        del_s[rr] = in ? __ldg(p.delta + idx) : 0.0f;
      }
      __syncwarp();
      if (leader && !*abort_flag) {
        issued = s + 1;
        const uint32_t dst = sRing + st * kKvStageBytes;
        mbar_arrive_expect_tx(b_full + 8 * st, 2 * kTileBytes);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          tma_load_2d(dst + ch * 16384, &tmQ, b_full + 8 * st, h * D + ch * 64, q0);
          tma_load_2d(dst + kTileBytes + ch * 16384, &tmDO, b_full + 8 * st, h * D + ch * 64, q0);
        }
      }
      __syncwarp();
    }
    if (leader && *abort_flag) {
      mbar_wait_drain(b_kvfull, 0, kWaitTimeoutNs);
      for (int u = (issued > kKvStages ? issued - kKvStages : 0); u < issued; ++u)
        mbar_wait_drain(b_full + 8 * (u % kKvStages), (u / kKvStages) & 1, kWaitTimeoutNs);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0);  // K / V (keys) x Q / dO (rows), K-major
      constexpr uint32_t idA = idesc_bf16_f32(128, D, 1);    // P^T / dS^T (TMEM) x dO / Q (MN-major)
      const uint64_t dK = sdesc_sw128(sK, 16, 1024), dV = sdesc_sw128(sV, 16, 1024);
      const uint64_t dR0 = sdesc_sw128(sRing, 16, 1024);
      const uint64_t dRmn0 = sdesc_sw128(sRing, 16384, 1024);
      KvWalk wk;
      int s = 0;
      bool more = wk.start(p, hk, krow);
      if (more) mbar_wait(b_kvfull, 0, abort_flag, p.err, kWaitTimeoutNs);
      for (; more && !*abort_flag; more = wk.next(p, hk, krow), ++s) {
        const int st = s % kKvStages;
        mbar_wait(b_full + 8 * st, (s / kKvStages) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (s >= 1) mbar_wait(b_accdone, (s - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (*abort_flag) break;
        tc_fence_after();
        const uint64_t dQs = dR0 + static_cast<uint64_t>((st * kKvStageBytes) >> 4);
        const uint64_t dDOs = dQs + static_cast<uint64_t>(kTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_bf16_ss(tmem + kColST, dK + off, dQs + off, idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_bf16_ss(tmem + kColDPT, dV + off, dDOs + off, idS, kk > 0);
        }
        umma_commit(b_sfull);
        mbar_wait(b_pdsfull, s & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (*abort_flag) break;
        tc_fence_after();
        const uint64_t dQmn = dRmn0 + static_cast<uint64_t>((st * kKvStageBytes) >> 4);
        const uint64_t dDOmn = dQmn + static_cast<uint64_t>(kTileBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // P^T / dS^T of query rows 16kk..16kk+15: compute warpgroup kk/4
          // packed them at the start of its own 64-column half
          const uint32_t acol = 64u * (kk >> 2) + 8u * (kk & 3);
          const uint64_t boff = static_cast<uint64_t>((kk * 2048) >> 4);
          umma_bf16_ts(tmem + kColDV, tmem + kColST + acol, dDOmn + boff, idA, (s > 0 || kk > 0) ? 1u : 0u);
          umma_bf16_ts(tmem + kColDK, tmem + kColDPT + acol, dQmn + boff, idA, (s > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(b_empty + 8 * st);
        umma_commit(b_accdone);
      }
      umma_commit(b_drain);
      mbar_wait_drain(b_drain, 0, kWaitTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2, t = threadIdx.x & 127;  // key t of the tile; query columns 64wg..64wg+63
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int k_local = kt * 128 + t;
    KvWalk wk;
    int s = 0;
    bool more = wk.start(p, hk, krow);
    for (; more && !*abort_flag; more = wk.next(p, hk, krow), ++s) {
      const int st = s % kKvStages;
      const bool partial = wk.partial();
      const int h = wk.head(p, hk);
      const int qt = (MODS && (p.flags & FA_MOD_ALIBI)) ? wk.qtile(p) : 0;
      const float slope_l2 = (MODS && (p.flags & FA_MOD_ALIBI)) ? p.slopes[h] * kLog2e : 0.0f;
      uint2 pw = make_uint2(~0u, ~0u);
      if (partial)
        pw = __ldg(reinterpret_cast<const uint2*>(p.kpayload + wk.entry(p) * 512 + t * 4) + wg);
      const float* lse_s = reinterpret_cast<const float*>(gbase + kKvOffRing + st * kKvStageBytes + 2 * kTileBytes);
      const float* del_s = lse_s + 128;
      mbar_wait(b_full + 8 * st, (s / kKvStages) & 1, abort_flag, p.err, kWaitTimeoutNs);  // LSE, Delta
      mbar_wait(b_sfull, s & 1, abort_flag, p.err, kWaitTimeoutNs);
      tc_fence_after();
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        float sv[32], dp[32];
        const uint32_t col = 64u * wg + 32u * h2;  // query columns of this pass
        tmem_ld32f(lane_addr + kColST + col, sv);
        tmem_ld32f(lane_addr + kColDPT + col, dp);
        const uint32_t bits = h2 ? pw.y : pw.x;
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float2 l2 = *reinterpret_cast<const float2*>(lse_s + col + c);
          const float2 de = *reinterpret_cast<const float2*>(del_s + col + c);
          const float al0 = slope_l2 * static_cast<float>(k_local - (qt * 128 + static_cast<int>(col) + c));
          float pv0, pv1, ds0, ds1;
          grad_elem<MODS>(p, sv[c], dp[c], l2.x, de.x, al0, (bits >> c) & 1u, pv0, ds0);
          grad_elem<MODS>(p, sv[c + 1], dp[c + 1], l2.y, de.y, al0 - slope_l2, (bits >> (c + 1)) & 1u, pv1, ds1);
          pp[c / 2] = pack_bf16x2(pv0, pv1);
          pd[c / 2] = pack_bf16x2(ds0, ds1);
        }
        tmem_st16(lane_addr + kColST + 64u * wg + 16u * h2, pp);
        tmem_st16(lane_addr + kColDPT + 64u * wg + 16u * h2, pd);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(b_pdsfull);
    }
    // ---------------------------------------------------------- epilogue
    if (s > 0) {
      mbar_wait(b_accdone, (s - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
      tc_fence_after();
    }
    const long long krow_g = static_cast<long long>(k_off) + kt * 128 + t;
    const bool key_ok = t < kv && bsm_ok(krow_g, p.total_k, p.err);
    __nv_bfloat16* dkrow = p.dk + (krow_g * p.Hk + hk) * D + wg * 64;
    __nv_bfloat16* dvrow = p.dv + (krow_g * p.Hk + hk) * D + wg * 64;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      float a[32], bsum[32];
      if (s > 0) {
        tmem_ld32f(lane_addr + kColDK + 64u * wg + 32u * h2, a);
        tmem_ld32f(lane_addr + kColDV + 64u * wg + 32u * h2, bsum);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) a[c] = bsum[c] = 0.0f;
      }
      if (key_ok) {
        uint32_t pk[16], pv[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          pk[c] = pack_bf16x2(a[2 * c] * p.scale, a[2 * c + 1] * p.scale);
          pv[c] = pack_bf16x2(bsum[2 * c], bsum[2 * c + 1]);
        }
        uint4* dk4 = reinterpret_cast<uint4*>(dkrow + 32 * h2);
        uint4* dv4 = reinterpret_cast<uint4*>(dvrow + 32 * h2);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dk4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          dv4[i] = make_uint4(pv[4 * i], pv[4 * i + 1], pv[4 * i + 2], pv[4 * i + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_bwd() {
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

// 2-D view [rows, heads*D] of a bf16 tensor, box 64 columns x 128 rows, 128-byte swizzle.
bool make_map_bwd(CUtensorMap* m, const void* ptr, int64_t rows, int64_t heads) {
  auto fn = encode_fn_bwd();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * D * 2)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class Kern>
cudaError_t launch_pdl(Kern kern, unsigned grid, int smem, cudaStream_t st, const CUtensorMap& a,
                       const CUtensorMap& b, const CUtensorMap& c, const CUtensorMap& d, const BwdParams& p) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, b, c, d, p);
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t st, const char** why) {
  const fa_plan* pl = a.plan;
  const Geometry& g = pl->geom;
  if (g.head_dim != D) {
    *why = "the backward supports head_dim 128";
    return cudaErrorInvalidValue;
  }
  const int64_t rows_q = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_q : g.total_q;
  const int64_t rows_k = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_k : g.total_k;
  // Delta = rowsum(dO * O), one warp per (row, head)
  if (rows_q > 0) {
    const long long warps = rows_q * g.heads_q;
    const unsigned blocks = static_cast<unsigned>((warps * 32 + 255) / 256);
    k_bwd_delta<<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(a.o),
                                        static_cast<const __nv_bfloat16*>(a.dout), a.delta, rows_q, g.heads_q);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      *why = "Delta kernel launch failed";
      return e;
    }
  }
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map_bwd(&mq, a.q, rows_q, g.heads_q) || !make_map_bwd(&mk, a.k, rows_k, g.heads_k) ||
      !make_map_bwd(&mv, a.v, rows_k, g.heads_k) || !make_map_bwd(&mdo, a.dout, rows_q, g.heads_q)) {
    *why = "cuTensorMapEncodeTiled failed (pointer alignment or driver entry point)";
    return cudaErrorInvalidValue;
  }
  BwdParams p{};
  p.work = pl->work_desc;
  p.seq = pl->seq_desc;
  p.p_off = pl->p_off;
  p.f_off = pl->f_off;
  p.p_idx = pl->p_idx;
  p.f_idx = pl->f_idx;
  p.payload = pl->payload;
  p.cu_krows = pl->cu_krows;
  p.krow_batch = pl->krow_batch;
  p.kp_off = pl->kp_off;
  p.kf_off = pl->kf_off;
  p.kp_idx = pl->kp_idx;
  p.kf_idx = pl->kf_idx;
  p.kpayload = pl->kpayload;
  p.lse = a.lse;
  p.delta = a.delta;
  p.dq = static_cast<__nv_bfloat16*>(a.dq);
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.err = fwd_error_word();
  p.Hq = g.heads_q;
  p.Hk = g.heads_k;
  p.Hmask = pl->Hmask;
  p.rows = static_cast<int>(pl->rows);
  p.k_rows = static_cast<int>(pl->k_rows);
  p.total_q = static_cast<int>(rows_q);
  p.ntasks = static_cast<int>(pl->tasks);
  p.B = g.batch;
  p.total_k = static_cast<int>(rows_k);
  p.nP = pl->P;
  p.nF = pl->F;
  p.kP = pl->kP;
  p.kF = pl->kF;
  p.flags = a.flags;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.y_scale = (a.softcap > 0.0f) ? a.scale / a.softcap : 0.0f;
  p.cap = a.softcap;
  if (a.flags & FA_MOD_ALIBI)
    for (int h = 0; h < g.heads_q; ++h) p.slopes[h] = a.slopes[h];
  if (p.err == nullptr) {
    *why = "error word not found";
    return cudaErrorInvalidValue;
  }
  const bool mods = (a.flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI)) != 0;
  cudaError_t e = cudaSuccess;
  if (pl->tasks > 0) {
    e = mods ? launch_pdl(k_bwd_dq<true>, static_cast<unsigned>(pl->tasks), kDqSmem, st, mq, mk, mv, mdo, p)
             : launch_pdl(k_bwd_dq<false>, static_cast<unsigned>(pl->tasks), kDqSmem, st, mq, mk, mv, mdo, p);
    if (e != cudaSuccess) {
      *why = "dQ kernel launch failed";
      return e;
    }
  }
  const long long kv_tasks = static_cast<long long>(pl->k_rows) * g.heads_k;
  if (kv_tasks > 0) {
    e = mods ? launch_pdl(k_bwd_dkdv<true>, static_cast<unsigned>(kv_tasks), kKvSmem, st, mq, mk, mv, mdo, p)
             : launch_pdl(k_bwd_dkdv<false>, static_cast<unsigned>(kv_tasks), kKvSmem, st, mq, mk, mv, mdo, p);
    if (e != cudaSuccess) *why = "dK/dV kernel launch failed";
  }
  return e;
}

}  // namespace bsm
