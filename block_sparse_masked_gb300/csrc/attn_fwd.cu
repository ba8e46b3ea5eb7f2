// attn_fwd.cu -- masked attention forward on sm_103a consuming a MaskPlan.
//
// Consumption protocol of "Flex Attention Mask Plan Design" §6.1: for one
// (sample, Q head, Q tile) task, the partial K tiles are processed with the
// packed predicate (§5: bit 1 keeps the score, bit 0 makes it -inf), then
// the full K tiles without it; empty tiles are never visited.  A row without
// any visible key ends with O = 0 and LSE = -inf.  The math is FlexAttention
// Eq. 1, softmax(mod(Q K^T * scale)) V, computed with an online softmax so
// the score matrix is never stored.
//
// One CTA per task (the plan's work_desc gives the execution order), 192
// threads, warp-specialised:
//   warp 4     TMA producer: Q once, then K and V tiles through a ring of
//              kStages shared-memory stages (mbarrier transaction counts).
//   warp 5     TMEM allocator and MMA issuer (one thread): S = Q K^T into a
//              double-buffered TMEM accumulator, O += P V into a TMEM
//              accumulator, completion signalled with tcgen05.commit.
//   warps 0-3  softmax warpgroup: thread r owns score row r (TMEM lane r),
//              applies scale, score_mods and the predicate, keeps the running
//              max / sum, writes P (bf16) to shared memory and rescales O in
//              TMEM when the max moves; epilogue writes O (bf16) and LSE.
// Every wait is bounded (global-timer limit); on a timeout the CTA sets an
// error bit, drains what it has in flight, frees TMEM and exits.
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

__device__ uint32_t g_fwd_err = 0;

namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;         // 64-column (128-byte) swizzle chunks
  static constexpr int kTileBytes = 128 * D * 2; // Q, K or V tile, bf16
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kPBytes = 128 * 128 * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffP = kOffV + kStages * kTileBytes;
  static constexpr int kOffBar = kOffP + 2 * kPBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = kOffBar + kBarBytes + 1024;  // + slack for 1 KB alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S buffers at columns 0 and 128
  static constexpr uint32_t kColO = 256;  // O accumulator
  static_assert(kSmem <= 232448, "shared memory budget");
};

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
  int Hq, Hk, Hmask, rows, total_q;
  int flags;
  float scale;       // multiplies Q K^T
  float scale_log2;  // scale * log2(e)
  float softcap, inv_softcap;
  float slopes[kMaxHeads];
};

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
__global__ void __launch_bounds__(192, 1)
    k_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kOffQ;
  const uint32_t sK = base + C::kOffK;
  const uint32_t sV = base + C::kOffV;
  const uint32_t sP = base + C::kOffP;
  const uint32_t bar0 = base + C::kOffBar;
  // barrier slots (8 bytes each)
  const uint32_t b_q = bar0;
  const uint32_t b_kfull = bar0 + 8;                // [S]
  const uint32_t b_vfull = b_kfull + 8 * S;         // [S]
  const uint32_t b_empty = b_vfull + 8 * S;         // [S]
  const uint32_t b_sfull = b_empty + 8 * S;         // [2]
  const uint32_t b_pfull = b_sfull + 16;            // [2]
  const uint32_t b_odone = b_pfull + 16;
  const uint32_t b_drain = b_odone + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBar + 8 * (3 * S + 8));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBar + 8 * (3 * S + 8) + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int* wd = p.work + 4LL * blockIdx.x;
  const int m_block = wd[0], h = wd[1], b = wd[2], qv = wd[3];
  const int* sq = p.seq + 8 * b;
  const int q_off = sq[0], k_off = sq[1], row_begin = sq[4];
  const int hm = (p.Hmask == 1) ? 0 : h;
  const int hk = h / (p.Hq / p.Hk);
  const long long flat = static_cast<long long>(hm) * p.rows + row_begin + m_block;
  const int p0 = p.p_off[flat], np_ = p.p_off[flat + 1] - p0;
  const int f0 = p.f_off[flat], nf = p.f_off[flat + 1] - f0;
  const int n = np_ + nf;
  const int q_row0 = q_off + m_block * kTile;

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(b_kfull + 8 * s, 1);
      mbar_init(b_vfull + 8 * s, 1);
      mbar_init(b_empty + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_pfull + 8 * i, 128);
    }
    mbar_init(b_odone, 1);
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(b_q, C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) tma_load_2d(sQ + c * 16384, &tmQ, b_q, h * D + c * 64, q_row0);
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j % S;
        if (j >= S && !mbar_wait(b_empty + 8 * st, ((j / S) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs))
          break;
        const int kt = (j < np_) ? __ldg(p.p_idx + p0 + j) : __ldg(p.f_idx + f0 + (j - np_));
        const int krow = k_off + kt * kTile;
        mbar_arrive_expect_tx(b_kfull + 8 * st, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_2d(sK + st * C::kTileBytes + c * 16384, &tmK, b_kfull + 8 * st, hk * D + c * 64, krow);
        mbar_arrive_expect_tx(b_vfull + 8 * st, C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_2d(sV + st * C::kTileBytes + c * 16384, &tmV, b_vfull + 8 * st, hk * D + c * 64, krow);
        issued = j + 1;
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA exits
        mbar_wait_drain(b_q, 0, kWaitTimeoutNs);
        for (int j = (issued > S ? issued - S : 0); j < issued; ++j) {
          mbar_wait_drain(b_kfull + 8 * (j % S), (j / S) & 1, kWaitTimeoutNs);
          mbar_wait_drain(b_vfull + 8 * (j % S), (j / S) & 1, kWaitTimeoutNs);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, 1);
      auto issue_s = [&](int buf, int st) {
        const uint32_t dcol = tmem + C::kColS + 128u * buf;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_bf16_ss(dcol, sdesc_sw128(sQ + off, 16, 1024),
                       sdesc_sw128(sK + st * C::kTileBytes + off, 16, 1024), idS, kk > 0);
        }
      };
      auto issue_pv = [&](int buf, int st, bool acc) {
        const uint32_t dcol = tmem + C::kColO;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_bf16_ss(dcol, sdesc_sw128(sP + buf * C::kPBytes + aoff, 16, 1024),
                       sdesc_sw128(sV + st * C::kTileBytes + kk * 2048, 16384, 1024), idO,
                       (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(b_q, 0, abort_flag, &g_fwd_err, kWaitTimeoutNs) &&
                mbar_wait(b_kfull, 0, abort_flag, &g_fwd_err, kWaitTimeoutNs);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        umma_commit(b_sfull);
        for (int j = 0; j < n; ++j) {
          if (j + 1 < n) {
            const int st1 = (j + 1) % S;
            if (!mbar_wait(b_kfull + 8 * st1, ((j + 1) / S) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs)) break;
            tc_fence_after();
            issue_s((j + 1) & 1, st1);
            umma_commit(b_sfull + 8 * ((j + 1) & 1));
          }
          const int st = j % S;
          if (!mbar_wait(b_pfull + 8 * (j & 1), (j >> 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs)) break;
          if (!mbar_wait(b_vfull + 8 * st, (j / S) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs)) break;
          tc_fence_after();
          issue_pv(j & 1, st, j > 0);
          umma_commit(b_empty + 8 * st);
          umma_commit(b_odone);
        }
      }
      // every MMA issued above completes before TMEM is released
      umma_commit(b_drain);
      mbar_wait_drain(b_drain, 0, kWaitTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // score row, TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int q_local = m_block * kTile + r;
    float m_run = -INFINITY, l_run = 0.0f;
    float slope = 0.0f;
    if (MODS && (p.flags & FA_MOD_ALIBI)) slope = p.slopes[h];
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int buf = j & 1;
      const bool partial = j < np_;
      uint4 pm = make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
      if (partial) pm = __ldg(reinterpret_cast<const uint4*>(p.payload) + static_cast<long long>(p0 + j) * kTile + r);
      int kt = 0;
      if (MODS) kt = partial ? __ldg(p.p_idx + p0 + j) : __ldg(p.f_idx + f0 + (j - np_));
      if (!__all_sync(0xffffffffu,
                      mbar_wait(b_sfull + 8 * buf, (j >> 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[128];
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t v[32];
        tmem_ld32(lane_addr + C::kColS + 128u * buf + 32u * c4, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c4 * 32 + i] = __uint_as_float(v[i]);
      }
      const uint32_t pw[4] = {pm.x, pm.y, pm.z, pm.w};
      float mx = -INFINITY;
      if (MODS) {
        const float fd0 = static_cast<float>(kt * kTile - q_local);  // k - q at column 0
        float amax = 0.0f;
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          x[c] *= p.scale;
          amax = fmaxf(amax, fabsf(x[c]));
        }
        if (p.flags & FA_MOD_SOFTCAP) {
          // warp-uniform choice between the series (|s/cap| < 0.5 everywhere)
          // and the exponential form of tanh
          if (__any_sync(0xffffffffu, amax >= 0.5f * p.softcap)) {
#pragma unroll
            for (int c = 0; c < 128; ++c) x[c] = softcap_exp(x[c], p.softcap, p.inv_softcap);
          } else {
#pragma unroll
            for (int c = 0; c < 128; ++c) x[c] = softcap_series(x[c], p.softcap, p.inv_softcap);
          }
        }
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          float s = fmaf(slope, fd0 + static_cast<float>(c), x[c]);
          if (partial && !((pw[c >> 5] >> (c & 31)) & 1u)) s = -INFINITY;
          x[c] = s;
          mx = fmaxf(mx, s);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          float s = x[c] * p.scale_log2;
          if (partial && !((pw[c >> 5] >> (c & 31)) & 1u)) s = -INFINITY;
          x[c] = s;
          mx = fmaxf(mx, s);
        }
      }
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      float alpha, rowsum = 0.0f;
      uint32_t pk[64];
      if (MODS) {
        alpha = ex2_approx((m_run - m_use) * kLog2e);
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          const float e0 = ex2_approx((x[c] - m_use) * kLog2e);
          const float e1 = ex2_approx((x[c + 1] - m_use) * kLog2e);
          rowsum += e0 + e1;
          pk[c >> 1] = pack_bf16x2(e0, e1);
        }
      } else {
        alpha = ex2_approx(m_run - m_use);
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          const float e0 = ex2_approx(x[c] - m_use);
          const float e1 = ex2_approx(x[c + 1] - m_use);
          rowsum += e0 + e1;
          pk[c >> 1] = pack_bf16x2(e0, e1);
        }
      }
      l_run = l_run * alpha + rowsum;
      m_run = m_new;
      // P(j) -> shared memory, 128-byte swizzled K-major layout (two 64-key chunks)
      {
        const uint32_t prow = sP + buf * C::kPBytes + r * 128;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int w0 = c * 32 + u * 4;  // packed word index (2 keys per word)
            st_shared_v4(prow + c * 16384 + ((u ^ (r & 7)) << 4), pk[w0], pk[w0 + 1], pk[w0 + 2], pk[w0 + 3]);
          }
      }
      if (j > 0) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(b_odone, (j - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(lane_addr + C::kColO + 32u * c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(lane_addr + C::kColO + 32u * c, v);
          }
          tmem_st_wait();
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(b_pfull + 8 * buf);
    }
    // ------------------------------------------------------------ epilogue
    const bool row_ok = r < qv;
    const long long grow = static_cast<long long>(q_row0) + r;
    __nv_bfloat16* orow = p.o + (grow * p.Hq + h) * D;
    bool have = (n > 0) && ok && (l_run > 0.0f);
    if (n > 0 && ok) {
      if (!__all_sync(0xffffffffu,
                      mbar_wait(b_odone, (n - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs))) {
        ok = false;
        have = false;
      }
    }
    if (n > 0 && ok) {
      tc_fence_after();
      const float inv_l = have ? 1.0f / l_run : 0.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(lane_addr + C::kColO + 32u * c, v);
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
    } else if (row_ok) {
      uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
    }
    if (row_ok && p.lse != nullptr) {
      float lse = -INFINITY;
      if (have) lse = MODS ? (m_run + __logf(l_run)) : (m_run + __log2f(l_run)) * kLn2;
      p.lse[static_cast<long long>(h) * p.total_q + grow] = lse;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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
  static thread_local int configured_dev = -1;  // attribute is per device
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem);
  (void)configured_dev;
  if (e != cudaSuccess) {
    *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  kern<<<static_cast<unsigned>(pl->tasks), 192, Cfg<D>::kSmem, st>>>(mq, mk, mv, p);
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
