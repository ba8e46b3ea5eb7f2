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
// Tasks are scheduled in work_desc order by the GPU's cluster launch control
// ("Flex Attention Mask Plan Design" §4.8: the SM100/SM103 forward takes its
// tasks from the hardware CLC queue): the kernel is launched with one CTA per
// task, shared memory keeps one CTA per SM, and each running CTA handles its
// own task and then takes over tasks of CTAs that have not started yet.  No
// state outlives a launch, so one plan serves concurrent calls on any
// streams.  320 threads, warp-specialised:
//   warp 8      TMA producer: Q tiles into a 2-deep ring; K and V tiles into
//               one ring, issued in the order the MMAs consume them (K of
//               tile g+1 before V of tile g).
//   warp 9      TMEM allocator and MMA issuer (one thread): S(g) = Q K^T into
//               one of three TMEM score buffers, then O += P(g-1) V with P
//               read from TMEM (it overwrites its score buffer in bf16).
//   warps 0-7   two softmax warpgroups; thread r of warpgroup w owns score
//               row r, columns 64w..64w+63 (TMEM lane r).  Per tile they
//               exchange the row max through shared memory, write P to TMEM,
//               rescale their half of O when the reference max moves, and
//               store their half of the output at the end of the task.
// Block-mask plans run in steps of two 64-key positions (next_step below):
// tiles with one live key half are paired, so that each step multiplies and
// exponentiates 128 keys.
// Every wait is an mbarrier wait with a global-timer limit (the softmax
// warps synchronise through an mbarrier too, not a named barrier).  After a
// timeout the CTA records an error bit, stops waiting, drains copies and
// MMAs in flight, frees TMEM and exits.
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
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold, log2 units

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;          // 64-column (128-byte) swizzle chunks
  static constexpr int kTileBytes = 128 * D * 2;  // Q, K or V tile, bf16
  static constexpr int kQStages = 2;
  static constexpr int kSlots = (D == 128) ? 5 : 12;  // one ring of K and V tiles
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + kQStages * kTileBytes;
  static constexpr int kOffSmall = kOffKV + kSlots * kTileBytes;
  static constexpr int kSmallBytes = 512 + 256 + 128 + 2 * 2 * 128 * 4;  // barriers, task ring, task broadcast, exchange
  static constexpr int kNeed = kOffSmall + kSmallBytes;
  // dynamic shared memory normally starts 1 KB-aligned; what is left up to the
  // per-block limit is slack for a misaligned start (checked at run time)
  static constexpr int kSmem = (kNeed + 1024 <= 232448) ? kNeed + 1024 : 232448;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 384;  // S buffers at 0, 128, 256; O after them
  static_assert(kColO + D <= kTmemCols, "TMEM budget");
  static_assert(kNeed <= 232448, "shared memory budget");
};

constexpr int kWG = 2;                     // softmax warpgroups, 64 score columns each
constexpr int kCols = 128 / kWG;
constexpr int kSoftmaxThreads = 128 * kWG;
constexpr int kWarpProducer = 4 * kWG, kWarpMma = 4 * kWG + 1;
constexpr int kThreads = kSoftmaxThreads + 64;
constexpr uint32_t kBarSoftmax = 1;  // named barrier of the softmax warps

struct FwdParams {
  const int32_t* work;
  const int32_t* seq;
  const int32_t* p_off;
  const int32_t* f_off;
  const int32_t* p_idx;
  const int32_t* f_idx;
  const uint32_t* payload;
  const uint8_t* halves;  // [P] bit s: key columns 64s..64s+63 of the entry hold a visible element
  __nv_bfloat16* o;
  float* lse;
  int Hq, Hk, Hmask, rows, total_q, ntasks;
  int B;             // samples
  long long nP, nF;  // partial and full entries of the plan (bounds of the checked build)
  int flags;
  float scale;       // multiplies Q K^T
  float scale_log2;  // scale * log2(e)
  float y_scale;     // scale / softcap: argument of tanh per unit of Q K^T
  float cap_log2;    // softcap * log2(e)
  float c1, c3, c5;  // cap_log2 * tanh(y_scale * s) ~ s * (c1 + s^2 * (c3 + s^2 * c5)) for small y
  float slopes[kMaxHeads];
};

// Per-task view of the plan shared by every role (decoded once by the
// producer and handed to the other roles through a shared-memory ring).
struct Task {
  int m_block, h, b, qv, q_off, k_off, hk, p0, np, f0, n, pad;
};
constexpr int kTaskRing = 2;  // tasks a CTA may hold ahead of its softmax warps

__device__ __forceinline__ Task load_task(const FwdParams& p, int t) {
  Task k;
  const int* wd = p.work + 4LL * t;
  k.m_block = wd[0];
  k.h = static_cast<int>(bsm_idx(wd[1], p.Hq, &g_fwd_err));
  k.b = static_cast<int>(bsm_idx(wd[2], p.B, &g_fwd_err));
  k.qv = wd[3];
  const int* sq = p.seq + 8 * k.b;
  k.q_off = sq[0];
  k.k_off = sq[1];
  const int row_begin = sq[4];
  const int hm = (p.Hmask == 1) ? 0 : k.h;
  k.hk = k.h / (p.Hq / p.Hk);
  const long long flat =
      bsm_idx(static_cast<long long>(hm) * p.rows + row_begin + k.m_block, static_cast<long long>(p.Hmask) * p.rows,
              &g_fwd_err);
  k.p0 = p.p_off[flat];
  k.np = p.p_off[flat + 1] - k.p0;
  k.f0 = p.f_off[flat];
  k.n = k.np + (p.f_off[flat + 1] - k.f0);
  return k;
}

__device__ __forceinline__ int tile_index(const FwdParams& p, const Task& k, int j) {
  return (j < k.np) ? __ldg(p.p_idx + bsm_idx(k.p0 + j, p.nP, &g_fwd_err))
                    : __ldg(p.f_idx + bsm_idx(k.f0 + (j - k.np), p.nF, &g_fwd_err));
}
// Key halves of tile j that hold a visible element (bit s: keys 64s..64s+63);
// full tiles use both.  A tile with one empty half loads, multiplies and
// exponentiates only the other half.
__device__ __forceinline__ int tile_halves(const FwdParams& p, const Task& k, int j) {
  return (j < k.np) ? static_cast<int>(__ldg(p.halves + bsm_idx(k.p0 + j, p.nP, &g_fwd_err))) : 3;
}

// Block-mask plans (HALVES): one ring slot, score buffer and P V step
// ("step") carries 128 keys in two 64-key positions.  A tile whose two
// halves are live fills both positions; tiles with one live half are paired
// in list order, the first at position 0 and the second at position 1, and
// an unpaired last one runs alone at position 0.  The producer, the MMA
// issuer and the softmax warps derive the same sequence from the plan.
// The walk is warp-uniform: lane l keeps the halves of entries base+l (hc)
// and base+32+l (hn, loaded one batch ahead), read by shuffle.
struct StepIter {
  int j;       // next plan entry to examine
  int pend;    // entry with one live half waiting for a partner, or -1
  int pend_h;  // its halves
  int base;    // first entry of the batch in hc
  int hc, hn;  // this lane's halves of entries base+lane, base+32+lane
};
__device__ __forceinline__ void step_begin(const FwdParams& p, const Task& k, StepIter& it, int lane) {
  it.j = 0;
  it.pend = -1;
  it.pend_h = 0;
  it.base = 0;
  it.hc = tile_halves(p, k, lane);
  it.hn = tile_halves(p, k, 32 + lane);
}
// Next step of the task: entries ea (position 0) and eb (position 1; eb ==
// ea for a tile with both halves live, -1 when position 1 is empty) and
// their halves ha, hb.  Returns false when the task has no step left.
__device__ __forceinline__ bool next_step(const FwdParams& p, const Task& k, StepIter& it, int lane, int& ea,
                                          int& eb, int& ha, int& hb) {
  while (it.j < k.n) {
    const int j = it.j++;
    while (j >= it.base + 32) {
      it.base += 32;
      it.hc = it.hn;
      it.hn = tile_halves(p, k, it.base + 32 + lane);
    }
    const int h = __shfl_sync(0xffffffffu, it.hc, j - it.base);
    if (h == 3) {
      ea = eb = j;
      ha = hb = 3;
      return true;
    }
    if (it.pend < 0) {
      it.pend = j;
      it.pend_h = h;
      continue;
    }
    ea = it.pend;
    ha = it.pend_h;
    eb = j;
    hb = h;
    it.pend = -1;
    return true;
  }
  if (it.pend >= 0) {
    ea = it.pend;
    ha = it.pend_h;
    eb = -1;
    hb = 0;
    it.pend = -1;
    return true;
  }
  return false;
}
// Slot tags written by the producer for the MMA issuer (HALVES).
constexpr int kPos0 = 1, kPos1 = 2, kLastStep = 4;

// tanh(y) for |y| < 0.5 on a pair of columns in packed fp32: Maclaurin
// series through y^13 (truncation error below 1e-6 relative at |y| = 0.5).
__device__ __forceinline__ uint64_t tanh_series13(uint64_t y) {
  const uint64_t y2 = f2_mul(y, y);
  uint64_t s = f2_pack(21844.0f / 6081075.0f, 21844.0f / 6081075.0f);
  s = f2_fma(s, y2, f2_pack(-1382.0f / 155925.0f, -1382.0f / 155925.0f));
  s = f2_fma(s, y2, f2_pack(62.0f / 2835.0f, 62.0f / 2835.0f));
  s = f2_fma(s, y2, f2_pack(-17.0f / 315.0f, -17.0f / 315.0f));
  s = f2_fma(s, y2, f2_pack(2.0f / 15.0f, 2.0f / 15.0f));
  s = f2_fma(s, y2, f2_pack(-1.0f / 3.0f, -1.0f / 3.0f));
  return f2_fma(f2_mul(s, y2), y, y);
}
// tanh(y) for any y, from tanh(y) = 1 - 2 / (exp(2y) + 1).
__device__ __forceinline__ float tanh_exp(float y) {
  const float e = ex2_approx(2.0f * kLog2e * y);
  return 1.0f - __fdividef(2.0f, e + 1.0f);
}

// HALVES: the plan may hold partial tiles with an empty 64-key half (block
// masks); those load, multiply and exponentiate only the live half.
template <int D, bool MODS, bool HALVES>
__global__ void __launch_bounds__(kThreads, 1)
    k_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
          const __grid_constant__ CUtensorMap tmKh, const __grid_constant__ CUtensorMap tmVh,
          const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  constexpr int NS = C::kSlots;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kOffQ;
  const uint32_t sKV = base + C::kOffKV;
  // barrier slots (8 bytes each)
  const uint32_t bar0 = base + C::kOffSmall;
  const uint32_t b_qfull = bar0;                 // [2]
  const uint32_t b_qempty = b_qfull + 16;        // [2]
  const uint32_t b_full = b_qempty + 16;         // [NS] K/V ring
  const uint32_t b_empty = b_full + 8 * NS;      // [NS]
  const uint32_t b_sfull = b_empty + 8 * NS;     // [3]
  const uint32_t b_pfull = b_sfull + 24;         // [3]
  const uint32_t b_pvdone = b_pfull + 24;        // [3] PV(g) done: P buffer g%3 free, O updated
  const uint32_t b_drain = b_pvdone + 24;
  const uint32_t b_tfull = b_drain + 8;          // [kTaskRing] task ring
  const uint32_t b_tempty = b_tfull + 8 * kTaskRing;
  const uint32_t b_clc = b_tempty + 8 * kTaskRing;  // cluster launch control response

  uint8_t* small = gbase + C::kOffSmall;
  int* slot_hm = reinterpret_cast<int*>(small + 400);  // [NS] key halves of the K tile in each ring slot
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(small + 480);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(small + 488);
  Task* tring = reinterpret_cast<Task*>(small + 512);    // [kTaskRing]
  Task* tdec = reinterpret_cast<Task*>(small + 768);     // [2] task as seen by the softmax warps
  float* xmax = reinterpret_cast<float*>(small + 896);  // [2 parity][kWG][128]; also the per-task sum exchange
  const uint32_t clc_resp = smem_u32(small + 864);      // [2] 16-byte cluster launch control responses
  static_assert(16 + 16 + 16 * C::kSlots + 3 * 24 + 8 + 16 * kTaskRing + 8 <= 400, "barrier slots");
  static_assert(768 + 2 * sizeof(Task) <= 864, "task broadcast");
  static_assert(C::kSlots * 4 <= 80, "slot tags");
  static_assert(sizeof(Task) * kTaskRing <= 256, "task ring");
  if ((base - raw) + C::kNeed > static_cast<uint32_t>(C::kSmem)) {
    // dynamic shared memory not aligned as expected: report and stop (uniform exit)
    if (threadIdx.x == 0) atomicOr(&g_fwd_err, DEVERR_SMEM_ALIGN);
    return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_qfull + 8 * i, 1);
      mbar_init(b_qempty + 8 * i, 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_full + 8 * s, 1);
      mbar_init(b_empty + 8 * s, 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_pfull + 8 * i, kSoftmaxThreads);
      mbar_init(b_pvdone + 8 * i, 1);
    }
    mbar_init(b_drain, 1);
    mbar_init(b_clc, 1);
    for (int i = 0; i < kTaskRing; ++i) {
      mbar_init(b_tfull + 8 * i, 1);
      mbar_init(b_tempty + 8 * i, 2);  // the MMA issuer and softmax thread 0
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // set-up above overlaps the previous kernel of the stream; the plan, the
  // task queue, Q/K/V and O belong to work that may still be finishing
  grid_dependency_wait();

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    // K and V tiles share one ring, filled in the order the MMA issuer
    // consumes them: K(0), then K(g) followed by V(g-1) for every later tile
    // (across task boundaries; at a boundary the previous task's last V goes
    // first), and V of the last tile at the end.  The whole warp walks the
    // loop: lanes fetch tile indices 32 at a time, lane 0 issues the copies.
    const bool leader = lane == 0;
    if (leader) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      if (HALVES) {
        tma_prefetch_desc(&tmKh);
        tma_prefetch_desc(&tmVh);
      }
    }
    int tq = 0, c = 0;               // tasks with tiles, ring loads
    int q_issued = 0, c_issued = 0;  // loads actually started (for the abort drain)
    bool pend = false;
    int pv_row = 0, pv_hk = 0, pv_hm = 3;
    // a whole 128-row tile, stored [chunk][128 rows][128 bytes]
    auto load_tile = [&](const CUtensorMap* map, int row, int hk) {
      if (leader) {
        const int slot = c % NS;
        if (c >= NS) mbar_wait(b_empty + 8 * slot, ((c / NS) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        if (!*abort_flag) {
          c_issued = c + 1;
          mbar_arrive_expect_tx(b_full + 8 * slot, C::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < C::kChunks; ++ch)
            tma_load_2d(sKV + slot * C::kTileBytes + ch * 16384, map, b_full + 8 * slot, hk * D + ch * 64, row);
        }
      }
      __syncwarp();
      ++c;
    };
    // HALVES: one step into a ring slot, position 0 from source row r0 and
    // (tag & kPos1) position 1 from r1; a position is one 64-row box per
    // 64-column chunk, stored where rows 0-63 (64-127) of a whole tile go
    auto load_step = [&](const CUtensorMap* map64, int r0, int r1, int hk, int tag) {
      if (leader) {
        const int slot = c % NS;
        if (c >= NS) mbar_wait(b_empty + 8 * slot, ((c / NS) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        if (!*abort_flag) {
          c_issued = c + 1;
          slot_hm[slot] = tag;  // published to the MMA issuer by the arrive below
          const bool two = (tag & kPos1) != 0;
          const uint32_t dst = sKV + slot * C::kTileBytes;
          mbar_arrive_expect_tx(b_full + 8 * slot, two ? C::kTileBytes : C::kTileBytes / 2);
#pragma unroll
          for (int ch = 0; ch < C::kChunks; ++ch) {
            tma_load_2d(dst + ch * 16384, map64, b_full + 8 * slot, hk * D + ch * 64, r0);
            if (two) tma_load_2d(dst + ch * 16384 + 8192, map64, b_full + 8 * slot, hk * D + ch * 64, r1);
          }
        }
      }
      __syncwarp();
      ++c;
    };
    int pv_r1 = 0;  // HALVES: source row of the pending V's position 1
    int ti = 0;  // task ring position
    auto publish = [&](const Task& k) {
      if (leader) {
        const int slot = ti % kTaskRing;
        if (ti >= kTaskRing)
          mbar_wait(b_tempty + 8 * slot, ((ti / kTaskRing) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        tring[slot] = k;
        mbar_arrive(b_tfull + 8 * slot);  // release: the task is visible to the waiters
      }
      __syncwarp();
      ++ti;
    };
    ClcTasks tasks{clc_resp, b_clc};
    for (;;) {
      int t = -1;
      if (leader) t = tasks.next(abort_flag, &g_fwd_err, kWaitTimeoutNs);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0 || t >= p.ntasks) break;
      const Task k = load_task(p, t);
      publish(k);
      if (k.n == 0) continue;
      const int qb = tq & 1;
      if (leader) {
        if (tq >= 2) mbar_wait(b_qempty + 8 * qb, ((tq >> 1) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        if (!*abort_flag) {
          q_issued = tq + 1;
          mbar_arrive_expect_tx(b_qfull + 8 * qb, C::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < C::kChunks; ++ch)
            tma_load_2d(sQ + qb * C::kTileBytes + ch * 16384, &tmQ, b_qfull + 8 * qb, k.h * D + ch * 64,
                        k.q_off + k.m_block * kTile);
        }
      }
      __syncwarp();
      // HALVES: steps in next_step order (K of step s, then V of step s-1)
      int pr_row = -1;  // source row of a one-half tile waiting for a partner
      bool first = true;
      auto emit = [&](int r0, int r1, int tag) {
        if (first && pend) {
          load_step(&tmVh, pv_row, pv_r1, pv_hk, pv_hm);
          pend = false;
        }
        first = false;
        load_step(&tmKh, r0, r1, k.hk, tag);
        if (pend) load_step(&tmVh, pv_row, pv_r1, pv_hk, pv_hm);
        pend = true;
        pv_row = r0;
        pv_r1 = r1;
        pv_hk = k.hk;
        pv_hm = tag;
      };
      for (int j0 = 0; j0 < k.n; j0 += 32) {
        int my_kt = 0, my_hm = 3;
        if (j0 + lane < k.n) {
          my_kt = tile_index(p, k, j0 + lane);
          if (HALVES) my_hm = tile_halves(p, k, j0 + lane);
        }
        const int cnt = min(32, k.n - j0);
        for (int jj = 0; jj < cnt; ++jj) {
          const int j = j0 + jj;
          const int krow = k.k_off + __shfl_sync(0xffffffffu, my_kt, jj) * kTile;
          const int hm = __shfl_sync(0xffffffffu, my_hm, jj);
          if constexpr (HALVES) {
            // the softmax warps read this entry's predicate words a few
            // steps from now: bring them into L2 (the payload is read once)
            if (leader && j < k.np)
              bulk_prefetch_l2(p.payload + static_cast<long long>(k.p0 + j) * kTile * 4, kTile * 4 * 4);
            const bool end = j == k.n - 1;
            if (hm == 3) {
              emit(krow, krow + 64, kPos0 | kPos1 | ((end && pr_row < 0) ? kLastStep : 0));
            } else if (pr_row < 0) {
              pr_row = krow + 64 * (hm >> 1);
            } else {
              const int r0 = pr_row;
              pr_row = -1;
              emit(r0, krow + 64 * (hm >> 1), kPos0 | kPos1 | (end ? kLastStep : 0));
            }
          } else {
            if (j == 0 && pend) {
              load_tile(&tmV, pv_row, pv_hk);
              pend = false;
            }
            load_tile(&tmK, krow, k.hk);
            if (pend) load_tile(&tmV, pv_row, pv_hk);
            pend = true;
            pv_row = krow;
            pv_hk = k.hk;
          }
        }
      }
      if (HALVES && pr_row >= 0) emit(pr_row, 0, kPos0 | kLastStep);
      ++tq;
    }
    if (pend) {
      if constexpr (HALVES) load_step(&tmVh, pv_row, pv_r1, pv_hk, pv_hm);
      else load_tile(&tmV, pv_row, pv_hk);
    }
    {
      Task end{};
      end.n = -1;  // end of this CTA's tasks
      publish(end);
    }
    if (leader && *abort_flag) {
      // let the copies already started land before the CTA exits (only the
      // last load of each slot can still be in flight)
      for (int u = (q_issued > 2 ? q_issued - 2 : 0); u < q_issued; ++u)
        mbar_wait_drain(b_qfull + 8 * (u & 1), (u >> 1) & 1, kWaitTimeoutNs);
      for (int u = (c_issued > NS ? c_issued - NS : 0); u < c_issued; ++u)
        mbar_wait_drain(b_full + 8 * (u % NS), (u / NS) & 1, kWaitTimeoutNs);
      tasks.drain(kWaitTimeoutNs);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t idS64 = idesc_bf16_f32(128, 64, 0);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, 1);
      // shared-memory descriptors of Q buffer 0 and ring slot 0 (K-major for
      // Q K^T, MN-major for P V), built once: a step inside the buffers adds
      // its byte offset / 16 to the start-address field, which stays below
      // 2^14 because shared memory is below 256 KB
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sKV, 16384, 1024);
      int g = 0, tq = 0, c = 0;  // tiles, tasks with tiles, ring slots consumed
      bool pend = false;
      int pg = 0, phm = 3;
      bool pacc = false;
      auto issue_pv = [&](int gp, bool acc, int hm) {
        const int sb = gp % 3, slot = c % NS;
        mbar_wait(b_pfull + 8 * sb, (gp / 3) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        mbar_wait(b_full + 8 * slot, (c / NS) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        ++c;
        if (*abort_flag) return;
        tc_fence_after();
        const uint32_t pcol = tmem + 128u * sb;
        const uint64_t dV = dV0 + static_cast<uint64_t>((slot * C::kTileBytes) >> 4);
        // 16-key steps (HALVES: of the occupied positions, hm = the slot tag)
        const int kk1 = (HALVES && !(hm & kPos1)) ? 4 : 8;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (kk < kk1)
            umma_bf16_ts(tmem + C::kColO, pcol + 8u * kk, dV + static_cast<uint64_t>((kk * 2048) >> 4), idO,
                         (acc || kk > 0) ? 1u : 0u);
        umma_commit(b_empty + 8 * slot);
        umma_commit(b_pvdone + 8 * sb);
      };
      for (int ti = 0;; ++ti) {
        const int tslot = ti % kTaskRing;
        mbar_wait(b_tfull + 8 * tslot, (ti / kTaskRing) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        const Task k = tring[tslot];
        mbar_arrive(b_tempty + 8 * tslot);
        if (k.n < 0 || *abort_flag) break;
        if (k.n == 0) continue;
        // the previous task's last PV first (the producer loads its V before
        // this task's K tiles), and before waiting for this task's Q tile:
        // that task's epilogue waits for it
        if (pend) {
          issue_pv(pg, pacc, phm);
          pend = false;
        }
        const int qb = tq & 1;  // (its buffer is handed back by the softmax epilogue)
        mbar_wait(b_qfull + 8 * qb, (tq >> 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        // HALVES: one step per slot until the producer's last-step tag (at
        // most one per plan entry)
        int nsteps = k.n;
        for (int j = 0; j < k.n; ++j) {
          const int gi = g + j;
          const int sb = gi % 3, slot = c % NS;
          mbar_wait(b_full + 8 * slot, (c / NS) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
          const int hm = HALVES ? slot_hm[slot] : 3;  // written by the producer before its arrive
          if (gi >= 3) mbar_wait(b_pvdone + 8 * sb, ((gi / 3) - 1) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
          ++c;
          if (!*abort_flag) {
            tc_fence_after();
            const uint64_t dQ = dQ0 + static_cast<uint64_t>((qb * C::kTileBytes) >> 4);
            const uint64_t dK = dK0 + static_cast<uint64_t>((slot * C::kTileBytes) >> 4);
            // a step with position 0 only multiplies 64 keys (N = 64)
            const uint32_t idQK = (HALVES && !(hm & kPos1)) ? idS64 : idS;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off16 = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
              umma_bf16_ss(tmem + 128u * sb, dQ + off16, dK + off16, idQK, kk > 0);
            }
            umma_commit(b_sfull + 8 * sb);
            umma_commit(b_empty + 8 * slot);
          }
          if (pend) issue_pv(pg, pacc, phm);
          pend = true;
          pg = gi;
          pacc = j > 0;
          phm = hm;
          if (HALVES && ((hm & kLastStep) || *abort_flag)) {
            nsteps = j + 1;
            break;
          }
        }
        g += nsteps;
        ++tq;
      }
      if (pend) issue_pv(pg, pacc, phm);
      // every MMA issued above completes before TMEM is released
      umma_commit(b_drain);
      mbar_wait_drain(b_drain, 0, kWaitTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wg = warp >> 2;                // score columns kCols*wg .. kCols*wg + kCols-1
    const int r = threadIdx.x & 127;         // score row, TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    constexpr int OC = D / kWG;              // output columns of this warpgroup
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    // Thread 0 takes each task from the ring (and turns a timeout into the
    // end marker) and broadcasts it through shared memory, so that every
    // softmax warp runs the same loops and reaches the same named barriers.
    auto group_sync = [&]() { named_bar_sync(kBarSoftmax, kSoftmaxThreads); };
    int g = 0, tq = 0;
    bool store_pending = false;  // thread 0: an output tile is being stored from Q buffer pend_qb
    int pend_qb = 0;
    for (int ti = 0;; ++ti) {
      if (threadIdx.x == 0) {
        const int tslot = ti % kTaskRing;
        mbar_wait(b_tfull + 8 * tslot, (ti / kTaskRing) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        Task kk = tring[tslot];
        mbar_arrive(b_tempty + 8 * tslot);
        if (*abort_flag) kk.n = -1;
        tdec[ti & 1] = kk;
      }
      group_sync();
      const Task k = tdec[ti & 1];
      if (k.n < 0) break;
      const long long grow = static_cast<long long>(k.q_off) + k.m_block * kTile + r;
      const bool row_ok = r < k.qv && bsm_ok(grow, p.total_q, &g_fwd_err);
      __nv_bfloat16* orow = p.o + (grow * p.Hq + k.h) * D + wg * OC;
      if (k.n == 0) {
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int i = 0; i < OC / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          if (wg == 0 && p.lse != nullptr) p.lse[static_cast<long long>(k.h) * p.total_q + grow] = -INFINITY;
        }
        continue;
      }
      const int qb = tq & 1;
      float slope2 = 0.0f;  // ALiBi slope in log2 units
      if (MODS && (p.flags & FA_MOD_ALIBI)) slope2 = p.slopes[k.h] * kLog2e;
      const int q_local = k.m_block * kTile + r;
      float m_run = -INFINITY, l_part = 0.0f;
      // predicate words of this warpgroup's 64 columns of this thread's row
      const uint2* pay = reinterpret_cast<const uint2*>(p.payload + static_cast<long long>(k.p0) * kTile * 4 + r * 4) + wg;
      // One step (tile) of the online softmax: plan entry e supplies these
      // 64 columns (-1: an empty position), hh is its 64-key half, pw the
      // predicate words of this row (all ones unless partial), kt its K tile.
      auto step = [&](const int j, const int e, const int hh, const bool partial, const uint2 pw, const int kt) {
        const int gi = g + j;
        const int sb = gi % 3;
        // a warp whose 32 rows see none of this warpgroup's 64 columns (an
        // empty position, or a key half with no visible key in these rows)
        // has nothing to exponentiate: its P is 0
        const bool dead = HALVES && (e < 0 || (partial && __all_sync(0xffffffffu, (pw.x | pw.y) == 0u)));
        mbar_wait(b_sfull + 8 * sb, (gi / 3) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
        tc_fence_after();
        float s[kCols];
        if (!dead) tmem_ld64(lane_addr + 128u * sb + kCols * wg, s);
        else {
#pragma unroll
          for (int c = 0; c < kCols; ++c) s[c] = -INFINITY;
        }
        if (MODS && !dead) {
          // scores in log2 units, log2(e) * (softcap(scale * s) + slope * (k - q)),
          // pairs of columns in packed fp32; the tanh series is chosen per warp
          // from the largest |y| = |scale * s / softcap| it holds
          if (p.flags & FA_MOD_SOFTCAP) {
            float amax = 0.0f;
#pragma unroll
            for (int c = 0; c < kCols; c += 2) amax = max3f(amax, fabsf(s[c]), fabsf(s[c + 1]));
            const float ya = amax * p.y_scale;
            const uint64_t ys = f2_pack(p.y_scale, p.y_scale), cl = f2_pack(p.cap_log2, p.cap_log2);
            if (__any_sync(0xffffffffu, ya >= 0.5f)) {
#pragma unroll
              for (int c = 0; c < kCols; ++c) s[c] = p.cap_log2 * tanh_exp(s[c] * p.y_scale);
            } else if (__any_sync(0xffffffffu, ya >= 0.125f)) {
#pragma unroll
              for (int c = 0; c < kCols; c += 2)
                f2_unpack(f2_mul(tanh_series13(f2_mul(f2_pack(s[c], s[c + 1]), ys)), cl), s[c], s[c + 1]);
            } else {
              // |y| < 0.125: the series through y^5 (the first omitted term,
              // 17 y^7 / 315, is below 3e-7 of y there), with y_scale and
              // cap_log2 folded into its coefficients: a polynomial in the
              // raw score s and u = s^2
              const uint64_t k1 = f2_pack(p.c1, p.c1), k3 = f2_pack(p.c3, p.c3), k5 = f2_pack(p.c5, p.c5);
#pragma unroll
              for (int c = 0; c < kCols; c += 2) {
                const uint64_t x = f2_pack(s[c], s[c + 1]);
                const uint64_t u = f2_mul(x, x);
                f2_unpack(f2_mul(x, f2_fma(u, f2_fma(u, k5, k3), k1)), s[c], s[c + 1]);
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < kCols; c += 2) f2_unpack(f2_mul(f2_pack(s[c], s[c + 1]), sc2), s[c], s[c + 1]);
          }
          if (p.flags & FA_MOD_ALIBI) {
            const float fd0 = static_cast<float>(kt * kTile + hh * kCols - q_local);  // k - q at column 0
            const uint64_t sl = f2_pack(slope2, slope2);
#pragma unroll
            for (int c = 0; c < kCols; c += 2) {
              const uint64_t kq = f2_pack(fd0 + static_cast<float>(c), fd0 + static_cast<float>(c + 1));
              f2_unpack(f2_fma(sl, kq, f2_pack(s[c], s[c + 1])), s[c], s[c + 1]);
            }
          }
        }
        // (a warp whose rows see every one of its 64 columns skips it)
        if (partial && !dead && !__all_sync(0xffffffffu, (pw.x & pw.y) == ~0u)) {
#pragma unroll
          for (int c = 0; c < kCols; ++c)
            if (!((((c < 32) ? pw.x : pw.y) >> (c & 31)) & 1u)) s[c] = -INFINITY;
        }
        // row max of this quarter (four independent chains), then of the row
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < kCols; c += 8) {
          m0 = max3f(m0, s[c], s[c + 1]);
          m1 = max3f(m1, s[c + 2], s[c + 3]);
          m2 = max3f(m2, s[c + 4], s[c + 5]);
          m3 = max3f(m3, s[c + 6], s[c + 7]);
        }
        float* xm = xmax + (gi & 1) * (kWG * 128);
        xm[wg * 128 + r] = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        tc_fence_before();
        group_sync();
        tc_fence_after();
        if (j == 0 && threadIdx.x == 0 && store_pending) {
          // the previous task's output tile has left shared memory by now:
          // hand its Q buffer back to the producer
          bulk_wait_read_all();
          mbar_arrive(b_qempty + 8 * pend_qb);
          store_pending = false;
        }
        const float mrow = fmaxf(xm[r], xm[128 + r]);
        // Running max in log2 units of the exponent (with mods the scores are
        // already in them; without, the scale is applied to the max and inside
        // the exponential).  The reference max only moves when the tile max
        // exceeds it by more than kRescaleLog2 (a factor 256): exp values stay
        // <= 256, and O and l are rescaled (after PV(g-1) completes) only when
        // it moves.
        const float m_tile = MODS ? mrow : mrow * p.scale_log2;
        float alpha = 1.0f;
        if (j == 0) {
          m_run = m_tile;
        } else if (m_tile > m_run + kRescaleLog2) {
          alpha = ex2_approx(m_run - m_tile);
          m_run = m_tile;
        }
        const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
        uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;  // packed partial sums
        uint32_t pk[kCols / 2];
        const uint64_t negm = f2_pack(-m_use, -m_use);
        if (dead) {
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c) pk[c] = 0u;
        } else {
#pragma unroll
          for (int c = 0; c < kCols; c += 2) {
            uint64_t x = f2_pack(s[c], s[c + 1]);
            x = MODS ? f2_add(x, negm) : f2_fma(x, sc2, negm);
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
        }
        float a0, a1;
        f2_unpack(f2_add(f2_add(acc0, acc1), f2_add(acc2, acc3)), a0, a1);
        l_part = l_part * alpha + (a0 + a1);
        // P (bf16 pairs) of this quarter's keys into the score buffer's first 64 columns
        tmem_st32(lane_addr + 128u * sb + (kCols / 2) * wg, pk);
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
          // O holds PV(g-1): wait for it before rescaling
          mbar_wait(b_pvdone + 8 * ((gi - 1) % 3), ((gi - 1) / 3) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < OC / 16; ++c) {
            uint32_t v[16];
            const uint32_t oa = lane_addr + C::kColO + wg * OC + 16u * c;
            tmem_ld16(oa, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st16(oa, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(b_pfull + 8 * sb);
      };
      if constexpr (HALVES) {
        // Block masks: the sources of the next two steps are held in two
        // buffers used in turn, so that predicate words (read once, from
        // HBM) are requested two steps before they are needed.
        struct Src {
          int e, h, kt;
          uint2 pw;
        };
        StepIter it;
        step_begin(p, k, it, lane);
        auto fetch = [&](Src& q) {
          int ea = -1, eb = -1, ha = 0, hb = 0;
          if (!next_step(p, k, it, lane, ea, eb, ha, hb)) return false;
          if (ea == eb) {
            q.e = ea;
            q.h = wg;
          } else {
            q.e = wg ? eb : ea;
            q.h = (wg ? hb : ha) >> 1;
          }
          q.pw = make_uint2(~0u, ~0u);
          if (q.e >= 0 && q.e < k.np) {
            const long long e = bsm_idx(k.p0 + q.e, p.nP, &g_fwd_err) - k.p0;
            q.pw = __ldg(pay - wg + e * kTile * 2 + q.h);
          }
          q.kt = (MODS && q.e >= 0) ? tile_index(p, k, q.e) : 0;
          return true;
        };
        Src qa, qb;
        bool va = fetch(qa);  // a task with tiles has at least one step
        bool vb = fetch(qb);
        int j = 0;
        for (;;) {
          if (!va) break;
          {
            const int e = qa.e, hh = qa.h, kt = qa.kt;
            const bool partial = e >= 0 && e < k.np;
            const uint2 pw = partial ? qa.pw : make_uint2(~0u, ~0u);
            va = fetch(qa);  // step j + 2
            step(j++, e, hh, partial, pw, kt);
          }
          if (!vb) break;
          {
            const int e = qb.e, hh = qb.h, kt = qb.kt;
            const bool partial = e >= 0 && e < k.np;
            const uint2 pw = partial ? qb.pw : make_uint2(~0u, ~0u);
            vb = fetch(qb);  // step j + 2
            step(j++, e, hh, partial, pw, kt);
          }
        }
        g += j;
      } else {
        // interval masks: predicate words and K tile fetched one tile ahead
        uint2 pw_next = (k.np > 0) ? __ldg(pay + (bsm_idx(k.p0, p.nP, &g_fwd_err) - k.p0) * kTile * 2)
                                   : make_uint2(~0u, ~0u);
        int kt_next = MODS ? tile_index(p, k, 0) : 0;
        for (int j = 0; j < k.n; ++j) {
          const bool partial = j < k.np;
          const uint2 pw = partial ? pw_next : make_uint2(~0u, ~0u);
          const int kt = kt_next;
          if (j + 1 < k.np) pw_next = __ldg(pay + (bsm_idx(k.p0 + j + 1, p.nP, &g_fwd_err) - k.p0) * kTile * 2);
          if (MODS && j + 1 < k.n) kt_next = tile_index(p, k, j + 1);
          step(j, j, wg, partial, pw, kt);
        }
        g += k.n;
      }
      // ---------------------------------------------------------- epilogue
      mbar_wait(b_pvdone + 8 * ((g - 1) % 3), ((g - 1) / 3) & 1, abort_flag, &g_fwd_err, kWaitTimeoutNs);
      tc_fence_after();
      // sum exchange through the max-exchange buffer of the next tile's parity
      // (its last readers passed the previous tile's barrier); a second
      // barrier keeps the next task's max exchange from overwriting it early
      float* xs = xmax + (g & 1) * (kWG * 128);
      xs[wg * 128 + r] = l_part;
      group_sync();
      const float l = xs[r] + xs[128 + r];
      const bool have = l > 0.0f;
      const float inv_l = have ? 1.0f / l : 0.0f;
      // A full 128-row tile is staged in its task's Q buffer (no S MMA reads it
      // any more: the last PV has completed) and written by one TMA store; a
      // tail tile is stored row by row so that no other task's rows are touched.
      const bool tma_out = (k.qv == kTile);
      const uint32_t stage = sQ + qb * C::kTileBytes;
#pragma unroll
      for (int c = 0; c < OC / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(lane_addr + C::kColO + wg * OC + 16u * c, v);
        uint32_t pkd[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          pkd[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l);
        if (tma_out) {
          const int col = wg * OC + 16 * c;         // first output column of these 16
          const int chunk = col >> 6, unit = (col & 63) >> 3;
          const uint32_t rowa = stage + chunk * 16384 + r * 128;
          st_shared_v4(rowa + (((unit) ^ (r & 7)) << 4), pkd[0], pkd[1], pkd[2], pkd[3]);
          st_shared_v4(rowa + (((unit + 1) ^ (r & 7)) << 4), pkd[4], pkd[5], pkd[6], pkd[7]);
        } else if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 16);
          dst[0] = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
          dst[1] = make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
        }
      }
      if (tma_out) fence_proxy_async_smem();
      group_sync();  // staging complete; also keeps the sum exchange slots alive until read
      if (threadIdx.x == 0) {
        if (tma_out) {
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_store_2d(&tmO, stage + c * 16384, k.h * D + c * 64, k.q_off + k.m_block * kTile);
          bulk_commit_group();
          store_pending = true;
          pend_qb = qb;
        } else {
          mbar_arrive(b_qempty + 8 * qb);
        }
      }
      if (wg == 0 && row_ok && p.lse != nullptr) {
        float lse = -INFINITY;
        if (have) lse = (m_run + __log2f(l)) * kLn2;
        p.lse[static_cast<long long>(k.h) * p.total_q + grow] = lse;
      }
      ++tq;
      tc_fence_before();
    }
    if (threadIdx.x == 0 && store_pending) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
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

// 2-D view [rows, heads*D] of a bf16 tensor, box 64 columns x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t heads, int D, uint32_t box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * D * 2)};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool MODS, bool HALVES>
cudaError_t launch_impl(const FwdLaunch& a, cudaStream_t st, const char** why) {
  const fa_plan* pl = a.plan;
  const Geometry& g = pl->geom;
  const int64_t rows_q = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_q : g.total_q;
  const int64_t rows_k = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_k : g.total_k;
  CUtensorMap mq, mk, mv, mo, mkh, mvh;
  bool ok = make_map(&mq, a.q, rows_q, g.heads_q, D) && make_map(&mk, a.k, rows_k, g.heads_k, D) &&
            make_map(&mv, a.v, rows_k, g.heads_k, D) && make_map(&mo, a.o, rows_q, g.heads_q, D);
  // 64-row boxes of K and V for block-mask plans (two per ring slot)
  if (HALVES) {
    ok = ok && make_map(&mkh, a.k, rows_k, g.heads_k, D, 64) && make_map(&mvh, a.v, rows_k, g.heads_k, D, 64);
  } else {
    mkh = mk;
    mvh = mv;
  }
  if (!ok) {
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
  p.halves = pl->halves;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.Hq = g.heads_q;
  p.Hk = g.heads_k;
  p.Hmask = pl->Hmask;
  p.rows = static_cast<int>(pl->rows);
  p.total_q = static_cast<int>(rows_q);
  p.B = g.batch;
  p.nP = pl->P;
  p.nF = pl->F;
  p.flags = a.flags;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.y_scale = (a.softcap > 0.0f) ? a.scale / a.softcap : 0.0f;
  p.cap_log2 = a.softcap * kLog2e;
  {
    const double ys = (a.softcap > 0.0f) ? static_cast<double>(a.scale) / a.softcap : 0.0;
    const double cl = static_cast<double>(a.softcap) * 1.4426950408889634;
    p.c1 = static_cast<float>(cl * ys);
    p.c3 = static_cast<float>(-cl * ys * ys * ys / 3.0);
    p.c5 = static_cast<float>(2.0 * cl * ys * ys * ys * ys * ys / 15.0);
  }
  if (a.flags & FA_MOD_ALIBI)
    for (int h = 0; h < g.heads_q; ++h) p.slopes[h] = a.slopes[h];
  auto kern = k_fwd<D, MODS, HALVES>;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmem);
  if (e != cudaSuccess) {
    *why = "device attribute / cudaFuncSetAttribute failed";
    return e;
  }
  // one CTA per task; shared memory keeps one per SM and the running CTAs
  // take over the rest (cluster launch control).  Launched with programmatic
  // stream serialization, so that its set-up overlaps the end of the
  // previous kernel in the stream.
  (void)sms;
  const unsigned grid = static_cast<unsigned>(pl->tasks);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mo, mkh, mvh, p);
  if (e != cudaSuccess) *why = "forward kernel launch failed";
  return e;
}

// Nothing ever arrives on this barrier: every thread's bounded wait gives up
// after timeout_ns, the first one records DEVERR_TIMEOUT, and the kernel ends.
__global__ void k_wait_selftest(uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(smem_u32(&bar), 0, &abort_flag, &g_fwd_err, timeout_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t st) {
  k_wait_selftest<<<1, 64, 0, st>>>(timeout_ns);
  return cudaGetLastError();
}

// Interval masks without score mods run in attn_fwd_pair.cu (see use_pair
// below), so every plan that reaches this kernel either has score mods or is
// a block-mask plan.
template <int D>
cudaError_t launch_d(const FwdLaunch& a, cudaStream_t st, const char** why) {
  const bool mods = (a.flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI)) != 0;
  const bool halves = a.plan->mask_kind == MASK_BLOCKS;
  if (mods) return halves ? launch_impl<D, true, true>(a, st, why) : launch_impl<D, true, false>(a, st, why);
  return launch_impl<D, false, true>(a, st, why);
}

// Interval-mask plans without score mods run two Q tiles per task
// (attn_fwd_pair.cu): neighbouring Q tiles see mostly the same K tiles, and
// the shared K/V stream halves the bytes each SM loads per score.  With score
// mods the softmax (tanh series, ALiBi) is the bound, and the kernel here,
// with two warpgroups per tile, runs it faster; block-mask plans also stay
// here, with empty 64-key halves skipped.
static bool use_pair(const FwdLaunch& a) {
  return a.plan->mask_kind == MASK_INTERVALS && (a.flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI | FA_FWD_ONE_TILE)) == 0;
}
cudaError_t launch_fwd_d64(const FwdLaunch& a, cudaStream_t st, const char** why) {
  if (use_pair(a)) return launch_fwd_pair_d64(a, st, why);
  return launch_d<64>(a, st, why);
}
cudaError_t launch_fwd_d128(const FwdLaunch& a, cudaStream_t st, const char** why) {
  if (use_pair(a)) return launch_fwd_pair_d128(a, st, why);
  // block masks of 64-aligned blocks: one 64-row half of a Q tile against
  // pairs of its live 64x64 quadrants (attn_fwd_kt.cu)
  if (fwd_kt_applies(a)) return launch_fwd_kt(a, st, why);
  return launch_d<128>(a, st, why);
}

uint32_t* fwd_error_word() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_fwd_err) != cudaSuccess) return nullptr;
  return static_cast<uint32_t*>(ptr);
}

}  // namespace bsm
