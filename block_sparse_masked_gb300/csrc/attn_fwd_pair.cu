// attn_fwd_pair.cu -- masked attention forward on sm_103a, two Q tiles per
// task sharing one K/V stream.
//
// Same mathematics and consumption protocol as attn_fwd.cu ("Flex Attention
// Mask Plan Design" §6.1: partial K tiles with the packed predicate, full K
// tiles without it, empty tiles never visited; FlexAttention Eq. 1 with an
// online softmax).  A task here is a pair of vertically adjacent Q tiles
// (m, m+1) of one (sample, Q head) -- "A" and "B" -- taken from work_desc
// entries with an even m (the odd ones are skipped; they are the B tiles).
// The CTA walks the union of the two tiles' K-tile lists in ascending K-tile
// order and loads each K/V tile once: for masks whose neighbouring Q tiles
// see mostly the same keys (sliding windows, causal, prefix) this halves the
// K/V bytes each SM takes in per score, and K/V loading (TMA into shared
// memory, about 60 bytes per cycle per SM) is what bounds one Q tile per task.
// Used for interval-mask plans without score mods (with mods the softmax is
// the bound and attn_fwd.cu, two warpgroups per tile, runs it faster).
//
// Tasks come from cluster launch control as in attn_fwd.cu (one CTA per
// work_desc entry; a running CTA takes over entries of CTAs that have not
// started), in the plan's consumer order: longest task first, so that the
// last tasks to start are the shortest (with a few tasks per SM, the §4.8
// order -- sections, then cost -- starts heavy tasks of the last sections
// last and the launch ends on them).  352 threads, warp-specialised:
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: thread r owns
//               score row r (TMEM lane r) and all 128 key columns, so the row
//               max and sum stay in the thread.  Each group walks its own
//               tiles (a merge of its partial and full lists) in the same
//               ascending order.
//   warp 8      producer (lane 0): takes tasks, loads the two Q tiles, and
//               K(u), V(u-1) of every union tile u into one ring, tagging each
//               K slot with the tiles that use it.
//   warp 9      TMEM allocator and issuer of the Q K^T MMAs (lane 0).
//   warp 10     issuer of the P V MMAs (lane 0): a second issuing thread, so
//               that QK^T of one tile is never queued behind the issue of the
//               other tile's PV (tcgen05.mma issue blocks while the tensor
//               pipe's queue is full).
// TMEM (D=128): O_A [0,128), O_B [128,256), one score buffer S [256,384)
// shared by both tiles, P_A [384,448), P_B [448,512) (P in bf16 pairs).  The
// score buffer passes between the tiles: a softmax group releases it as soon
// as it has read its scores into registers, so QK^T of the other tile runs
// while the first group computes.  Per union tile the MMA issuer orders
// S_A(u), PV_A(u-1), S_B(u), PV_B(u-1): each PV fills the gap while the
// score buffer makes its round trip.  K(u) and V(u) follow each other in one
// ring; both slots carry the use tag.
// Every wait is a bounded mbarrier wait; after a timeout the CTA records an
// error bit, stops waiting, drains copies and MMAs in flight, frees TMEM and
// exits.  The softmax warps never meet at a named barrier.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace bsm {
namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold, log2 units

constexpr int kThreads = 352;
constexpr int kWarpProducer = 8, kWarpMma = 9, kWarpPv = 10;
constexpr int kTaskRing = 2;
constexpr uint32_t kTaskConsumers = 2 + 8;  // the two MMA issuers and lane 0 of every softmax warp

template <int D>
struct PCfg {
  static constexpr int kChunks = D / 64;          // 64-column (128-byte) swizzle chunks
  static constexpr int kTileBytes = 128 * D * 2;  // Q, K or V tile, bf16
  static constexpr int kSlots = (D == 128) ? 5 : 12;  // one ring of K and V tiles
  static constexpr int kOffQ = 0;                 // Q_A, Q_B
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOffSmall = kOffKV + kSlots * kTileBytes;
  static constexpr int kSmallBytes = 1024;
  static constexpr int kNeed = kOffSmall + kSmallBytes;
  static constexpr int kSmem = (kNeed + 1024 <= 232448) ? kNeed + 1024 : 232448;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 0;            // O_A at 0, O_B at D
  static constexpr uint32_t kColS = 2 * D;        // the shared score buffer (128 columns)
  static constexpr uint32_t kColP = 2 * D + 128;  // P_A, then P_B 64 columns later
  static_assert(kColP + 128 <= kTmemCols, "TMEM budget");
  static_assert(kNeed <= 232448, "shared memory budget");
};

struct PairParams {
  const int32_t* work;
  const int32_t* lpt;  // the order in which tasks are taken: work_desc positions, longest first
  const int32_t* seq;
  const int32_t* p_off;
  const int32_t* f_off;
  const int32_t* p_idx;
  const int32_t* f_idx;
  const uint32_t* payload;
  __nv_bfloat16* o;
  float* lse;
  uint32_t* err;     // the forward kernels' error word
  int Hq, Hk, Hmask, rows, total_q, ntasks;
  int B;             // samples
  long long nP, nF;  // partial and full entries of the plan (bounds of the checked build)
  float scale_log2;  // scale * log2(e)
};

// One Q tile of a pair: its rows and its partial/full lists.
struct Half {
  int qv;       // valid rows (0: the tile does not exist)
  int m;        // m_block
  int p0, np;   // partial entries [p0, p0+np)
  int f0, nf;   // full entries [f0, f0+nf)
};
struct PairTask {
  int skip;     // 1: not a pair (odd m_block, claimed and dropped), -1: end marker
  int h, b, hk, q_off, k_off;
  Half t[2];
};

__device__ __forceinline__ PairTask load_pair(const PairParams& p, int t) {
  PairTask k{};
  const int* wd = p.work + 4LL * t;
  const int m = wd[0];
  if (m & 1) {
    k.skip = 1;
    return k;
  }
  k.h = static_cast<int>(bsm_idx(wd[1], p.Hq, p.err));
  k.b = static_cast<int>(bsm_idx(wd[2], p.B, p.err));
  const int* sq = p.seq + 8 * k.b;
  k.q_off = sq[0];
  k.k_off = sq[1];
  const int q_len = sq[2], row_begin = sq[4], nrows = sq[5];
  k.hk = k.h / (p.Hq / p.Hk);
  const int hm = (p.Hmask == 1) ? 0 : k.h;
  for (int x = 0; x < 2; ++x) {
    Half& s = k.t[x];
    s.m = m + x;
    if (s.m >= nrows) continue;  // no B tile (qv stays 0, lists empty)
    s.qv = min(128, q_len - s.m * 128);
    const long long flat = bsm_idx(static_cast<long long>(hm) * p.rows + row_begin + s.m,
                                   static_cast<long long>(p.Hmask) * p.rows, p.err);
    s.p0 = p.p_off[flat];
    s.np = p.p_off[flat + 1] - s.p0;
    s.f0 = p.f_off[flat];
    s.nf = p.f_off[flat + 1] - s.f0;
  }
  return k;
}

__device__ __forceinline__ int p_entry(const PairParams& p, long long i) {
  return __ldg(p.p_idx + bsm_idx(i, p.nP, p.err));
}
__device__ __forceinline__ int f_entry(const PairParams& p, long long i) {
  return __ldg(p.f_idx + bsm_idx(i, p.nF, p.err));
}

// Ascending walk over one tile's K tiles: a merge of its partial list and
// its full list (each ascending).  The next entry of each list is fetched
// one step ahead.
struct OwnWalk {
  int ip, jf;        // positions in the partial and full lists
  int kp, kf;        // current heads (INT_MAX once exhausted)
  int kp_nx, kf_nx;  // the entries after them
  __device__ __forceinline__ void init(const PairParams& p, const Half& s) {
    ip = 0;
    jf = 0;
    kp = (s.np > 0) ? p_entry(p, s.p0) : INT_MAX;
    kf = (s.nf > 0) ? f_entry(p, s.f0) : INT_MAX;
    kp_nx = (s.np > 1) ? p_entry(p, s.p0 + 1) : INT_MAX;
    kf_nx = (s.nf > 1) ? f_entry(p, s.f0 + 1) : INT_MAX;
  }
  __device__ __forceinline__ int head() const { return min(kp, kf); }
  // Takes the head: returns its K tile; *partial_entry = its payload entry or -1
  __device__ __forceinline__ int take(const PairParams& p, const Half& s, int* partial_entry) {
    if (kp < kf) {
      const int kt = kp;
      *partial_entry = s.p0 + ip;
      ++ip;
      kp = kp_nx;
      kp_nx = (ip + 1 < s.np) ? p_entry(p, s.p0 + ip + 1) : INT_MAX;
      return kt;
    }
    const int kt = kf;
    *partial_entry = -1;
    ++jf;
    kf = kf_nx;
    kf_nx = (jf + 1 < s.nf) ? f_entry(p, s.f0 + jf + 1) : INT_MAX;
    return kt;
  }
};

// Slot tag written by the producer before the K copy's arrive: bits 0-1 how
// tile A uses the union tile (0 not, 1 partial, 2 full), bits 2-3 tile B,
// bit 4 last union tile of the task.
constexpr int kTagLast = 16;

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    k_fwd_pair(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ PairParams p) {
  using C = PCfg<D>;
  constexpr int NS = C::kSlots;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  if ((base - raw) + C::kNeed > static_cast<uint32_t>(C::kSmem)) {
    if (threadIdx.x == 0) atomicOr(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  const uint32_t sQ = base + C::kOffQ;
  const uint32_t sKV = base + C::kOffKV;
  const uint32_t bar0 = base + C::kOffSmall;
  const uint32_t b_qfull = bar0;                // Q_A and Q_B of the current task
  const uint32_t b_qempty = b_qfull + 8;        // released with the task's last S
  const uint32_t b_full = b_qempty + 8;         // [NS] K/V ring
  const uint32_t b_empty = b_full + 8 * NS;     // [NS]
  const uint32_t b_sfull = b_empty + 8 * NS;    // [2] S of tile A / B in the score buffer
  const uint32_t b_sfree = b_sfull + 16;        // the score buffer has been read (4 arrives)
  const uint32_t b_pfull = b_sfree + 8;         // [2] P of tile A / B written (4 arrives)
  const uint32_t b_pvdone = b_pfull + 16;       // [2] PV of tile A / B complete
  const uint32_t b_drain = b_pvdone + 16;       // [2] S issuer, PV issuer
  const uint32_t b_tfull = b_drain + 16;        // [kTaskRing]
  const uint32_t b_tempty = b_tfull + 8 * kTaskRing;
  const uint32_t b_clc = b_tempty + 8 * kTaskRing;  // cluster launch control response
  uint8_t* small = gbase + C::kOffSmall;
  int* slot_tag = reinterpret_cast<int*>(small + 400);            // [NS]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(small + 464);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(small + 468);
  PairTask* tring = reinterpret_cast<PairTask*>(small + 512);     // [kTaskRing]
  const uint32_t clc_resp = smem_u32(small + 672);                 // [2] 16-byte cluster launch control responses
  static_assert(8 + 8 + 16 * NS + 16 + 8 + 16 + 16 + 16 + 16 * kTaskRing + 8 <= 400, "barrier slots");
  static_assert(512 + sizeof(PairTask) * kTaskRing <= 672 && 672 + 32 <= C::kSmallBytes, "task ring, responses");
  static_assert(NS * 4 <= 64, "slot tags");
  static_assert(sizeof(PairTask) * kTaskRing <= 512, "task ring");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_full + 8 * s, 1);
      mbar_init(b_empty + 8 * s, 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(b_sfull + 8 * x, 1);
      mbar_init(b_pfull + 8 * x, 4);
      mbar_init(b_pvdone + 8 * x, 1);
    }
    mbar_init(b_sfree, 4);
    mbar_init(b_drain, 1);
    mbar_init(b_drain + 8, 1);
    mbar_init(b_clc, 1);
    for (int i = 0; i < kTaskRing; ++i) {
      mbar_init(b_tfull + 8 * i, 1);
      mbar_init(b_tempty + 8 * i, kTaskConsumers);
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
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int c = 0, c_issued = 0;     // ring loads
      int tq = 0, q_issued = 0;    // tasks with tiles, Q loads
      auto load = [&](const CUtensorMap* map, int row, int hk, int tag) {
        const int slot = c % NS;
        if (c >= NS) mbar_wait(b_empty + 8 * slot, ((c / NS) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (!*abort_flag) {
          c_issued = c + 1;
          slot_tag[slot] = tag;  // published to the MMA issuers by the arrive below
          mbar_arrive_expect_tx(b_full + 8 * slot, C::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < C::kChunks; ++ch)
            tma_load_2d(sKV + slot * C::kTileBytes + ch * 16384, map, b_full + 8 * slot, hk * D + ch * 64, row);
        }
        ++c;
      };
      int ti = 0;
      auto publish = [&](const PairTask& k) {
        const int slot = ti % kTaskRing;
        if (ti >= kTaskRing)
          mbar_wait(b_tempty + 8 * slot, ((ti / kTaskRing) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        tring[slot] = k;
        mbar_arrive(b_tfull + 8 * slot);
        ++ti;
      };
      ClcTasks tasks{clc_resp, b_clc};
      for (;;) {
        const int t = tasks.next(abort_flag, p.err, kWaitTimeoutNs);
        if (t < 0 || t >= p.ntasks) break;
        const PairTask k = load_pair(p, __ldg(p.lpt + bsm_idx(t, p.ntasks, p.err)));
        if (k.skip) continue;
        publish(k);
        const int nA = k.t[0].np + k.t[0].nf, nB = k.t[1].np + k.t[1].nf;
        if (nA + nB == 0) continue;
        if (tq >= 1) mbar_wait(b_qempty, (tq - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (!*abort_flag) {
          q_issued = tq + 1;
          const int nq = (k.t[1].qv > 0) ? 2 : 1;
          mbar_arrive_expect_tx(b_qfull, nq * C::kTileBytes);
          for (int x = 0; x < nq; ++x)
#pragma unroll
            for (int ch = 0; ch < C::kChunks; ++ch)
              tma_load_2d(sQ + x * C::kTileBytes + ch * 16384, &tmQ, b_qfull, k.h * D + ch * 64,
                          k.q_off + k.t[x].m * 128);
        }
        OwnWalk wa, wb;
        wa.init(p, k.t[0]);
        wb.init(p, k.t[1]);
        for (;;) {
          const int ha = wa.head(), hb = wb.head();
          const int kt = min(ha, hb);
          if (kt == INT_MAX) break;
          int tag = 0, e;
          if (ha == kt) tag |= (wa.take(p, k.t[0], &e), e >= 0 ? 1 : 2);
          if (hb == kt) tag |= (wb.take(p, k.t[1], &e), e >= 0 ? 1 : 2) << 2;
          if (min(wa.head(), wb.head()) == INT_MAX) tag |= kTagLast;
          const int row = k.k_off + kt * 128;
          load(&tmK, row, k.hk, tag);
          load(&tmV, row, k.hk, tag);
        }
        ++tq;
      }
      PairTask end{};
      end.skip = -1;
      publish(end);
      if (*abort_flag) {
        // let the copies already started land before the CTA exits
        if (q_issued > 0) mbar_wait_drain(b_qfull, (q_issued - 1) & 1, kWaitTimeoutNs);
        for (int u = (c_issued > NS ? c_issued - NS : 0); u < c_issued; ++u)
          mbar_wait_drain(b_full + 8 * (u % NS), (u / NS) & 1, kWaitTimeoutNs);
        tasks.drain(kWaitTimeoutNs);
      }
    }
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ------------------------------------------------------------ MMA issuers
    // Ring position 2u holds K(u) of the CTA's u-th union tile, 2u+1 holds
    // V(u).  The S issuer takes the K slots: per union tile S_A(u), S_B(u) for
    // the tiles that use it, each once the previous S has been read out of
    // the shared score buffer.  The PV issuer takes the V slots: PV_A(u),
    // PV_B(u) once the tile's P is written.
    const bool is_s = warp == kWarpMma;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, 1);
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = sdesc_sw128(sKV, 16, 1024);
      const uint64_t dV0 = sdesc_sw128(sKV, 16384, 1024);
      int u = 0;         // union tiles taken
      int tq = 0;        // tasks with tiles
      int s_uses = 0;    // S issued into the score buffer
      int g_pv[2] = {0, 0};  // PVs issued per tile (A, B), over all tasks
      for (int ti = 0;; ++ti) {
        const int tslot = ti % kTaskRing;
        mbar_wait(b_tfull + 8 * tslot, (ti / kTaskRing) & 1, abort_flag, p.err, kWaitTimeoutNs);
        const PairTask k = tring[tslot];
        mbar_arrive(b_tempty + 8 * tslot);
        if (k.skip < 0 || *abort_flag) break;
        if (k.t[0].np + k.t[0].nf + k.t[1].np + k.t[1].nf == 0) continue;
        if (is_s) mbar_wait(b_qfull, tq & 1, abort_flag, p.err, kWaitTimeoutNs);
        bool acc[2] = {false, false};  // the tile's O already holds a PV of this task
        for (;;) {
          const int pos = 2 * u + (is_s ? 0 : 1);
          const int slot = pos % NS;
          mbar_wait(b_full + 8 * slot, (pos / NS) & 1, abort_flag, p.err, kWaitTimeoutNs);
          const int tag = slot_tag[slot];  // written by the producer before its arrive
          const bool last = (tag & kTagLast) != 0;
          ++u;
          for (int x = 0; x < 2; ++x) {
            if (!((tag >> (2 * x)) & 3)) continue;
            if (is_s) {
              if (s_uses > 0) mbar_wait(b_sfree, (s_uses - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
              ++s_uses;
              if (*abort_flag) continue;
              tc_fence_after();
              const uint64_t dQ = dQ0 + static_cast<uint64_t>((x * C::kTileBytes) >> 4);
              const uint64_t dK = dK0 + static_cast<uint64_t>((slot * C::kTileBytes) >> 4);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off16 = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                umma_bf16_ss(tmem + C::kColS, dQ + off16, dK + off16, idS, kk > 0);
              }
              umma_commit(b_sfull + 8 * x);
            } else {
              mbar_wait(b_pfull + 8 * x, g_pv[x] & 1, abort_flag, p.err, kWaitTimeoutNs);
              ++g_pv[x];
              if (*abort_flag) continue;
              tc_fence_after();
              const uint64_t dV = dV0 + static_cast<uint64_t>((slot * C::kTileBytes) >> 4);
              const uint32_t pcol = tmem + C::kColP + 64u * x;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_bf16_ts(tmem + C::kColO + D * x, pcol + 8u * kk, dV + static_cast<uint64_t>((kk * 2048) >> 4),
                             idO, (acc[x] || kk > 0) ? 1u : 0u);
              umma_commit(b_pvdone + 8 * x);
              acc[x] = true;
            }
          }
          // every MMA reading this slot is issued: refill it once they complete;
          // the task's last S also frees the Q tiles
          if (!*abort_flag) {
            umma_commit(b_empty + 8 * slot);
            if (is_s && last) umma_commit(b_qempty);
          }
          if (last || *abort_flag) break;
        }
        ++tq;
      }
      umma_commit(b_drain + (is_s ? 0 : 8));
      mbar_wait_drain(b_drain + (is_s ? 0 : 8), 0, kWaitTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;             // 0: tile A, 1: tile B
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;        // score row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::kColS;
    const uint32_t tP = tmem + lane_off + C::kColP + 64u * x;
    const uint32_t tO = tmem + lane_off + C::kColO + D * x;
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    int g = 0;  // this tile's own K tiles processed, over all tasks
    for (int ti = 0;; ++ti) {
      const int tslot = ti % kTaskRing;
      if (lane == 0) mbar_wait(b_tfull + 8 * tslot, (ti / kTaskRing) & 1, abort_flag, p.err, kWaitTimeoutNs);
      __syncwarp();
      const PairTask k = tring[tslot];
      int stop = k.skip < 0;
      if (lane == 0 && *abort_flag) stop = 1;
      stop = __shfl_sync(0xffffffffu, stop, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(b_tempty + 8 * tslot);
      if (stop) break;
      const Half& hx = k.t[x];
      if (hx.qv <= 0) continue;  // no B tile in this pair
      const int n = hx.np + hx.nf;
      const long long grow = static_cast<long long>(k.q_off) + hx.m * 128 + r;
      const bool row_ok = r < hx.qv && bsm_ok(grow, p.total_q, p.err);
      __nv_bfloat16* orow = p.o + (grow * p.Hq + k.h) * D;
      if (n == 0) {
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          if (p.lse != nullptr) p.lse[static_cast<long long>(k.h) * p.total_q + grow] = -INFINITY;
        }
        continue;
      }
      float m_run = -INFINITY, l_run = 0.0f;
      OwnWalk walk;
      walk.init(p, hx);
      const uint4* pay = reinterpret_cast<const uint4*>(p.payload) + r;  // + entry * 128
      int e_next;
      walk.take(p, hx, &e_next);
      uint4 pw_next = (e_next >= 0) ? __ldg(pay + bsm_idx(e_next, p.nP, p.err) * 128)
                                    : make_uint4(~0u, ~0u, ~0u, ~0u);
      for (int j = 0; j < n; ++j) {
        const bool partial = e_next >= 0;
        const uint4 pw = pw_next;
        if (j + 1 < n) {  // next own tile, fetched one step ahead
          walk.take(p, hx, &e_next);
          pw_next = (e_next >= 0) ? __ldg(pay + bsm_idx(e_next, p.nP, p.err) * 128)
                                  : make_uint4(~0u, ~0u, ~0u, ~0u);
        }
        mbar_wait(b_sfull + 8 * x, g & 1, abort_flag, p.err, kWaitTimeoutNs);
        tc_fence_after();
        float sv[128];
        tmem_ld128(tS, sv);
        // scores are in registers: hand the buffer to the other tile's QK^T
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sfree);
        if (partial) {
          const uint32_t words[4] = {pw.x, pw.y, pw.z, pw.w};
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (!((words[c >> 5] >> (c & 31)) & 1u)) sv[c] = -INFINITY;
        }
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          m0 = max3f(m0, sv[c], sv[c + 1]);
          m1 = max3f(m1, sv[c + 2], sv[c + 3]);
          m2 = max3f(m2, sv[c + 4], sv[c + 5]);
          m3 = max3f(m3, sv[c + 6], sv[c + 7]);
        }
        const float mrow = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        // Running max in log2 units; it only moves when the tile max exceeds
        // it by more than kRescaleLog2 (exp values stay <= 256), and O and l
        // are rescaled only then.
        const float m_tile = mrow * p.scale_log2;
        float alpha = 1.0f;
        if (j == 0) {
          m_run = m_tile;
        } else if (m_tile > m_run + kRescaleLog2) {
          alpha = ex2_approx(m_run - m_tile);
          m_run = m_tile;
        }
        const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
        const uint64_t negm = f2_pack(-m_use, -m_use);
        uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
        // the P buffer (and O) were last used by this tile's previous PV
        if (g > 0) mbar_wait(b_pvdone + 8 * x, (g - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            uint64_t v = f2_pack(sv[32 * ch + c], sv[32 * ch + c + 1]);
            v = f2_fma(v, sc2, negm);
            float x0, x1;
            f2_unpack(v, x0, x1);
            const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
            const uint64_t ev = f2_pack(e0, e1);
            switch ((c >> 1) & 3) {
              case 0: acc0 = f2_add(acc0, ev); break;
              case 1: acc1 = f2_add(acc1, ev); break;
              case 2: acc2 = f2_add(acc2, ev); break;
              default: acc3 = f2_add(acc3, ev); break;
            }
            pk[c >> 1] = pack_bf16x2(e0, e1);
          }
          tmem_st16(tP + 16u * ch, pk);
        }
        float a0, a1;
        f2_unpack(f2_add(f2_add(acc0, acc1), f2_add(acc2, acc3)), a0, a1);
        l_run = l_run * alpha + (a0 + a1);
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tO + 32u * c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(tO + 32u * c, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull + 8 * x);
        ++g;
      }
      // ---------------------------------------------------------- epilogue
      mbar_wait(b_pvdone + 8 * x, (g - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
      tc_fence_after();
      const bool have = l_run > 0.0f;
      const float inv_l = have ? 1.0f / l_run : 0.0f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + 32u * c, v);
        uint32_t pkd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pkd[i] = pack_bf16x2(__uint_as_float(v[2 * i]) * inv_l, __uint_as_float(v[2 * i + 1]) * inv_l);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pkd[4 * i], pkd[4 * i + 1], pkd[4 * i + 2], pkd[4 * i + 3]);
        }
      }
      if (row_ok && p.lse != nullptr) {
        float lse = -INFINITY;
        if (have) lse = (m_run + __log2f(l_run)) * kLn2;
        p.lse[static_cast<long long>(k.h) * p.total_q + grow] = lse;
      }
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_pair() {
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
bool make_map_pair(CUtensorMap* m, const void* ptr, int64_t rows, int64_t heads, int D) {
  auto fn = encode_fn_pair();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * D * 2)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_pair_impl(const FwdLaunch& a, cudaStream_t st, const char** why) {
  const fa_plan* pl = a.plan;
  const Geometry& g = pl->geom;
  const int64_t rows_q = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_q : g.total_q;
  const int64_t rows_k = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_k : g.total_k;
  CUtensorMap mq, mk, mv;
  if (!make_map_pair(&mq, a.q, rows_q, g.heads_q, D) || !make_map_pair(&mk, a.k, rows_k, g.heads_k, D) ||
      !make_map_pair(&mv, a.v, rows_k, g.heads_k, D)) {
    *why = "cuTensorMapEncodeTiled failed (pointer alignment or driver entry point)";
    return cudaErrorInvalidValue;
  }
  if (pl->lpt == nullptr) {  // built for every interval plan, the only plans routed here
    *why = "the plan carries no longest-first task order";
    return cudaErrorInvalidValue;
  }
  PairParams p{};
  p.work = pl->work_desc;
  p.lpt = pl->lpt;
  p.seq = pl->seq_desc;
  p.p_off = pl->p_off;
  p.f_off = pl->f_off;
  p.p_idx = pl->p_idx;
  p.f_idx = pl->f_idx;
  p.payload = pl->payload;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.err = fwd_error_word();
  p.Hq = g.heads_q;
  p.Hk = g.heads_k;
  p.Hmask = pl->Hmask;
  p.rows = static_cast<int>(pl->rows);
  p.total_q = static_cast<int>(rows_q);
  p.ntasks = static_cast<int>(pl->tasks);
  p.B = g.batch;
  p.nP = pl->P;
  p.nF = pl->F;
  p.scale_log2 = a.scale * kLog2e;
  if (a.flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI)) {
    *why = "score mods are not supported by the two-tile forward";
    return cudaErrorInvalidValue;
  }
  if (p.err == nullptr) {
    *why = "forward error word not found";
    return cudaErrorInvalidValue;
  }
  auto kern = k_fwd_pair<D>;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PCfg<D>::kSmem);
  if (e != cudaSuccess) {
    *why = "device attribute / cudaFuncSetAttribute failed";
    return e;
  }
  // one CTA per work_desc entry (the odd ones find nothing to do and take
  // over others at once); shared memory keeps one per SM and the running
  // CTAs take over the rest (cluster launch control).  Launched with
  // programmatic stream serialization, so that its set-up overlaps the end
  // of the previous kernel in the stream.
  (void)sms;
  const unsigned grid = static_cast<unsigned>(pl->tasks);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = PCfg<D>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, p);
  if (e != cudaSuccess) *why = "forward kernel launch failed";
  return e;
}


}  // namespace

cudaError_t launch_fwd_pair_d64(const FwdLaunch& a, cudaStream_t st, const char** why) {
  return launch_pair_impl<64>(a, st, why);
}
cudaError_t launch_fwd_pair_d128(const FwdLaunch& a, cudaStream_t st, const char** why) {
  return launch_pair_impl<128>(a, st, why);
}

}  // namespace bsm
