// attn_fwd_kt.cu -- keys-major masked attention forward for block-mask plans
// whose logical blocks are multiples of 64 in both directions (sm_103a, d=128).
//
// Consumption protocol of "Flex Attention Mask Plan Design" §6.1 (partial
// tiles with the packed predicate of §5, full tiles without it, empty tiles
// never visited; a row without a visible key gets O = 0 and LSE = -inf),
// with the math of FlexAttention Eq. 1 and an online softmax.
//
// Why keys-major.  With 64x64 logical blocks ("Decoupling Logical Masks from
// GPU Execution for Dynamic Block-Sparse Attention" §2: the effective set
// E(M) of a block mask) a 128x128 physical tile holds four 64x64 quadrants,
// and at low density a live quadrant almost never has a live neighbour in
// the same 64 keys.  A 128-row Q tile times a 64-key half therefore computes
// about twice the visible scores.  This kernel instead works on one 64-row
// half of the Q tile at a time (a "sub-task") and on pairs of its live 64-key
// quadrants (a "step"):
//   S^T = K Q^T     tcgen05 M=128 (the two quadrants' keys) x N=64 (queries),
//                   into TMEM, one key per lane: every score is visible
//                   (except at sequence tails, where the plan's predicate
//                   words mask the rest);
//   P^T             exponentials written by the thread of each key to shared
//                   memory, one 128-byte row per key;
//   O^T += V^T P^T  tcgen05 M=128 (head dimension) x N=64 (queries), V read
//                   MN-major from the ring slot that holds it, into TMEM.
// The plan is the ordinary one (physical tiles 128x128); its per-entry
// quadrant bits say which quadrants are live and which need no predicate.
//
// Online softmax per query column.  Columns never mix, so two softmax
// warpgroups own 32 query columns each and run independently.  The
// reference max of a column only moves when a score exceeds it by more than
// 2^8 (one barrier reduction per warpgroup and step decides); the first step
// of each sub-task and every such rare step take the exact column max across
// the 128 keys (warp reduce-scatter by shuffles, then shared memory), rescale
// the running sums and O^T, and continue.  The column sums are reduced the
// same way once per sub-task.
//
// Tasks are work_desc entries taken through cluster launch control (the
// SM100/SM103 hardware queue of §4.8), each split into its two 64-row
// halves.  352 threads; every hand-off is an mbarrier:
//   warps 0-7  softmax: warpgroup w owns query columns 32w..32w+31; thread
//              t of a warpgroup = TMEM lane t = key t of a step, and in the
//              epilogue head-dimension column t of O.
//   warp 8     walks the plan: sub-task records, step descriptors, Q halves
//              (2-deep ring) and each step's K rows (K ring); an empty second
//              position is loaded from rows past the tensor (zero fill, no
//              memory traffic).
//   warp 9     TMEM allocation and the S^T issuer.
//   warp 10    the V loads (V ring, up to its depth ahead) and the P V issuer.
// K and V have rings of their own so that a V load waiting for its slot (which
// frees only after the softmax) never holds back a K load.  Every wait is an
// mbarrier wait with a global-timer limit; after a timeout the CTA records an
// error bit, stops waiting, drains what is in flight, frees TMEM and exits.
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
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold, log2 units
constexpr float kNoMax = -1.0e30f;    // reference max of a column before its first visible score

constexpr int D = 128;
constexpr int kHalf = 64;                       // Q rows per sub-task, keys per position
constexpr int kGroups = 2;                      // softmax warpgroups (each 128 threads, one key per thread)
constexpr int kCols = kHalf / kGroups;          // query columns per softmax warpgroup
constexpr int kHalfBytes = kHalf * D * 2;       // 16 KB
constexpr int kSlotBytes = 2 * kHalfBytes;      // ring slot: two positions
constexpr int kKSlots = 3, kVSlots = 2;
constexpr int kSBuf = 2;                        // TMEM S^T buffers, 64 columns each
constexpr int kPBuf = 2;                        // shared-memory P^T buffers
constexpr int kDescRing = 8;                    // step descriptors ahead of the consumers
constexpr int kSubRing = 2;                     // sub-task records
constexpr uint32_t kColO = kSBuf * kHalf;       // O^T buffers (two, 64 columns each) after S^T
constexpr uint32_t kTmemCols = 512;
static_assert(kColO + 2 * kHalf <= kTmemCols, "TMEM budget");

constexpr int kOffQ = 0;                                   // 2 Q halves: [chunk][64 rows][128 B]
constexpr int kOffK = kOffQ + 2 * kHalfBytes;              // K ring: [chunk][128 rows][128 B]
constexpr int kOffV = kOffK + kKSlots * kSlotBytes;        // V ring, same layout
constexpr int kOffP = kOffV + kVSlots * kSlotBytes;        // P^T: [128 keys][64 queries] bf16
constexpr int kOffSmall = kOffP + kPBuf * kHalfBytes;
// small area: barriers, records, exchange
constexpr int kNumBars = 2 + 2 + 2 * kKSlots + 2 * kVSlots + 2 * kSBuf + 2 * kPBuf + 2 + 2 * kDescRing +
                         2 * kSubRing + 3;
constexpr int kSmTmem = 8 * kNumBars;
constexpr int kSmAbort = kSmTmem + 4;
constexpr int kSmClc = (kSmAbort + 4 + 15) & ~15;        // 2 x 16-byte responses
constexpr int kSmSub = kSmClc + 32;                      // kSubRing records
constexpr int kSmBcast = kSmSub + kSubRing * 32;         // one record copy per softmax warpgroup
constexpr int kSmDesc = kSmBcast + kGroups * 32;         // kDescRing step descriptors
constexpr int kSmM = kSmDesc + kDescRing * 32;           // [64] floats: reference max of each query column
constexpr int kSmM2 = kSmM + 64 * 4;                     // [64] floats: new reference max, then 1/l
constexpr int kSmXch = kSmM2 + 64 * 4;                   // [warpgroups][4 warps][kCols] floats
constexpr int kSmallBytes = kSmXch + kGroups * 4 * kCols * 4;
constexpr int kNeed = kOffSmall + kSmallBytes;
// dynamic shared memory starts 1 KB-aligned in practice; what is left up to
// the per-block limit is slack for a misaligned start (checked at run time)
constexpr int kSmem = (kNeed + 1024 <= 232448) ? kNeed + 1024 : 232448;
static_assert(kNeed <= 232448, "shared memory budget");

constexpr int kWarpProducer = 4 * kGroups, kWarpS = kWarpProducer + 1, kWarpPV = kWarpProducer + 2;
constexpr int kThreads = 32 * (kWarpPV + 1);
constexpr int kSoftmaxThreads = 128 * kGroups;

struct KtParams {
  const int32_t* work;
  const int32_t* seq;
  const int32_t* p_off;
  const int32_t* f_off;
  const int32_t* p_idx;
  const int32_t* f_idx;
  const uint32_t* payload;
  const uint8_t* quads;  // [P] bit 2a+s: quadrant (row half a, key half s) live; bit 4+2a+s: all visible
  __nv_bfloat16* o;
  float* lse;
  uint32_t* err;
  int Hq, Hk, Hmask, rows, total_q, rows_k, ntasks;
  int B;             // samples
  long long nP, nF;  // partial and full entries of the plan (bounds of the checked build)
  float scale_log2;
};

// One 64-row half of a work_desc entry, as the producer publishes it.
struct Sub {
  int h, q0, qv, nsteps, qh, pad[3];  // nsteps < 0: end of the CTA's work
};
static_assert(sizeof(Sub) == 32, "record size");
// One step: the K/V rows of its two positions (the second may lie past the
// tensor: an empty position, zero-filled), the K/V head, and per position
// the predicate source: kFullPos (no predicate), kEmptyPos, or
// (partial entry << 1 | key half of the tile).
struct StepDesc {
  int r0, r1, hk, e0, e1, pad[3];
};
static_assert(sizeof(StepDesc) == 32, "descriptor size");
constexpr int kFullPos = -1, kEmptyPos = -2;

__device__ __forceinline__ int tile_of(const KtParams& p, int p0, int np, int f0, int j) {
  return (j < np) ? __ldg(p.p_idx + bsm_idx(p0 + j, p.nP, p.err))
                  : __ldg(p.f_idx + bsm_idx(f0 + (j - np), p.nF, p.err));
}
__device__ __forceinline__ int quads_of(const KtParams& p, int p0, int np, int j) {
  return (j < np) ? static_cast<int>(__ldg(p.quads + bsm_idx(p0 + j, p.nP, p.err))) : 0xFF;  // full tiles: every quadrant full
}

// Instruction descriptor, kind::f16 with A and B both MN-major (the P V step:
// A = V^T from the ring slot, B = P^T from shared memory).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_mn(int M, int N) {
  return idesc_bf16_f32(M, N, 1) | (1u << 15);
}

// Barrier reduction over one softmax warpgroup (named barrier `id`, 128
// threads): every thread passes v, all get the OR.
__device__ __forceinline__ bool group_any(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, 128, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}

// Warp reduce-scatter of kCols per-lane values: afterwards lane l holds, in
// v[0], the reduction over the warp of column l % kCols.
template <bool MAX>
__device__ __forceinline__ void warp_reduce_scatter32(float (&v)[kCols], int lane) {
#pragma unroll
  for (int half = kCols / 2; half >= 1; half >>= 1) {
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float a = v[i], b = v[i + half];
      const float send = upper ? a : b, keep = upper ? b : a;
      const float got = __shfl_xor_sync(0xffffffffu, send, half);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int o = kCols; o < 32; o <<= 1) {  // fewer columns than lanes: fold the lane groups
    const float got = __shfl_xor_sync(0xffffffffu, v[0], o);
    v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
  }
}

// kCols fp32 columns of this thread's TMEM lane, and their store.
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&x)[kCols]) {
  if constexpr (kCols == 32) {
    tmem_ld32f(taddr, *reinterpret_cast<float(*)[32]>(&x[0]));
  } else {
    tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(&x[0]));
  }
}
__device__ __forceinline__ void st_cols(uint32_t taddr, const float (&x)[kCols]) {
#pragma unroll
  for (int c = 0; c < kCols; c += 16) tmem_st16(taddr + c, *reinterpret_cast<const uint32_t(*)[16]>(&x[c]));
}

// 32 scores of this thread's TMEM lane in log2 units, -inf where the
// predicate bits pm are 0 (bit c: column c).
__device__ __forceinline__ void load_scores(uint32_t taddr, float (&x)[kCols], uint32_t pm, uint64_t sc2,
                                            float scale_log2) {
  ld_cols(taddr, x);
  if (pm == ~0u) {
#pragma unroll
    for (int c = 0; c < kCols; c += 2) f2_unpack(f2_mul(f2_pack(x[c], x[c + 1]), sc2), x[c], x[c + 1]);
  } else {
#pragma unroll
    for (int c = 0; c < kCols; ++c) x[c] = ((pm >> c) & 1u) ? x[c] * scale_log2 : -INFINITY;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    k_fwd_kt(const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmKh,
             const __grid_constant__ CUtensorMap tmVh, const __grid_constant__ CUtensorMap tmOq,
             const __grid_constant__ KtParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  if ((base - raw) + kNeed > static_cast<uint32_t>(kSmem)) {
    if (threadIdx.x == 0) atomicOr(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  const uint32_t sQ = base + kOffQ, sK = base + kOffK, sV = base + kOffV, sP = base + kOffP;
  uint8_t* small = gbase + kOffSmall;
  const uint32_t bars = base + kOffSmall;
  const uint32_t b_qfull = bars, b_qempty = b_qfull + 16;  // [2]
  const uint32_t b_kfull = b_qempty + 16, b_kempty = b_kfull + 8 * kKSlots;
  const uint32_t b_vfull = b_kempty + 8 * kKSlots, b_vempty = b_vfull + 8 * kVSlots;
  const uint32_t b_sfull = b_vempty + 8 * kVSlots, b_sfree = b_sfull + 8 * kSBuf;
  const uint32_t b_pfull = b_sfree + 8 * kSBuf, b_pvdone = b_pfull + 8 * kPBuf;
  const uint32_t b_ofree = b_pvdone + 8 * kPBuf;  // [2]
  const uint32_t b_dfull = b_ofree + 16, b_dempty = b_dfull + 8 * kDescRing;
  const uint32_t b_tfull = b_dempty + 8 * kDescRing, b_tempty = b_tfull + 8 * kSubRing;
  const uint32_t b_clc = b_tempty + 8 * kSubRing, b_drain = b_clc + 8, b_drain2 = b_drain + 8;
  static_assert(8 * kNumBars == kSmTmem, "barrier count");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(small + kSmTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(small + kSmAbort);
  const uint32_t clc_resp = smem_u32(small + kSmClc);
  Sub* sring = reinterpret_cast<Sub*>(small + kSmSub);
  StepDesc* dring = reinterpret_cast<StepDesc*>(small + kSmDesc);
  float* mref = reinterpret_cast<float*>(small + kSmM);
  float* mnew = reinterpret_cast<float*>(small + kSmM2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_qfull + 8 * i, 1);
      mbar_init(b_qempty + 8 * i, kGroups);  // thread 0 of each softmax warpgroup
      mbar_init(b_ofree + 8 * i, kSoftmaxThreads);
    }
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(b_kfull + 8 * s, 1);
      mbar_init(b_kempty + 8 * s, 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(b_vfull + 8 * s, 1);
      mbar_init(b_vempty + 8 * s, 1);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_sfree + 8 * i, kSoftmaxThreads);
    }
    for (int i = 0; i < kPBuf; ++i) {
      mbar_init(b_pfull + 8 * i, kSoftmaxThreads);
      mbar_init(b_pvdone + 8 * i, 1);
    }
    for (int i = 0; i < kDescRing; ++i) {
      mbar_init(b_dfull + 8 * i, 1);
      mbar_init(b_dempty + 8 * i, kGroups + 1);  // thread 0 of each softmax warpgroup and the V loader
    }
    for (int i = 0; i < kSubRing; ++i) {
      mbar_init(b_tfull + 8 * i, 1);
      mbar_init(b_tempty + 8 * i, kGroups + 2);  // S issuer, P V issuer, thread 0 of each softmax warpgroup
    }
    mbar_init(b_clc, 1);
    mbar_init(b_drain, 1);
    mbar_init(b_drain2, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpS) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the set-up above overlaps the previous kernel of the stream (programmatic
  // stream serialization); everything below may read its results
  grid_dependency_wait();

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the plan (lanes hold 32 entries); lane 0 issues
    // the copies and publishes records and step descriptors.
    const bool leader = lane == 0;
    if (leader) {
      tma_prefetch_desc(&tmQh);
      tma_prefetch_desc(&tmKh);
      tma_prefetch_desc(&tmOq);
    }
    int g = 0, k_issued = 0;   // steps (K loads)
    int si = 0, q_issued = 0;  // sub-tasks with steps (Q halves loaded)
    int ti = 0;                // sub-task records
    auto publish = [&](const Sub& s) {
      if (leader) {
        const int slot = ti % kSubRing;
        if (ti >= kSubRing) mbar_wait(b_tempty + 8 * slot, ((ti / kSubRing) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        sring[slot] = s;
        mbar_arrive(b_tfull + 8 * slot);
      }
      __syncwarp();
      ++ti;
    };
    // one step: its descriptor, then its K rows
    auto emit = [&](int r0, int e0, int r1, int e1, int hk) {
      if (leader) {
        const int di = g % kDescRing;
        if (g >= kDescRing) mbar_wait(b_dempty + 8 * di, ((g / kDescRing) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        StepDesc d{};
        d.r0 = r0;
        d.r1 = r1;
        d.hk = hk;
        d.e0 = e0;
        d.e1 = e1;
        dring[di] = d;
        mbar_arrive(b_dfull + 8 * di);
        const int slot = g % kKSlots;
        if (g >= kKSlots) mbar_wait(b_kempty + 8 * slot, ((g / kKSlots) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (!*abort_flag) {
          k_issued = g + 1;
          const uint32_t dst = sK + slot * kSlotBytes;
          mbar_arrive_expect_tx(b_kfull + 8 * slot, kSlotBytes);
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            tma_load_2d(dst + ch * 16384, &tmKh, b_kfull + 8 * slot, hk * D + ch * 64, r0);
            tma_load_2d(dst + ch * 16384 + 8192, &tmKh, b_kfull + 8 * slot, hk * D + ch * 64, r1);
          }
        }
      }
      __syncwarp();
      ++g;
    };
    ClcTasks tasks{clc_resp, b_clc};
    for (;;) {
      int t = -1;
      if (leader) t = tasks.next(abort_flag, p.err, kWaitTimeoutNs);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0 || t >= p.ntasks || *abort_flag) break;
      const int* wd = p.work + 4LL * t;
      const int m_block = __ldg(wd + 0), qv = __ldg(wd + 3);
      const int h = static_cast<int>(bsm_idx(__ldg(wd + 1), p.Hq, p.err));
      const int b = static_cast<int>(bsm_idx(__ldg(wd + 2), p.B, p.err));
      const int* sq = p.seq + 8 * b;
      const int q_off = __ldg(sq + 0), k_off = __ldg(sq + 1), row_begin = __ldg(sq + 4);
      const int hm = (p.Hmask == 1) ? 0 : h;
      const int hk = h / (p.Hq / p.Hk);
      const long long flat = bsm_idx(static_cast<long long>(hm) * p.rows + row_begin + m_block,
                                     static_cast<long long>(p.Hmask) * p.rows, p.err);
      const int p0 = __ldg(p.p_off + flat), np = __ldg(p.p_off + flat + 1) - p0;
      const int f0 = __ldg(p.f_off + flat), n = np + (__ldg(p.f_off + flat + 1) - f0);
      for (int qh = 0; qh < 2; ++qh) {
        const int qv_h = min(max(qv - kHalf * qh, 0), kHalf);
        if (qv_h == 0) continue;
        // live quadrants of this half
        int nlive = 0;
        for (int j0 = 0; j0 < n; j0 += 32) {
          const int j = j0 + lane;
          const int q = (j < n) ? quads_of(p, p0, np, j) : 0;
          nlive += __reduce_add_sync(0xffffffffu, __popc((q >> (2 * qh)) & 3));
        }
        Sub s{};
        s.h = h;
        s.q0 = q_off + m_block * 128 + kHalf * qh;
        s.qv = qv_h;
        s.nsteps = (nlive + 1) / 2;
        s.qh = qh;
        publish(s);
        if (s.nsteps == 0) continue;
        const int qb = si & 1;
        if (leader) {
          if (si >= 2) mbar_wait(b_qempty + 8 * qb, ((si >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (!*abort_flag) {
            q_issued = si + 1;
            mbar_arrive_expect_tx(b_qfull + 8 * qb, kHalfBytes);
#pragma unroll
            for (int ch = 0; ch < 2; ++ch)
              tma_load_2d(sQ + qb * kHalfBytes + ch * 8192, &tmQh, b_qfull + 8 * qb, h * D + ch * 64, s.q0);
          }
        }
        __syncwarp();
        ++si;
        // steps: live quadrants in list order (key half 0 before 1), two per step
        int hold_r = -1, hold_e = 0;
        for (int j0 = 0; j0 < n; j0 += 32) {
          const int j = j0 + lane;
          int my_q = 0, my_kt = 0;
          if (j < n) {
            my_q = quads_of(p, p0, np, j);
            my_kt = tile_of(p, p0, np, f0, j);
          }
          const int cnt = min(32, n - j0);
          for (int jj = 0; jj < cnt; ++jj) {
            const int q = __shfl_sync(0xffffffffu, my_q, jj);
            const int kt = __shfl_sync(0xffffffffu, my_kt, jj);
#pragma unroll
            for (int kh = 0; kh < 2; ++kh) {
              const int bit = 2 * qh + kh;
              if (!((q >> bit) & 1)) continue;
              const int r = k_off + kt * 128 + kHalf * kh;
              const int e = ((q >> (4 + bit)) & 1) ? kFullPos : (((p0 + j0 + jj) << 1) | kh);
              if (hold_r < 0) {
                hold_r = r;
                hold_e = e;
              } else {
                emit(hold_r, hold_e, r, e, hk);
                hold_r = -1;
              }
            }
          }
        }
        if (hold_r >= 0) emit(hold_r, hold_e, p.rows_k, kEmptyPos, hk);  // rows past the tensor: zeros
      }
    }
    {
      Sub end{};
      end.nsteps = -1;
      publish(end);
    }
    if (leader && *abort_flag) {
      // let copies already started land before the CTA exits
      for (int u = (q_issued > 2 ? q_issued - 2 : 0); u < q_issued; ++u)
        mbar_wait_drain(b_qfull + 8 * (u & 1), (u >> 1) & 1, kWaitTimeoutNs);
      for (int u = (k_issued > kKSlots ? k_issued - kKSlots : 0); u < k_issued; ++u)
        mbar_wait_drain(b_kfull + 8 * (u % kKSlots), (u / kKSlots) & 1, kWaitTimeoutNs);
      tasks.drain(kWaitTimeoutNs);
    }
  } else if (warp == kWarpS) {
    // ------------------------------------------------------------ S^T issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kHalf, 0);  // K (M=128 keys) x Q half (N=64), K-major
      const uint64_t dK0 = sdesc_sw128(sK, 16, 1024);
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);
      int g = 0, si = 0;
      for (int ti = 0;; ++ti) {
        const int tslot = ti % kSubRing;
        mbar_wait(b_tfull + 8 * tslot, (ti / kSubRing) & 1, abort_flag, p.err, kWaitTimeoutNs);
        const Sub s = sring[tslot];
        mbar_arrive(b_tempty + 8 * tslot);
        if (s.nsteps < 0 || *abort_flag) break;
        if (s.nsteps == 0) continue;
        const int qb = si & 1;
        mbar_wait(b_qfull + 8 * qb, (si >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        const uint64_t dQ = dQ0 + static_cast<uint64_t>((qb * kHalfBytes) >> 4);
        for (int j = 0; j < s.nsteps; ++j, ++g) {
          const int sb = g % kSBuf, slot = g % kKSlots;
          mbar_wait(b_kfull + 8 * slot, (g / kKSlots) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (g >= kSBuf) mbar_wait(b_sfree + 8 * sb, ((g / kSBuf) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (*abort_flag) break;
          tc_fence_after();
          const uint64_t dK = dK0 + static_cast<uint64_t>((slot * kSlotBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t offK = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            const uint32_t offQ = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tmem + kHalf * sb, dK + offK, dQ + offQ, idS, kk > 0);
          }
          umma_commit(b_sfull + 8 * sb);
          umma_commit(b_kempty + 8 * slot);
        }
        ++si;
      }
      // every MMA issued above completes before TMEM is released
      umma_commit(b_drain);
      mbar_wait_drain(b_drain, 0, kWaitTimeoutNs);
    }
  } else if (warp == kWarpPV) {
    // ------------------------------------------------ V loads and P V issuer
    // V(g) is requested as soon as its descriptor exists and the P V that
    // last used its slot has completed, up to kVSlots steps ahead.
    if (lane == 0) {
      tma_prefetch_desc(&tmVh);
      constexpr uint32_t idO = idesc_bf16_f32_mn(128, kHalf);  // V^T (M=128 dims) x P^T (N=64), MN-major
      const uint64_t dV0 = sdesc_sw128(sV, 16384, 1024);
      const uint64_t dP0 = sdesc_sw128(sP, 16384, 1024);
      int gl = 0, v_issued = 0;  // V loads requested
      int g = 0, si = 0;         // P V steps, sub-tasks with steps
      // request V(gl) while it is within the ring's reach of step `need`
      // (blocking only for V(need) itself)
      auto top_up = [&](int need) {
        while (gl < need + kVSlots && !*abort_flag) {
          const int di = gl % kDescRing, slot = gl % kVSlots;
          if (gl > need) {
            // optional look-ahead: only if nothing has to be waited for
            if (!mbar_try_wait(b_dfull + 8 * di, (gl / kDescRing) & 1)) return;
            if (gl >= kVSlots && !mbar_try_wait(b_vempty + 8 * slot, ((gl / kVSlots) - 1) & 1)) return;
          } else {
            mbar_wait(b_dfull + 8 * di, (gl / kDescRing) & 1, abort_flag, p.err, kWaitTimeoutNs);
            if (gl >= kVSlots) mbar_wait(b_vempty + 8 * slot, ((gl / kVSlots) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
            if (*abort_flag) return;
          }
          const StepDesc dsc = dring[di];
          mbar_arrive(b_dempty + 8 * di);
          v_issued = gl + 1;
          const uint32_t dst = sV + slot * kSlotBytes;
          mbar_arrive_expect_tx(b_vfull + 8 * slot, kSlotBytes);
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            tma_load_2d(dst + ch * 16384, &tmVh, b_vfull + 8 * slot, dsc.hk * D + ch * 64, dsc.r0);
            tma_load_2d(dst + ch * 16384 + 8192, &tmVh, b_vfull + 8 * slot, dsc.hk * D + ch * 64, dsc.r1);
          }
          ++gl;
        }
      };
      for (int ti = 0;; ++ti) {
        const int tslot = ti % kSubRing;
        mbar_wait(b_tfull + 8 * tslot, (ti / kSubRing) & 1, abort_flag, p.err, kWaitTimeoutNs);
        const Sub s = sring[tslot];
        mbar_arrive(b_tempty + 8 * tslot);
        if (s.nsteps < 0 || *abort_flag) break;
        if (s.nsteps == 0) continue;
        const int ob = si & 1;
        for (int j = 0; j < s.nsteps; ++j, ++g) {
          top_up(g);
          const int pb = g % kPBuf, slot = g % kVSlots;
          mbar_wait(b_pfull + 8 * pb, (g / kPBuf) & 1, abort_flag, p.err, kWaitTimeoutNs);
          mbar_wait(b_vfull + 8 * slot, (g / kVSlots) & 1, abort_flag, p.err, kWaitTimeoutNs);
          // the first P V of a sub-task overwrites its O^T buffer: the
          // epilogue of the sub-task two before must have read it
          if (j == 0 && si >= 2) mbar_wait(b_ofree + 8 * ob, ((si >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (*abort_flag) break;
          tc_fence_after();
          const uint64_t dV = dV0 + static_cast<uint64_t>((slot * kSlotBytes) >> 4);
          const uint64_t dP = dP0 + static_cast<uint64_t>((pb * kHalfBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_bf16_ss(tmem + kColO + kHalf * ob, dV + static_cast<uint64_t>((kk * 2048) >> 4),
                         dP + static_cast<uint64_t>((kk * 2048) >> 4), idO, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(b_vempty + 8 * slot);
          umma_commit(b_pvdone + 8 * pb);
        }
        ++si;
      }
      // every MMA issued above completes before TMEM is released
      umma_commit(b_drain2);
      mbar_wait_drain(b_drain2, 0, kWaitTimeoutNs);
      if (*abort_flag) {
        for (int u = (v_issued > kVSlots ? v_issued - kVSlots : 0); u < v_issued; ++u)
          mbar_wait_drain(b_vfull + 8 * (u % kVSlots), (u / kVSlots) & 1, kWaitTimeoutNs);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wg = warp >> 2;         // query columns kCols wg .. kCols wg + kCols - 1
    const int t = threadIdx.x & 127;  // key t of a step; head-dimension column t in the epilogue
    const int cb = kCols * wg;
    const uint32_t bar_id = 1 + wg;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    float* xch = reinterpret_cast<float*>(small + kSmXch) + wg * 4 * kCols;  // [4 warps][kCols]
    Sub* bcast = reinterpret_cast<Sub*>(small + kSmBcast) + wg;
    const int pos = t >> 6;
    int g = 0, si = 0;
    bool store_pending = false;
    int pend_qb = 0;
    auto group_sync = [&]() { named_bar_sync(bar_id, 128); };
    for (int ti = 0;; ++ti) {
      if (t == 0) {
        const int tslot = ti % kSubRing;
        mbar_wait(b_tfull + 8 * tslot, (ti / kSubRing) & 1, abort_flag, p.err, kWaitTimeoutNs);
        Sub s = sring[tslot];
        mbar_arrive(b_tempty + 8 * tslot);
        if (*abort_flag) s.nsteps = -1;
        *bcast = s;
      }
      group_sync();
      const Sub s = *bcast;
      group_sync();  // every thread has its copy before the next record lands
      if (s.nsteps < 0) break;
      if (s.nsteps == 0) {
        // no visible key for any row of this half: O = 0, LSE = -inf
        const int row = cb + t;
        if (t < kCols && row < s.qv && bsm_ok(s.q0 + row, p.total_q, p.err)) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + (static_cast<long long>(s.q0 + row) * p.Hq + s.h) * D);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          if (p.lse != nullptr) p.lse[static_cast<long long>(s.h) * p.total_q + s.q0 + row] = -INFINITY;
        }
        continue;
      }
      const int qb = si & 1, ob = si & 1;
      uint64_t l2[kCols / 2];  // this key's share of the column sums, pairs of columns
#pragma unroll
      for (int c = 0; c < kCols / 2; ++c) l2[c] = 0;
      if (t < kCols) mref[cb + t] = kNoMax;
      group_sync();
      for (int j = 0; j < s.nsteps; ++j, ++g) {
        const int di = g % kDescRing, sb = g % kSBuf, pb = g % kPBuf;
        mbar_wait(b_dfull + 8 * di, (g / kDescRing) & 1, abort_flag, p.err, kWaitTimeoutNs);
        const int e = pos ? dring[di].e1 : dring[di].e0;
        if (j == 0 && t == 0 && store_pending) {
          // this warpgroup's previous output rows have left shared memory:
          // its share of the Q buffer goes back to the producer
          bulk_wait_read_all();
          mbar_arrive(b_qempty + 8 * pend_qb);
          store_pending = false;
        }
        // predicate bits of this key for the warpgroup's 32 queries (partial
        // quadrants only: sequence tails); the word is the same for the warp
        uint32_t pm = ~0u;
        if (e == kEmptyPos) {
          pm = 0u;
        } else if (e >= 0) {
          const int kc = kHalf * (e & 1) + (t & 63);
          const uint32_t* pw =
              p.payload + bsm_idx(e >> 1, p.nP, p.err) * 512 + (kHalf * s.qh + cb) * 4 + (kc >> 5);
          uint32_t bits = 0u;
#pragma unroll 8
          for (int r = 0; r < kCols; ++r) bits |= ((__ldg(pw + 4 * r) >> (kc & 31)) & 1u) << r;
          pm = bits;
        }
        mbar_wait(b_sfull + 8 * sb, (g / kSBuf) & 1, abort_flag, p.err, kWaitTimeoutNs);
        // the P V that last read P buffer pb (step g - 2) has completed
        if (g >= kPBuf) mbar_wait(b_pvdone + 8 * pb, ((g / kPBuf) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        tc_fence_after();
        float x[kCols];
        load_scores(lane_addr + kHalf * sb + cb, x, pm, sc2, p.scale_log2);
        // does a score exceed its column's reference max by more than 2^8?
        float amax = -INFINITY;
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(mref + cb + c);
          amax = max3f(amax, x[c] - m4.x, x[c + 1] - m4.y);
          amax = max3f(amax, x[c + 2] - m4.z, x[c + 3] - m4.w);
        }
        const bool need = (j == 0) | group_any(bar_id, amax > kRescaleLog2);
        if (t == 0) mbar_arrive(b_dempty + 8 * di);  // every thread of the group has read it
        if (need) {
          // exact column max over the 128 keys (x is reloaded afterwards)
          warp_reduce_scatter32<true>(x, lane);
          if (lane < kCols) xch[(warp & 3) * kCols + lane] = x[0];
          group_sync();
          if (t < kCols) {
            const float cm = fmaxf(fmaxf(xch[t], xch[kCols + t]), fmaxf(xch[2 * kCols + t], xch[3 * kCols + t]));
            mnew[cb + t] = fmaxf(mref[cb + t], cm);
          }
          group_sync();
          // rescale factors 2^(old - new) per column: the sums, and O^T once
          // it holds P V of earlier steps
          bool moved = false;
#pragma unroll
          for (int c = 0; c < kCols; c += 2) {
            const float2 mo = *reinterpret_cast<const float2*>(mref + cb + c);
            const float2 mn = *reinterpret_cast<const float2*>(mnew + cb + c);
            moved |= (mo.x != mn.x) | (mo.y != mn.y);
            l2[c / 2] = f2_mul(l2[c / 2], f2_pack(ex2_approx(mo.x - mn.x), ex2_approx(mo.y - mn.y)));
          }
          if (j > 0 && group_any(bar_id, moved)) {
            // wait for the last P V, then scale column (query) c of this
            // thread's O^T row (head dimension t)
            mbar_wait(b_pvdone + 8 * ((g - 1) % kPBuf), ((g - 1) / kPBuf) & 1, abort_flag, p.err, kWaitTimeoutNs);
            tc_fence_after();
            ld_cols(lane_addr + kColO + kHalf * ob + cb, x);
#pragma unroll
            for (int c = 0; c < kCols; c += 2) {
              const float2 mo = *reinterpret_cast<const float2*>(mref + cb + c);
              const float2 mn = *reinterpret_cast<const float2*>(mnew + cb + c);
              x[c] *= ex2_approx(mo.x - mn.x);
              x[c + 1] *= ex2_approx(mo.y - mn.y);
            }
            st_cols(lane_addr + kColO + kHalf * ob + cb, x);
            tmem_st_wait();
          }
          group_sync();  // every thread has read the old maxima
          if (t < kCols) mref[cb + t] = mnew[cb + t];
          group_sync();
          load_scores(lane_addr + kHalf * sb + cb, x, pm, sc2, p.scale_log2);
        }
        tc_fence_before();
        mbar_arrive(b_sfree + 8 * sb);
        // this key's P^T row for the group's 32 queries (bf16), and the sums
        uint32_t pk[kCols / 2];
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(mref + cb + c);
          float d[4];
          f2_unpack(f2_add(f2_pack(x[c], x[c + 1]), f2_pack(-m4.x, -m4.y)), d[0], d[1]);
          f2_unpack(f2_add(f2_pack(x[c + 2], x[c + 3]), f2_pack(-m4.z, -m4.w)), d[2], d[3]);
          const float e0 = ex2_approx(d[0]), e1 = ex2_approx(d[1]), e2 = ex2_approx(d[2]), e3 = ex2_approx(d[3]);
          l2[c / 2] = f2_add(l2[c / 2], f2_pack(e0, e1));
          l2[c / 2 + 1] = f2_add(l2[c / 2 + 1], f2_pack(e2, e3));
          pk[c / 2] = pack_bf16x2(e0, e1);
          pk[c / 2 + 1] = pack_bf16x2(e2, e3);
        }
        const uint32_t prow = sP + pb * kHalfBytes + t * 128;
#pragma unroll
        for (int u = 0; u < kCols / 8; ++u)
          st_shared_v4(prow + ((((kCols / 8) * wg + u) ^ (t & 7)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                       pk[4 * u + 3]);
        fence_proxy_async_smem();
        mbar_arrive(b_pfull + 8 * pb);
      }
      // ---------------------------------------------------------- epilogue
      // the sub-task's last P V has completed: O^T is final
      mbar_wait(b_pvdone + 8 * ((g - 1) % kPBuf), ((g - 1) / kPBuf) & 1, abort_flag, p.err, kWaitTimeoutNs);
      tc_fence_after();
      {
        float v[kCols];
#pragma unroll
        for (int c = 0; c < kCols; c += 2) f2_unpack(l2[c / 2], v[c], v[c + 1]);
        warp_reduce_scatter32<false>(v, lane);
        if (lane < kCols) xch[(warp & 3) * kCols + lane] = v[0];
        group_sync();
        if (t < kCols) {
          const float l = (xch[t] + xch[kCols + t]) + (xch[2 * kCols + t] + xch[3 * kCols + t]);
          const bool have = l > 0.0f;
          mnew[cb + t] = have ? 1.0f / l : 0.0f;
          if (cb + t < s.qv && p.lse != nullptr && bsm_ok(s.q0 + cb + t, p.total_q, p.err))
            p.lse[static_cast<long long>(s.h) * p.total_q + s.q0 + cb + t] =
                have ? (mref[cb + t] + __log2f(l)) * kLn2 : -INFINITY;
        }
        group_sync();
      }
      float o[kCols];
      ld_cols(lane_addr + kColO + kHalf * ob + cb, o);
      tc_fence_before();
      mbar_arrive(b_ofree + 8 * ob);
#pragma unroll
      for (int c = 0; c < kCols; c += 4) {
        const float4 il = *reinterpret_cast<const float4*>(mnew + cb + c);
        o[c] *= il.x;
        o[c + 1] *= il.y;
        o[c + 2] *= il.z;
        o[c + 3] *= il.w;
      }
      if (s.qv == kHalf) {
        // stage this group's kCols output rows (row cb + c, column t) in the
        // half's Q buffer (no MMA reads it any more: the last P V has
        // completed) and store them with TMA
        const uint32_t stage = sQ + qb * kHalfBytes + (t >> 6) * 8192;
        const uint32_t unit = (t & 63) >> 3, byte = (t & 7) * 2;
#pragma unroll
        for (int c = 0; c < kCols; ++c) {
          const int row = cb + c;
          const __nv_bfloat16 hv = __float2bfloat16_rn(o[c]);
          const uint32_t a = stage + row * 128 + ((unit ^ (row & 7)) << 4) + byte;
          asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(*reinterpret_cast<const uint16_t*>(&hv)) : "memory");
        }
        fence_proxy_async_smem();
        group_sync();
        if (t == 0) {
          if (bsm_ok(s.q0 + cb + kCols - 1, p.total_q, p.err))
#pragma unroll
            for (int ch = 0; ch < 2; ++ch)
              tma_store_2d(&tmOq, sQ + qb * kHalfBytes + ch * 8192 + cb * 128, s.h * D + ch * 64, s.q0 + cb);
          bulk_commit_group();
          store_pending = true;
          pend_qb = qb;
        }
      } else {
        // a tail half: rows past the sample belong to another sample; store
        // the valid rows directly (column t of each)
        __nv_bfloat16* orow = p.o + static_cast<long long>(s.q0 + cb) * p.Hq * D + s.h * D + t;
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          if (cb + c < s.qv && bsm_ok(s.q0 + cb + c, p.total_q, p.err))
            orow[static_cast<long long>(c) * p.Hq * D] = __float2bfloat16_rn(o[c]);
        group_sync();
        if (t == 0) mbar_arrive(b_qempty + 8 * qb);
      }
      ++si;
    }
    if (t == 0 && store_pending) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpS) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_kt() {
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

// 2-D view [rows, heads*D] of a bf16 tensor, box 64 columns x box_rows rows, 128-byte swizzle.
bool make_map64(CUtensorMap* m, const void* ptr, int64_t rows, int64_t heads, uint32_t box_rows = 64) {
  auto fn = encode_fn_kt();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(heads * D), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(heads * D * 2)};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fwd_kt_applies(const FwdLaunch& a) {
  const fa_plan* pl = a.plan;
  return pl->mask_kind == MASK_BLOCKS && pl->geom.head_dim == D &&
         (a.flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI | FA_FWD_COARSENED)) == 0 && pl->block_q > 0 && pl->block_kv > 0 &&
         pl->block_q % kHalf == 0 && pl->block_kv % kHalf == 0;
}

cudaError_t launch_fwd_kt(const FwdLaunch& a, cudaStream_t st, const char** why) {
  const fa_plan* pl = a.plan;
  const Geometry& g = pl->geom;
  const int64_t rows_q = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_q : g.total_q;
  const int64_t rows_k = (g.layout == FA_LAYOUT_BSHD) ? int64_t(g.batch) * g.seqlen_k : g.total_k;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map64(&mq, a.q, rows_q, g.heads_q) || !make_map64(&mk, a.k, rows_k, g.heads_k) ||
      !make_map64(&mv, a.v, rows_k, g.heads_k) || !make_map64(&mo, a.o, rows_q, g.heads_q, kCols)) {
    *why = "cuTensorMapEncodeTiled failed (pointer alignment or driver entry point)";
    return cudaErrorInvalidValue;
  }
  KtParams p{};
  p.work = pl->work_desc;
  p.seq = pl->seq_desc;
  p.p_off = pl->p_off;
  p.f_off = pl->f_off;
  p.p_idx = pl->p_idx;
  p.f_idx = pl->f_idx;
  p.payload = pl->payload;
  p.quads = pl->quads;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.err = fwd_error_word();
  p.Hq = g.heads_q;
  p.Hk = g.heads_k;
  p.Hmask = pl->Hmask;
  p.rows = static_cast<int>(pl->rows);
  p.total_q = static_cast<int>(rows_q);
  p.rows_k = static_cast<int>(rows_k);
  p.ntasks = static_cast<int>(pl->tasks);
  p.B = g.batch;
  p.nP = pl->P;
  p.nF = pl->F;
  p.scale_log2 = a.scale * kLog2e;
  if (p.err == nullptr) {
    *why = "forward error word not found";
    return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(k_fwd_kt, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) {
    *why = "cudaFuncSetAttribute failed";
    return e;
  }
  // one CTA per work_desc entry; shared memory keeps one per SM and the
  // running CTAs take over the rest (cluster launch control); programmatic
  // stream serialization lets its set-up overlap the previous kernel
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(pl->tasks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_fwd_kt, mq, mk, mv, mo, p);
  if (e != cudaSuccess) *why = "forward kernel launch failed";
  return e;
}

}  // namespace bsm
