// attn_decode.cu -- decoding attention over a paged KV cache (sm_103a).
//
// "FlexAttention: A Programming Model for Generating Optimized Attention
// Kernels" (summary page), §3.4 Paged Attention Integration and Modification
// Conversion for Inference:
//   * the query rows are the newest tokens of each sequence, at absolute
//     position offset + q_idx (offset = k_len - q_len); their interval
//     endpoints are given at that position, so the plan built from them over
//     the logical keys is the converted mask, and the plan's K tile lists
//     say which logical tiles a query row needs;
//   * logical key j of sequence b lives in page page_table[b][j / page_size]
//     at row j % page_size.  The page lookup is a data transformation of the
//     plan's index lists, done once per call by k_decode_prep (every K tile
//     of every list gets the physical start row of each of its pages), not
//     in the attention loop, which only sees physical rows.  The predicate
//     payload stays indexed by list entry and needs no conversion.
//
// Three launches:
//   k_decode_prep     converts every list entry to the physical rows of its
//                     pages through the page table (one thread per entry),
//                     and in its first CTA scans the rows' entry counts;
//   k_decode<N>       persistent, one CTA per SM.  The K tiles of all rows
//                     and K/V heads, concatenated, are cut into C equal
//                     ranges, one per CTA (the Split-K partition of
//                     "Decoupling Logical Masks from GPU Execution for Dynamic
//                     Block-Sparse Attention", Split-K paragraph, sized so
//                     that every CTA streams the same number of tiles); a
//                     range falls into pieces, one per (row, K/V head) it
//                     touches.  The G = Hq/Hk query heads of the K/V head (the
//                     GQA group; N = G rounded up to 16) form the N columns of
//                     keys-major products on the tensor cores:
//                       S^T = K Q^T (M = 128 keys) into TMEM,
//                       P^T = exp2(S^T - m) (bf16, shared memory, K-major),
//                       O^T += V^T P^T (M = 128 head dims),
//                     with a lazily updated per-column reference max; each
//                     piece's unnormalised O, reference max m and sum l go to
//                     a workspace slot;
//   k_decode_combine  one warp per (query row, head): merges the pieces of
//                     the row with weights 2^(m - max m), divides by the
//                     merged l, writes O (bf16) and LSE (natural log).
// The path is bound by HBM bandwidth (every visible K/V byte is read once per
// K/V head); the tensor cores keep the arithmetic off the issue slots.
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
constexpr int kTileBytes = kTile * D * 2;       // 32 KB: one K or V tile, [2 halves][128 rows][128 B]
constexpr int kStageBytes = 2 * kTileBytes;     // K then V
constexpr int kThreads = 224;  // warps 0-3 softmax, 4 producer, 5 S^T issuer, 6 P V issuer
constexpr int kWarpProducer = 4, kWarpMma = 5, kWarpPV = 6;

struct DecParams {
  // plan
  const int32_t* seq;
  const int32_t* p_off;
  const int32_t* f_off;
  const int32_t* p_idx;
  const int32_t* f_idx;
  const uint32_t* payload;
  // k_decode_prep outputs
  const int32_t* remap;    // [(P + F) * chunks]: physical start row of each page chunk, -1 past k_len
  const int32_t* cu_rows;  // [R + 1]: prefix of the rows' entry counts (row r = mask head * B + sequence)
  // piece results
  float* part_o;           // [slots][G][D]: unnormalised O
  float* part_ml;          // [slots][2][G]: reference max (log2 units), sum l
  uint32_t* err;
  int B, Hq, Hk, Hmask, rows, G, gy, chunks, chunk_rows, oob_row, R;
  long long nP, nF;
  float scale_log2;
  // score mods (FA_MOD_SOFTCAP, FA_MOD_ALIBI) at the query's absolute position
  int flags;
  float y_scale, cap_log2;      // softcap: log2(e) * cap * tanh(y_scale * s)
  float slopes_l2[kMaxHeads];   // ALiBi slope * log2(e) per Q head
};

// tanh(y) = 1 - 2 / (exp(2y) + 1); absolute error ~1e-7, which the softcap
// scales by the cap
__device__ __forceinline__ float tanh_exp2(float y) {
  const float e = ex2_approx(2.0f * kLog2e * y);
  return 1.0f - __fdividef(2.0f, e + 1.0f);
}

template <int N>
struct DecLayout {
  static_assert(N % 16 == 0 && N >= 16 && N <= 64, "query columns");
  static constexpr int kStages = (N <= 32) ? 3 : 2;  // K/V ring depth within the shared-memory budget
  static constexpr int kOffRing = 0;
  static constexpr int kOffQ = kStages * kStageBytes;        // [2 buffers][2 halves][N rows][128 B]
  static constexpr int kQBytes = 2 * N * 128;
  static constexpr int kOffP = kOffQ + 2 * kQBytes;          // P: [2 buffers][2 key halves][N rows][128 B]
  static constexpr int kOffSmall = kOffP + 2 * kQBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * 8;
  static constexpr int kSmTmem = 8 * kNumBars;
  static constexpr int kSmAbort = kSmTmem + 4;
  static constexpr int kSmRed = (kSmAbort + 4 + 15) & ~15;  // [4 warps][N] floats
  static constexpr int kSmMref = kSmRed + 4 * N * 4;        // [N]
  static constexpr int kSmAlpha = kSmMref + N * 4;          // [N]
  static constexpr int kSmallBytes = kSmAlpha + N * 4;
  static constexpr int kNeed = kOffSmall + kSmallBytes;
  static constexpr int kSmem = (kNeed + 1024 <= 232448) ? kNeed + 1024 : 232448;
  static constexpr uint32_t kTmemCols = (4 * N <= 64) ? 64 : (4 * N <= 128 ? 128 : 256);
  static_assert(kNeed <= 232448, "shared memory budget");
};

// The work is the sequence of segments s = r * gy + gi, row r = hm * B + b
// (mask head, sequence), gi the K/V head of the GQA group (always 0 for
// per-head masks): segment s holds the K tiles of row r for that K/V head.
// CTA c of C takes the tiles [W c / C, W (c + 1) / C) of the concatenation
// (W tiles in all), so every CTA streams the same number of K/V tiles; its
// range falls into pieces, one per segment it touches.  A piece's results
// go to slot s + c, which no other piece uses.
__device__ __forceinline__ long long seg_start(const int32_t* cu_rows, int R, int gy, long long s) {
  if (s >= static_cast<long long>(R) * gy) return static_cast<long long>(gy) * __ldg(cu_rows + R);
  const long long r = s / gy, gi = s % gy;
  const long long a = __ldg(cu_rows + r), n = __ldg(cu_rows + r + 1) - a;
  return gy * a + gi * n;
}
__device__ __forceinline__ long long seg_start(const DecParams& p, long long s) {
  return seg_start(p.cu_rows, p.R, p.gy, s);
}

// One piece as every role sees it.
struct Unit {
  int hm, b, hk, e0, n;   // mask head, sequence, K/V head, first list entry, entries
  int p0, np, f0;         // the row's partial and full lists
  int q_off, k_len;
  long long slot;         // workspace slot of the piece's results
};

struct Pieces {
  long long pos, end, s, S;
  int c;
  __device__ __forceinline__ void init(const DecParams& p, int cta, int C) {
    const long long W = static_cast<long long>(p.gy) * __ldg(p.cu_rows + p.R);
    c = cta;
    pos = W * cta / C;
    end = W * (cta + 1) / C;
    S = static_cast<long long>(p.R) * p.gy;
    // the last segment starting at or before pos
    long long lo = 0, hi = S;
    while (hi - lo > 1) {
      const long long mid = (lo + hi) >> 1;
      if (seg_start(p, mid) <= pos) lo = mid; else hi = mid;
    }
    s = lo;
  }
  // the next piece of this CTA's range; false at its end
  __device__ __forceinline__ bool next(const DecParams& p, Unit* x) {
    if (pos >= end) return false;
    while (s + 1 < S && seg_start(p, s + 1) <= pos) ++s;  // past empty segments
    const long long a = seg_start(p, s), z = seg_start(p, s + 1);
    const long long r = s / p.gy;
    const int gi = static_cast<int>(s % p.gy);
    x->hm = static_cast<int>(r / p.B);
    x->b = static_cast<int>(bsm_idx(r % p.B, p.B, p.err));
    x->hk = (p.Hmask == 1) ? gi : x->hm;
    x->e0 = static_cast<int>(pos - a);
    x->n = static_cast<int>((z < end ? z : end) - pos);
    const int32_t* sq = p.seq + 8 * x->b;
    x->q_off = __ldg(sq + 0);
    x->k_len = __ldg(sq + 3);
    const long long flat = bsm_idx(static_cast<long long>(x->hm) * p.rows + __ldg(sq + 4),
                                   static_cast<long long>(p.Hmask) * p.rows, p.err);
    x->p0 = __ldg(p.p_off + flat);
    x->np = __ldg(p.p_off + flat + 1) - x->p0;
    x->f0 = __ldg(p.f_off + flat);
    x->slot = s + c;
    pos += x->n;
    return true;
  }
};

// Warp reduction of 16 columns: on return every lane holds, for column
// (lane & 15), the max (or sum) over the 32 lanes.  v is consumed.
template <bool MAX>
__device__ __forceinline__ float reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int half = 8 >> r;
    const bool upper = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float a = v[i], b = v[i + half];
      const float send = upper ? a : b, keep = upper ? b : a;
      const float got = __shfl_xor_sync(0xffffffffu, send, half);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  const float got = __shfl_xor_sync(0xffffffffu, v[0], 16);
  return MAX ? fmaxf(v[0], got) : v[0] + got;
}

// N fp32 columns of this thread's TMEM lane.
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&f)[N]) {
  if constexpr (N == 16) {
    tmem_ld16(taddr, reinterpret_cast<uint32_t (&)[16]>(f));
  } else {
#pragma unroll
    for (int c = 0; c < N; c += 32) tmem_ld32(taddr + c, *reinterpret_cast<uint32_t(*)[32]>(f + c));
  }
}
template <int N>
__device__ __forceinline__ void st_cols(uint32_t taddr, const float (&f)[N]) {
#pragma unroll
  for (int c = 0; c < N; c += 16) tmem_st16(taddr + c, *reinterpret_cast<const uint32_t(*)[16]>(f + c));
}

// Per-column reduction of v[N] over the 128 softmax threads (thread t =
// 32 warp + lane); red is the [4][N] exchange area.  Thread t < N gets the
// result for column t; the others get 0.  The caller passes another barrier
// of the 128 threads before red is written again.
template <int N, bool MAX>
__device__ __forceinline__ float group_reduce(const float (&v)[N], float* red, int warp, int lane) {
#pragma unroll
  for (int g = 0; g < N / 16; ++g) {
    float w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = v[16 * g + i];
    const float r = reduce16<MAX>(w, lane);
    if (lane < 16) red[warp * N + 16 * g + lane] = r;
  }
  named_bar_sync(1, 128);
  const int t = warp * 32 + lane;
  float out = 0.0f;
  if (t < N) {
    const float a = red[t], b = red[N + t], x = red[2 * N + t], y = red[3 * N + t];
    out = MAX ? fmaxf(fmaxf(a, b), fmaxf(x, y)) : (a + b) + (x + y);
  }
  return out;
}

// OR of v over the 128 softmax threads (named barrier `id`); also a barrier.
__device__ __forceinline__ bool group_or(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, %2, 128, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id)
      : "memory");
  return r != 0;
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1)
    k_decode(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ DecParams p) {
  using L = DecLayout<N>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  if ((base - raw) + L::kNeed > static_cast<uint32_t>(L::kSmem)) {
    if (threadIdx.x == 0) atomicOr(p.err, DEVERR_SMEM_ALIGN);
    return;
  }
  const uint32_t sRing = base + L::kOffRing, sQ = base + L::kOffQ, sP = base + L::kOffP;
  uint8_t* small = gbase + L::kOffSmall;
  const uint32_t bars = base + L::kOffSmall;
  const uint32_t b_full = bars, b_empty = b_full + 8 * L::kStages;
  const uint32_t b_qfull = b_empty + 8 * L::kStages, b_qempty = b_qfull + 16;
  const uint32_t b_sfull = b_qempty + 16, b_sfree = b_sfull + 16;
  const uint32_t b_pfull = b_sfree + 16, b_pvdone = b_pfull + 16;  // [2] each: one per P buffer
  const uint32_t b_ofree = b_pvdone + 16, b_drain = b_ofree + 16, b_drain2 = b_drain + 8;
  static_assert(8 * L::kNumBars == L::kSmTmem, "barrier count");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(small + L::kSmTmem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(small + L::kSmAbort);
  float* red = reinterpret_cast<float*>(small + L::kSmRed);
  float* mref = reinterpret_cast<float*>(small + L::kSmMref);
  float* alpha = reinterpret_cast<float*>(small + L::kSmAlpha);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(b_full + 8 * s, 1);
      mbar_init(b_empty + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b_qfull + 8 * i, 1);
      mbar_init(b_qempty + 8 * i, 1);
      mbar_init(b_sfull + 8 * i, 1);
      mbar_init(b_sfree + 8 * i, 4);  // lane 0 of each softmax warp
      mbar_init(b_ofree + 8 * i, 4);
      mbar_init(b_pfull + 8 * i, 4);
      mbar_init(b_pvdone + 8 * i, 1);
    }
    mbar_init(b_drain, 1);
    mbar_init(b_drain2, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
    tmem_relinquish();
  }
  // P rows of query columns past the group stay zero: only rows < G are written
  for (int i = threadIdx.x; i < 2 * L::kQBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(gbase + L::kOffP)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S^T buffers at 0 and N, O^T buffers at 2N and 3N

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int g = 0, issued = 0, ui = 0, q_issued = 0;
      Pieces it;
      it.init(p, blockIdx.x, gridDim.x);
      Unit x;
      for (; !*abort_flag && it.next(p, &x); ++ui) {
        const int qb = ui & 1;
        if (ui >= 2) mbar_wait(b_qempty + 8 * qb, ((ui >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        if (*abort_flag) break;
        mbar_arrive_expect_tx(b_qfull + 8 * qb, L::kQBytes);
        const int qrow = x.q_off * p.Hq + x.hk * p.G;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
          tma_load_2d(sQ + qb * L::kQBytes + h2 * N * 128, &tmQ, b_qfull + 8 * qb, h2 * 64, qrow);
        q_issued = ui + 1;
        for (int j = 0; j < x.n; ++j, ++g) {
          const int st = g % L::kStages;
          if (g >= L::kStages) mbar_wait(b_empty + 8 * st, ((g / L::kStages) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (*abort_flag) break;
          const int e = x.e0 + j;
          const long long ri = (e < x.np) ? bsm_idx(static_cast<long long>(x.p0) + e, p.nP, p.err)
                                          : p.nP + bsm_idx(static_cast<long long>(x.f0) + (e - x.np), p.nF, p.err);
          const uint32_t dst = sRing + st * kStageBytes;
          mbar_arrive_expect_tx(b_full + 8 * st, kStageBytes);
          for (int c = 0; c < p.chunks; ++c) {
            int r = __ldg(p.remap + ri * p.chunks + c);
            if (r < 0) r = p.oob_row;  // past the sequence: rows beyond the cache read as zeros
            const uint32_t off = static_cast<uint32_t>(c * p.chunk_rows * 128);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              tma_load_2d(dst + h2 * 16384 + off, &tmK, b_full + 8 * st, x.hk * D + h2 * 64, r);
              tma_load_2d(dst + kTileBytes + h2 * 16384 + off, &tmV, b_full + 8 * st, x.hk * D + h2 * 64, r);
            }
          }
          issued = g + 1;
        }
      }
      if (*abort_flag) {
        // let copies already started land before the CTA exits
        for (int v = (issued > L::kStages ? issued - L::kStages : 0); v < issued; ++v)
          mbar_wait_drain(b_full + 8 * (v % L::kStages), (v / L::kStages) & 1, kWaitTimeoutNs);
        for (int v = (q_issued > 2 ? q_issued - 2 : 0); v < q_issued; ++v)
          mbar_wait_drain(b_qfull + 8 * (v & 1), (v >> 1) & 1, kWaitTimeoutNs);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ S^T issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, N, 0);  // K (128 keys) x Q (N), both K-major
      const uint64_t dK0 = sdesc_sw128(sRing, 16, 1024);
      const uint64_t dQ0 = sdesc_sw128(sQ, 16, 1024);
      int g = 0, ui = 0;
      Pieces it;
      it.init(p, blockIdx.x, gridDim.x);
      Unit x;
      for (; !*abort_flag && it.next(p, &x); ++ui) {
        const int n = x.n, qb = ui & 1;
        mbar_wait(b_qfull + 8 * qb, (ui >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        const uint64_t dQ = dQ0 + static_cast<uint64_t>((qb * L::kQBytes) >> 4);
        for (int j = 0; j < n; ++j, ++g) {
          const int st = g % L::kStages, sb = g & 1;
          mbar_wait(b_full + 8 * st, (g / L::kStages) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (g >= 2) mbar_wait(b_sfree + 8 * sb, ((g >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (*abort_flag) break;
          tc_fence_after();
          const uint64_t dK = dK0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t offK = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            const uint32_t offQ = ((kk >> 2) * (N * 128) + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tmem + N * sb, dK + offK, dQ + offQ, idS, kk > 0);
          }
          umma_commit(b_sfull + 8 * sb);
        }
        // the piece's Q buffer is free once its last S^T completes
        umma_commit(b_qempty + 8 * qb);
      }
      // every MMA issued above completes before TMEM is released
      umma_commit(b_drain);
      mbar_wait_drain(b_drain, 0, kWaitTimeoutNs);
    }
  } else if (warp == kWarpPV) {
    // ------------------------------------------------------------ P V issuer
    // Issued as soon as P lands: it does not wait for the next K tile.
    if (lane == 0) {
      constexpr uint32_t idO = idesc_bf16_f32(128, N, 0) | (1u << 15);  // V^T (MN-major) x P (K-major)
      const uint64_t dV0 = sdesc_sw128(sRing + kTileBytes, 16384, 1024);
      const uint64_t dP0 = sdesc_sw128(sP, 16, 1024);
      int g = 0, ui = 0;
      Pieces it;
      it.init(p, blockIdx.x, gridDim.x);
      Unit x;
      for (; !*abort_flag && it.next(p, &x); ++ui) {
        const int n = x.n, ob = ui & 1;
        // the piece's first P V overwrites its O^T buffer: the epilogue of the
        // piece two before must have read it
        if (ui >= 2) mbar_wait(b_ofree + 8 * ob, ((ui >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        for (int j = 0; j < n; ++j, ++g) {
          const int st = g % L::kStages, pb = g & 1;
          mbar_wait(b_pfull + 8 * pb, (g >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
          if (*abort_flag) break;
          tc_fence_after();
          const uint64_t dV = dV0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
          const uint64_t dP = dP0 + static_cast<uint64_t>((pb * L::kQBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t offP = ((kk >> 2) * (N * 128) + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tmem + 2 * N + N * ob, dV + static_cast<uint64_t>((kk * 2048) >> 4), dP + offP, idO,
                         (j > 0 || kk > 0) ? 1u : 0u);
          }
          // the stage (its K was read by S^T, which completed before P was written) and P are free
          umma_commit(b_empty + 8 * st);
          umma_commit(b_pvdone + 8 * pb);
        }
      }
      umma_commit(b_drain2);
      mbar_wait_drain(b_drain2, 0, kWaitTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // thread t: key t of each K tile, and head dimension t of O^T.  Every
    // decision to stop is taken by all 128 threads together (an OR over a
    // barrier), so that none is left waiting at a named barrier.
    const int t = threadIdx.x;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int g = 0, ui = 0;
    bool stop = false;
    Pieces it;
    it.init(p, blockIdx.x, gridDim.x);
    Unit x;
    for (; !stop && it.next(p, &x); ++ui) {
      const int ob = ui & 1;
      float l_part[N];
#pragma unroll
      for (int c = 0; c < N; ++c) l_part[c] = 0.0f;
      if (t < N) mref[t] = kNoMax;
      named_bar_sync(1, 128);
      for (int j = 0; j < x.n; ++j, ++g) {
        const int sb = g & 1, st = g % L::kStages;
        const int e = x.e0 + j;
        const bool partial = e < x.np;
        const long long ep = partial ? bsm_idx(static_cast<long long>(x.p0) + e, p.nP, p.err)
                                     : bsm_idx(static_cast<long long>(x.f0) + (e - x.np), p.nF, p.err);
        const int lt = partial ? __ldg(p.p_idx + ep) : __ldg(p.f_idx + ep);
        // row 0 of the tile is the sequence's query row (one query per sequence)
        const uint32_t word = partial ? __ldg(p.payload + ep * (kTile * kPayloadWords) + (t >> 5)) : ~0u;
        const int kpos = lt * kTile + t;
        const bool vis = ((word >> (t & 31)) & 1u) && kpos < x.k_len;
        bool ok = mbar_wait(b_sfull + 8 * sb, (g >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
        tc_fence_after();
        float s[N];
        ld_cols<N>(lane_addr + N * sb, s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_sfree + 8 * sb);
        if (p.flags) {
          // softcap(scale * s), then ALiBi slope * (k - q) with the query at k_len - 1
          const float dk = static_cast<float>(kpos - (x.k_len - 1));
#pragma unroll
          for (int c = 0; c < N; ++c) {
            float z = (p.flags & FA_MOD_SOFTCAP) ? p.cap_log2 * tanh_exp2(s[c] * p.y_scale) : s[c] * p.scale_log2;
            if ((p.flags & FA_MOD_ALIBI) && c < p.G) z += p.slopes_l2[x.hk * p.G + c] * dk;
            s[c] = (vis && c < p.G) ? z : -INFINITY;
          }
        } else {
#pragma unroll
          for (int c = 0; c < N; ++c) s[c] = (vis && c < p.G) ? s[c] * p.scale_log2 : -INFINITY;
        }
        const float tmax = group_reduce<N, true>(s, red, warp, lane);
        // reference max per column: raised when a score exceeds it by more than 2^8
        bool need = false;
        if (t < N) {
          const float mo = mref[t];
          need = tmax > mo + kRescaleLog2;
          const float mn = need ? tmax : mo;
          alpha[t] = need ? exp2f(mo - mn) : 1.0f;
          mref[t] = mn;
        }
        // P buffer g & 1 is free once the P V of step g - 2 has completed
        const int pb = g & 1;
        if (g >= 2) ok = mbar_wait(b_pvdone + 8 * pb, ((g >> 1) - 1) & 1, abort_flag, p.err, kWaitTimeoutNs) && ok;
        // one barrier in the common case: stop and rescale are both rare
        bool any = false;
        if (group_or(2, need || !ok || *abort_flag)) {
          stop = group_or(2, !ok || *abort_flag);
          if (stop) break;
          any = true;  // no thread had a failed wait, so some column's max rose
        }
        if (any) {
#pragma unroll
          for (int c = 0; c < N; ++c) l_part[c] *= alpha[c];
          if (j > 0) {
            // O^T is rescaled between the P V of step g - 1 and that of step g
            ok = mbar_wait(b_pvdone + 8 * (pb ^ 1), ((g - 1) >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
            stop = group_or(2, !ok || *abort_flag);
            if (stop) break;
            tc_fence_after();
            float o[N];
            ld_cols<N>(lane_addr + 2 * N + N * ob, o);
#pragma unroll
            for (int c = 0; c < N; ++c) o[c] *= alpha[c];
            st_cols<N>(lane_addr + 2 * N + N * ob, o);
            tmem_st_wait();
          }
        }
        // P (bf16) into the K-major P buffer: row c, column (key) t; rows of
        // columns past the group stay zero
        const uint32_t prow = sP + pb * L::kQBytes + (t >> 6) * (N * 128);
        const uint32_t chunk = static_cast<uint32_t>((t & 63) >> 3), byte = static_cast<uint32_t>((t & 7) * 2);
#pragma unroll
        for (int c = 0; c < N; ++c) {
          if (c < p.G) {
            const float pv = exp2f(s[c] - mref[c]);
            l_part[c] += pv;
            const __nv_bfloat16 hv = __float2bfloat16_rn(pv);
            const uint32_t a = prow + c * 128 + ((chunk ^ static_cast<uint32_t>(c & 7)) << 4) + byte;
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(*reinterpret_cast<const uint16_t*>(&hv)) : "memory");
          }
        }
        // keys past the sequence: their V rows (unused cache memory) become
        // zeros, so that 0 * V stays 0 in the product
        if (kpos >= x.k_len) {
          uint8_t* vrow = gbase + L::kOffRing + st * kStageBytes + kTileBytes + t * 128;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int i = 0; i < 8; ++i) reinterpret_cast<uint4*>(vrow + h2 * 16384)[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_pfull + 8 * pb);
      }
      if (stop) break;
      // piece epilogue: O^T and the column sums
      const bool ok = mbar_wait(b_pvdone + 8 * ((g - 1) & 1), ((g - 1) >> 1) & 1, abort_flag, p.err, kWaitTimeoutNs);
      stop = group_or(2, !ok || *abort_flag);
      if (stop) break;
      tc_fence_after();
      float o[N];
      ld_cols<N>(lane_addr + 2 * N + N * ob, o);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_ofree + 8 * ob);
      const float lsum = group_reduce<N, false>(l_part, red, warp, lane);
      float* po = p.part_o + x.slot * p.G * D;
#pragma unroll
      for (int c = 0; c < N; ++c)
        if (c < p.G) po[c * D + t] = o[c];
      if (t < p.G) {
        p.part_ml[x.slot * 2 * p.G + t] = mref[t];
        p.part_ml[x.slot * 2 * p.G + p.G + t] = lsum;
      }
      named_bar_sync(1, 128);  // mref is reset for the next piece only after every thread read it
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// ------------------------------------------------------------ prep
struct PrepParams {
  const int32_t* seq;
  const int32_t* p_off;
  const int32_t* f_off;
  const int32_t* p_idx;
  const int32_t* f_idx;
  const int32_t* entry_row;  // [P] flat plan row of each partial entry
  const int32_t* cu_q_rows;  // [B+1] plan row prefix of the sequences
  const int32_t* page_table;
  int32_t* remap;
  int32_t* cu_rows;  // [Hmask*B + 1]: prefix of the rows' entry counts
  uint32_t* err;
  long long nP, nF, num_pages;
  int B, Hmask, rows, pages_per_seq, page_size, chunks, chunk_rows;
};

// K tile entries of (mask head, sequence) row r = hm * B + b.
__device__ __forceinline__ int row_entries(const PrepParams& p, int r, int* p0, int* np, int* f0, int* b_out) {
  const int hm = r / p.B, b = r % p.B;
  const int32_t* sq = p.seq + 8 * b;
  *b_out = b;
  if (__ldg(sq + 5) == 0) {  // no query row: nothing to compute
    *p0 = *np = *f0 = 0;
    return 0;
  }
  const long long flat = static_cast<long long>(hm) * p.rows + __ldg(sq + 4);
  *p0 = __ldg(p.p_off + flat);
  *np = __ldg(p.p_off + flat + 1) - *p0;
  *f0 = __ldg(p.f_off + flat);
  return *np + (__ldg(p.f_off + flat + 1) - *f0);
}

// Largest i in [lo, hi) with a[i] <= x (a ascending, a[lo] <= x).
__device__ __forceinline__ int last_le(const int32_t* a, int lo, int hi, long long x) {
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Block 0: entries per row, exclusive scan into cu_rows.  Every other block: the page conversion of 256 list entries
// (partial entries first, then full ones), one thread each.
__global__ void __launch_bounds__(256) k_decode_prep(PrepParams p) {
  if (blockIdx.x > 0) {
    const long long e = static_cast<long long>(blockIdx.x - 1) * blockDim.x + threadIdx.x;
    if (e >= p.nP + p.nF) return;
    const bool partial = e < p.nP;
    long long flat;
    int lt;
    if (partial) {
      flat = __ldg(p.entry_row + e);
      lt = __ldg(p.p_idx + e);
    } else {
      const long long ef = e - p.nP;
      flat = last_le(p.f_off, 0, p.Hmask * p.rows, ef);  // the last row starting at or before ef holds it
      lt = __ldg(p.f_idx + ef);
    }
    const int row = static_cast<int>(flat % p.rows);
    const int b = last_le(p.cu_q_rows, 0, p.B, row);
    const int k_len = __ldg(p.seq + 8 * b + 3);
    const int32_t* table = p.page_table + static_cast<long long>(b) * p.pages_per_seq;
    int32_t* out = p.remap + e * p.chunks;
    for (int c = 0; c < p.chunks; ++c) {
      const long long lrow = static_cast<long long>(lt) * kTile + static_cast<long long>(c) * p.chunk_rows;
      int32_t phys = -1;
      if (lrow < k_len) {
        const long long pg = lrow / p.page_size;
        const int page = (pg < p.pages_per_seq) ? __ldg(table + pg) : -1;
        if (page < 0 || page >= p.num_pages)
          atomicOr(p.err, DEVERR_PAGE);
        else
          phys = static_cast<int32_t>(static_cast<long long>(page) * p.page_size + lrow % p.page_size);
      }
      out[c] = phys;
    }
    return;
  }
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_carry;
  const int R = p.B * p.Hmask;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < R; base += blockDim.x) {
    const int r = base + threadIdx.x;
    int cnt = 0;
    if (r < R) {
      int p0, np, f0, b;
      cnt = row_entries(p, r, &p0, &np, &f0, &b);
    }
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int v = lane < nw ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      s_warp[lane] = v;
    }
    __syncthreads();
    if (r < R) p.cu_rows[r] = s_carry + (wid ? s_warp[wid - 1] : 0) + x - cnt;
    __syncthreads();
    if (threadIdx.x == 0) s_carry += s_warp[nw - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) p.cu_rows[R] = s_carry;
}

// ------------------------------------------------------------ combine
struct CombineParams {
  const float* part_o;
  const float* part_ml;
  const int32_t* cu_rows;
  __nv_bfloat16* o;
  float* lse;
  int B, Hq, Hk, Hmask, G, gy, total_q, R, C;
};

// The CTA of k_decode (C of them over W tiles) whose range holds tile x.
__device__ __forceinline__ int cta_of(long long x, long long W, int C) {
  long long c = x * C / W;
  while (c + 1 < C && W * (c + 1) / C <= x) ++c;
  while (c > 0 && W * c / C > x) --c;
  return static_cast<int>(c);
}

// One warp per (query row, head): the pieces of its segment are those of
// the CTAs whose ranges meet the segment, in slots s + c.
__global__ void __launch_bounds__(256) k_decode_combine(CombineParams p) {
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<long long>(p.total_q) * p.Hq) return;
  const int qr = static_cast<int>(wid / p.Hq), h = static_cast<int>(wid % p.Hq);
  const int b = qr;  // one query row per sequence
  const int hm = (p.Hmask == 1) ? 0 : h;
  const int gi = (p.Hmask == 1) ? h / p.G : 0, c = h % p.G;
  const long long sg = static_cast<long long>(hm * p.B + b) * p.gy + gi;
  const long long x0 = seg_start(p.cu_rows, p.R, p.gy, sg), x1 = seg_start(p.cu_rows, p.R, p.gy, sg + 1);
  const long long W = static_cast<long long>(p.gy) * __ldg(p.cu_rows + p.R);
  const int c0 = (x1 > x0) ? cta_of(x0, W, p.C) : 0, c1 = (x1 > x0) ? cta_of(x1 - 1, W, p.C) : -1;
  float M = -INFINITY;
  for (int k = c0; k <= c1; ++k) {
    const long long slot = sg + k;
    const float l = __ldg(p.part_ml + slot * 2 * p.G + p.G + c);
    if (l > 0.0f) M = fmaxf(M, __ldg(p.part_ml + slot * 2 * p.G + c));
  }
  float Lsum = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int k = c0; k <= c1; ++k) {
    const long long slot = sg + k;
    const float l = __ldg(p.part_ml + slot * 2 * p.G + p.G + c);
    if (!(l > 0.0f)) continue;
    const float w = exp2f(__ldg(p.part_ml + slot * 2 * p.G + c) - M);
    Lsum += w * l;
    const float4 v = __ldg(reinterpret_cast<const float4*>(p.part_o + (slot * p.G + c) * D) + lane);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
  }
  const float inv = (Lsum > 0.0f) ? 1.0f / Lsum : 0.0f;
  const uint32_t lo = pack_bf16x2(acc.x * inv, acc.y * inv), hi = pack_bf16x2(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(p.o + (static_cast<long long>(qr) * p.Hq + h) * D)[lane] = make_uint2(lo, hi);
  if (lane == 0 && p.lse != nullptr)
    p.lse[static_cast<long long>(h) * p.total_q + qr] = (Lsum > 0.0f) ? (M + __log2f(Lsum)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn_dec() {
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

// 2-D view [rows, cols] of a bf16 tensor (row pitch cols * 2 bytes), box 64 x box_rows, 128-byte swizzle.
bool make_map_dec(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, uint32_t box_rows) {
  auto fn = encode_fn_dec();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
cudaError_t launch_decode_n(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                            const DecParams& p, int grid, cudaStream_t st) {
  using L = DecLayout<N>;
  cudaError_t e = cudaFuncSetAttribute(k_decode<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  k_decode<N><<<grid, kThreads, L::kSmem, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

size_t decode_workspace_bytes(const DecodeLaunch& a, DecodeSizes* z) {
  const fa_plan* pl = a.plan;
  const Geometry& g = pl->geom;
  DecodeSizes s{};
  s.G = (pl->Hmask == 1) ? g.heads_q / g.heads_k : 1;
  s.gy = (pl->Hmask == 1) ? g.heads_k : 1;
  s.chunk_rows = a.page_size < kTile ? a.page_size : kTile;
  s.chunks = kTile / s.chunk_rows;
  const long long entries = pl->P + pl->F;
  const long long work = entries * s.gy;  // K/V tiles over every segment
  // one persistent CTA per SM, fewer when there are fewer tiles
  s.C = static_cast<int>(work < a.num_sms ? (work > 0 ? work : 1) : a.num_sms);
  const long long rows = static_cast<long long>(pl->Hmask) * g.batch;
  s.slots = rows * s.gy + s.C;  // piece slots s + c
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  size_t off = 0;
  s.off_remap = off;
  off += al(4ull * static_cast<size_t>(entries > 0 ? entries : 1) * s.chunks);
  s.off_cu = off;
  off += al(4ull * static_cast<size_t>(rows + 1));
  s.off_part_o = off;
  off += al(4ull * static_cast<size_t>(s.slots) * s.G * D);
  s.off_part_ml = off;
  off += al(8ull * static_cast<size_t>(s.slots) * s.G);
  s.bytes = off;
  *z = s;
  return off;
}

cudaError_t launch_decode(const DecodeLaunch& a, const DecodeSizes& s, void* ws, cudaStream_t st,
                          const char** why) {
  const fa_plan* pl = a.plan;
  const Geometry& g = pl->geom;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* remap = reinterpret_cast<int32_t*>(w + s.off_remap);
  int32_t* cu = reinterpret_cast<int32_t*>(w + s.off_cu);
  float* part_o = reinterpret_cast<float*>(w + s.off_part_o);
  float* part_ml = reinterpret_cast<float*>(w + s.off_part_ml);
  uint32_t* err = fwd_error_word();
  if (err == nullptr) {
    *why = "device error word not found";
    return cudaErrorInvalidValue;
  }

  PrepParams pp{};
  pp.seq = pl->seq_desc;
  pp.p_off = pl->p_off;
  pp.f_off = pl->f_off;
  pp.p_idx = pl->p_idx;
  pp.f_idx = pl->f_idx;
  pp.entry_row = pl->entry_row;
  pp.cu_q_rows = pl->cu_q_rows;
  pp.page_table = a.page_table;
  pp.remap = remap;
  pp.cu_rows = cu;
  pp.err = err;
  pp.nP = pl->P;
  pp.nF = pl->F;
  pp.num_pages = a.num_pages;
  pp.B = g.batch;
  pp.Hmask = pl->Hmask;
  pp.rows = static_cast<int>(pl->rows);
  pp.pages_per_seq = a.pages_per_seq;
  pp.page_size = a.page_size;
  pp.chunks = s.chunks;
  pp.chunk_rows = s.chunk_rows;
  const long long entries = pl->P + pl->F;
  k_decode_prep<<<static_cast<unsigned>(1 + (entries + 255) / 256), 256, 0, st>>>(pp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    *why = "decode prep launch failed";
    return e;
  }

  const int N = (s.G <= 16) ? 16 : (s.G <= 32 ? 32 : 64);
  const int64_t rows_q = g.total_q;
  const int64_t cache_rows = a.num_pages * static_cast<int64_t>(a.page_size);
  CUtensorMap mq, mk, mv;
  if (!make_map_dec(&mq, a.q, rows_q * g.heads_q, D, static_cast<uint32_t>(N)) ||
      !make_map_dec(&mk, a.k_cache, cache_rows, static_cast<int64_t>(g.heads_k) * D, static_cast<uint32_t>(s.chunk_rows)) ||
      !make_map_dec(&mv, a.v_cache, cache_rows, static_cast<int64_t>(g.heads_k) * D, static_cast<uint32_t>(s.chunk_rows))) {
    *why = "cuTensorMapEncodeTiled failed (pointer alignment or driver entry point)";
    return cudaErrorInvalidValue;
  }
  DecParams p{};
  p.seq = pl->seq_desc;
  p.p_off = pl->p_off;
  p.f_off = pl->f_off;
  p.p_idx = pl->p_idx;
  p.f_idx = pl->f_idx;
  p.payload = pl->payload;
  p.remap = remap;
  p.cu_rows = cu;
  p.part_o = part_o;
  p.part_ml = part_ml;
  p.err = err;
  p.B = g.batch;
  p.Hq = g.heads_q;
  p.Hk = g.heads_k;
  p.Hmask = pl->Hmask;
  p.rows = static_cast<int>(pl->rows);
  p.G = s.G;
  p.gy = s.gy;
  p.chunks = s.chunks;
  p.chunk_rows = s.chunk_rows;
  p.oob_row = static_cast<int>(cache_rows);
  p.nP = pl->P;
  p.nF = pl->F;
  p.R = pl->Hmask * g.batch;
  p.scale_log2 = a.scale * kLog2e;
  p.flags = a.flags;
  p.y_scale = (a.flags & FA_MOD_SOFTCAP) ? a.scale / a.softcap : 0.0f;
  p.cap_log2 = a.softcap * kLog2e;
  if (a.flags & FA_MOD_ALIBI)
    for (int h = 0; h < g.heads_q; ++h) p.slopes_l2[h] = a.slopes[h] * kLog2e;
  const int grid = s.C;
  if (N == 16)
    e = launch_decode_n<16>(mq, mk, mv, p, grid, st);
  else if (N == 32)
    e = launch_decode_n<32>(mq, mk, mv, p, grid, st);
  else
    e = launch_decode_n<64>(mq, mk, mv, p, grid, st);
  if (e != cudaSuccess) {
    *why = "decode kernel launch failed";
    return e;
  }

  CombineParams cp{};
  cp.part_o = part_o;
  cp.part_ml = part_ml;
  cp.cu_rows = cu;
  cp.R = pl->Hmask * g.batch;
  cp.C = s.C;
  cp.o = static_cast<__nv_bfloat16*>(a.o);
  cp.lse = a.lse;
  cp.B = g.batch;
  cp.Hq = g.heads_q;
  cp.Hk = g.heads_k;
  cp.Hmask = pl->Hmask;
  cp.G = s.G;
  cp.gy = s.gy;
  cp.total_q = static_cast<int>(rows_q);
  const long long warps = rows_q * g.heads_q;
  if (warps > 0) {
    k_decode_combine<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, st>>>(cp);
    e = cudaGetLastError();
    if (e != cudaSuccess) *why = "decode combine launch failed";
  }
  return e;
}

}  // namespace bsm
