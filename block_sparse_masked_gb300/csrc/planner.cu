// planner.cu -- GPU mask planner: mask -> MaskPlan.
//
// Stages follow "Flex Attention Mask Plan Design" (cuDNN frontend docs):
//   k_geometry         §4.2 compact row prefixes + §3.2 prefix validation,
//                      sequence descriptors of §4.8
//   k_classify_*       §4.3 Q2K classification into visible/full bitsets and
//                      per-row partial/full counts; endpoints validated and
//                      clamped (§3.3); block masks use the logical-block
//                      expansion E(M) of "Decoupling Logical Masks from GPU
//                      Execution for Dynamic Block-Sparse Attention" §2
//   k_scan_header      §4.5 exclusive scans and the 8-value allocation header
//   k_materialize      §4.6 independent partial / full CSR index lists
//   k_payload          §5 packed predicate payload, bit-packed with warp ballots
//   k_sched_*          §4.8 forward task order by bounded counting
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace bsm {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Set bits [lo, hi] (tile indices, inclusive) that fall into word w.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi, int w) {
  const int base = w * 32;
  const int L = max(lo, base), H = min(hi, base + 31);
  if (L > H) return 0u;
  const uint64_t m = ((uint64_t(2) << (H - base)) - 1) & ~((uint64_t(1) << (L - base)) - 1);
  return static_cast<uint32_t>(m);
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ long long block_excl_scan(long long v, long long* total) {
  __shared__ long long s_warp[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    long long s = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(kFull, s, o);
      if (lane >= o) s += y;
    }
    s_warp[lane] = s;
  }
  __syncthreads();
  const long long warp_prefix = wid ? s_warp[wid - 1] : 0;
  *total = s_warp[31];
  __syncthreads();
  return warp_prefix + x - v;
}

// ------------------------------------------------------------ geometry
struct GeoParams {
  int layout, B, Sq, Sk, total_q, total_k;
  const int32_t* cu_q;
  const int32_t* cu_k;
  int32_t* cu_rows;
  int32_t* seq;
  int32_t* row_batch;
  uint32_t* err;
  int rows_ub;
};

__global__ void __launch_bounds__(1024) k_geometry(GeoParams g) {
  if (threadIdx.x == 0) *g.err = 0;  // the build's error word starts here
  __syncthreads();
  long long carry = 0;
  for (int base = 0; base < g.B; base += 1024) {
    const int b = base + threadIdx.x;
    int q_off = 0, k_off = 0, q_len = 0, k_len = 0;
    if (b < g.B) {
      if (g.layout == FA_LAYOUT_BSHD) {
        q_off = b * g.Sq;
        k_off = b * g.Sk;
        q_len = g.Sq;
        k_len = g.Sk;
      } else {
        const int a = g.cu_q[b], e = g.cu_q[b + 1];
        const int c = g.cu_k[b], f = g.cu_k[b + 1];
        bool bad = false;
        if (b == 0 && (a != 0 || c != 0)) bad = true;
        if (b == g.B - 1 && (e != g.total_q || f != g.total_k)) bad = true;
        if (e < a || f < c) bad = true;
        if (e - a > g.Sq || f - c > g.Sk) bad = true;
        if (a < 0 || c < 0 || e > g.total_q || f > g.total_k) bad = true;
        if (bad) atomicOr(g.err, PLANERR_SEQLENS);
        // clamp so that later stages index safely before the error is read
        q_off = min(max(a, 0), g.total_q);
        k_off = min(max(c, 0), g.total_k);
        q_len = min(max(e - a, 0), min(g.Sq, g.total_q - q_off));
        k_len = min(max(f - c, 0), min(g.Sk, g.total_k - k_off));
      }
    }
    const int nrows = (b < g.B) ? cdiv(q_len, kTile) : 0;
    long long tot;
    const long long begin = carry + block_excl_scan(nrows, &tot);
    if (b < g.B) {
      int32_t* s = g.seq + 8 * b;
      s[0] = q_off;
      s[1] = k_off;
      s[2] = q_len;
      s[3] = k_len;
      s[4] = static_cast<int32_t>(begin);
      s[5] = nrows;
      s[6] = cdiv(k_len, kTile);
      s[7] = 0;
      g.cu_rows[b] = static_cast<int32_t>(begin);
    }
    carry += tot;
  }
  if (threadIdx.x == 0) g.cu_rows[g.B] = static_cast<int32_t>(carry);
  __syncthreads();
  for (int b = threadIdx.x; b < g.B; b += 1024) {
    const int begin = g.seq[8 * b + 4], n = g.seq[8 * b + 5];
    for (int r = 0; r < n && begin + r < g.rows_ub; ++r) g.row_batch[begin + r] = b;
  }
}

// ------------------------------------------------------------ classify
struct ClassifyParams {
  const int32_t* seq;
  const int32_t* row_batch;
  const int32_t* cu_rows;
  int B;
  // intervals
  const int32_t* mask_func;
  int nfunc, total_q;
  // blocks
  const uint8_t* block_mask;
  int block_q, block_kv, nbq, nbk;
  // outputs
  uint32_t* vis_bits;
  uint32_t* full_bits;
  int32_t* p_cnt;
  int32_t* f_cnt;
  uint32_t* err;
  int rows_ub, words;
};

// One CTA per (Q plan row, mask head); thread t owns Q row t of the tile.
// Per row, each K tile is "touched" if a non-empty interval intersects it and
// "covered" if one maximal run of merged intervals contains the whole tile;
// visible = OR over valid rows of touched, full = AND over all 128 rows of
// covered (rows past the sample's q_len cover nothing, so a Q tail is never full).
__global__ void __launch_bounds__(128) k_classify_intervals(ClassifyParams p) {
  const int row = blockIdx.x, hm = blockIdx.y, t = threadIdx.x;
  const int lane = t & 31, wid = t >> 5;
  const long long ws_row = static_cast<long long>(hm) * p.rows_ub + row;
  __shared__ uint32_t s_v[4], s_f[4];
  const int rows_total = p.cu_rows[p.B];
  if (row >= rows_total) {
    for (int w = t; w < p.words; w += 128) {
      p.vis_bits[ws_row * p.words + w] = 0;
      p.full_bits[ws_row * p.words + w] = 0;
    }
    if (t == 0) {
      p.p_cnt[ws_row] = 0;
      p.f_cnt[ws_row] = 0;
    }
    return;
  }
  const int b = p.row_batch[row];
  const int32_t* s = p.seq + 8 * b;
  const int q_off = s[0], q_len = s[2], k_len = s[3], row_begin = s[4];
  const int q_local = (row - row_begin) * kTile + t;
  const bool valid = q_local < q_len;
  const int32_t* F = p.mask_func + static_cast<long long>(hm) * p.nfunc * p.total_q + q_off + q_local;
  const long long fstride = p.total_q;

  // validation: 0 <= F0 <= ... <= F(n-1) <= k_len
  if (valid) {
    int prev = 0;
    bool bad = false;
    for (int f = 0; f < p.nfunc; ++f) {
      const int e = __ldg(F + f * fstride);
      if (e < prev || e > k_len) bad = true;  // e < 0 is caught by e < prev (prev starts at 0)
      prev = max(prev, e);
    }
    if (bad) atomicOr(p.err, PLANERR_MASK);
  }

  int pc = 0, fc = 0;
  for (int w = 0; w < p.words; ++w) {
    uint32_t vrow = 0, frow = 0;
    if (valid) {
      // clamped, monotone endpoints (equal to the input when it is valid)
      int prev = min(max(__ldg(F), 0), k_len);
      int ma = 0, mb = prev;  // current merged run [ma, mb)
      if (prev > 0) vrow |= range_bits(0, (prev - 1) / kTile, w);
      for (int i = 1; i + 1 < p.nfunc; i += 2) {
        const int a = min(max(__ldg(F + i * fstride), prev), k_len);
        const int e = min(max(__ldg(F + (i + 1) * fstride), a), k_len);
        prev = e;
        if (a < e) {
          vrow |= range_bits(a / kTile, (e - 1) / kTile, w);
          if (a == mb) {
            mb = e;
          } else {
            if (mb > ma) frow |= range_bits(cdiv(ma, kTile), mb / kTile - 1, w);
            ma = a;
            mb = e;
          }
        }
      }
      if (mb > ma) frow |= range_bits(cdiv(ma, kTile), mb / kTile - 1, w);
    }
    const uint32_t wv = __reduce_or_sync(kFull, vrow);
    const uint32_t wf = __reduce_and_sync(kFull, frow);
    if (lane == 0) {
      s_v[wid] = wv;
      s_f[wid] = wf;
    }
    __syncthreads();
    if (t == 0) {
      const uint32_t v = s_v[0] | s_v[1] | s_v[2] | s_v[3];
      const uint32_t f = s_f[0] & s_f[1] & s_f[2] & s_f[3];
      p.vis_bits[ws_row * p.words + w] = v;
      p.full_bits[ws_row * p.words + w] = f;
      pc += __popc(v & ~f);
      fc += __popc(f);
    }
    __syncthreads();
  }
  if (t == 0) {
    p.p_cnt[ws_row] = pc;
    p.f_cnt[ws_row] = fc;
  }
}

// Block masks (fixed length): thread per K tile.  Tile (i, j) touches the
// logical blocks [r0, r1] x [c0, c1] that overlap its in-bounds part; it is
// visible if any is active and full if all are and the tile has no Q/K tail.
// Words are bit-packed with warp ballots.
__global__ void __launch_bounds__(256) k_classify_blocks(ClassifyParams p) {
  const int row = blockIdx.x, hm = blockIdx.y, t = threadIdx.x;
  const int lane = t & 31;
  const long long ws_row = static_cast<long long>(hm) * p.rows_ub + row;
  __shared__ int s_pc, s_fc;
  if (t == 0) {
    s_pc = 0;
    s_fc = 0;
  }
  __syncthreads();
  const int b = p.row_batch[row];
  const int32_t* s = p.seq + 8 * b;
  const int q_len = s[2], k_len = s[3], row_begin = s[4], nk = s[6];
  const int q0 = (row - row_begin) * kTile, q1 = min(q0 + kTile, q_len);
  const bool qtail = (q1 - q0) < kTile;
  const int r0 = q0 / p.block_q, r1 = (q1 - 1) / p.block_q;
  const uint8_t* M = p.block_mask + static_cast<long long>(hm) * p.nbq * p.nbk;
  const int nwords_used = p.words * 32;
  for (int j0 = 0; j0 < nwords_used; j0 += 256) {
    const int j = j0 + t;
    bool vis = false, full = false;
    if (j < nk) {
      const int k0 = j * kTile, k1 = min(k0 + kTile, k_len);
      const bool ktail = (k1 - k0) < kTile;
      const int c0 = k0 / p.block_kv, c1 = (k1 - 1) / p.block_kv;
      bool any = false, all = true;
      for (int r = r0; r <= r1; ++r) {
        const uint8_t* Mr = M + static_cast<long long>(r) * p.nbk;
        for (int c = c0; c <= c1; ++c) {
          const bool x = __ldg(Mr + c) != 0;
          any |= x;
          all &= x;
        }
      }
      vis = any;
      full = any && all && !qtail && !ktail;
    }
    const uint32_t vb = __ballot_sync(kFull, vis);
    const uint32_t fb = __ballot_sync(kFull, full);
    const int w = j >> 5;
    if (lane == 0 && w < p.words) {
      p.vis_bits[ws_row * p.words + w] = vb;
      p.full_bits[ws_row * p.words + w] = fb;
      atomicAdd(&s_pc, __popc(vb & ~fb));
      atomicAdd(&s_fc, __popc(fb));
    }
  }
  __syncthreads();
  if (t == 0) {
    p.p_cnt[ws_row] = s_pc;
    p.f_cnt[ws_row] = s_fc;
  }
}

// ------------------------------------------------------------ scan + header
struct ScanParams {
  const int32_t* p_cnt;
  const int32_t* f_cnt;
  const int32_t* cu_rows;
  int32_t* p_off;
  int32_t* f_off;
  long long* header;
  const uint32_t* err;
  int B, Hmask, rows_ub;
};

__global__ void __launch_bounds__(1024) k_scan_header(ScanParams p) {
  const int rows = p.cu_rows[p.B];
  const long long n = static_cast<long long>(p.Hmask) * rows;
  long long cp = 0, cf = 0;
  for (long long base = 0; base < n; base += 1024) {
    const long long i = base + threadIdx.x;
    int vp = 0, vf = 0;
    if (i < n) {
      const long long hm = i / rows, r = i % rows;
      vp = p.p_cnt[hm * p.rows_ub + r];
      vf = p.f_cnt[hm * p.rows_ub + r];
    }
    long long tp, tf;
    const long long ep = block_excl_scan(vp, &tp);
    const long long ef = block_excl_scan(vf, &tf);
    if (i < n) {
      p.p_off[i] = static_cast<int32_t>(cp + ep);
      p.f_off[i] = static_cast<int32_t>(cf + ef);
    }
    cp += tp;
    cf += tf;
  }
  if (threadIdx.x == 0) {
    p.p_off[n] = static_cast<int32_t>(cp);
    p.f_off[n] = static_cast<int32_t>(cf);
    uint32_t e = *p.err;
    if (cp > 0x3fffffffLL || cf > 0x3fffffffLL) e |= PLANERR_OVERFLOW;
    p.header[0] = rows;
    p.header[1] = cp;
    p.header[2] = cf;
    p.header[3] = 0;
    p.header[4] = 0;
    p.header[5] = 0;
    p.header[6] = 0;
    p.header[7] = e;
  }
}

// ------------------------------------------------------------ materialize
struct MatParams {
  const uint32_t* vis_bits;
  const uint32_t* full_bits;
  const int32_t* p_off;  // workspace offsets, exact [Hmask*rows+1] layout
  const int32_t* f_off;
  int32_t* p_idx;
  int32_t* f_idx;
  int32_t* entry_row;  // [P]: flat (hm*rows + row) of each partial entry
  int rows, rows_ub, words;
  // exact-size copies into the plan, done by the same launch
  const int32_t* src[6];
  int32_t* dst[6];
  long long count[6];
};

// One warp per (row, mask head): lane w handles bitset word w; ranks come
// from a warp scan of popcounts, so indices come out ascending.
__global__ void __launch_bounds__(32) k_materialize(MatParams p) {
  {
    const long long tid = (static_cast<long long>(blockIdx.y) * gridDim.x + blockIdx.x) * 32 + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * gridDim.y * 32;
#pragma unroll
    for (int a = 0; a < 6; ++a)
      for (long long i = tid; i < p.count[a]; i += nthreads) p.dst[a][i] = p.src[a][i];
  }
  const int row = blockIdx.x, hm = blockIdx.y, lane = threadIdx.x;
  if (row >= p.rows) return;
  const long long flat = static_cast<long long>(hm) * p.rows + row;
  const long long ws_row = static_cast<long long>(hm) * p.rows_ub + row;
  int pbase = p.p_off[flat], fbase = p.f_off[flat];
  for (int w0 = 0; w0 < p.words; w0 += 32) {
    const int w = w0 + lane;
    uint32_t vb = 0, fb = 0;
    if (w < p.words) {
      vb = p.vis_bits[ws_row * p.words + w];
      fb = p.full_bits[ws_row * p.words + w];
    }
    uint32_t pb = vb & ~fb;
    const int np = __popc(pb), nf = __popc(fb);
    int xp = np, xf = nf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yp = __shfl_up_sync(kFull, xp, o), yf = __shfl_up_sync(kFull, xf, o);
      if (lane >= o) {
        xp += yp;
        xf += yf;
      }
    }
    int pp = pbase + xp - np, pf = fbase + xf - nf;
    while (pb) {
      const int bit = __ffs(pb) - 1;
      pb &= pb - 1;
      p.p_idx[pp] = w * 32 + bit;
      p.entry_row[pp] = static_cast<int32_t>(flat);
      ++pp;
    }
    while (fb) {
      const int bit = __ffs(fb) - 1;
      fb &= fb - 1;
      p.f_idx[pf++] = w * 32 + bit;
    }
    pbase += __shfl_sync(kFull, xp, 31);
    fbase += __shfl_sync(kFull, xf, 31);
  }
}

// ------------------------------------------------------------ payload
struct PayloadParams {
  const int32_t* entry_row;
  const int32_t* p_idx;
  const int32_t* row_batch;
  const int32_t* seq;
  uint32_t* payload;
  uint8_t* halves;  // [P] bit s: column half s of the entry has a visible element
  int rows, P;
  // intervals
  const int32_t* mask_func;
  int nfunc, total_q;
  // blocks
  const uint8_t* block_mask;
  int block_q, block_kv, nbq, nbk;
};

template <int KIND>
__device__ __forceinline__ bool visible_at(const PayloadParams& p, int hm, int q_off, int q_local,
                                           int col) {
  if (KIND == MASK_INTERVALS) {
    const int32_t* F = p.mask_func + static_cast<long long>(hm) * p.nfunc * p.total_q + q_off + q_local;
    const long long fs = p.total_q;
    bool in = col < __ldg(F);
    for (int i = 1; i + 1 < p.nfunc; i += 2)
      in |= (col >= __ldg(F + i * fs)) && (col < __ldg(F + (i + 1) * fs));
    return in;
  } else {
    const uint8_t* M = p.block_mask + static_cast<long long>(hm) * p.nbq * p.nbk;
    return __ldg(M + static_cast<long long>(q_local / p.block_q) * p.nbk + col / p.block_kv) != 0;
  }
}

// Interval masks: one CTA (4 warps) per partial entry; warp wi packs rows
// 32*wi .. 32*wi+31.  For each row the 32 lanes test 32 consecutive columns
// and a ballot forms one uint32 word; lane i keeps the 4 words of row i and
// the warp stores 32 rows x 16 bytes contiguously.  With at most kMaxFuncFast
// endpoints per row, lane i loads row i's endpoints once and the warp
// broadcasts them with shuffles; otherwise every lane reads them per row.
constexpr int kMaxFuncFast = 9;

template <bool FAST>
__global__ void __launch_bounds__(128) k_payload_intervals(PayloadParams p) {
  const long long e = blockIdx.x;
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int flat = p.entry_row[e];
  const int hm = flat / p.rows, row = flat % p.rows;
  const int j = p.p_idx[e];
  const int b = p.row_batch[row];
  const int32_t* s = p.seq + 8 * b;
  const int q_off = s[0], q_len = s[2], k_len = s[3], row_begin = s[4];
  const int q0 = (row - row_begin) * kTile;
  const int c0 = j * kTile;
  const int32_t* Fbase = p.mask_func + static_cast<long long>(hm) * p.nfunc * p.total_q + q_off;
  const long long fs = p.total_q;
  int myF[kMaxFuncFast];
  if (FAST) {
    const int q_mine = q0 + wi * 32 + lane;
#pragma unroll
    for (int f = 0; f < kMaxFuncFast; ++f)
      myF[f] = (f < p.nfunc && q_mine < q_len) ? __ldg(Fbase + f * fs + q_mine) : 0;
  }
  uint32_t mine[kPayloadWords] = {0, 0, 0, 0};
  for (int i = 0; i < 32; ++i) {
    const int q_local = q0 + wi * 32 + i;
    if (q_local >= q_len) break;  // uniform: rows past the sample stay 0
    bool in[kPayloadWords];
    if (FAST) {
      int F[kMaxFuncFast];
#pragma unroll
      for (int f = 0; f < kMaxFuncFast; ++f) F[f] = __shfl_sync(kFull, myF[f], i);
#pragma unroll
      for (int wd = 0; wd < kPayloadWords; ++wd) {
        const int col = c0 + wd * 32 + lane;
        bool v = col < F[0];
#pragma unroll
        for (int f = 1; f + 1 < kMaxFuncFast; f += 2)
          if (f + 1 < p.nfunc) v |= (col >= F[f]) && (col < F[f + 1]);
        in[wd] = v && (col < k_len);
      }
    } else {
#pragma unroll
      for (int wd = 0; wd < kPayloadWords; ++wd) {
        const int col = c0 + wd * 32 + lane;
        in[wd] = (col < k_len) && visible_at<MASK_INTERVALS>(p, hm, q_off, q_local, col);
      }
    }
#pragma unroll
    for (int wd = 0; wd < kPayloadWords; ++wd) {
      const uint32_t word = __ballot_sync(kFull, in[wd]);
      if (lane == i) mine[wd] = word;
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(p.payload) + e * kTile + wi * 32 + lane;
  *dst = make_uint4(mine[0], mine[1], mine[2], mine[3]);
  // which 64-column halves hold a visible element (OR over the 128 rows)
  __shared__ uint32_t s_half[4];
  const uint32_t hb = ((mine[0] | mine[1]) ? 1u : 0u) | ((mine[2] | mine[3]) ? 2u : 0u);
  const uint32_t hw = __reduce_or_sync(kFull, hb);
  if (lane == 0) s_half[wi] = hw;
  __syncthreads();
  if (threadIdx.x == 0) p.halves[e] = static_cast<uint8_t>(s_half[0] | s_half[1] | s_half[2] | s_half[3]);
}

// Block masks: one warp per partial entry.  The rows of a tile that fall in
// the same logical block row have identical predicate words, so the warp
// walks the tile's row segments (one per logical block row, clipped to the
// sample) and forms each segment's 4 words with 4 ballots over the columns;
// lane l then stores rows l, l+32, l+64, l+96 (16 bytes each, coalesced).
__global__ void __launch_bounds__(128) k_payload_blocks(PayloadParams p) {
  const long long e = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (e >= p.P) return;
  const int flat = p.entry_row[e];
  const int hm = flat / p.rows, row = flat % p.rows;
  const int j = p.p_idx[e];
  const int b = p.row_batch[row];
  const int32_t* s = p.seq + 8 * b;
  const int q_len = s[2], k_len = s[3], row_begin = s[4];
  const int q0 = (row - row_begin) * kTile;
  const uint8_t* M = p.block_mask + static_cast<long long>(hm) * p.nbq * p.nbk;
  int cb[kPayloadWords];
  bool cin[kPayloadWords];
#pragma unroll
  for (int wd = 0; wd < kPayloadWords; ++wd) {
    const int col = j * kTile + wd * 32 + lane;
    cin[wd] = col < k_len;
    cb[wd] = cin[wd] ? col / p.block_kv : 0;
  }
  uint32_t mine[4][kPayloadWords];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int wd = 0; wd < kPayloadWords; ++wd) mine[i][wd] = 0;
  const int r_end = min(kTile, q_len - q0);  // rows past the sample stay 0
  for (int r = 0; r < r_end;) {
    const int rb = (q0 + r) / p.block_q;
    const int seg_end = min(r_end, (rb + 1) * p.block_q - q0);
    const uint8_t* Mr = M + static_cast<long long>(rb) * p.nbk;
    uint32_t words[kPayloadWords];
#pragma unroll
    for (int wd = 0; wd < kPayloadWords; ++wd)
      words[wd] = __ballot_sync(kFull, cin[wd] && __ldg(Mr + cb[wd]) != 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int R = lane + 32 * i;
      if (R >= r && R < seg_end)
#pragma unroll
        for (int wd = 0; wd < kPayloadWords; ++wd) mine[i][wd] = words[wd];
    }
    r = seg_end;
  }
  uint4* dst = reinterpret_cast<uint4*>(p.payload) + e * kTile + lane;
  uint32_t hb = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dst[32 * i] = make_uint4(mine[i][0], mine[i][1], mine[i][2], mine[i][3]);
    hb |= ((mine[i][0] | mine[i][1]) ? 1u : 0u) | ((mine[i][2] | mine[i][3]) ? 2u : 0u);
  }
  hb = __reduce_or_sync(kFull, hb);
  if (lane == 0) p.halves[e] = static_cast<uint8_t>(hb);
}

// ------------------------------------------------------------ schedule
struct SchedParams {
  const int32_t* seq;
  const int32_t* p_off;
  const int32_t* f_off;
  int32_t* hist;     // [NS*(C+1)]
  int32_t* cursors;  // [NS*(C+1)]
  int32_t* work;     // [tasks*4]
  int B, Hq, Hk, Hmask, rows, C, NS;
};

__device__ __forceinline__ int task_cost(const SchedParams& p, int h, int row) {
  const long long flat = static_cast<long long>(p.Hmask == 1 ? 0 : h) * p.rows + row;
  return (p.p_off[flat + 1] - p.p_off[flat]) + (p.f_off[flat + 1] - p.f_off[flat]);
}

// Bucket of a task inside its section: C - cost for cost in [1, C], C for cost 0.
__device__ __forceinline__ int task_bucket(const SchedParams& p, int cost) {
  return cost > 0 ? (p.C - min(cost, p.C)) : p.C;
}

// One CTA builds the whole schedule with bounded counting:
//  1. histogram of (section, cost bucket) over every task, one warp per section;
//  2. offsets: positive-cost tasks of section s start after every positive
//     task of sections < s, ordered by bucket (cost descending); zero-cost
//     tasks follow every positive task, sections in order (section totals
//     and bucket cursors one warp per section, starts by a block scan);
//  3. scatter: one warp per section walks its tasks in tie order (head in the
//     section's group, then m_block), 32 at a time; lanes with the same
//     bucket take consecutive slots in lane order, so the sort is stable.
// Section s = (sample b, K/V head hk).
__global__ void __launch_bounds__(1024) k_schedule(SchedParams p) {
  const int C = p.C;
  const int group = p.Hq / p.Hk;
  const long long nb = static_cast<long long>(p.NS) * (C + 1);
  for (long long i = threadIdx.x; i < nb; i += blockDim.x) p.hist[i] = 0;
  __syncthreads();
  // one warp per section (the sections are many and small: one per sample
  // and K/V head, a few dozen tasks each)
  for (int sct = threadIdx.x >> 5; sct < p.NS; sct += blockDim.x >> 5) {
    const int b = sct / p.Hk, hk = sct % p.Hk;
    const int begin = p.seq[8 * b + 4], nrows = p.seq[8 * b + 5];
    const int n = group * nrows;
    for (int t = threadIdx.x & 31; t < n; t += 32) {
      const int h = hk * group + t / nrows, m = t % nrows;
      atomicAdd(&p.hist[static_cast<long long>(sct) * (C + 1) + task_bucket(p, task_cost(p, h, begin + m))], 1);
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  // 2a. positive-cost tasks per section (one warp per section, lanes over
  //     buckets); kept in the section's bucket-0 cursor until 2b
  for (int sct = threadIdx.x >> 5; sct < p.NS; sct += blockDim.x >> 5) {
    const int32_t* h = p.hist + static_cast<long long>(sct) * (C + 1);
    long long tot = 0;
    for (int c = lane; c < C; c += 32) tot += h[c];
#pragma unroll
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(kFull, tot, o);
    if (lane == 0) p.cursors[static_cast<long long>(sct) * (C + 1)] = static_cast<int32_t>(tot);
  }
  __syncthreads();
  // 2b. section starts: positive tasks of section s after those of sections
  //     < s; zero-cost tasks after every positive task, sections in order
  __shared__ long long s_tot_pos;
  long long carry_pos = 0;
  for (int base = 0; base < p.NS; base += 1024) {
    const int sct = base + threadIdx.x;
    const long long pos = (sct < p.NS) ? p.cursors[static_cast<long long>(sct) * (C + 1)] : 0;
    long long tot;
    const long long start = carry_pos + block_excl_scan(pos, &tot);
    if (sct < p.NS) p.cursors[static_cast<long long>(sct) * (C + 1)] = static_cast<int32_t>(start);
    carry_pos += tot;
  }
  if (threadIdx.x == 0) s_tot_pos = carry_pos;
  __syncthreads();
  long long carry_zero = s_tot_pos;
  for (int base = 0; base < p.NS; base += 1024) {
    const int sct = base + threadIdx.x;
    const long long z = (sct < p.NS) ? p.hist[static_cast<long long>(sct) * (C + 1) + C] : 0;
    long long tot;
    const long long start = carry_zero + block_excl_scan(z, &tot);
    if (sct < p.NS) p.cursors[static_cast<long long>(sct) * (C + 1) + C] = static_cast<int32_t>(start);
    carry_zero += tot;
  }
  __syncthreads();
  // 2c. bucket cursors inside each section: its start plus an exclusive scan
  //     of its bucket counts (one warp per section, 32 buckets at a time)
  for (int sct = threadIdx.x >> 5; sct < p.NS; sct += blockDim.x >> 5) {
    const int32_t* h = p.hist + static_cast<long long>(sct) * (C + 1);
    int32_t* cur = p.cursors + static_cast<long long>(sct) * (C + 1);
    long long run = cur[0];
    __syncwarp();
    for (int c0 = 0; c0 < C; c0 += 32) {
      const int c = c0 + lane;
      const long long v = (c < C) ? h[c] : 0;
      long long x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (c < C) cur[c] = static_cast<int32_t>(run + x - v);
      run += __shfl_sync(kFull, x, 31);
    }
  }
  for (int sct = threadIdx.x >> 5; sct < p.NS; sct += blockDim.x >> 5) {
    const int b = sct / p.Hk, hk = sct % p.Hk;
    const int begin = p.seq[8 * b + 4], nrows = p.seq[8 * b + 5], q_len = p.seq[8 * b + 2];
    const int n = group * nrows;
    int32_t* cur = p.cursors + static_cast<long long>(sct) * (C + 1);
    for (int t0 = 0; t0 < n; t0 += 32) {
      const int t = t0 + lane;
      const bool act = t < n;
      const unsigned amask = __ballot_sync(kFull, act);
      if (act) {
        const int h = hk * group + t / nrows, m = t % nrows;
        const int bucket = task_bucket(p, task_cost(p, h, begin + m));
        const unsigned same = __match_any_sync(amask, bucket);
        const int rank = __popc(same & ((1u << lane) - 1));
        const int pos = cur[bucket] + rank;
        int32_t* wd = p.work + 4LL * pos;
        wd[0] = m;
        wd[1] = h;
        wd[2] = b;
        wd[3] = min(kTile, q_len - m * kTile);
        __syncwarp(amask);
        if (rank == 0) cur[bucket] += __popc(same);
      }
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------ statistics
__global__ void k_count_visible(const uint32_t* payload, long long nwords, long long full_tiles,
                                unsigned long long* out) {
  unsigned long long acc = 0;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < nwords; i += 256LL * gridDim.x)
    acc += __popc(payload[i]);
  for (int o = 16; o; o >>= 1) acc += __shfl_down_sync(kFull, acc, o);
  if ((threadIdx.x & 31) == 0) atomicAdd(out, acc);
  if (blockIdx.x == 0 && threadIdx.x == 0)
    atomicAdd(out, static_cast<unsigned long long>(full_tiles) * kTile * kTile);
}

}  // namespace

// ====================================================================== host
cudaError_t launch_geometry(const Geometry& g, const int32_t* cu_q, const int32_t* cu_k,
                            const PlanWorkspace& ws, cudaStream_t st) {
  GeoParams p{g.layout, g.batch, g.seqlen_q, g.seqlen_k, g.total_q, g.total_k, cu_q, cu_k,
              ws.cu_rows, ws.seq, ws.row_batch, ws.err, ws.rows_ub};
  k_geometry<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_classify(const Geometry& g, const MaskArgs& m, const PlanWorkspace& ws,
                            cudaStream_t st) {
  ClassifyParams p{};
  p.seq = ws.seq;
  p.row_batch = ws.row_batch;
  p.cu_rows = ws.cu_rows;
  p.B = g.batch;
  p.mask_func = m.mask_func;
  p.nfunc = m.nfunc;
  p.total_q = g.total_q;
  p.block_mask = m.block_mask;
  p.block_q = m.block_q;
  p.block_kv = m.block_kv;
  p.nbq = m.nbq;
  p.nbk = m.nbk;
  p.vis_bits = ws.vis_bits;
  p.full_bits = ws.full_bits;
  p.p_cnt = ws.p_cnt;
  p.f_cnt = ws.f_cnt;
  p.err = ws.err;
  p.rows_ub = ws.rows_ub;
  p.words = ws.words;
  if (ws.rows_ub == 0) return cudaSuccess;
  dim3 grid(ws.rows_ub, m.Hmask);
  if (m.kind == MASK_INTERVALS)
    k_classify_intervals<<<grid, 128, 0, st>>>(p);
  else
    k_classify_blocks<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_scan_header(const Geometry& g, int Hmask, const PlanWorkspace& ws,
                               cudaStream_t st) {
  ScanParams p{ws.p_cnt, ws.f_cnt, ws.cu_rows, ws.p_off, ws.f_off, ws.header, ws.err,
               g.batch, Hmask, ws.rows_ub};
  k_scan_header<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_materialize(const Geometry& g, const MaskArgs& m, const PlanWorkspace& ws,
                               fa_plan* plan, const int32_t* cu_q_src, const int32_t* cu_k_src,
                               cudaStream_t st) {
  const int rows = static_cast<int>(plan->rows);
  const long long nflat = static_cast<long long>(m.Hmask) * rows;
  MatParams mp{};
  mp.vis_bits = ws.vis_bits;
  mp.full_bits = ws.full_bits;
  mp.p_off = ws.p_off;
  mp.f_off = ws.f_off;
  mp.p_idx = plan->p_idx;
  mp.f_idx = plan->f_idx;
  mp.entry_row = plan->entry_row;
  mp.rows = rows;
  mp.rows_ub = ws.rows_ub;
  mp.words = ws.words;
  const int32_t* src[6] = {ws.cu_rows, ws.seq, ws.p_off, ws.f_off, cu_q_src, cu_k_src};
  int32_t* dst[6] = {plan->cu_q_rows, plan->seq_desc, plan->p_off, plan->f_off, plan->cu_seqlens_q,
                     plan->cu_seqlens_k};
  const long long cnt[6] = {g.batch + 1LL, 8LL * g.batch, nflat + 1, nflat + 1,
                            (g.layout == FA_LAYOUT_THD) ? g.batch + 1LL : 0,
                            (g.layout == FA_LAYOUT_THD) ? g.batch + 1LL : 0};
  for (int a = 0; a < 6; ++a) {
    mp.src[a] = src[a];
    mp.dst[a] = dst[a];
    mp.count[a] = cnt[a];
  }
  k_materialize<<<dim3(rows > 0 ? rows : 1, rows > 0 ? m.Hmask : 1), 32, 0, st>>>(mp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || plan->P == 0) return e;
  PayloadParams pp{};
  pp.entry_row = plan->entry_row;
  pp.p_idx = plan->p_idx;
  pp.row_batch = ws.row_batch;
  pp.seq = ws.seq;
  pp.payload = plan->payload;
  pp.halves = plan->halves;
  pp.rows = rows;
  pp.P = static_cast<int>(plan->P);
  pp.mask_func = m.mask_func;
  pp.nfunc = m.nfunc;
  pp.total_q = g.total_q;
  pp.block_mask = m.block_mask;
  pp.block_q = m.block_q;
  pp.block_kv = m.block_kv;
  pp.nbq = m.nbq;
  pp.nbk = m.nbk;
  if (m.kind == MASK_INTERVALS && m.nfunc <= kMaxFuncFast)
    k_payload_intervals<true><<<static_cast<unsigned>(plan->P), 128, 0, st>>>(pp);
  else if (m.kind == MASK_INTERVALS)
    k_payload_intervals<false><<<static_cast<unsigned>(plan->P), 128, 0, st>>>(pp);
  else
    k_payload_blocks<<<static_cast<unsigned>((plan->P + 3) / 4), 128, 0, st>>>(pp);
  return cudaGetLastError();
}

cudaError_t launch_schedule(const Geometry& g, fa_plan* plan, int32_t* hist, int32_t* cursors,
                            int num_sections, int max_cost, cudaStream_t st) {
  if (plan->tasks == 0) return cudaSuccess;
  SchedParams p{plan->seq_desc, plan->p_off, plan->f_off, hist, cursors, plan->work_desc,
                g.batch, g.heads_q, g.heads_k, plan->Hmask, static_cast<int>(plan->rows),
                max_cost, num_sections};
  k_schedule<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_count_visible(const fa_plan* plan, unsigned long long* out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(unsigned long long), st);
  if (e != cudaSuccess) return e;
  const long long nwords = plan->P * kTile * kPayloadWords;
  k_count_visible<<<1024, 256, 0, st>>>(plan->payload, nwords, plan->F, out);
  return cudaGetLastError();
}

}  // namespace bsm

// ================================================= allocation-free sizing
// Scratch of fa_plan_header_noalloc: the geometry, classification and scan
// stages above write their workspace here instead of into memory obtained
// from an allocator.  Every device on which the library is loaded holds
// this array until the process exits.
static constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace bsm {
namespace {

// Device address of g_noalloc_scratch for device `dev`, looked up once per
// device (with that device current) and cached.  In host code the symbol
// itself is only a host-side stand-in, so kernels must get this address.
void* noalloc_scratch_address(int dev, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[128] = {};
  *err = cudaSuccess;
  if (dev < 0 || dev >= 128) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace bsm

extern "C" int fa_plan_header_noalloc(const fa_geometry* geom, const int32_t* mask_func,
                                      int32_t Hmask, int32_t nfunc, int64_t* header_out,
                                      void* stream) {
  using namespace bsm;
  clear_last_error();
  if (int e = check_geometry_public(geom)) return e;
  if (nfunc < 1 || nfunc % 2 != 1) return report_error(FA_ERR_INVALID_ARG, "nfunc must be a positive odd integer");
  if (Hmask != 1 && Hmask != geom->heads_q) return report_error(FA_ERR_INVALID_ARG, "Hmask must be 1 or heads_q");
  if (!header_out || reinterpret_cast<uintptr_t>(header_out) % 8 != 0)
    return report_error(FA_ERR_INVALID_ARG, "header_out must be a non-NULL, 8-byte aligned device pointer");
  const Geometry g = geometry_public(geom);
  if (!mask_func && g.total_q > 0) return report_error(FA_ERR_INVALID_ARG, "mask_func is NULL");
  const int B = g.batch;
  const long long nq_max = (static_cast<long long>(g.seqlen_q) + kTile - 1) / kTile;
  const long long kt_ub = (static_cast<long long>(g.seqlen_k) + kTile - 1) / kTile;
  const long long rows_ub = static_cast<long long>(B) * nq_max;
  const long long words = kt_ub > 0 ? (kt_ub + 31) / 32 : 1;
  const long long nflat = static_cast<long long>(Hmask) * rows_ub;
  // same sub-arrays as the allocating build's first workspace
  const size_t sizes[] = {4, 64, 4ull * (B + 1), 32ull * B, 4ull * rows_ub, 4ull * nflat * words,
                          4ull * nflat * words, 4ull * nflat, 4ull * nflat, 4ull * (nflat + 1),
                          4ull * (nflat + 1)};
  size_t off[11], need = 0;
  for (int i = 0; i < 11; ++i) {
    off[i] = need;
    need += round256(sizes[i]);
  }
  if (need > kNoAllocScratchBytes)
    return report_error(FA_ERR_UNSUPPORTED,
                        "this mask needs %zu bytes of planner scratch; the allocation-free entry point "
                        "has %zu (use fa_plan_build_intervals)",
                        need, kNoAllocScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return report_error(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  uint8_t* base = static_cast<uint8_t*>(noalloc_scratch_address(dev, &e));
  if (!base) return report_error(FA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
  PlanWorkspace ws{};
  ws.err = reinterpret_cast<uint32_t*>(base + off[0]);
  ws.header = reinterpret_cast<long long*>(header_out);  // the scan writes the header straight to the output
  ws.cu_rows = reinterpret_cast<int32_t*>(base + off[2]);
  ws.seq = reinterpret_cast<int32_t*>(base + off[3]);
  ws.row_batch = reinterpret_cast<int32_t*>(base + off[4]);
  ws.vis_bits = reinterpret_cast<uint32_t*>(base + off[5]);
  ws.full_bits = reinterpret_cast<uint32_t*>(base + off[6]);
  ws.p_cnt = reinterpret_cast<int32_t*>(base + off[7]);
  ws.f_cnt = reinterpret_cast<int32_t*>(base + off[8]);
  ws.p_off = reinterpret_cast<int32_t*>(base + off[9]);
  ws.f_off = reinterpret_cast<int32_t*>(base + off[10]);
  ws.rows_ub = static_cast<int>(rows_ub);
  ws.kt_ub = static_cast<int>(kt_ub);
  ws.words = static_cast<int>(words);
  MaskArgs m{};
  m.kind = MASK_INTERVALS;
  m.mask_func = mask_func;
  m.nfunc = nfunc;
  m.Hmask = Hmask;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the error word must start at zero
  e = cudaMemsetAsync(ws.err, 0, 4, st);
  if (e == cudaSuccess) e = launch_geometry(g, geom->cu_seqlens_q, geom->cu_seqlens_k, ws, st);
  if (e == cudaSuccess) e = launch_classify(g, m, ws, st);
  if (e == cudaSuccess) e = launch_scan_header(g, Hmask, ws, st);
  if (e != cudaSuccess) return report_error(FA_ERR_CUDA, "allocation-free planner stages: %s", cudaGetErrorString(e));
  return FA_OK;
}

