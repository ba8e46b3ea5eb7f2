// planner.cu -- GPU mask planner: mask -> MaskPlan, in three launches.
//
// Stages follow "Flex Attention Mask Plan Design" (cuDNN frontend docs):
//   k_front_*   one CTA per (mask head, sample, Q tile row of the sample):
//               §4.3 Q2K classification into visible/full bitsets and
//               per-row partial/full counts, endpoints validated and clamped
//               (§3.3); block masks use the logical-block expansion E(M) of
//               "Decoupling Logical Masks from GPU Execution for Dynamic
//               Block-Sparse Attention" §2.  Every CTA adds its rows'
//               counts to the §4.5 entry totals; the last CTA to finish
//               builds the §4.2 compact row prefixes with the §3.2 prefix
//               validation and the §4.8 sequence descriptors and writes the
//               8-value allocation header from the totals (for backward
//               plans after the K2Q scans), also straight into host memory
//               for the one host read-back.
//   k_schedule  §4.5 exclusive scans of the per-row counts into the
//               partial/full offsets, then the §4.8 forward task order by
//               bounded counting (runs while the host reads the header and
//               allocates the plan).
//   k_back_*    one CTA per (Q tile row, mask head): exact-size copies into
//               the plan, §4.6 partial / full CSR index lists and the §5
//               packed predicate payload of the row's partial tiles.
// Every GPU launch costs a few microseconds of device time on its own, so
// the stages are fused into as few launches as their data dependences
// allow: only the totals size the plan, so the header goes out before the
// offsets are scanned, and the plan can only be written once the host has
// sized and allocated it.
#include <cuda_runtime.h>

#include <atomic>
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

// Block-wide exclusive scan of one value per thread (blockDim.x a multiple
// of 32, at most 1024); *total receives the block's sum.
__device__ __forceinline__ long long block_excl_scan(long long v, long long* total) {
  __shared__ long long s_warp[32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    long long s = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(kFull, s, o);
      if (lane >= o) s += y;
    }
    s_warp[lane] = s;
  }
  __syncthreads();
  const long long warp_prefix = wid ? s_warp[wid - 1] : 0;
  *total = s_warp[nw - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

// ------------------------------------------------------------ front
struct FrontParams {
  int layout, B, Sq, Sk, total_q, total_k, nq_max;
  const int32_t* cu_q;
  const int32_t* cu_k;
  // intervals
  const int32_t* mask_func;
  int nfunc;
  // blocks
  const uint8_t* block_mask;
  int block_q, block_kv, nbq, nbk;
  int Hmask;
  // per padded row (mask head, sample, Q tile row of the sample): flat index
  // hm * rows_ub + b * nq_max + lr
  uint32_t* vis_bits;  // [Hmask*rows_ub*words]
  uint32_t* full_bits;
  int32_t* p_cnt;      // [Hmask*rows_ub]
  int32_t* f_cnt;
  int rows_ub, words;
  // written by the last CTA
  int32_t* cu_rows;    // [B+1]
  int32_t* seq;        // [B*8]
  int32_t* row_batch;  // [rows]
  int32_t* p_off;      // [Hmask*rows+1], compact order (hm, row)
  int32_t* f_off;
  long long* header;   // device, 8 values
  long long* host_header;  // host memory, 8 values then the ticket; may be null
  long long ticket;
  unsigned* ctl;       // [0] CTAs arrived, [1] error bits; zero at launch, zero again at exit
  unsigned long long* tot;  // [2] partial and full entries of every row; zero at launch, zero again at exit
  // backward K2Q view (§4.4); kp_cnt is null when it is not built
  int32_t* kp_cnt;     // [Hmask*B*kt_ub] per padded K row (hm, b, K tile): zero at launch
  int32_t* kf_cnt;
  int kt_ub;
  int32_t* cu_krows;   // [B+1], written by the last CTA
  int32_t* krow_batch; // [k_rows]
  int32_t* kp_off;     // [Hmask*k_rows+1], compact order (hm, K row)
  int32_t* kf_off;
};

// K2Q counts (§4.4): the tile (Q row, K tile j) of sample b adds one
// partial or full Q contributor to K row (hm, b, j).
__device__ __forceinline__ void count_k2q(const FrontParams& p, int hm, int b, int j, bool partial, bool full) {
  const long long r = (static_cast<long long>(hm) * p.B + b) * p.kt_ub + j;
  if (partial) atomicAdd(p.kp_cnt + r, 1);
  if (full) atomicAdd(p.kf_cnt + r, 1);
}

struct SampleGeo {
  int q_off, k_off, q_len, k_len;
  bool bad;
};

// Sample b's offsets and lengths.  THD prefixes are validated (§3.2) and
// clamped, so that every stage indexes safely before the host reads the
// error bits.
__device__ __forceinline__ SampleGeo sample_geo(const FrontParams& p, int b) {
  SampleGeo s{};
  if (p.layout == FA_LAYOUT_BSHD) {
    s.q_off = b * p.Sq;
    s.k_off = b * p.Sk;
    s.q_len = p.Sq;
    s.k_len = p.Sk;
    s.bad = false;
    return s;
  }
  const int a = __ldg(p.cu_q + b), e = __ldg(p.cu_q + b + 1);
  const int c = __ldg(p.cu_k + b), f = __ldg(p.cu_k + b + 1);
  bool bad = false;
  if (b == 0 && (a != 0 || c != 0)) bad = true;
  if (b == p.B - 1 && (e != p.total_q || f != p.total_k)) bad = true;
  if (e < a || f < c) bad = true;
  if (e - a > p.Sq || f - c > p.Sk) bad = true;
  if (a < 0 || c < 0 || e > p.total_q || f > p.total_k) bad = true;
  s.q_off = min(max(a, 0), p.total_q);
  s.k_off = min(max(c, 0), p.total_k);
  s.q_len = min(max(e - a, 0), min(p.Sq, p.total_q - s.q_off));
  s.k_len = min(max(f - c, 0), min(p.Sk, p.total_k - s.k_off));
  s.bad = bad;
  return s;
}

// Interval masks, 128 threads: thread t owns Q row t of the tile.  Per row,
// each K tile is "touched" if a non-empty interval intersects it and
// "covered" if one maximal run of merged intervals contains the whole tile;
// visible = OR over valid rows of touched, full = AND over all 128 rows of
// covered (rows past the sample's q_len cover nothing, so a Q tail is never full).
__device__ __forceinline__ void classify_intervals(const FrontParams& p, const SampleGeo& sg, int b,
                                                   int lr, int hm, long long ws_row) {
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  __shared__ uint32_t s_v[4], s_f[4];
  const int q_local = lr * kTile + t;
  const int k_len = sg.k_len;
  const bool valid = q_local < sg.q_len;
  const int32_t* F = p.mask_func + static_cast<long long>(hm) * p.nfunc * p.total_q + sg.q_off + q_local;
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
    if (bad) atomicOr(&p.ctl[1], PLANERR_MASK);
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
      if (p.kp_cnt) {
        for (uint32_t x = v; x; x &= x - 1) {
          const int bit = __ffs(x) - 1;
          count_k2q(p, hm, b, 32 * w + bit, !((f >> bit) & 1u), (f >> bit) & 1u);
        }
      }
    }
    __syncthreads();
  }
  if (t == 0) {
    p.p_cnt[ws_row] = pc;
    p.f_cnt[ws_row] = fc;
    atomicAdd(&p.tot[0], static_cast<unsigned long long>(pc));
    atomicAdd(&p.tot[1], static_cast<unsigned long long>(fc));
  }
}

// Block masks (fixed length), 256 threads: thread per K tile, the CTA's R
// padded Q tile rows x0 .. x0+R-1 together.  Tile (i, j) touches the
// logical blocks [r0, r1] x [c0, c1] that overlap its in-bounds part; it is
// visible if any is active and full if all are and the tile has no Q/K
// tail.  Words are bit-packed with warp ballots.  When a tile touches at
// most two blocks each way (blocks of 64 or more that divide the tile), the
// four mask bytes of every row are requested before any is used, so the
// rows share one memory latency; wider spans take a loop.
template <int R>
__device__ __forceinline__ void classify_blocks_rows(const FrontParams& p, int hm, int x0) {
  const int t = threadIdx.x, lane = t & 31;
  __shared__ int s_pc[R], s_fc[R];
  if (t < R) {
    s_pc[t] = 0;
    s_fc[t] = 0;
  }
  __syncthreads();
  const uint8_t* M = p.block_mask + static_cast<long long>(hm) * p.nbq * p.nbk;
  int rb[R], lrr[R], qlen[R], klen[R], r0[R], r1[R];
  bool ok[R], qtail[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int x = x0 + i;
    ok[i] = false;
    rb[i] = 0;
    lrr[i] = 0;
    qlen[i] = klen[i] = 0;
    r0[i] = r1[i] = 0;
    qtail[i] = false;
    if (x < p.rows_ub) {
      const int b = x / p.nq_max, lr = x % p.nq_max;
      const SampleGeo sg = sample_geo(p, b);
      if (lr < cdiv(sg.q_len, kTile)) {
        ok[i] = true;
        rb[i] = b;
        lrr[i] = lr;
        qlen[i] = sg.q_len;
        klen[i] = sg.k_len;
        const int q0 = lr * kTile, q1 = min(q0 + kTile, sg.q_len);
        qtail[i] = (q1 - q0) < kTile;
        r0[i] = q0 / p.block_q;
        r1[i] = (q1 - 1) / p.block_q;
      }
    }
  }
  const int nwords_used = p.words * 32;
  for (int j0 = 0; j0 < nwords_used; j0 += blockDim.x) {
    const int j = j0 + t;
    int c0[R], c1[R];
    bool in[R], ktail[R], two[R];
    uint32_t m4[R];  // bytes (r0, c0), (r0, c1), (r1, c0), (r1, c1), nonzero -> 1
#pragma unroll
    for (int i = 0; i < R; ++i) {
      in[i] = ok[i] && j < cdiv(klen[i], kTile);
      c0[i] = c1[i] = 0;
      ktail[i] = false;
      two[i] = false;
      m4[i] = 0u;
      if (in[i]) {
        const int k0 = j * kTile, k1 = min(k0 + kTile, klen[i]);
        ktail[i] = (k1 - k0) < kTile;
        c0[i] = k0 / p.block_kv;
        c1[i] = (k1 - 1) / p.block_kv;
        two[i] = (r1[i] - r0[i] <= 1) && (c1[i] - c0[i] <= 1);
        if (two[i]) {
          const uint8_t* A = M + static_cast<long long>(r0[i]) * p.nbk;
          const uint8_t* Bm = M + static_cast<long long>(r1[i]) * p.nbk;
          m4[i] = (__ldg(A + c0[i]) ? 1u : 0u) | (__ldg(A + c1[i]) ? 2u : 0u) | (__ldg(Bm + c0[i]) ? 4u : 0u) |
                  (__ldg(Bm + c1[i]) ? 8u : 0u);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      bool vis = false, full = false;
      if (in[i]) {
        bool any, all;
        if (two[i]) {
          any = m4[i] != 0u;
          all = m4[i] == 0xFu;
        } else {
          any = false;
          all = true;
          for (int r = r0[i]; r <= r1[i]; ++r) {
            const uint8_t* Mr = M + static_cast<long long>(r) * p.nbk;
            for (int c = c0[i]; c <= c1[i]; ++c) {
              const bool xv = __ldg(Mr + c) != 0;
              any |= xv;
              all &= xv;
            }
          }
        }
        vis = any;
        full = any && all && !qtail[i] && !ktail[i];
        if (p.kp_cnt && vis) count_k2q(p, hm, rb[i], j, !full, full);
      }
      const uint32_t vb = __ballot_sync(kFull, vis);
      const uint32_t fb = __ballot_sync(kFull, full);
      const int w = j >> 5;
      if (ok[i] && lane == 0 && w < p.words) {
        const long long ws_row = static_cast<long long>(hm) * p.rows_ub + x0 + i;
        p.vis_bits[ws_row * p.words + w] = vb;
        p.full_bits[ws_row * p.words + w] = fb;
        atomicAdd(&s_pc[i], __popc(vb & ~fb));
        atomicAdd(&s_fc[i], __popc(fb));
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < R; ++i) {
    if (t == i && ok[i]) {
      const long long ws_row = static_cast<long long>(hm) * p.rows_ub + x0 + i;
      p.p_cnt[ws_row] = s_pc[i];
      p.f_cnt[ws_row] = s_fc[i];
    }
  }
  if (t == 0) {
    unsigned long long a = 0, c = 0;
#pragma unroll
    for (int i = 0; i < R; ++i) {
      a += ok[i] ? s_pc[i] : 0;
      c += ok[i] ? s_fc[i] : 0;
    }
    if (a) atomicAdd(&p.tot[0], a);
    if (c) atomicAdd(&p.tot[1], c);
  }
}

// Work of the last CTA of the front launch: sample descriptors, compact row
// prefixes and the row -> sample map; exclusive scans of the per-row counts
// in compact (mask head, row) order; the header; reset of the control words.
constexpr int kScanItems = 8;

// q = i / d, r = i % d for 0 <= i, in 32-bit arithmetic when i fits.
__device__ __forceinline__ void div_idx(long long i, int d, int& q, int& r) {
  if (i <= 0x7fffffffLL) {
    const int ii = static_cast<int>(i);
    q = ii / d;
    r = ii - q * d;
  } else {
    q = static_cast<int>(i / d);
    r = static_cast<int>(i % d);
  }
}

// Exclusive scans, by the whole CTA, of two per-row counts over padded rows
// x in [0, npad).  at(x, ci) says whether row x exists and gives its
// position ci in compact order, which is the padded order without the rows
// that do not exist; so the scan over padded rows, with zeros for those,
// is the compact scan.  The counts are read (cnt_a/cnt_c at x) only for rows
// that exist: the others were never written.  Offsets to off_a/off_c [n + 1]
// at the compact positions; totals added to tot_a/tot_c.  Each thread takes
// kScanItems consecutive rows, whose loads are independent.
template <class At>
__device__ void scan_pair_padded(long long npad, long long n, const int32_t* cnt_a, const int32_t* cnt_c,
                                 int32_t* off_a, int32_t* off_c, long long& tot_a, long long& tot_c, At at) {
  const int nt = blockDim.x;
  long long ca = 0, cc = 0;
  for (long long base = 0; base < npad; base += static_cast<long long>(nt) * kScanItems) {
    const long long i0 = base + static_cast<long long>(threadIdx.x) * kScanItems;
    int va[kScanItems], vc[kScanItems];
    long long ci[kScanItems];
    long long sa = 0, sc = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
      const long long i = i0 + k;
      va[k] = 0;
      vc[k] = 0;
      ci[k] = -1;
      if (i < npad && at(i, ci[k])) {
        va[k] = __ldcg(cnt_a + i);
        vc[k] = __ldcg(cnt_c + i);
      }
      sa += va[k];
      sc += vc[k];
    }
    long long ta, tc;
    long long ea = ca + block_excl_scan(sa, &ta);
    long long ec = cc + block_excl_scan(sc, &tc);
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
      if (ci[k] >= 0) {
        off_a[ci[k]] = static_cast<int32_t>(ea);
        off_c[ci[k]] = static_cast<int32_t>(ec);
      }
      ea += va[k];
      ec += vc[k];
    }
    ca += ta;
    cc += tc;
  }
  if (threadIdx.x == 0) {
    off_a[n] = static_cast<int32_t>(ca);
    off_c[n] = static_cast<int32_t>(cc);
  }
  __syncthreads();
  tot_a += ca;
  tot_c += cc;
}

// Sample prefixes (cu_rows or cu_krows) staged in shared memory for the
// padded scans when there are at most this many samples.
constexpr int kCuSmem = 1024;

// The same scans, staged through shared memory (buf_a/buf_c: ITEMS *
// blockDim.x ints each, 16-byte aligned): a pass loads its counts with
// coalesced loads, all issued before any is used; each thread then scans
// ITEMS consecutive rows out of shared memory; the offsets go back through
// shared memory and out with coalesced stores (the compact positions of
// consecutive existing rows are consecutive).
template <int ITEMS, class At>
__device__ void scan_pair_staged(long long npad, long long n, const int32_t* __restrict__ cnt_a,
                                 const int32_t* __restrict__ cnt_c, int32_t* off_a, int32_t* off_c,
                                 int32_t* buf_a, int32_t* buf_c, long long& tot_a, long long& tot_c, At at) {
  static_assert(ITEMS == 4, "one int4 per thread");
  const int nt = blockDim.x, t = threadIdx.x;
  const long long P = static_cast<long long>(nt) * ITEMS;
  long long ca = 0, cc = 0;
  for (long long base = 0; base < npad; base += P) {
    int la[ITEMS], lc[ITEMS];
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      const long long x = base + static_cast<long long>(u) * nt + t;
      long long ci;
      const bool ok = x < npad && at(x, ci);
      la[u] = ok ? __ldcg(cnt_a + x) : 0;
      lc[u] = ok ? __ldcg(cnt_c + x) : 0;
    }
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      buf_a[u * nt + t] = la[u];
      buf_c[u * nt + t] = lc[u];
    }
    __syncthreads();
    const int4 a4 = reinterpret_cast<const int4*>(buf_a)[t];
    const int4 c4 = reinterpret_cast<const int4*>(buf_c)[t];
    long long ta, tc;
    const long long ea = ca + block_excl_scan(static_cast<long long>(a4.x) + a4.y + a4.z + a4.w, &ta);
    const long long ec = cc + block_excl_scan(static_cast<long long>(c4.x) + c4.y + c4.z + c4.w, &tc);
    reinterpret_cast<int4*>(buf_a)[t] =
        make_int4(static_cast<int32_t>(ea), static_cast<int32_t>(ea + a4.x), static_cast<int32_t>(ea + a4.x + a4.y),
                  static_cast<int32_t>(ea + a4.x + a4.y + a4.z));
    reinterpret_cast<int4*>(buf_c)[t] =
        make_int4(static_cast<int32_t>(ec), static_cast<int32_t>(ec + c4.x), static_cast<int32_t>(ec + c4.x + c4.y),
                  static_cast<int32_t>(ec + c4.x + c4.y + c4.z));
    __syncthreads();
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      const long long x = base + static_cast<long long>(u) * nt + t;
      long long ci;
      if (x < npad && at(x, ci)) {
        off_a[ci] = buf_a[u * nt + t];
        off_c[ci] = buf_c[u * nt + t];
      }
    }
    ca += ta;
    cc += tc;
    __syncthreads();  // the buffers are read before the next pass writes them
  }
  if (t == 0) {
    off_a[n] = static_cast<int32_t>(ca);
    off_c[n] = static_cast<int32_t>(cc);
  }
  __syncthreads();
  tot_a += ca;
  tot_c += cc;
}

__device__ void front_finish(const FrontParams& p) {
  const int nt = blockDim.x;
  long long carry = 0;
  uint32_t err_local = 0;
  for (int base = 0; base < p.B; base += nt) {
    const int b = base + threadIdx.x;
    SampleGeo sg{};
    int nrows = 0;
    if (b < p.B) {
      sg = sample_geo(p, b);
      nrows = cdiv(sg.q_len, kTile);
      if (sg.bad) err_local |= PLANERR_SEQLENS;
    }
    long long tot;
    const long long begin = carry + block_excl_scan(nrows, &tot);
    if (b < p.B) {
      int32_t* s = p.seq + 8 * b;
      s[0] = sg.q_off;
      s[1] = sg.k_off;
      s[2] = sg.q_len;
      s[3] = sg.k_len;
      s[4] = static_cast<int32_t>(begin);
      s[5] = nrows;
      s[6] = cdiv(sg.k_len, kTile);
      s[7] = 0;
      p.cu_rows[b] = static_cast<int32_t>(begin);
    }
    carry += tot;
  }
  if (err_local) atomicOr(&p.ctl[1], err_local);
  const int rows = static_cast<int>(carry);
  if (threadIdx.x == 0) p.cu_rows[p.B] = rows;
  __syncthreads();
  // row -> sample: the last sample whose first row is <= r (a sample without
  // rows shares its start with the next one, so it is never chosen)
  for (int r = threadIdx.x; r < rows; r += nt) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.cu_rows[mid] <= r) lo = mid; else hi = mid - 1;
    }
    p.row_batch[r] = lo;
  }
  __syncthreads();
  __shared__ int32_t s_cu[kCuSmem + 1];
  const bool cu_smem = p.B <= kCuSmem;
  // backward K2Q view (§4.2 backward prefix, §4.4 counts, §4.5 scan): K plan
  // rows per sample, K row -> sample, and the K2Q offsets
  long long k_rows = 0, kp = 0, kf = 0;
  if (p.kp_cnt) {
    for (int base = 0; base < p.B; base += nt) {
      const int b = base + threadIdx.x;
      const int nk = (b < p.B) ? cdiv(sample_geo(p, b).k_len, kTile) : 0;
      long long tot;
      const long long begin = k_rows + block_excl_scan(nk, &tot);
      if (b < p.B) p.cu_krows[b] = static_cast<int32_t>(begin);
      k_rows += tot;
    }
    if (threadIdx.x == 0) p.cu_krows[p.B] = static_cast<int32_t>(k_rows);
    __syncthreads();
    for (long long r = threadIdx.x; r < k_rows; r += nt) {
      int lo = 0, hi = p.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cu_krows[mid] <= r) lo = mid; else hi = mid - 1;
      }
      p.krow_batch[r] = lo;
    }
    __syncthreads();
    const long long nk_flat = static_cast<long long>(p.Hmask) * k_rows;
    if (cu_smem)
      for (int b = threadIdx.x; b <= p.B; b += nt) s_cu[b] = p.cu_krows[b];
    __syncthreads();
    // padded K rows (hm, b, K tile) in the layout of kp_cnt
    scan_pair_padded(static_cast<long long>(p.Hmask) * p.B * p.kt_ub, nk_flat, p.kp_cnt, p.kf_cnt, p.kp_off,
                     p.kf_off, kp, kf, [&](long long x, long long& ci) {
                       int hb, j;
                       div_idx(x, p.kt_ub, hb, j);
                       const int hm = hb / p.B, b = hb - hm * p.B;
                       const int c0 = cu_smem ? s_cu[b] : p.cu_krows[b];
                       const int c1 = cu_smem ? s_cu[b + 1] : p.cu_krows[b + 1];
                       if (j >= c1 - c0) return false;
                       ci = static_cast<long long>(hm) * k_rows + c0 + j;
                       return true;
                     });
  }
  if (threadIdx.x == 0) {
    // entry totals of the Q2K view: every CTA added its rows' counts (the
    // offsets themselves are scanned by the schedule stage, which runs next)
    const long long cp = static_cast<long long>(__ldcg(&p.tot[0]));
    const long long cf = static_cast<long long>(__ldcg(&p.tot[1]));
    uint32_t e = atomicExch(&p.ctl[1], 0u);  // read and reset the error bits
    if (cp > 0x3fffffffLL || cf > 0x3fffffffLL || kp > 0x3fffffffLL || kf > 0x3fffffffLL) e |= PLANERR_OVERFLOW;
    // {fwd Q rows, fwd partial, fwd full, bwd Q rows, bwd K rows, bwd partial,
    // bwd full, error}: the dQ consumer reads the forward Q2K view, which has
    // the backward geometry, so bwd Q rows = fwd Q rows
    const long long h[8] = {rows, cp, cf, p.kp_cnt ? rows : 0, k_rows, kp, kf, static_cast<long long>(e)};
#pragma unroll
    for (int k = 0; k < 8; ++k) p.header[k] = h[k];
    p.ctl[0] = 0u;  // every CTA has arrived: the control words are free again
    p.tot[0] = 0ull;
    p.tot[1] = 0ull;
    if (p.host_header) {
      volatile long long* hh = p.host_header;
#pragma unroll
      for (int k = 0; k < 8; ++k) hh[k] = h[k];
      __threadfence_system();
      hh[8] = p.ticket;  // published last: the host reads the values after seeing it
    }
  }
}

// Padded rows per CTA of the front stage: one for interval masks; four for
// block masks, whose rows are cheap (a few bytes of the block mask per K
// tile), so that fewer CTAs pay the device-wide fence and the arrival.
template <int KIND>
constexpr int kFrontRows = (KIND == MASK_INTERVALS) ? 1 : 4;

// kFrontRows padded rows per CTA: x = blockIdx.x * kFrontRows + i =
// b * nq_max + lr (rows past a sample's end, and x >= rows_ub, only arrive),
// blockIdx.y = mask head.  The last CTA to arrive (atomic count after a
// device-wide fence) finishes the stage.
template <int KIND>
__global__ void __launch_bounds__(KIND == MASK_INTERVALS ? 128 : 256) k_front(FrontParams p) {
  const int hm = blockIdx.y;
  if constexpr (KIND == MASK_INTERVALS) {
    const int x = blockIdx.x;
    if (x < p.rows_ub) {
      const int b = x / p.nq_max, lr = x % p.nq_max;
      const SampleGeo sg = sample_geo(p, b);
      if (lr < cdiv(sg.q_len, kTile))
        classify_intervals(p, sg, b, lr, hm, static_cast<long long>(hm) * p.rows_ub + x);
    }
  } else {
    classify_blocks_rows<kFrontRows<KIND>>(p, hm, blockIdx.x * kFrontRows<KIND>);
  }
  __shared__ unsigned s_last;
  __threadfence();  // every thread's outputs are visible device-wide before the CTA arrives
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned total = gridDim.x * gridDim.y;
    s_last = (atomicAdd(&p.ctl[0], 1u) == total - 1) ? 1u : 0u;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  front_finish(p);
}

// ------------------------------------------------------------ back
struct BackParams {
  // exact-size copies from the workspace (and the caller's cu_seqlens)
  const int32_t* src[8];
  int32_t* dst[8];
  long long count[8];
  // workspace
  const uint32_t* vis_bits;
  const uint32_t* full_bits;
  const int32_t* p_off;  // compact [Hmask*rows+1]
  const int32_t* f_off;
  const int32_t* row_batch;
  const int32_t* seq;
  // plan
  int32_t* p_idx;
  int32_t* f_idx;
  int32_t* entry_row;  // [P]: flat (hm*rows + row) of each partial entry
  uint32_t* payload;   // [P*128*4]
  uint8_t* halves;     // [P] bit s: column half s of the entry has a visible element
  uint8_t* quads;      // [P] bit 2a+s / 4+2a+s: quadrant (row half a, column half s) any / all visible
  int rows, rows_ub, nq_max, words;
  // intervals
  const int32_t* mask_func;
  int nfunc, total_q;
  // blocks
  const uint8_t* block_mask;
  int block_q, block_kv, nbq, nbk;
  // bounds of the checked build: plan entries, and the device error word
  long long nP, nF;
  uint32_t* err;
};

// Quadrant bits of one partial entry, per lane and then reduced over the
// warp: quadrant (a, s) = tile rows 64a..64a+63 x columns 64s..64s+63;
// `live` bit 2a+s: a visible element, `full` bit 2a+s: every element visible.
struct QuadBits {
  uint32_t live = 0u, full = 0xFu;
  // add tile row (lane + 32 i)'s four payload words
  __device__ __forceinline__ void add(int i, const uint32_t (&w)[kPayloadWords]) {
    const int a = i >> 1;
    const uint32_t l = ((w[0] | w[1]) ? 1u : 0u) | ((w[2] | w[3]) ? 2u : 0u);
    const uint32_t f = (((w[0] & w[1]) == kFull) ? 1u : 0u) | (((w[2] & w[3]) == kFull) ? 2u : 0u);
    live |= l << (2 * a);
    full &= ~((f ^ 3u) << (2 * a));
  }
  __device__ __forceinline__ void reduce() {
    live = __reduce_or_sync(kFull, live);
    full = __reduce_and_sync(kFull, full);
  }
  __device__ __forceinline__ uint32_t halves() const { return ((live & 5u) ? 1u : 0u) | ((live & 10u) ? 2u : 0u); }
  __device__ __forceinline__ uint32_t quads() const { return live | (full << 4); }
};

// Endpoints of the CTA's 128 Q rows kept in shared memory for the payload
// when a row has at most this many.
constexpr int kSmemFuncs = 16;

// OR the columns [lo, hi) of tile columns [c0, c0 + 128) into w[0..3]
// (bit l of word wd = column c0 + 32 wd + l).
__device__ __forceinline__ void add_columns(uint32_t (&w)[kPayloadWords], int c0, int lo, int hi) {
  lo = max(lo, c0);
  hi = min(hi, c0 + kTile);
#pragma unroll
  for (int wd = 0; wd < kPayloadWords; ++wd) {
    const int base = c0 + 32 * wd;
    const int L = max(lo, base), H = min(hi, base + 32);
    if (L < H) w[wd] |= static_cast<uint32_t>(((uint64_t(1) << (H - L)) - 1) << (L - base));
  }
}

// Interval payload of one partial entry (tile column j), one warp: lane l
// forms the 4 words of rows l, l+32, l+64, l+96 from the row's intervals
// [0, F0), [F1, F2), ... clipped to the tile and to k_len; rows past the
// sample stay 0.  Returns this lane's quadrant bits (not yet reduced).
__device__ __forceinline__ QuadBits payload_intervals_entry(const BackParams& p, long long e, int j,
                                                            int q_len, int k_len, int q0, int hm,
                                                            int q_off, const int32_t (*sF)[kTile],
                                                            bool smem) {
  const int lane = threadIdx.x & 31;
  const int c0 = j * kTile;
  const int32_t* Fg = p.mask_func + static_cast<long long>(hm) * p.nfunc * p.total_q + q_off;
  QuadBits qb;
  uint4* dst = reinterpret_cast<uint4*>(p.payload) + e * kTile;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = lane + 32 * i;
    uint32_t w[kPayloadWords] = {0, 0, 0, 0};
    if (q0 + t < q_len) {
      auto F = [&](int f) { return smem ? sF[f][t] : __ldg(Fg + static_cast<long long>(f) * p.total_q + q0 + t); };
      add_columns(w, c0, 0, min(F(0), k_len));
      for (int f = 1; f + 1 < p.nfunc; f += 2) add_columns(w, c0, F(f), min(F(f + 1), k_len));
    }
    dst[t] = make_uint4(w[0], w[1], w[2], w[3]);
    qb.add(i, w);
  }
  return qb;
}

// Block payload of one partial entry, one warp.  The rows of a tile that
// fall in the same logical block row have identical predicate words, so the
// warp walks the tile's row segments (one per logical block row, clipped to
// the sample) and forms each segment's 4 words with 4 ballots over the
// columns; lane l then stores rows l, l+32, l+64, l+96 (16 bytes each,
// coalesced).
__device__ __forceinline__ QuadBits payload_blocks_entry(const BackParams& p, long long e, int j,
                                                         int q_len, int k_len, int q0, int hm) {
  const int lane = threadIdx.x & 31;
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
  // a plan that keeps only quadrant bits has no payload words to write
  uint4* dst = p.payload ? reinterpret_cast<uint4*>(p.payload) + e * kTile + lane : nullptr;
  QuadBits qb;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (dst) dst[32 * i] = make_uint4(mine[i][0], mine[i][1], mine[i][2], mine[i][3]);
    qb.add(i, mine[i]);
  }
  return qb;
}

// One CTA (4 warps) per (Q plan row, mask head).  All CTAs share the
// exact-size copies.  Warp 0 turns the row's bitsets into its CSR entries
// (lane w handles bitset word w; ranks come from a warp scan of popcounts,
// so indices come out ascending); then the 4 warps take the row's partial
// entries in turn and write their payloads.
template <int KIND>
__global__ void __launch_bounds__(128) k_back(BackParams p) {
  {
    const long long tid = (static_cast<long long>(blockIdx.y) * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * gridDim.y * blockDim.x;
#pragma unroll
    for (int a = 0; a < 8; ++a)
      for (long long i = tid; i < p.count[a]; i += nthreads) p.dst[a][i] = __ldg(p.src[a] + i);
  }
  const int row = blockIdx.x, hm = blockIdx.y;
  if (row >= p.rows) return;
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int b = __ldg(p.row_batch + row);
  const int32_t* s = p.seq + 8 * b;
  const int q_off = __ldg(s + 0), q_len = __ldg(s + 2), k_len = __ldg(s + 3), row_begin = __ldg(s + 4);
  const int lr = row - row_begin;
  const long long flat = static_cast<long long>(hm) * p.rows + row;
  const long long ws_row = static_cast<long long>(hm) * p.rows_ub + static_cast<long long>(b) * p.nq_max + lr;
  const int pstart = __ldg(p.p_off + flat), np = __ldg(p.p_off + flat + 1) - pstart;
  if (KIND == MASK_BLOCKS && p.payload == nullptr) {
    // Quadrant bits only (64-aligned logical blocks over 64-multiple
    // lengths): each 64x64 quadrant lies inside one logical block pair and
    // inside or outside the sample as a whole, so it is wholly visible or
    // wholly masked.  Thread t takes tile j = j0 + t of each 128-tile chunk:
    // its four block-mask bytes are requested with the row's bitset words,
    // and its list position is its rank among the row's partial (or full)
    // tiles -- earlier chunks, earlier warps, lower lanes -- so the lists
    // come out ascending, as warp 0 writes them below for the other plans.
    const uint8_t* M = p.block_mask + static_cast<long long>(hm) * p.nbq * p.nbk;
    const int q0 = lr * kTile, t = threadIdx.x;
    __shared__ int s_np[4], s_nf[4];
    int pc = pstart, fc = __ldg(p.f_off + flat);
    for (int j0 = 0; j0 < p.words * 32; j0 += 128) {
      const int j = j0 + t, w = j >> 5;
      uint32_t vb = 0u, fb = 0u, live = 0u;
      if (w < p.words) {
        vb = __ldg(p.vis_bits + ws_row * p.words + w);
        fb = __ldg(p.full_bits + ws_row * p.words + w);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int qr = q0 + 64 * a, kc = j * kTile + 64 * s2;
          if (qr < q_len && kc < k_len && __ldg(M + static_cast<long long>(qr / p.block_q) * p.nbk + kc / p.block_kv))
            live |= 1u << (2 * a + s2);
        }
      const uint32_t pb = vb & ~fb;
      const uint32_t below = (1u << lane) - 1u;
      if (lane == 0) {
        s_np[wi] = __popc(pb);
        s_nf[wi] = __popc(fb);
      }
      __syncthreads();
      int pre_p = 0, pre_f = 0, all_p = 0, all_f = 0;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        if (x < wi) {
          pre_p += s_np[x];
          pre_f += s_nf[x];
        }
        all_p += s_np[x];
        all_f += s_nf[x];
      }
      __syncthreads();  // s_np / s_nf are read before the next chunk writes them
      if ((pb >> lane) & 1u) {
        const long long e = bsm_idx(pc + pre_p + __popc(pb & below), p.nP, p.err);
        p.p_idx[e] = j;
        p.entry_row[e] = static_cast<int32_t>(flat);
        p.halves[e] = static_cast<uint8_t>(((live & 5u) ? 1u : 0u) | ((live & 10u) ? 2u : 0u));
        p.quads[e] = static_cast<uint8_t>(live | (live << 4));
      }
      if ((fb >> lane) & 1u) p.f_idx[bsm_idx(fc + pre_f + __popc(fb & below), p.nF, p.err)] = j;
      pc += all_p;
      fc += all_f;
    }
    return;
  }
  if (wi == 0) {
    int pbase = pstart, fbase = __ldg(p.f_off + flat);
    for (int w0 = 0; w0 < p.words; w0 += 32) {
      const int w = w0 + lane;
      uint32_t vb = 0, fb = 0;
      if (w < p.words) {
        vb = __ldg(p.vis_bits + ws_row * p.words + w);
        fb = __ldg(p.full_bits + ws_row * p.words + w);
      }
      uint32_t pb = vb & ~fb;
      const int npw = __popc(pb), nfw = __popc(fb);
      int xp = npw, xf = nfw;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yp = __shfl_up_sync(kFull, xp, o), yf = __shfl_up_sync(kFull, xf, o);
        if (lane >= o) {
          xp += yp;
          xf += yf;
        }
      }
      int pp = pbase + xp - npw, pf = fbase + xf - nfw;
      while (pb) {
        const int bit = __ffs(pb) - 1;
        pb &= pb - 1;
        const long long at = bsm_idx(pp, p.nP, p.err);
        p.p_idx[at] = w * 32 + bit;
        p.entry_row[at] = static_cast<int32_t>(flat);
        ++pp;
      }
      while (fb) {
        const int bit = __ffs(fb) - 1;
        fb &= fb - 1;
        p.f_idx[bsm_idx(pf++, p.nF, p.err)] = w * 32 + bit;
      }
      pbase += __shfl_sync(kFull, xp, 31);
      fbase += __shfl_sync(kFull, xf, 31);
    }
  }
  const int q0 = lr * kTile;
  __shared__ int32_t sF[KIND == MASK_INTERVALS ? kSmemFuncs : 1][kTile];
  const bool smem = KIND == MASK_INTERVALS && p.nfunc <= kSmemFuncs;
  if (KIND == MASK_INTERVALS && smem) {
    const int t = threadIdx.x;
    const int32_t* Fg = p.mask_func + static_cast<long long>(hm) * p.nfunc * p.total_q + q_off;
    for (int f = 0; f < p.nfunc; ++f)
      sF[f][t] = (q0 + t < q_len) ? __ldg(Fg + static_cast<long long>(f) * p.total_q + q0 + t) : 0;
  }
  __syncthreads();  // the row's p_idx (written by warp 0) and sF are visible to the CTA
  for (int k = wi; k < np; k += 4) {
    const long long e = bsm_idx(pstart + k, p.nP, p.err);
    const int j = p.p_idx[e];
    QuadBits qb;
    if (KIND == MASK_INTERVALS)
      qb = payload_intervals_entry(p, e, j, q_len, k_len, q0, hm, q_off, sF, smem);
    else
      qb = payload_blocks_entry(p, e, j, q_len, k_len, q0, hm);
    qb.reduce();
    if (lane == 0) {
      p.halves[e] = static_cast<uint8_t>(qb.halves());
      p.quads[e] = static_cast<uint8_t>(qb.quads());
    }
  }
}

// ------------------------------------------------------------ K2Q view
// §4.7 K2Q materialisation, one CTA (4 warps) per (K row, mask head), after
// the Q2K back stage: warp 0 reads the row's K tile bit out of the Q-major
// bitsets of every Q row of the sample, 32 Q rows per ballot, and writes the
// ascending partial and full Q tile lists with each entry's dQ write rank
// (the K tile's rank among the Q row's non-empty tiles: ascending K order);
// then the 4 warps transpose each partial entry's Q2K predicate words into
// the key-major layout of the K-major consumer (one word per key and 32
// queries, 32 ballots per 32x32 bit block).
struct K2QParams {
  // exact-size copies into the plan
  const int32_t* src[4];
  int32_t* dst[4];
  long long count[4];
  // workspace
  const uint32_t* vis_bits;
  const uint32_t* full_bits;
  const int32_t* seq;
  const int32_t* cu_krows;
  const int32_t* krow_batch;
  const int32_t* kp_off;
  const int32_t* kf_off;
  int rows_ub, nq_max, words;
  // plan
  const int32_t* p_off;      // Q2K partial offsets [Hmask*rows+1]
  const uint32_t* payload;   // Q2K payload [P*128*4]
  int32_t* kp_idx;
  int32_t* kf_idx;
  int32_t* dq_order;
  int32_t* dq_order_full;
  uint32_t* kpayload;        // [P'*128*4]: key c, word w, bit l = (query 32w+l, key c) visible
  // quadrant-exact block plans (64-aligned blocks, 64-multiple lengths): the
  // Q2K quadrant bits, from which the key-major words follow directly
  const uint8_t* quads;
  int rows, k_rows;
  // bounds of the checked build: Q2K partial entries, K2Q partial and full
  // entries, and the device error word
  long long nP, kP, kF;
  uint32_t* err;
};

__device__ __forceinline__ int popc_below(const uint32_t* wv, int j) {
  int n = 0;
  for (int w = 0; w < (j >> 5); ++w) n += __popc(__ldg(wv + w));
  return n + __popc(__ldg(wv + (j >> 5)) & ((1u << (j & 31)) - 1u));
}
__device__ __forceinline__ int popc_partial_below(const uint32_t* wv, const uint32_t* wf, int j) {
  int n = 0;
  for (int w = 0; w < (j >> 5); ++w) n += __popc(__ldg(wv + w) & ~__ldg(wf + w));
  return n + __popc((__ldg(wv + (j >> 5)) & ~__ldg(wf + (j >> 5))) & ((1u << (j & 31)) - 1u));
}

__global__ void __launch_bounds__(128) k_back_k2q(K2QParams p) {
  {
    const long long tid = (static_cast<long long>(blockIdx.y) * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nthreads = static_cast<long long>(gridDim.x) * gridDim.y * blockDim.x;
#pragma unroll
    for (int a = 0; a < 4; ++a)
      for (long long i = tid; i < p.count[a]; i += nthreads) p.dst[a][i] = __ldg(p.src[a] + i);
  }
  const int krow = blockIdx.x, hm = blockIdx.y;
  if (krow >= p.k_rows) return;
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int b = __ldg(p.krow_batch + krow);
  const int j = krow - __ldg(p.cu_krows + b);  // sample-local K tile
  const int nq = __ldg(p.seq + 8 * b + 5), row_begin = __ldg(p.seq + 8 * b + 4);
  const long long flat = static_cast<long long>(hm) * p.k_rows + krow;
  const int pstart = __ldg(p.kp_off + flat), np = __ldg(p.kp_off + flat + 1) - pstart;
  const long long qrow0 = static_cast<long long>(hm) * p.rows_ub + static_cast<long long>(b) * p.nq_max;
  if (wi == 0) {
    int pb = pstart, fb = __ldg(p.kf_off + flat);
    for (int i0 = 0; i0 < nq; i0 += 32) {
      const int i = i0 + lane;
      bool isp = false, isf = false;
      int rank = 0;
      if (i < nq) {
        const uint32_t* wv = p.vis_bits + (qrow0 + i) * p.words;
        const uint32_t* wf = p.full_bits + (qrow0 + i) * p.words;
        const bool v = (__ldg(wv + (j >> 5)) >> (j & 31)) & 1u;
        isf = (__ldg(wf + (j >> 5)) >> (j & 31)) & 1u;
        isp = v && !isf;
        if (v) rank = popc_below(wv, j);
      }
      const uint32_t bp = __ballot_sync(kFull, isp), bf = __ballot_sync(kFull, isf);
      const uint32_t below = (1u << lane) - 1u;
      if (isp) {
        const long long e = bsm_idx(pb + __popc(bp & below), p.kP, p.err);
        p.kp_idx[e] = i;
        p.dq_order[e] = rank;
      }
      if (isf) {
        const long long e = bsm_idx(fb + __popc(bf & below), p.kF, p.err);
        p.kf_idx[e] = i;
        p.dq_order_full[e] = rank;
      }
      pb += __popc(bp);
      fb += __popc(bf);
    }
  }
  __syncthreads();  // warp 0's Q tile lists are visible to the CTA
  for (int k = wi; k < np; k += 4) {
    const long long e = bsm_idx(pstart + k, p.kP, p.err);
    const int i = p.kp_idx[e];
    const uint32_t* wv = p.vis_bits + (qrow0 + i) * p.words;
    const uint32_t* wf = p.full_bits + (qrow0 + i) * p.words;
    const long long eq = bsm_idx(__ldg(p.p_off + static_cast<long long>(hm) * p.rows + row_begin + i) +
                                     popc_partial_below(wv, wf, j),
                                 p.nP, p.err);
    uint4* dst = reinterpret_cast<uint4*>(p.kpayload + e * (kTile * kPayloadWords));
    if (p.quads) {
      // each 64x64 quadrant is wholly visible or wholly masked: key 32 kc +
      // lane (key half kc / 2) sees query word w (query half w / 2) in full
      // exactly when the quadrant's "all visible" bit is set
      const uint32_t q = __ldg(p.quads + eq);
#pragma unroll
      for (int kc = 0; kc < kPayloadWords; ++kc) {
        uint32_t w4[kPayloadWords];
#pragma unroll
        for (int w = 0; w < kPayloadWords; ++w) w4[w] = ((q >> (4 + 2 * (w >> 1) + (kc >> 1))) & 1u) ? kFull : 0u;
        dst[32 * kc + lane] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      continue;
    }
    const uint32_t* src = p.payload + eq * (kTile * kPayloadWords);
    uint32_t mine[kPayloadWords][kPayloadWords];  // [key chunk][query word] for key 32 chunk + lane
#pragma unroll
    for (int wq = 0; wq < kPayloadWords; ++wq)
#pragma unroll
      for (int kc = 0; kc < kPayloadWords; ++kc) {
        const uint32_t v = __ldg(src + (32 * wq + lane) * kPayloadWords + kc);  // query 32 wq + lane, keys 32 kc..
        uint32_t got = 0;
#pragma unroll
        for (int bit = 0; bit < 32; ++bit) {
          const uint32_t word = __ballot_sync(kFull, (v >> bit) & 1u);  // key 32 kc + bit, queries 32 wq..
          if (lane == bit) got = word;
        }
        mine[kc][wq] = got;
      }
#pragma unroll
    for (int kc = 0; kc < kPayloadWords; ++kc)
      dst[32 * kc + lane] = make_uint4(mine[kc][0], mine[kc][1], mine[kc][2], mine[kc][3]);
  }
}

// Quotient by a divisor fixed for the whole kernel, 1 <= d < 2^31, of
// 0 <= x < 2^31, by one multiply and a shift ("Division by Invariant
// Integers using Multiplication", Granlund and Montgomery, 1994): with
// L = ceil(log2 d) and m = ceil(2^(31+L) / d), m d - 2^(31+L) < 2^L, so
// floor(x m / 2^(31+L)) = floor(x / d) for every x below 2^31.  The single
// CTA of the schedule stage is bound by instruction issue, and a 32-bit
// integer division, which the GPU carries out in software, costs it dozens
// of instructions per task.
// The multiplier costs a 64-bit division: the host forms those of divisors
// it knows, and one thread those of the rest.
struct InvDiv {
  uint32_t m;
  int sh;
  __host__ __device__ static InvDiv of(int d) {
    int L = 0;
    while ((1u << L) < static_cast<uint32_t>(d)) ++L;
    const uint64_t two = 1ull << (31 + L);
    return InvDiv{static_cast<uint32_t>((two + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d)), 31 + L};
  }
  __device__ __forceinline__ int q(int x) const {
    return static_cast<int>((static_cast<uint64_t>(static_cast<uint32_t>(x)) * m) >> sh);
  }
};

// ------------------------------------------------------------ schedule
// Reads the front stage's outputs in the workspace (the number of rows
// included) and writes work_desc there; the back stage copies it into the plan.
struct SchedParams {
  const int32_t* seq;
  const int32_t* cu_rows;
  const int32_t* row_batch;  // [rows]
  const int32_t* p_cnt;      // per padded row (mask head, sample, Q tile row): the front stage's counts
  const int32_t* f_cnt;
  int32_t* p_off;            // compact [Hmask*rows+1]: scanned here
  int32_t* f_off;
  int32_t* hist;     // [NS*(C+1)]
  int32_t* cursors;  // [NS*(C+1)]
  int32_t* work;     // [tasks*4]
  int32_t* lpt;      // [tasks] consumer order (null: not built)
  int32_t* lbkt;     // [tasks] scratch: bucket of every work_desc position
  int32_t* lhist;    // [32*(C+1)] scratch: per-warp bucket counts, then starts
  int B, Hq, Hk, Hmask, C, NS;
  int rows_ub, nq_max;
  InvDiv by_rows_ub, by_nq, by_group;  // of rows_ub, nq_max, Hq / Hk
  int in_smem;       // 1: histogram and cursors live in dynamic shared memory (2*NS*(C+1) ints)
  int bkt_smem;      // 1: the task buckets follow them there (Hq*rows_ub ints); 0: in lbkt
  uint32_t* err;     // device error word (checked build)
};

__device__ __forceinline__ int task_cost(const SchedParams& p, int rows, int h, int row) {
  const long long flat = static_cast<long long>(p.Hmask == 1 ? 0 : h) * rows + row;
  return (p.p_off[flat + 1] - p.p_off[flat]) + (p.f_off[flat + 1] - p.f_off[flat]);
}

// Bucket of a task inside its section: C - cost for cost in [1, C], C for cost 0.
__device__ __forceinline__ int task_bucket(const SchedParams& p, int cost) {
  return cost > 0 ? (p.C - min(cost, p.C)) : p.C;
}

// Lanes of `amask` whose v equals this lane's (v in [0, 2^nbits)), by one
// ballot per bit of v; the calling lane must be in amask.
__device__ __forceinline__ unsigned lanes_with_same(unsigned amask, int v, int nbits) {
  unsigned same = amask;
  for (int k = 0; k < nbits; ++k) {
    const unsigned bal = __ballot_sync(amask, (v >> k) & 1);
    same &= ((v >> k) & 1) ? bal : ~bal;
  }
  return same;
}

// One CTA builds the whole schedule with bounded counting:
//  1. every task's cost bucket, kept per (head, row), and the histogram of
//     (section, cost bucket), the whole CTA over the tasks (four per thread
//     and pass, their loads issued together; lanes with the same histogram
//     cell add once);
//  2. offsets: positive-cost tasks of section s start after every positive
//     task of sections < s, ordered by bucket (cost descending); zero-cost
//     tasks follow every positive task, sections in order (section totals
//     and bucket cursors one warp per section, starts by a block scan);
//  3. scatter: one warp per section walks its tasks in tie order (head in the
//     section's group, then m_block), 32 at a time, reading the buckets of
//     step 1; lanes with the same bucket take consecutive slots in lane
//     order, so the sort is stable.
// Section s = (sample b, K/V head hk).
__global__ void __launch_bounds__(1024) k_schedule(SchedParams p) {
  const int C = p.C;
  const int nbits = 32 - __clz(C);  // buckets lie in [0, C]
  const int group = p.Hq / p.Hk;
  const int rows = p.cu_rows[p.B];
  const long long nb = static_cast<long long>(p.NS) * (C + 1);
  extern __shared__ int32_t s_counts[];
  int32_t* const hist = p.in_smem ? s_counts : p.hist;
  int32_t* const cursors = p.in_smem ? s_counts + nb : p.cursors;
  int32_t* const bkt = p.bkt_smem ? s_counts + 2 * nb : p.lbkt;  // [Hq*rows]: bucket of task (head, row)
  for (long long i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0;
  {
    // 0. the Q2K offsets (the plan's partial/full offsets): exclusive scans
    //    of the front stage's per-row counts, padded rows in compact order
    __shared__ int32_t s_cu[kCuSmem + 1];
    __shared__ __align__(16) int32_t s_sa[4 * 1024], s_sc[4 * 1024];  // staging of the scan (blockDim.x <= 1024)
    const bool cu_smem = p.B <= kCuSmem;
    if (cu_smem)
      for (int b = threadIdx.x; b <= p.B; b += blockDim.x) s_cu[b] = p.cu_rows[b];
    __syncthreads();
    long long cp = 0, cf = 0;
    const InvDiv by_rows_ub = p.by_rows_ub, by_nq = p.by_nq;
    scan_pair_staged<4>(static_cast<long long>(p.Hmask) * p.rows_ub, static_cast<long long>(p.Hmask) * rows, p.p_cnt,
                        p.f_cnt, p.p_off, p.f_off, s_sa, s_sc, cp, cf, [&](long long x, long long& ci) {
                       // x < Hmask * rows_ub < 2^31 (bounded on the host)
                       const int xi = static_cast<int>(x);
                       const int hm = by_rows_ub.q(xi), xr = xi - hm * p.rows_ub;
                       const int b = by_nq.q(xr), lr = xr - b * p.nq_max;
                       const int c0 = cu_smem ? s_cu[b] : p.cu_rows[b];
                       const int c1 = cu_smem ? s_cu[b + 1] : p.cu_rows[b + 1];
                       if (lr >= c1 - c0) return false;
                       ci = static_cast<long long>(hm) * rows + c0 + lr;
                       return true;
                     });
  }
  const int lane = threadIdx.x & 31;
  const int T = p.Hq * rows;  // fits: the host bounds Hq * rows_ub below 2^31
  constexpr int kPer = 4;
  __shared__ InvDiv s_by_rows;
  if (threadIdx.x == 0) s_by_rows = InvDiv::of(max(rows, 1));
  __syncthreads();
  const InvDiv by_rows = s_by_rows, by_group = p.by_group;
  for (int base = 0; base < T; base += kPer * static_cast<int>(blockDim.x)) {
    int cost[kPer], sct[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int f = base + u * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
      cost[u] = 0;
      sct[u] = 0;
      if (f < T) {
        const int h = by_rows.q(f), r = f - h * rows;
        cost[u] = task_cost(p, rows, h, r);
        sct[u] = __ldg(p.row_batch + r) * p.Hk + by_group.q(h);
      }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int f = base + u * static_cast<int>(blockDim.x) + static_cast<int>(threadIdx.x);
      if (f < T) {
        const int bucket = task_bucket(p, cost[u]);
        bkt[f] = bucket;
        atomicAdd(&hist[static_cast<long long>(sct[u]) * (C + 1) + bucket], 1);
      }
    }
  }
  __syncthreads();
  // 2a. positive-cost tasks per section (one warp per section, lanes over
  //     buckets); kept in the section's bucket-0 cursor until 2b
  for (int sct = threadIdx.x >> 5; sct < p.NS; sct += blockDim.x >> 5) {
    const int32_t* h = hist + static_cast<long long>(sct) * (C + 1);
    long long tot = 0;
    for (int c = lane; c < C; c += 32) tot += h[c];
#pragma unroll
    for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(kFull, tot, o);
    if (lane == 0) cursors[static_cast<long long>(sct) * (C + 1)] = static_cast<int32_t>(tot);
  }
  __syncthreads();
  // 2b. section starts: positive tasks of section s after those of sections
  //     < s; zero-cost tasks after every positive task, sections in order
  __shared__ long long s_tot_pos;
  long long carry_pos = 0;
  for (int base = 0; base < p.NS; base += 1024) {
    const int sct = base + threadIdx.x;
    const long long pos = (sct < p.NS) ? cursors[static_cast<long long>(sct) * (C + 1)] : 0;
    long long tot;
    const long long start = carry_pos + block_excl_scan(pos, &tot);
    if (sct < p.NS) cursors[static_cast<long long>(sct) * (C + 1)] = static_cast<int32_t>(start);
    carry_pos += tot;
  }
  if (threadIdx.x == 0) s_tot_pos = carry_pos;
  __syncthreads();
  long long carry_zero = s_tot_pos;
  for (int base = 0; base < p.NS; base += 1024) {
    const int sct = base + threadIdx.x;
    const long long z = (sct < p.NS) ? hist[static_cast<long long>(sct) * (C + 1) + C] : 0;
    long long tot;
    const long long start = carry_zero + block_excl_scan(z, &tot);
    if (sct < p.NS) cursors[static_cast<long long>(sct) * (C + 1) + C] = static_cast<int32_t>(start);
    carry_zero += tot;
  }
  __syncthreads();
  // 2c. bucket cursors inside each section: its start plus an exclusive scan
  //     of its bucket counts (one warp per section, 32 buckets at a time)
  for (int sct = threadIdx.x >> 5; sct < p.NS; sct += blockDim.x >> 5) {
    const int32_t* h = hist + static_cast<long long>(sct) * (C + 1);
    int32_t* cur = cursors + static_cast<long long>(sct) * (C + 1);
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
    int32_t* cur = cursors + static_cast<long long>(sct) * (C + 1);
    InvDiv by_nrows{0u, 0};
    if (lane == 0) by_nrows = InvDiv::of(max(nrows, 1));
    by_nrows.m = __shfl_sync(kFull, by_nrows.m, 0);
    by_nrows.sh = __shfl_sync(kFull, by_nrows.sh, 0);
    for (int t0 = 0; t0 < n; t0 += 32) {
      const int t = t0 + lane;
      const bool act = t < n;
      const unsigned amask = __ballot_sync(kFull, act);
      if (act) {
        const int hg = by_nrows.q(t), m = t - hg * nrows;
        const int h = hk * group + hg;
        const int bucket = bkt[h * rows + begin + m];
        const unsigned same = lanes_with_same(amask, bucket, nbits);
        const int rank = __popc(same & ((1u << lane) - 1));
        const int pos = cur[bucket] + rank;
        // one 16-byte store per entry (work_desc is 16-byte aligned)
        *reinterpret_cast<int4*>(p.work + 4LL * bsm_idx(pos, static_cast<long long>(p.Hq) * rows, p.err)) =
            make_int4(m, h, b, min(kTile, q_len - m * kTile));
        __syncwarp(amask);
        if (rank == 0) cur[bucket] += __popc(same);
      }
      __syncwarp();
    }
  }
  // 4. the consumer order (lpt): every work_desc position by cost bucket
  //    (cost descending, zero-cost tasks last), stable in work_desc order --
  //    the longest-first order in which a consumer with few tasks per SM
  //    takes them.  Per-warp bucket counts over contiguous chunks of
  //    positions, a scan over (bucket, warp), then each warp scatters its
  //    chunk in order.
  if (p.lpt != nullptr) {
    __syncthreads();  // every work_desc entry is written
    const long long T = static_cast<long long>(p.Hq) * rows;
    const int nw = blockDim.x >> 5, w = threadIdx.x >> 5;
    const long long chunk = (T + nw - 1) / nw;
    const long long c0 = min(T, static_cast<long long>(w) * chunk), c1 = min(T, c0 + chunk);
    int32_t* wh = p.lhist + static_cast<long long>(w) * (C + 1);
    for (int c = lane; c <= C; c += 32) wh[c] = 0;
    __syncwarp();
    for (long long i = c0 + lane; i < c1; i += 32) {
      const int32_t* wd = p.work + 4 * i;
      const int b = wd[2];
      const int row = p.seq[8 * b + 4] + wd[0];
      // (the buckets of step 1 when they are in shared memory; lbkt is
      // rewritten here, by position)
      const int bucket = p.bkt_smem ? bkt[wd[1] * rows + row] : task_bucket(p, task_cost(p, rows, wd[1], row));
      p.lbkt[i] = bucket;
      atomicAdd(&wh[bucket], 1);
    }
    __syncthreads();
    // start of (bucket c, warp w): the positions of buckets < c, then those
    // of warps < w in bucket c
    long long carry = 0;
    for (int cb = 0; cb <= C; cb += blockDim.x) {
      const int c = cb + threadIdx.x;
      long long tot_c = 0;
      if (c <= C)
        for (int ww = 0; ww < nw; ++ww) tot_c += p.lhist[static_cast<long long>(ww) * (C + 1) + c];
      long long all;
      const long long base_c = carry + block_excl_scan(tot_c, &all);
      if (c <= C) {
        long long run = base_c;
        for (int ww = 0; ww < nw; ++ww) {
          int32_t* cell = p.lhist + static_cast<long long>(ww) * (C + 1) + c;
          const int v = *cell;
          *cell = static_cast<int32_t>(run);
          run += v;
        }
      }
      carry += all;
    }
    __syncthreads();
    for (long long i0 = c0; i0 < c1; i0 += 32) {
      const long long i = i0 + lane;
      const bool act = i < c1;
      const unsigned amask = __ballot_sync(kFull, act);
      if (act) {
        const int bucket = p.lbkt[i];
        const unsigned same = lanes_with_same(amask, bucket, nbits);
        const int rank = __popc(same & ((1u << lane) - 1));
        p.lpt[bsm_idx(wh[bucket] + rank, T, p.err)] = static_cast<int32_t>(i);
        __syncwarp(amask);
        if (rank == 0) wh[bucket] += __popc(same);
      }
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------ statistics
// Visible pairs of a plan: set payload bits of the partial entries (or,
// for a plan that keeps only quadrant bits, 64 x 64 per fully visible
// quadrant) plus 128 x 128 per full entry.
__global__ void k_count_visible(const uint32_t* payload, long long nwords, const uint8_t* quads,
                                long long nquads, long long full_tiles, unsigned long long* out) {
  unsigned long long acc = 0;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < nwords; i += 256LL * gridDim.x)
    acc += __popc(payload[i]);
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < nquads; i += 256LL * gridDim.x)
    acc += 64ull * 64ull * __popc(static_cast<uint32_t>(quads[i]) >> 4);
  for (int o = 16; o; o >>= 1) acc += __shfl_down_sync(kFull, acc, o);
  if ((threadIdx.x & 31) == 0) atomicAdd(out, acc);
  if (blockIdx.x == 0 && threadIdx.x == 0)
    atomicAdd(out, static_cast<unsigned long long>(full_tiles) * kTile * kTile);
}

}  // namespace


// ====================================================================== host
cudaError_t launch_front(const Geometry& g, const MaskArgs& m, const PlanWorkspace& ws,
                         const int32_t* cu_q, const int32_t* cu_k, long long* host_header,
                         long long ticket, cudaStream_t st) {
  FrontParams p{};
  p.layout = g.layout;
  p.B = g.batch;
  p.Sq = g.seqlen_q;
  p.Sk = g.seqlen_k;
  p.total_q = g.total_q;
  p.total_k = g.total_k;
  p.nq_max = ws.nq_max;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.mask_func = m.mask_func;
  p.nfunc = m.nfunc;
  p.block_mask = m.block_mask;
  p.block_q = m.block_q;
  p.block_kv = m.block_kv;
  p.nbq = m.nbq;
  p.nbk = m.nbk;
  p.Hmask = m.Hmask;
  p.vis_bits = ws.vis_bits;
  p.full_bits = ws.full_bits;
  p.p_cnt = ws.p_cnt;
  p.f_cnt = ws.f_cnt;
  p.rows_ub = ws.rows_ub;
  p.words = ws.words;
  p.cu_rows = ws.cu_rows;
  p.seq = ws.seq;
  p.row_batch = ws.row_batch;
  p.p_off = ws.p_off;
  p.f_off = ws.f_off;
  p.header = ws.header;
  p.host_header = host_header;
  p.ticket = ticket;
  p.ctl = ws.ctl;
  p.tot = reinterpret_cast<unsigned long long*>(ws.ctl + 2);
  p.kp_cnt = ws.kp_cnt;
  p.kf_cnt = ws.kf_cnt;
  p.kt_ub = ws.kt_ub;
  p.cu_krows = ws.cu_krows;
  p.krow_batch = ws.krow_batch;
  p.kp_off = ws.kp_off;
  p.kf_off = ws.kf_off;
  // at least one CTA, so that the last-CTA stage also runs without rows
  if (m.kind == MASK_INTERVALS) {
    const dim3 grid(ws.rows_ub > 0 ? ws.rows_ub : 1, m.Hmask);
    k_front<MASK_INTERVALS><<<grid, 128, 0, st>>>(p);
  } else {
    constexpr int R = kFrontRows<MASK_BLOCKS>;
    const dim3 grid(ws.rows_ub > 0 ? (ws.rows_ub + R - 1) / R : 1, m.Hmask);
    k_front<MASK_BLOCKS><<<grid, 256, 0, st>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_schedule(const Geometry& g, const PlanWorkspace& ws, int Hmask, int num_sections,
                            int max_cost, cudaStream_t st) {
  if (ws.rows_ub == 0) return cudaSuccess;
  SchedParams p{ws.seq, ws.cu_rows, ws.row_batch, ws.p_cnt, ws.f_cnt, ws.p_off, ws.f_off, ws.hist, ws.cursors,
                ws.work, ws.lpt, ws.lbkt, ws.lhist, g.batch, g.heads_q, g.heads_k, Hmask, max_cost, num_sections,
                ws.rows_ub, ws.nq_max, InvDiv::of(ws.rows_ub), InvDiv::of(ws.nq_max),
                InvDiv::of(g.heads_q / g.heads_k), 0, 0, checked_error_word()};
  // histogram and cursors in shared memory when they fit (shared-memory
  // atomics and the single CTA's scans then stay on chip), and the task
  // buckets after them when those fit too
  constexpr size_t kSchedSmemMax = 160 * 1024;
  const size_t bytes = 8ull * num_sections * (max_cost + 1);
  const size_t bkt_bytes = 4ull * g.heads_q * ws.rows_ub;
  size_t dyn = 0;
  if (bytes <= kSchedSmemMax) {
    static std::atomic<bool> attr_set[128];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
      if (cudaFuncSetAttribute(k_schedule, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSchedSmemMax)) != cudaSuccess)
        return cudaGetLastError();
      attr_set[dev].store(true, std::memory_order_release);
    }
    p.in_smem = 1;
    dyn = bytes;
    if (bytes + bkt_bytes <= kSchedSmemMax) {
      p.bkt_smem = 1;
      dyn += bkt_bytes;
    }
  }
  k_schedule<<<1, 1024, dyn, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_back(const Geometry& g, const MaskArgs& m, const PlanWorkspace& ws, fa_plan* plan,
                        const int32_t* cu_q_src, const int32_t* cu_k_src, cudaStream_t st) {
  const int rows = static_cast<int>(plan->rows);
  const long long nflat = static_cast<long long>(m.Hmask) * rows;
  BackParams p{};
  const int32_t* src[8] = {ws.cu_rows, ws.seq, ws.p_off, ws.f_off, cu_q_src, cu_k_src, ws.work, ws.lpt};
  int32_t* dst[8] = {plan->cu_q_rows, plan->seq_desc, plan->p_off, plan->f_off, plan->cu_seqlens_q,
                     plan->cu_seqlens_k, plan->work_desc, plan->lpt};
  const long long cnt[8] = {g.batch + 1LL, 8LL * g.batch, nflat + 1, nflat + 1,
                            (g.layout == FA_LAYOUT_THD) ? g.batch + 1LL : 0,
                            (g.layout == FA_LAYOUT_THD) ? g.batch + 1LL : 0, 4LL * plan->tasks,
                            (ws.lpt != nullptr) ? plan->tasks : 0};
  for (int a = 0; a < 8; ++a) {
    p.src[a] = src[a];
    p.dst[a] = dst[a];
    p.count[a] = cnt[a];
  }
  p.vis_bits = ws.vis_bits;
  p.full_bits = ws.full_bits;
  p.p_off = ws.p_off;
  p.f_off = ws.f_off;
  p.row_batch = ws.row_batch;
  p.seq = ws.seq;
  p.p_idx = plan->p_idx;
  p.f_idx = plan->f_idx;
  p.entry_row = plan->entry_row;
  p.payload = plan->payload;
  p.halves = plan->halves;
  p.quads = plan->quads;
  p.rows = rows;
  p.rows_ub = ws.rows_ub;
  p.nq_max = ws.nq_max;
  p.words = ws.words;
  p.mask_func = m.mask_func;
  p.nfunc = m.nfunc;
  p.total_q = g.total_q;
  p.block_mask = m.block_mask;
  p.block_q = m.block_q;
  p.block_kv = m.block_kv;
  p.nbq = m.nbq;
  p.nbk = m.nbk;
  p.nP = plan->P;
  p.nF = plan->F;
  p.err = checked_error_word();
  const dim3 grid(rows > 0 ? rows : 1, rows > 0 ? m.Hmask : 1);
  if (m.kind == MASK_INTERVALS)
    k_back<MASK_INTERVALS><<<grid, 128, 0, st>>>(p);
  else
    k_back<MASK_BLOCKS><<<grid, 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_back_k2q(const Geometry& g, const PlanWorkspace& ws, fa_plan* plan, cudaStream_t st) {
  K2QParams p{};
  const long long nflat = static_cast<long long>(plan->Hmask) * plan->k_rows + 1;
  p.src[0] = ws.cu_krows;   p.dst[0] = plan->cu_krows;   p.count[0] = g.batch + 1;
  p.src[1] = ws.krow_batch; p.dst[1] = plan->krow_batch; p.count[1] = plan->k_rows;
  p.src[2] = ws.kp_off;     p.dst[2] = plan->kp_off;     p.count[2] = nflat;
  p.src[3] = ws.kf_off;     p.dst[3] = plan->kf_off;     p.count[3] = nflat;
  p.vis_bits = ws.vis_bits;
  p.full_bits = ws.full_bits;
  p.seq = ws.seq;
  p.cu_krows = ws.cu_krows;
  p.krow_batch = ws.krow_batch;
  p.kp_off = ws.kp_off;
  p.kf_off = ws.kf_off;
  p.rows_ub = ws.rows_ub;
  p.nq_max = ws.nq_max;
  p.words = ws.words;
  p.p_off = plan->p_off;
  p.payload = plan->payload;
  p.kp_idx = plan->kp_idx;
  p.kf_idx = plan->kf_idx;
  p.dq_order = plan->dq_order;
  p.dq_order_full = plan->dq_order_full;
  p.kpayload = plan->kpayload;
  p.rows = static_cast<int>(plan->rows);
  p.k_rows = static_cast<int>(plan->k_rows);
  p.nP = plan->P;
  p.kP = plan->kP;
  p.kF = plan->kF;
  p.err = checked_error_word();
  const bool exact = plan->mask_kind == MASK_BLOCKS && plan->block_q % 64 == 0 && plan->block_kv % 64 == 0 &&
                     plan->geom.seqlen_q % 64 == 0 && plan->geom.seqlen_k % 64 == 0;
  p.quads = exact ? plan->quads : nullptr;
  const dim3 grid(plan->k_rows > 0 ? static_cast<unsigned>(plan->k_rows) : 1u, plan->Hmask);
  k_back_k2q<<<grid, 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_count_visible(const fa_plan* plan, unsigned long long* out, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(unsigned long long), st);
  if (e != cudaSuccess) return e;
  const long long nwords = plan->quads_only ? 0 : plan->P * kTile * kPayloadWords;
  const long long nquads = plan->quads_only ? plan->P : 0;
  k_count_visible<<<1024, 256, 0, st>>>(plan->payload, nwords, plan->quads, nquads, plan->F, out);
  return cudaGetLastError();
}

}  // namespace bsm

// ================================================= allocation-free sizing
// Scratch of fa_plan_header_noalloc: the front stage above writes its
// workspace here instead of into memory obtained from an allocator.  Every device on which the library is loaded holds
// this array until the process exits.
static constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace bsm {
namespace {

// Device address of g_noalloc_scratch for device `dev` (current).  In host
// code the symbol itself is only a host-side stand-in, so kernels must get
// this address.  Outside stream capture it is looked up on every call (a
// cheap host-side query), so that a device reset or another context on the
// device is picked up; during capture, where the lookup might have to load
// the module, the address from the last call outside capture is used.
void* noalloc_scratch_address(int dev, cudaStream_t st, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[128] = {};
  *err = cudaSuccess;
  if (dev < 0 || dev >= 128) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const bool capturing = cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lk(mu);
  if (!capturing || !addr[dev]) {
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
  const size_t sizes[] = {24, 64, 4ull * (B + 1), 32ull * B, 4ull * rows_ub, 4ull * nflat * words,
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
  uint8_t* base = static_cast<uint8_t*>(noalloc_scratch_address(dev, static_cast<cudaStream_t>(stream), &e));
  if (!base) return report_error(FA_ERR_CUDA, "cudaGetSymbolAddress of the scratch array: %s", cudaGetErrorString(e));
  PlanWorkspace ws{};
  ws.ctl = reinterpret_cast<unsigned*>(base + off[0]);
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
  ws.nq_max = static_cast<int>(nq_max);
  ws.kt_ub = static_cast<int>(kt_ub);
  ws.words = static_cast<int>(words);
  MaskArgs m{};
  m.kind = MASK_INTERVALS;
  m.mask_func = mask_func;
  m.nfunc = nfunc;
  m.Hmask = Hmask;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the front stage leaves its control words at zero, but a call whose
  // launch failed half-way is not known to have: start from zero every time
  e = cudaMemsetAsync(ws.ctl, 0, 24, st);
  if (e == cudaSuccess)
    e = launch_front(g, m, ws, geom->cu_seqlens_q, geom->cu_seqlens_k, nullptr, 0, st);
  if (e != cudaSuccess) return report_error(FA_ERR_CUDA, "allocation-free planner stage: %s", cudaGetErrorString(e));
  return FA_OK;
}

