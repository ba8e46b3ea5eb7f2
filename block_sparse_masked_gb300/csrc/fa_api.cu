// fa_api.cu -- the C ABI declared in include/fa.h: host validation,
// consumer resolution, plan ownership and the single header readback of the
// planner ("Flex Attention Mask Plan Design" §4.1, §4.5, §7, §8).
#include <cuda_runtime.h>

#include <chrono>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

namespace {

thread_local std::string t_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- memory
// Default allocator: one stream-ordered pool per device that keeps its
// memory (release threshold = max), so repeated plan builds do not go back
// to the driver.
cudaMemPool_t pool_for(int dev) {
  static std::mutex mu;
  static cudaMemPool_t pools[128] = {};
  if (dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pl = nullptr;
    if (cudaMemPoolCreate(&pl, &props) != cudaSuccess) return nullptr;
    uint64_t thr = ~0ull;
    cudaMemPoolSetAttribute(pl, cudaMemPoolAttrReleaseThreshold, &thr);
    pools[dev] = pl;
  }
  return pools[dev];
}

struct Alloc {
  const fa_allocator* custom;
  int dev;
  cudaStream_t st;
  void* get(size_t bytes) {
    if (bytes == 0) bytes = 256;
    if (custom && custom->alloc) return custom->alloc(bytes, st, custom->ctx);
    cudaMemPool_t pl = pool_for(dev);
    if (!pl) return nullptr;
    void* p = nullptr;
    if (cudaMallocFromPoolAsync(&p, bytes, pl, st) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return p;
  }
  void put(void* p, size_t bytes) {
    if (!p) return;
    if (bytes == 0) bytes = 256;
    if (custom && custom->free) {
      custom->free(p, bytes, st, custom->ctx);
      return;
    }
    cudaFreeAsync(p, st);
  }
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Carves consecutive 256-byte-aligned sub-arrays out of one allocation.
struct Carver {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  }
};

// Host memory the front stage writes the header into: 8 values, then the
// build's ticket, published last.  One per host thread: a thread waits for
// its header before it starts another build.
long long* pinned_header() {
  thread_local long long* h = nullptr;
  if (!h) {
    void* p = nullptr;
    if (cudaMallocHost(&p, 16 * sizeof(long long)) != cudaSuccess) return nullptr;
    h = static_cast<long long*>(p);
    for (int i = 0; i < 16; ++i) h[i] = 0;
  }
  return h;
}

// Event recorded after the front launch, per host thread and device: the
// header wait polls it to notice a failed launch.
cudaEvent_t front_event(int dev) {
  thread_local cudaEvent_t ev[128] = {};
  if (dev < 0 || dev >= 128) return nullptr;
  if (!ev[dev] && cudaEventCreateWithFlags(&ev[dev], cudaEventDisableTiming) != cudaSuccess) return nullptr;
  return ev[dev];
}

// Control words of the front stage (two 32-bit words, then two 64-bit
// entry totals; zero at launch and left at zero by it): a per-device free
// list hands each in-flight build its own set.  New sets are zeroed in
// stream order before their first use.
std::mutex g_ctl_mu;
std::vector<unsigned*> g_ctl_free[128];

unsigned* ctl_take(int dev, cudaStream_t st) {
  if (dev < 0 || dev >= 128) return nullptr;
  {
    std::lock_guard<std::mutex> lk(g_ctl_mu);
    if (!g_ctl_free[dev].empty()) {
      unsigned* p = g_ctl_free[dev].back();
      g_ctl_free[dev].pop_back();
      return p;
    }
  }
  void* p = nullptr;
  if (cudaMalloc(&p, 256) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (cudaMemsetAsync(p, 0, 24, st) != cudaSuccess) {
    cudaFree(p);
    return nullptr;
  }
  return static_cast<unsigned*>(p);
}

void ctl_give(int dev, unsigned* p) {
  std::lock_guard<std::mutex> lk(g_ctl_mu);
  g_ctl_free[dev].push_back(p);
}

// Waits until the front stage has published `ticket`, polling host memory;
// every 64 polls the event after the launch is checked, so that a failed
// launch or a kernel that ended without publishing returns an error.
cudaError_t wait_header(long long* hh, long long ticket, cudaEvent_t ev) {
  for (unsigned spin = 1;; ++spin) {
    if (__atomic_load_n(hh + 8, __ATOMIC_ACQUIRE) == ticket) return cudaSuccess;
    if ((spin & 63) == 0) {
      const cudaError_t q = cudaEventQuery(ev);
      if (q == cudaErrorNotReady) continue;
      if (q != cudaSuccess) return q;
      if (__atomic_load_n(hh + 8, __ATOMIC_ACQUIRE) == ticket) return cudaSuccess;
      return cudaErrorUnknown;
    }
  }
}

int cdiv(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

int check_geometry(const fa_geometry* g) {
  if (!g) return fail(FA_ERR_INVALID_ARG, "geometry is NULL");
  if (g->layout != FA_LAYOUT_BSHD && g->layout != FA_LAYOUT_THD)
    return fail(FA_ERR_INVALID_ARG, "layout must be FA_LAYOUT_BSHD or FA_LAYOUT_THD");
  if (g->dtype != FA_DTYPE_BF16) return fail(FA_ERR_UNSUPPORTED, "dtype must be FA_DTYPE_BF16");
  if (g->batch < 1) return fail(FA_ERR_INVALID_ARG, "batch must be >= 1");
  if (g->seqlen_q < 0 || g->seqlen_k < 0) return fail(FA_ERR_INVALID_ARG, "negative sequence length");
  if (g->heads_q < 1 || g->heads_k < 1 || g->heads_q % g->heads_k != 0)
    return fail(FA_ERR_INVALID_ARG, "heads_q must be a positive multiple of heads_k");
  if (g->heads_q > bsm::kMaxHeads) return fail(FA_ERR_UNSUPPORTED, "heads_q > %d", bsm::kMaxHeads);
  if (g->head_dim != 64 && g->head_dim != 128) return fail(FA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (g->layout == FA_LAYOUT_THD) {
    if (!g->cu_seqlens_q || !g->cu_seqlens_k) return fail(FA_ERR_INVALID_ARG, "THD needs cu_seqlens_q/k");
    if (g->total_q < 0 || g->total_k < 0) return fail(FA_ERR_INVALID_ARG, "negative token totals");
  } else {
    const long long tq = static_cast<long long>(g->batch) * g->seqlen_q;
    const long long tk = static_cast<long long>(g->batch) * g->seqlen_k;
    if (tq > 0x7fffffffLL || tk > 0x7fffffffLL) return fail(FA_ERR_UNSUPPORTED, "more than 2^31 rows");
  }
  return FA_OK;
}

bsm::Geometry to_geom(const fa_geometry* g) {
  bsm::Geometry r{};
  r.layout = g->layout;
  r.batch = g->batch;
  r.seqlen_q = g->seqlen_q;
  r.seqlen_k = g->seqlen_k;
  if (g->layout == FA_LAYOUT_BSHD) {
    r.total_q = g->batch * g->seqlen_q;
    r.total_k = g->batch * g->seqlen_k;
  } else {
    r.total_q = g->total_q;
    r.total_k = g->total_k;
  }
  r.heads_q = g->heads_q;
  r.heads_k = g->heads_k;
  r.head_dim = g->head_dim;
  r.dtype = g->dtype;
  return r;
}

uint64_t fnv(uint64_t h, int64_t v) {
  for (int i = 0; i < 8; ++i) {
    h ^= static_cast<uint64_t>((v >> (8 * i)) & 0xff);
    h *= 1099511628211ull;
  }
  return h;
}

void free_plan_mem(fa_plan* p, cudaStream_t st) {
  Alloc al{p->custom_alloc ? &p->alloc : nullptr, p->device, st};
  al.put(p->mem.ptr, p->mem.bytes);
  p->mem.ptr = nullptr;
  al.put(p->bmem.ptr, p->bmem.bytes);
  p->bmem.ptr = nullptr;
}

int build_common(const fa_geometry* gi, const bsm::MaskArgs& margs, uint32_t flags,
                 const fa_allocator* allocator, void* stream, fa_plan** out) {
  const auto t0 = std::chrono::steady_clock::now();
  if (!out) return fail(FA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (int e = check_geometry(gi)) return e;
  const bsm::Geometry g = to_geom(gi);
  const int B = g.batch;

  // upper bounds of the planner workspace (§4.5: exact sizes come from the header)
  const int nq_max = cdiv(g.seqlen_q, bsm::kTile);
  const int kt_ub = cdiv(g.seqlen_k, bsm::kTile);
  // B * ceil(max_q / 128) bounds the rows even for prefixes that fail validation,
  // because the geometry stage clamps every sample length to max_seqlen_q.
  const long long rows_ub_ll = static_cast<long long>(B) * nq_max;
  if (rows_ub_ll > (1LL << 26)) return fail(FA_ERR_UNSUPPORTED, "too many Q tiles");
  if (rows_ub_ll * margs.Hmask >= (1LL << 31)) return fail(FA_ERR_UNSUPPORTED, "too many Q tiles x mask heads");
  // forward tasks (Q tiles x Q heads) are indexed in 32-bit arithmetic
  if (rows_ub_ll * g.heads_q >= (1LL << 31)) return fail(FA_ERR_UNSUPPORTED, "too many Q tiles x Q heads");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return cuda_fail(e, "cudaGetDevice");
  const int rows_ub = static_cast<int>(rows_ub_ll);
  const int words = std::max(1, cdiv(kt_ub, 32));
  const int Hmask = margs.Hmask;

  bsm::PlanWorkspace ws{};
  ws.rows_ub = rows_ub;
  ws.nq_max = nq_max;
  ws.kt_ub = kt_ub;
  ws.words = words;
  const long long nflat_ub = static_cast<long long>(Hmask) * rows_ub;
  const int NS = B * g.heads_k;  // schedule sections
  const int C = kt_ub;           // largest task cost
  Carver c1;
  const size_t o_hdr = c1.take(64), o_cur = c1.take(4ull * (B + 1)),
               o_seq = c1.take(32ull * B), o_rb = c1.take(4ull * rows_ub),
               o_vis = c1.take(4ull * nflat_ub * words), o_full = c1.take(4ull * nflat_ub * words),
               o_pc = c1.take(4ull * nflat_ub), o_fc = c1.take(4ull * nflat_ub),
               o_po = c1.take(4ull * (nflat_ub + 1)), o_fo = c1.take(4ull * (nflat_ub + 1)),
               o_hist = c1.take(4ull * NS * (C + 1)), o_cursor = c1.take(4ull * NS * (C + 1)),
               o_work = c1.take(16ull * rows_ub * g.heads_q), o_lpt = c1.take(4ull * rows_ub * g.heads_q),
               o_lbkt = c1.take(4ull * rows_ub * g.heads_q), o_lhist = c1.take(4ull * 32 * (C + 1));
  // backward K2Q view: padded K rows (mask head, sample, K tile)
  const bool bwd = (flags & FA_PLAN_BACKWARD) != 0;
  const long long kflat_ub = bwd ? static_cast<long long>(Hmask) * B * kt_ub : 0;
  const size_t o_kpc = c1.take(4ull * kflat_ub), o_kfc = c1.take(4ull * kflat_ub),
               o_ckr = c1.take(bwd ? 4ull * (B + 1) : 0), o_krb = c1.take(bwd ? 4ull * B * kt_ub : 0),
               o_kpo = c1.take(bwd ? 4ull * (kflat_ub + 1) : 0), o_kfo = c1.take(bwd ? 4ull * (kflat_ub + 1) : 0);
  Alloc al{allocator, dev, st};
  uint8_t* w1 = static_cast<uint8_t*>(al.get(c1.off));
  if (!w1) return fail(FA_ERR_ALLOC, "workspace allocation of %zu bytes failed", c1.off);
  ws.header = reinterpret_cast<long long*>(w1 + o_hdr);
  ws.cu_rows = reinterpret_cast<int32_t*>(w1 + o_cur);
  ws.seq = reinterpret_cast<int32_t*>(w1 + o_seq);
  ws.row_batch = reinterpret_cast<int32_t*>(w1 + o_rb);
  ws.vis_bits = reinterpret_cast<uint32_t*>(w1 + o_vis);
  ws.full_bits = reinterpret_cast<uint32_t*>(w1 + o_full);
  ws.p_cnt = reinterpret_cast<int32_t*>(w1 + o_pc);
  ws.f_cnt = reinterpret_cast<int32_t*>(w1 + o_fc);
  ws.p_off = reinterpret_cast<int32_t*>(w1 + o_po);
  ws.f_off = reinterpret_cast<int32_t*>(w1 + o_fo);
  ws.hist = reinterpret_cast<int32_t*>(w1 + o_hist);
  ws.cursors = reinterpret_cast<int32_t*>(w1 + o_cursor);
  ws.work = reinterpret_cast<int32_t*>(w1 + o_work);
  // the longest-first order is built for interval plans only: block plans
  // are taken in work_desc order, whose sections keep each head's K/V in L2
  ws.lpt = (margs.kind == bsm::MASK_INTERVALS) ? reinterpret_cast<int32_t*>(w1 + o_lpt) : nullptr;
  ws.lbkt = reinterpret_cast<int32_t*>(w1 + o_lbkt);
  ws.lhist = reinterpret_cast<int32_t*>(w1 + o_lhist);
  if (bwd) {
    ws.kp_cnt = reinterpret_cast<int32_t*>(w1 + o_kpc);
    ws.kf_cnt = reinterpret_cast<int32_t*>(w1 + o_kfc);
    ws.cu_krows = reinterpret_cast<int32_t*>(w1 + o_ckr);
    ws.krow_batch = reinterpret_cast<int32_t*>(w1 + o_krb);
    ws.kp_off = reinterpret_cast<int32_t*>(w1 + o_kpo);
    ws.kf_off = reinterpret_cast<int32_t*>(w1 + o_kfo);
  }

  auto bail = [&](int code) {
    al.put(w1, c1.off);
    return code;
  };

  long long* hh = pinned_header();
  if (!hh) return bail(fail(FA_ERR_ALLOC, "pinned header buffer"));
  cudaEvent_t ev = front_event(dev);
  if (!ev) return bail(fail(FA_ERR_CUDA, "event creation failed"));
  ws.ctl = ctl_take(dev, st);
  if (!ws.ctl) return bail(fail(FA_ERR_ALLOC, "planner control words"));
  thread_local long long t_ticket = 0;
  const long long ticket = ++t_ticket;
  // front stage, then the schedule, which the GPU runs while this thread
  // waits for the header, sizes the plan and allocates it
  // the K2Q counts start at zero (two adjacent sub-arrays)
  cudaError_t e = bwd ? cudaMemsetAsync(ws.kp_cnt, 0, o_ckr - o_kpc, st) : cudaSuccess;
  if (!e) e = bsm::launch_front(g, margs, ws, gi->cu_seqlens_q, gi->cu_seqlens_k, hh, ticket, st);
  if (!e) e = cudaEventRecord(ev, st);
  if (!e) e = bsm::launch_schedule(g, ws, Hmask, NS, C, st);
  if (!e) e = wait_header(hh, ticket, ev);  // the one host/device synchronisation of a build
  // after a failure the control words are not known to be zero: they are not reused
  if (e) return bail(cuda_fail(e, "planner (front stage/header)"));
  ctl_give(dev, ws.ctl);
  long long hdr[8];
  std::memcpy(hdr, hh, sizeof(hdr));
  const uint32_t err = static_cast<uint32_t>(hdr[7]);
  if (err & bsm::PLANERR_SEQLENS)
    return bail(fail(FA_ERR_INVALID_SEQLENS, "cu_seqlens failed validation (start 0, end total, "
                                             "nondecreasing, within max_seqlen)"));
  if (err & bsm::PLANERR_MASK)
    return bail(fail(FA_ERR_INVALID_MASK, "mask endpoints out of range or out of order "
                                          "(need 0 <= F0 <= ... <= F(n-1) <= k_len)"));
  if (err & bsm::PLANERR_OVERFLOW) return bail(fail(FA_ERR_UNSUPPORTED, "more than 2^30 plan entries"));
  if (bwd && (hdr[5] != hdr[1] || hdr[6] != hdr[2]))
    return bail(fail(FA_ERR_CUDA, "planner inconsistency: K2Q and Q2K entry counts differ"));

  fa_plan* plan = new (std::nothrow) fa_plan();
  if (!plan) return bail(fail(FA_ERR_ALLOC, "host allocation"));
  plan->geom = g;
  plan->Hmask = Hmask;
  plan->mask_kind = margs.kind;
  plan->rows = hdr[0];
  plan->P = hdr[1];
  plan->F = hdr[2];
  plan->tasks = plan->rows * g.heads_q;
  std::memcpy(plan->header, hdr, sizeof(hdr));
  plan->device = dev;
  plan->signature = bsm::Signature{}.hash();
  // quadrant bits alone describe every partial entry of a 64-aligned block
  // plan over 64-multiple lengths: the predicate words are then left out
  plan->quads_only = (flags & FA_PLAN_QUADRANT_PAYLOAD) && !bwd && margs.kind == bsm::MASK_BLOCKS &&
                     margs.block_q % 64 == 0 && margs.block_kv % 64 == 0 && g.seqlen_q % 64 == 0 &&
                     g.seqlen_k % 64 == 0;
  if (allocator) {
    plan->alloc = *allocator;
    plan->custom_alloc = true;
  }
  const long long nflat = static_cast<long long>(Hmask) * plan->rows;
  Carver c2;
  const size_t q_cur = c2.take(4ull * (B + 1)), q_seq = c2.take(32ull * B),
               q_po = c2.take(4ull * (nflat + 1)), q_fo = c2.take(4ull * (nflat + 1)),
               q_pi = c2.take(4ull * plan->P), q_fi = c2.take(4ull * plan->F),
               q_pay = c2.take(plan->quads_only ? 0 : 16ull * bsm::kTile * plan->P), q_work = c2.take(16ull * plan->tasks),
               q_cq = c2.take(g.layout == FA_LAYOUT_THD ? 4ull * (B + 1) : 0),
               q_ck = c2.take(g.layout == FA_LAYOUT_THD ? 4ull * (B + 1) : 0),
               q_er = c2.take(4ull * plan->P), q_hv = c2.take(plan->P), q_qd = c2.take(plan->P),
               q_lpt = c2.take(margs.kind == bsm::MASK_INTERVALS ? 4ull * plan->tasks : 0);
  uint8_t* pm = static_cast<uint8_t*>(al.get(c2.off));
  if (!pm) {
    delete plan;
    return bail(fail(FA_ERR_ALLOC, "plan allocation of %zu bytes failed", c2.off));
  }
  plan->mem.ptr = pm;
  plan->mem.bytes = c2.off;
  plan->cu_q_rows = reinterpret_cast<int32_t*>(pm + q_cur);
  plan->seq_desc = reinterpret_cast<int32_t*>(pm + q_seq);
  plan->p_off = reinterpret_cast<int32_t*>(pm + q_po);
  plan->f_off = reinterpret_cast<int32_t*>(pm + q_fo);
  plan->p_idx = reinterpret_cast<int32_t*>(pm + q_pi);
  plan->f_idx = reinterpret_cast<int32_t*>(pm + q_fi);
  plan->payload = plan->quads_only ? nullptr : reinterpret_cast<uint32_t*>(pm + q_pay);
  plan->work_desc = reinterpret_cast<int32_t*>(pm + q_work);
  plan->lpt = (margs.kind == bsm::MASK_INTERVALS) ? reinterpret_cast<int32_t*>(pm + q_lpt) : nullptr;
  if (g.layout == FA_LAYOUT_THD) {
    plan->cu_seqlens_q = reinterpret_cast<int32_t*>(pm + q_cq);
    plan->cu_seqlens_k = reinterpret_cast<int32_t*>(pm + q_ck);
  }
  plan->entry_row = reinterpret_cast<int32_t*>(pm + q_er);
  plan->halves = pm + q_hv;
  plan->quads = pm + q_qd;
  plan->block_q = margs.block_q;
  plan->block_kv = margs.block_kv;
  if (bwd) {
    plan->backward = true;
    plan->k_rows = hdr[4];
    plan->kP = hdr[5];
    plan->kF = hdr[6];
    const long long kflat = static_cast<long long>(Hmask) * plan->k_rows;
    Carver c3;
    const size_t r_ckr = c3.take(4ull * (B + 1)), r_krb = c3.take(4ull * plan->k_rows),
                 r_kpo = c3.take(4ull * (kflat + 1)), r_kfo = c3.take(4ull * (kflat + 1)),
                 r_kpi = c3.take(4ull * plan->kP), r_kfi = c3.take(4ull * plan->kF),
                 r_dq = c3.take(4ull * plan->kP), r_dqf = c3.take(4ull * plan->kF),
                 r_kpay = c3.take(16ull * bsm::kTile * plan->kP);
    uint8_t* bm = static_cast<uint8_t*>(al.get(c3.off));
    if (!bm) {
      free_plan_mem(plan, st);
      delete plan;
      return bail(fail(FA_ERR_ALLOC, "backward view allocation of %zu bytes failed", c3.off));
    }
    plan->bmem.ptr = bm;
    plan->bmem.bytes = c3.off;
    plan->cu_krows = reinterpret_cast<int32_t*>(bm + r_ckr);
    plan->krow_batch = reinterpret_cast<int32_t*>(bm + r_krb);
    plan->kp_off = reinterpret_cast<int32_t*>(bm + r_kpo);
    plan->kf_off = reinterpret_cast<int32_t*>(bm + r_kfo);
    plan->kp_idx = reinterpret_cast<int32_t*>(bm + r_kpi);
    plan->kf_idx = reinterpret_cast<int32_t*>(bm + r_kfi);
    plan->dq_order = reinterpret_cast<int32_t*>(bm + r_dq);
    plan->dq_order_full = reinterpret_cast<int32_t*>(bm + r_dqf);
    plan->kpayload = reinterpret_cast<uint32_t*>(bm + r_kpay);
  }

  // exact-size copies (the schedule included), CSR lists, payloads: one launch
  e = bsm::launch_back(g, margs, ws, plan, gi->cu_seqlens_q, gi->cu_seqlens_k, st);
  if (!e && bwd) e = bsm::launch_back_k2q(g, ws, plan, st);
  if (e) {
    free_plan_mem(plan, st);
    delete plan;
    return bail(cuda_fail(e, "planner (back stage)"));
  }
  al.put(w1, c1.off);
  plan->build_us =
      std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
  *out = plan;
  return FA_OK;
}

}  // namespace

namespace bsm {
void clear_last_error() { t_err.clear(); }
int report_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}
int check_geometry_public(const fa_geometry* g) { return check_geometry(g); }
Geometry geometry_public(const fa_geometry* g) { return to_geom(g); }

uint64_t Signature::hash() const {
  uint64_t h = 1469598103934665603ull;
  for (int64_t v : {int64_t(arch), int64_t(direction), int64_t(kernel_family), int64_t(tile_q),
                    int64_t(tile_k), int64_t(q_stage), int64_t(cta_group), int64_t(pack_gqa),
                    int64_t(payload_layout), int64_t(scheduler_layout)})
    h = fnv(h, v);
  return h;
}
}  // namespace bsm

extern "C" {

int fa_plan_build_intervals(const fa_geometry* geom, const int32_t* mask_func, int32_t Hmask,
                            int32_t nfunc, const fa_allocator* allocator, void* stream, fa_plan** out) {
  return fa_plan_build_intervals_ex(geom, mask_func, Hmask, nfunc, 0u, allocator, stream, out);
}

int fa_plan_build_intervals_ex(const fa_geometry* geom, const int32_t* mask_func, int32_t Hmask,
                               int32_t nfunc, uint32_t flags, const fa_allocator* allocator, void* stream,
                               fa_plan** out) {
  t_err.clear();
  if (out) *out = nullptr;
  if (int e = check_geometry(geom)) return e;
  if (nfunc < 1 || nfunc % 2 != 1) return fail(FA_ERR_INVALID_ARG, "nfunc must be a positive odd integer");
  if (Hmask != 1 && Hmask != geom->heads_q) return fail(FA_ERR_INVALID_ARG, "Hmask must be 1 or heads_q");
  const bsm::Geometry g = to_geom(geom);
  if (!mask_func && g.total_q > 0) return fail(FA_ERR_INVALID_ARG, "mask_func is NULL");
  bsm::MaskArgs m{};
  m.kind = bsm::MASK_INTERVALS;
  m.mask_func = mask_func;
  m.nfunc = nfunc;
  m.Hmask = Hmask;
  if (flags & ~static_cast<uint32_t>(FA_PLAN_BACKWARD | FA_PLAN_QUADRANT_PAYLOAD))
    return fail(FA_ERR_INVALID_ARG, "unknown plan flags");
  return build_common(geom, m, flags, allocator, stream, out);
}

int fa_plan_build_blocks(const fa_geometry* geom, const uint8_t* block_mask, int32_t Hmask,
                         int32_t block_q, int32_t block_kv, const fa_allocator* allocator, void* stream,
                         fa_plan** out) {
  return fa_plan_build_blocks_ex(geom, block_mask, Hmask, block_q, block_kv, 0u, allocator, stream, out);
}

int fa_plan_build_blocks_ex(const fa_geometry* geom, const uint8_t* block_mask, int32_t Hmask,
                            int32_t block_q, int32_t block_kv, uint32_t flags, const fa_allocator* allocator,
                            void* stream, fa_plan** out) {
  t_err.clear();
  if (out) *out = nullptr;
  if (int e = check_geometry(geom)) return e;
  if (geom->layout != FA_LAYOUT_BSHD) return fail(FA_ERR_UNSUPPORTED, "block masks need FA_LAYOUT_BSHD");
  if (block_q < 1 || block_kv < 1) return fail(FA_ERR_INVALID_ARG, "block sizes must be >= 1");
  if (Hmask != 1 && Hmask != geom->heads_q) return fail(FA_ERR_INVALID_ARG, "Hmask must be 1 or heads_q");
  if (!block_mask && geom->seqlen_q > 0 && geom->seqlen_k > 0)
    return fail(FA_ERR_INVALID_ARG, "block_mask is NULL");
  bsm::MaskArgs m{};
  m.kind = bsm::MASK_BLOCKS;
  m.block_mask = block_mask;
  m.block_q = block_q;
  m.block_kv = block_kv;
  m.nbq = cdiv(geom->seqlen_q, block_q);
  m.nbk = cdiv(geom->seqlen_k, block_kv);
  m.Hmask = Hmask;
  if (flags & ~static_cast<uint32_t>(FA_PLAN_BACKWARD | FA_PLAN_QUADRANT_PAYLOAD))
    return fail(FA_ERR_INVALID_ARG, "unknown plan flags");
  return build_common(geom, m, flags, allocator, stream, out);
}

int fa_plan_free(fa_plan* plan, void* stream) {
  t_err.clear();
  if (!plan) return FA_OK;
  free_plan_mem(plan, static_cast<cudaStream_t>(stream));
  delete plan;
  return FA_OK;
}

int fa_fwd(const fa_plan* plan, const void* q, const void* k, const void* v, void* o, float* lse,
           const fa_geometry* geom, float scale, const fa_mods* mods, void* stream) {
  t_err.clear();
  if (!plan) return fail(FA_ERR_INVALID_ARG, "plan is NULL");
  if (int e = check_geometry(geom)) return e;
  const bsm::Geometry g = to_geom(geom);
  const bsm::Geometry& pg = plan->geom;
  if (g.layout != pg.layout || g.batch != pg.batch || g.seqlen_q != pg.seqlen_q || g.seqlen_k != pg.seqlen_k ||
      g.total_q != pg.total_q || g.total_k != pg.total_k || g.heads_q != pg.heads_q ||
      g.heads_k != pg.heads_k || g.head_dim != pg.head_dim || g.dtype != pg.dtype)
    return fail(FA_ERR_PLAN_MISMATCH, "geometry differs from the plan's");
  if (plan->signature != bsm::Signature{}.hash())
    return fail(FA_ERR_PLAN_MISMATCH, "plan signature differs from this consumer's");
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != plan->device) return fail(FA_ERR_PLAN_MISMATCH, "plan was built on device %d", plan->device);
  if (!(scale > 0.0f) || !std::isfinite(scale))
    return fail(FA_ERR_INVALID_ARG, "scale must be positive and finite");
  if (plan->quads_only &&
      ((mods && (mods->flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI | FA_FWD_COARSENED))) || g.head_dim != 128))
    return fail(FA_ERR_UNSUPPORTED,
                "a plan built with FA_PLAN_QUADRANT_PAYLOAD runs only the Direct 64x64 forward (head_dim 128, no mods)");
  if (plan->tasks == 0) return FA_OK;  // nothing to compute (e.g. no Q rows)
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  for (const void* ptr : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return fail(FA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  bsm::FwdLaunch a{};
  a.plan = plan;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.scale = scale;
  if (mods) {
    a.flags = mods->flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI | FA_FWD_ONE_TILE | FA_FWD_COARSENED);
    a.softcap = mods->softcap;
    a.slopes = mods->alibi_slopes;
    if ((a.flags & FA_MOD_SOFTCAP) && !(mods->softcap > 0.0f))
      return fail(FA_ERR_INVALID_ARG, "softcap must be > 0 when FA_MOD_SOFTCAP is set");
    if ((a.flags & FA_MOD_ALIBI) && !mods->alibi_slopes)
      return fail(FA_ERR_INVALID_ARG, "FA_MOD_ALIBI needs alibi_slopes");
  }
  const char* why = "";
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one launch: tasks are scheduled on the device (cluster launch control), no per-call state
  const cudaError_t e = (g.head_dim == 64) ? bsm::launch_fwd_d64(a, st, &why) : bsm::launch_fwd_d128(a, st, &why);
  if (e) return fail(FA_ERR_CUDA, "%s: %s", why, cudaGetErrorString(e));
  return FA_OK;
}

int fa_bwd(const fa_plan* plan, const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, const fa_geometry* geom, float scale,
           const fa_mods* mods, void* stream) {
  t_err.clear();
  if (!plan) return fail(FA_ERR_INVALID_ARG, "plan is NULL");
  if (!plan->backward) return fail(FA_ERR_PLAN_MISMATCH, "the plan was built without FA_PLAN_BACKWARD");
  if (int e = check_geometry(geom)) return e;
  const bsm::Geometry g = to_geom(geom);
  const bsm::Geometry& pg = plan->geom;
  if (g.layout != pg.layout || g.batch != pg.batch || g.seqlen_q != pg.seqlen_q || g.seqlen_k != pg.seqlen_k ||
      g.total_q != pg.total_q || g.total_k != pg.total_k || g.heads_q != pg.heads_q ||
      g.heads_k != pg.heads_k || g.head_dim != pg.head_dim || g.dtype != pg.dtype)
    return fail(FA_ERR_PLAN_MISMATCH, "geometry differs from the plan's");
  if (plan->signature != bsm::Signature{}.hash())
    return fail(FA_ERR_PLAN_MISMATCH, "plan signature differs from this consumer's");
  if (g.head_dim != 128) return fail(FA_ERR_UNSUPPORTED, "the backward supports head_dim 128");
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != plan->device) return fail(FA_ERR_PLAN_MISMATCH, "plan was built on device %d", plan->device);
  if (!(scale > 0.0f) || !std::isfinite(scale))
    return fail(FA_ERR_INVALID_ARG, "scale must be positive and finite");
  const long long rows_q = (g.layout == FA_LAYOUT_BSHD) ? static_cast<long long>(g.batch) * g.seqlen_q : g.total_q;
  const long long rows_k = (g.layout == FA_LAYOUT_BSHD) ? static_cast<long long>(g.batch) * g.seqlen_k : g.total_k;
  if (rows_q == 0 && rows_k == 0) return FA_OK;
  for (const void* ptr : {q, k, v, o, dout, static_cast<const void*>(lse), static_cast<const void*>(dq),
                          static_cast<const void*>(dk), static_cast<const void*>(dv)}) {
    if (!ptr) return fail(FA_ERR_INVALID_ARG, "q, k, v, o, dout, lse, dq, dk and dv must be non-NULL");
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return fail(FA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  }
  bsm::BwdLaunch a{};
  a.plan = plan;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.scale = scale;
  if (mods) {
    a.flags = mods->flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI);
    a.softcap = mods->softcap;
    a.slopes = mods->alibi_slopes;
    if ((a.flags & FA_MOD_SOFTCAP) && !(mods->softcap > 0.0f))
      return fail(FA_ERR_INVALID_ARG, "softcap must be > 0 when FA_MOD_SOFTCAP is set");
    if ((a.flags & FA_MOD_ALIBI) && !mods->alibi_slopes)
      return fail(FA_ERR_INVALID_ARG, "FA_MOD_ALIBI needs alibi_slopes");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Delta workspace [heads_q, total_q], stream-ordered, from the plan's allocator
  Alloc al{plan->custom_alloc ? &plan->alloc : nullptr, plan->device, st};
  const size_t dbytes = 4ull * static_cast<size_t>(g.heads_q) * static_cast<size_t>(rows_q > 0 ? rows_q : 1);
  a.delta = static_cast<float*>(al.get(dbytes));
  if (!a.delta) return fail(FA_ERR_ALLOC, "backward workspace of %zu bytes", dbytes);
  const char* why = "";
  const cudaError_t e = bsm::launch_bwd(a, st, &why);
  al.put(a.delta, dbytes);
  if (e) return fail(FA_ERR_CUDA, "%s: %s", why, cudaGetErrorString(e));
  return FA_OK;
}

int fa_decode_paged(const fa_plan* plan, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* page_table, int32_t pages_per_seq, int32_t page_size, int64_t num_pages,
                    void* o, float* lse, const fa_geometry* geom, float scale, const fa_mods* mods,
                    void* stream) {
  t_err.clear();
  if (!plan) return fail(FA_ERR_INVALID_ARG, "plan is NULL");
  if (int e = check_geometry(geom)) return e;
  const bsm::Geometry g = to_geom(geom);
  const bsm::Geometry& pg = plan->geom;
  if (g.layout != pg.layout || g.batch != pg.batch || g.seqlen_q != pg.seqlen_q || g.seqlen_k != pg.seqlen_k ||
      g.total_q != pg.total_q || g.total_k != pg.total_k || g.heads_q != pg.heads_q ||
      g.heads_k != pg.heads_k || g.head_dim != pg.head_dim || g.dtype != pg.dtype)
    return fail(FA_ERR_PLAN_MISMATCH, "geometry differs from the plan's");
  if (plan->signature != bsm::Signature{}.hash())
    return fail(FA_ERR_PLAN_MISMATCH, "plan signature differs from this consumer's");
  if (plan->mask_kind != bsm::MASK_INTERVALS)
    return fail(FA_ERR_UNSUPPORTED, "decoding takes interval-mask plans");
  if (g.layout != FA_LAYOUT_THD || g.seqlen_q != 1 || g.total_q != g.batch)
    return fail(FA_ERR_UNSUPPORTED, "decoding takes one query row per sequence (THD, max_seqlen_q = 1, total_q = batch)");
  if (g.head_dim != 128) return fail(FA_ERR_UNSUPPORTED, "decoding supports head_dim 128");
  const int G = g.heads_q / g.heads_k;
  if (!(plan->Hmask == 1 || (plan->Hmask == g.heads_q && G == 1)))
    return fail(FA_ERR_UNSUPPORTED, "decoding takes one mask for every head, or per-head masks without GQA");
  if (G > 64) return fail(FA_ERR_UNSUPPORTED, "decoding supports at most 64 query heads per K/V head");
  int mod_flags = 0;
  if (mods) {
    mod_flags = mods->flags & (FA_MOD_SOFTCAP | FA_MOD_ALIBI);
    if ((mod_flags & FA_MOD_SOFTCAP) && !(mods->softcap > 0.0f))
      return fail(FA_ERR_INVALID_ARG, "softcap must be > 0 when FA_MOD_SOFTCAP is set");
    if ((mod_flags & FA_MOD_ALIBI) && !mods->alibi_slopes)
      return fail(FA_ERR_INVALID_ARG, "FA_MOD_ALIBI needs alibi_slopes");
    if ((mod_flags & FA_MOD_ALIBI) && g.heads_q > bsm::kMaxHeads)
      return fail(FA_ERR_UNSUPPORTED, "ALiBi supports at most %d query heads", bsm::kMaxHeads);
  }
  if (page_size < 16 || (page_size & (page_size - 1)) != 0)
    return fail(FA_ERR_INVALID_ARG, "page_size must be a power of two >= 16");
  if (pages_per_seq < 1 || num_pages < 1 || num_pages * static_cast<int64_t>(page_size) + 128 > INT32_MAX)
    return fail(FA_ERR_INVALID_ARG, "pages_per_seq and num_pages must be >= 1 and num_pages * page_size < 2^31");
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != plan->device) return fail(FA_ERR_PLAN_MISMATCH, "plan was built on device %d", plan->device);
  if (!(scale > 0.0f) || !std::isfinite(scale))
    return fail(FA_ERR_INVALID_ARG, "scale must be positive and finite");
  if (g.total_q == 0) return FA_OK;
  for (const void* ptr : {q, k_cache, v_cache, static_cast<const void*>(o), static_cast<const void*>(page_table)})
    if (!ptr) return fail(FA_ERR_INVALID_ARG, "q, k_cache, v_cache, o and page_table must be non-NULL");
  for (const void* ptr : {q, k_cache, v_cache, static_cast<const void*>(o), static_cast<const void*>(lse)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return fail(FA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) sms = 1;
  bsm::DecodeLaunch a{};
  a.plan = plan;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.page_table = page_table;
  a.pages_per_seq = pages_per_seq;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.o = o;
  a.lse = lse;
  a.scale = scale;
  a.num_sms = sms;
  a.flags = mod_flags;
  a.softcap = mods ? mods->softcap : 0.0f;
  a.slopes = mods ? mods->alibi_slopes : nullptr;
  bsm::DecodeSizes z{};
  const size_t bytes = bsm::decode_workspace_bytes(a, &z);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Alloc al{plan->custom_alloc ? &plan->alloc : nullptr, plan->device, st};
  void* ws = al.get(bytes);
  if (!ws) return fail(FA_ERR_ALLOC, "decode workspace of %zu bytes", bytes);
  const char* why = "";
  const cudaError_t e = bsm::launch_decode(a, z, ws, st, &why);
  al.put(ws, bytes);
  if (e) return fail(FA_ERR_CUDA, "%s: %s", why, cudaGetErrorString(e));
  return FA_OK;
}

int fa_plan_info_get(const fa_plan* plan, int32_t count_visible, void* stream, fa_plan_info* info) {
  t_err.clear();
  if (!plan || !info) return fail(FA_ERR_INVALID_ARG, "plan and info must be non-NULL");
  std::memset(info, 0, sizeof(*info));
  std::memcpy(info->header, plan->header, sizeof(info->header));
  info->tile_q = bsm::kTile;
  info->tile_k = bsm::kTile;
  info->mask_heads = plan->Hmask;
  info->batch = plan->geom.batch;
  info->heads_q = plan->geom.heads_q;
  info->heads_k = plan->geom.heads_k;
  info->head_dim = plan->geom.head_dim;
  info->layout = plan->geom.layout;
  info->num_tasks = plan->tasks;
  info->payload_bytes = plan->quads_only ? 0 : plan->P * bsm::kTile * bsm::kPayloadWords * 4;
  info->plan_bytes = static_cast<int64_t>(plan->mem.bytes + plan->bmem.bytes);
  info->signature = plan->signature;
  info->build_us = plan->build_us;
  info->visible_pairs = -1;
  if (count_visible) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Alloc al{plan->custom_alloc ? &plan->alloc : nullptr, plan->device, st};
    unsigned long long* d = static_cast<unsigned long long*>(al.get(8));
    if (!d) return fail(FA_ERR_ALLOC, "8-byte counter");
    unsigned long long hv = 0;
    cudaError_t e = bsm::launch_count_visible(plan, d, st);
    if (!e) e = cudaMemcpyAsync(&hv, d, 8, cudaMemcpyDeviceToHost, st);
    if (!e) e = cudaStreamSynchronize(st);
    al.put(d, 8);
    if (e) return cuda_fail(e, "visible-pair count");
    info->visible_pairs = static_cast<int64_t>(hv);
  }
  return FA_OK;
}

int fa_plan_export(const fa_plan* plan, fa_plan_host_view* dst) {
  t_err.clear();
  if (!plan || !dst) return fail(FA_ERR_INVALID_ARG, "plan and dst must be non-NULL");
  const long long B = plan->geom.batch, nflat = static_cast<long long>(plan->Hmask) * plan->rows;
  struct Item {
    void* d;
    const void* s;
    size_t n;
  } items[] = {
      {dst->cu_q_rows, plan->cu_q_rows, 4ull * (B + 1)},
      {dst->sequence_desc, plan->seq_desc, 32ull * B},
      {dst->partial_offset, plan->p_off, 4ull * (nflat + 1)},
      {dst->partial_idx, plan->p_idx, 4ull * plan->P},
      {dst->full_offset, plan->f_off, 4ull * (nflat + 1)},
      {dst->full_idx, plan->f_idx, 4ull * plan->F},
      {dst->payload, plan->payload, plan->quads_only ? 0 : 16ull * bsm::kTile * plan->P},
      {dst->work_desc, plan->work_desc, 16ull * plan->tasks},
      {dst->halves, plan->halves, static_cast<size_t>(plan->P)},
      {dst->quads, plan->quads, static_cast<size_t>(plan->P)},
      {dst->lpt, plan->lpt, plan->lpt ? 4ull * plan->tasks : 0},
  };
  if (dst->lpt && !plan->lpt)  // block plans: work_desc order
    for (long long t = 0; t < plan->tasks; ++t) dst->lpt[t] = static_cast<int32_t>(t);
  for (auto& it : items) {
    if (!it.d || it.n == 0) continue;
    cudaError_t e = cudaMemcpy(it.d, it.s, it.n, cudaMemcpyDeviceToHost);
    if (e) return cuda_fail(e, "plan export");
  }
  return FA_OK;
}

int fa_plan_export_backward(const fa_plan* plan, fa_plan_bwd_host_view* dst) {
  t_err.clear();
  if (!plan || !dst) return fail(FA_ERR_INVALID_ARG, "plan and dst must be non-NULL");
  if (!plan->backward) return fail(FA_ERR_INVALID_ARG, "the plan was built without FA_PLAN_BACKWARD");
  const long long B = plan->geom.batch, nflat = static_cast<long long>(plan->Hmask) * plan->k_rows;
  struct Item {
    void* d;
    const void* s;
    size_t n;
  } items[] = {
      {dst->cu_k_rows, plan->cu_krows, 4ull * (B + 1)},
      {dst->partial_offset, plan->kp_off, 4ull * (nflat + 1)},
      {dst->partial_idx, plan->kp_idx, 4ull * plan->kP},
      {dst->full_offset, plan->kf_off, 4ull * (nflat + 1)},
      {dst->full_idx, plan->kf_idx, 4ull * plan->kF},
      {dst->payload, plan->kpayload, 16ull * bsm::kTile * plan->kP},
      {dst->dq_write_order, plan->dq_order, 4ull * plan->kP},
      {dst->dq_write_order_full, plan->dq_order_full, 4ull * plan->kF},
  };
  for (auto& it : items) {
    if (!it.d || it.n == 0) continue;
    cudaError_t e = cudaMemcpy(it.d, it.s, it.n, cudaMemcpyDeviceToHost);
    if (e) return cuda_fail(e, "backward view export");
  }
  return FA_OK;
}

int fa_device_error_flags(void* stream, uint32_t* flags) {
  t_err.clear();
  if (!flags) return fail(FA_ERR_INVALID_ARG, "flags is NULL");
  uint32_t* d = bsm::fwd_error_word();
  if (!d) return fail(FA_ERR_CUDA, "error word address");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flags, d, 4, cudaMemcpyDeviceToHost, st);
  if (!e) e = cudaStreamSynchronize(st);
  if (!e) e = cudaMemsetAsync(d, 0, 4, st);
  if (!e) e = cudaStreamSynchronize(st);
  if (e) return cuda_fail(e, "reading device error flags");
  return FA_OK;
}

int fa_selftest_wait_timeout(uint64_t timeout_ns, void* stream) {
  t_err.clear();
  if (timeout_ns < 1000 || timeout_ns > 100000000ull)
    return fail(FA_ERR_INVALID_ARG, "timeout_ns must be in [1 us, 100 ms]");
  cudaError_t e = bsm::launch_wait_selftest(timeout_ns, static_cast<cudaStream_t>(stream));
  if (e) return cuda_fail(e, "self-test launch");
  return FA_OK;
}

int fa_debug_set_work_desc(fa_plan* plan, int64_t task, int32_t field, int32_t value, void* stream) {
  t_err.clear();
#ifdef BSM_CHECKED
  if (plan == nullptr || task < 0 || task >= plan->tasks || field < 0 || field > 3)
    return fail(FA_ERR_INVALID_ARG, "task or field out of range");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(plan->work_desc + 4 * task + field, &value, sizeof(value),
                                  cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e) return cuda_fail(e, "work_desc write");
  return FA_OK;
#else
  (void)plan;
  (void)task;
  (void)field;
  (void)value;
  (void)stream;
  return fail(FA_ERR_UNSUPPORTED, "fa_debug_set_work_desc exists only in the bounds-checked build");
#endif
}

const char* fa_last_error(void) { return t_err.c_str(); }

const char* fa_version(void) {
#ifdef BSM_CHECKED
  return "block_sparse_masked_gb300 0.1 (sm_103a, bounds-checked)";
#else
  return "block_sparse_masked_gb300 0.1 (sm_103a)";
#endif
}

}  // extern "C"
