// internal.h -- host-side plan object and kernel launchers shared by the
// C ABI (fa_api.cu), the planner (planner.cu) and the attention forward
// (attn_fwd*.cu).  Not part of the public interface.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/fa.h"

namespace bsm {

constexpr int kTile = 128;            // physical tile, Q rows and K columns
constexpr int kPayloadWords = 4;      // uint32 words per tile row
constexpr int kMaxHeads = 256;        // heads_q limit of the forward kernel parameters

enum PlanErr : uint32_t { PLANERR_MASK = 1u, PLANERR_SEQLENS = 2u, PLANERR_OVERFLOW = 4u };
enum MaskKind : int { MASK_INTERVALS = 0, MASK_BLOCKS = 1 };

// Error bits reported by kernels (the device error word).
enum : uint32_t { DEVERR_TIMEOUT = 1u, DEVERR_SMEM_ALIGN = 2u, DEVERR_BOUNDS = 4u, DEVERR_PAGE = 8u };

// Debug builds (-DBSM_CHECKED): every plan-derived global index goes through
// bsm_idx(i, n, err), which returns i when 0 <= i < n and otherwise records
// DEVERR_BOUNDS in *err and returns 0, so that a read stays in bounds and a
// guarded write (bsm_ok) is skipped; nothing traps.  Release builds compile
// both to the plain index.
#if defined(__CUDACC__) && defined(BSM_CHECKED)
__device__ __forceinline__ long long bsm_idx(long long i, long long n, uint32_t* err) {
  if (i >= 0 && i < n) return i;
  atomicOr(err, DEVERR_BOUNDS);
  return 0;
}
__device__ __forceinline__ bool bsm_ok(long long i, long long n, uint32_t* err) {
  if (i >= 0 && i < n) return true;
  atomicOr(err, DEVERR_BOUNDS);
  return false;
}
#elif defined(__CUDACC__)
__device__ __forceinline__ long long bsm_idx(long long i, long long, uint32_t*) { return i; }
__device__ __forceinline__ bool bsm_ok(long long, long long, uint32_t*) { return true; }
#endif

// Consumer signature ("Flex Attention Mask Plan Design" §7): every field
// that fixes how the plan's topology and payload are laid out for the one
// consumer this library ships.
struct Signature {
  int32_t arch = 103;        // sm_103a
  int32_t direction = 0;     // forward
  int32_t kernel_family = 1; // tcgen05/TMEM forward, one Q tile per CTA
  int32_t tile_q = kTile, tile_k = kTile;
  int32_t q_stage = 1, cta_group = 1, pack_gqa = 0;
  int32_t payload_layout = 1;   // one TMEM lane per row, 4 words, bit l = column 32w+l
  int32_t scheduler_layout = 1; // work_desc in execution order, one task per CTA
  uint64_t hash() const;
};

struct Geometry {
  int32_t layout, batch, seqlen_q, seqlen_k, total_q, total_k, heads_q, heads_k, head_dim, dtype;
};

struct DeviceMem {
  void* ptr = nullptr;
  size_t bytes = 0;
};

}  // namespace bsm

struct fa_plan {
  bsm::Geometry geom;
  int32_t Hmask = 1;
  int32_t mask_kind = 0;
  int64_t rows = 0, P = 0, F = 0, tasks = 0;
  int64_t header[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  uint64_t signature = 0;
  int device = 0;
  double build_us = 0;
  fa_allocator alloc{};
  bool custom_alloc = false;
  bsm::DeviceMem mem;
  bsm::DeviceMem bmem;  // backward view (FA_PLAN_BACKWARD)
  // views into mem
  int32_t* cu_q_rows = nullptr;     // [B+1]
  int32_t* seq_desc = nullptr;      // [B*8]
  int32_t* p_off = nullptr;         // [Hmask*rows+1]
  int32_t* f_off = nullptr;
  int32_t* p_idx = nullptr;         // [P]
  int32_t* f_idx = nullptr;         // [F]
  uint32_t* payload = nullptr;      // [P*128*4]
  int32_t* work_desc = nullptr;     // [tasks*4]
  int32_t* lpt = nullptr;           // [tasks] work_desc positions, cost descending (stable)
  int32_t* cu_seqlens_q = nullptr;  // clones (THD)
  int32_t* cu_seqlens_k = nullptr;
  int32_t* entry_row = nullptr;     // [P] planner scratch kept with the plan: flat row of each entry
  uint8_t* halves = nullptr;        // [P] bit s: key columns 64s..64s+63 of the entry hold a visible element
  // [P] quadrant (a, s) = rows 64a.. x key columns 64s..: bit 2a+s any element visible, bit 4+2a+s all
  uint8_t* quads = nullptr;
  int32_t block_q = 0, block_kv = 0;  // logical block geometry of a block-mask plan
  bool quads_only = false;  // FA_PLAN_QUADRANT_PAYLOAD took effect: payload is null, quads describe the entries
  // backward K2Q view ("Flex Attention Mask Plan Design" §4.4, §4.7); absent
  // (k_rows = 0, null pointers) unless the plan was built with FA_PLAN_BACKWARD
  bool backward = false;
  int64_t k_rows = 0, kP = 0, kF = 0;
  int32_t* cu_krows = nullptr;       // [B+1] K plan row prefix
  int32_t* krow_batch = nullptr;     // [k_rows] sample of each K row
  int32_t* kp_off = nullptr;         // [Hmask*k_rows+1]
  int32_t* kf_off = nullptr;
  int32_t* kp_idx = nullptr;         // [kP] sample-local Q tiles, ascending per K row
  int32_t* kf_idx = nullptr;         // [kF]
  int32_t* dq_order = nullptr;       // [kP] dQ write rank (ascending K order within the Q tile)
  int32_t* dq_order_full = nullptr;  // [kF]
  uint32_t* kpayload = nullptr;      // [kP*128*4] key c, word w, bit l = (query 32w+l, key c) visible
};

namespace bsm {

// ---- planner launchers (planner.cu) -------------------------------------
// Padded rows: rows_ub = batch * nq_max (nq_max = Q tiles of the longest
// sample); padded row (b, lr) is b * nq_max + lr.
struct PlanWorkspace {
  unsigned* ctl;          // front stage control words [2]: zero before and after its launch
  long long* header;      // 8 values
  int32_t* cu_rows;       // [B+1]
  int32_t* seq;           // [B*8]
  int32_t* row_batch;     // [rows_ub]
  uint32_t* vis_bits;     // [Hmask*rows_ub*words], padded rows
  uint32_t* full_bits;
  int32_t* p_cnt;         // [Hmask*rows_ub], padded rows
  int32_t* f_cnt;
  int32_t* p_off;         // [Hmask*rows+1], compact rows
  int32_t* f_off;
  int32_t* hist;          // schedule counting buffers [num_sections*(max_cost+1)]
  int32_t* cursors;
  int32_t* work;          // schedule output [rows_ub*heads_q*4]
  int32_t* lpt;           // consumer order: work_desc positions by cost [rows_ub*heads_q]
  int32_t* lbkt;          // its scratch: cost bucket of every position [rows_ub*heads_q]
  int32_t* lhist;         // and per-warp bucket counts [32*(max_cost+1)]
  int rows_ub, nq_max, kt_ub, words;
  // backward K2Q view; kp_cnt null when not built
  int32_t* kp_cnt = nullptr;  // [Hmask*B*kt_ub], zero before the front stage
  int32_t* kf_cnt = nullptr;
  int32_t* cu_krows = nullptr;    // [B+1]
  int32_t* krow_batch = nullptr;  // [B*kt_ub]
  int32_t* kp_off = nullptr;      // [Hmask*B*kt_ub+1]
  int32_t* kf_off = nullptr;
};

struct MaskArgs {
  int kind;
  const int32_t* mask_func;   // intervals
  int nfunc;
  const uint8_t* block_mask;  // blocks
  int block_q, block_kv, nbq, nbk;
  int Hmask;
};

// Front stage (one launch): classification, then in its last CTA the
// sample descriptors, row prefixes, count scans and the header, which also
// goes to host_header[0..7] followed by host_header[8] = ticket when
// host_header is not null.  ws.ctl must be zero at launch (it is again after).
cudaError_t launch_front(const Geometry& g, const MaskArgs& m, const PlanWorkspace& ws,
                         const int32_t* cu_q, const int32_t* cu_k, long long* host_header,
                         long long ticket, cudaStream_t st);
// Task order into ws.work; needs only the front stage's outputs.
cudaError_t launch_schedule(const Geometry& g, const PlanWorkspace& ws, int Hmask, int num_sections,
                            int max_cost, cudaStream_t st);
// Back stage (one launch), once the plan is allocated from the header:
// exact-size copies into the plan, CSR lists, the entry->row map, payloads.
cudaError_t launch_back(const Geometry& g, const MaskArgs& m, const PlanWorkspace& ws, fa_plan* plan,
                        const int32_t* cu_q_src, const int32_t* cu_k_src, cudaStream_t st);
// K2Q view (FA_PLAN_BACKWARD plans), after launch_back: exact-size copies,
// Q tile lists with dQ write ranks, key-major payload.
cudaError_t launch_back_k2q(const Geometry& g, const PlanWorkspace& ws, fa_plan* plan, cudaStream_t st);
cudaError_t launch_count_visible(const fa_plan* plan, unsigned long long* out, cudaStream_t st);

// ---- forward (attn_fwd*.cu) ---------------------------------------------
struct FwdLaunch {
  const fa_plan* plan;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  float scale;
  int flags;
  float softcap;
  const float* slopes;  // host, heads_q
};
cudaError_t launch_fwd_d64(const FwdLaunch& a, cudaStream_t st, const char** why);
cudaError_t launch_fwd_d128(const FwdLaunch& a, cudaStream_t st, const char** why);
// two Q tiles per task sharing one K/V stream (attn_fwd_pair.cu; interval masks)
cudaError_t launch_fwd_pair_d64(const FwdLaunch& a, cudaStream_t st, const char** why);
cudaError_t launch_fwd_pair_d128(const FwdLaunch& a, cudaStream_t st, const char** why);
// keys-major forward for block-mask plans with 64-aligned logical blocks,
// d = 128, no score mods (attn_fwd_kt.cu)
bool fwd_kt_applies(const FwdLaunch& a);
cudaError_t launch_fwd_kt(const FwdLaunch& a, cudaStream_t st, const char** why);
// ---- backward (attn_bwd.cu), FA_PLAN_BACKWARD plans, head_dim 128 -----------
struct BwdLaunch {
  const fa_plan* plan;
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  float* delta;  // workspace [heads_q, total_q]
  void* dq;
  void* dk;
  void* dv;
  float scale;
  int flags;
  float softcap;
  const float* slopes;  // host, heads_q
};
// Delta, then the dQ kernel (forward Q2K view), then the dK/dV kernel (K2Q view).
cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t st, const char** why);

// Decoding over a paged KV cache (attn_decode.cu).
struct DecodeLaunch {
  const fa_plan* plan;
  const void* q;          // [total_q, heads_q, 128]
  const void* k_cache;    // [num_pages, page_size, heads_k, 128]
  const void* v_cache;
  const int32_t* page_table;  // device [batch, pages_per_seq]
  int pages_per_seq, page_size;
  int64_t num_pages;
  void* o;
  float* lse;
  float scale;
  int num_sms;
  int flags;             // FA_MOD_SOFTCAP | FA_MOD_ALIBI
  float softcap;
  const float* slopes;   // host, heads_q
};
struct DecodeSizes {
  int G, gy, chunks, chunk_rows, C;  // C: CTAs of the decode kernel
  long long slots;                   // piece result slots
  size_t off_remap, off_cu, off_part_o, off_part_ml, bytes;
};
// Workspace layout of one decode call; returns its size in bytes.
size_t decode_workspace_bytes(const DecodeLaunch& a, DecodeSizes* s);
// Page conversion and unit split, the decode kernel, the unit merge.
cudaError_t launch_decode(const DecodeLaunch& a, const DecodeSizes& s, void* ws, cudaStream_t st,
                          const char** why);
uint32_t* fwd_error_word();  // device address of the forward kernels' error word
// The error word the bounds checks of a checked build (-DBSM_CHECKED)
// report into; nullptr in a release build, whose checks compile away.
inline uint32_t* checked_error_word() {
#ifdef BSM_CHECKED
  return fwd_error_word();
#else
  return nullptr;
#endif
}
cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t st);

// ---- error reporting and argument checks shared with fa_plan_header_noalloc
void clear_last_error();
int report_error(int code, const char* fmt, ...);
int check_geometry_public(const fa_geometry* g);
Geometry geometry_public(const fa_geometry* g);

}  // namespace bsm
