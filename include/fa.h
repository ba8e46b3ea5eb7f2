/*
 * fa.h -- C ABI of the interval-masked / block-sparse attention forward
 * library for NVIDIA GB300 (sm_103a).
 *
 * Two steps, both on one GPU:
 *
 *   1. A GPU planner turns a mask into an immutable, reusable MaskPlan
 *      ("Flex Attention Mask Plan Design", cuDNN frontend documentation,
 *      §4 Planner Overview, §8 Plan Ownership and Reuse).
 *   2. fa_fwd consumes the plan and computes
 *          O = softmax(mod(Q K^T * scale)) V   and   LSE = ln sum exp(mod(.))
 *      (FlexAttention Eq. 1, and the same page §6.1 Forward for the
 *      consumption protocol).
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" must point to memory of the current CUDA
 *     device; pointers marked "host" to ordinary host memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All GPU work is enqueued on it.
 *   - Return value: FA_OK (0) or a negative FA_ERR_* code.  On error no
 *     output is produced (`*out` stays NULL) and nothing leaks;
 *     fa_last_error() gives a message for the calling thread.
 *   - Head dimension 64 or 128, bf16 Q/K/V/O, fp32 LSE, physical tiles of
 *     128 x 128 (Q rows x K columns).
 */
#ifndef BSM_FA_H
#define BSM_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1,     /* host-side structural check failed           */
  FA_ERR_INVALID_MASK = -2,    /* an endpoint is out of range / out of order  */
  FA_ERR_INVALID_SEQLENS = -3, /* cu_seqlens prefix check failed on the GPU   */
  FA_ERR_PLAN_MISMATCH = -4,   /* plan signature or geometry differs          */
  FA_ERR_ALLOC = -5,           /* device or host allocation failed            */
  FA_ERR_CUDA = -6,            /* a CUDA runtime / driver call failed         */
  FA_ERR_DEVICE_TIMEOUT = -7,  /* a bounded in-kernel wait ran out            */
  FA_ERR_UNSUPPORTED = -8      /* valid request outside what the library runs */
};

enum { FA_LAYOUT_BSHD = 0, FA_LAYOUT_THD = 1 };
enum { FA_DTYPE_BF16 = 0 };
enum { FA_MOD_SOFTCAP = 1, FA_MOD_ALIBI = 2 };
/* Physical plan choices of fa_fwd, also passed in fa_mods.flags ("Decoupling
 * Logical Masks from GPU Execution for Dynamic Block-Sparse Attention",
 * physical mappings and task organisation).  By default interval plans
 * without mods run two vertically adjacent Q tiles per task, and block plans
 * whose logical blocks are multiples of 64 (head_dim 128, no mods) run the
 * Direct mapping: one 64-row half of a Q tile per task, stepping through
 * its live 64x64 blocks.  FA_FWD_ONE_TILE runs one Q tile per task
 * instead; FA_FWD_COARSENED runs a block plan on whole 128x128 tiles (the
 * Coarsened mapping).  Results agree within the forward's tolerance. */
enum { FA_FWD_ONE_TILE = 16, FA_FWD_COARSENED = 32 };

/* Physical tile of the library's consumers. */
#define FA_TILE_Q 128
#define FA_TILE_K 128
/* uint32 words of packed predicate per tile row (128 columns / 32). */
#define FA_PAYLOAD_WORDS 4

typedef struct fa_plan fa_plan; /* opaque, immutable after build */

/*
 * Problem geometry ("Flex Attention Mask Plan Design" §3.1 Fixed Length,
 * §3.2 Varlen).
 *   layout FA_LAYOUT_BSHD: Q is [batch, seqlen_q, heads_q, head_dim] and K/V
 *     are [batch, seqlen_k, heads_k, head_dim], contiguous; total_q/total_k
 *     and cu_seqlens_* are ignored.
 *   layout FA_LAYOUT_THD: Q is [total_q, heads_q, head_dim], K/V are
 *     [total_k, heads_k, head_dim]; sample b owns Q rows
 *     [cu_seqlens_q[b], cu_seqlens_q[b+1]) and K rows likewise.
 *     cu_seqlens_q/k are device int32 [batch+1]; seqlen_q/k are the maximum
 *     sample lengths (max_seqlen_q/k).  The planner validates the prefixes
 *     on the GPU (start 0, end total, nondecreasing, within the maxima) and
 *     the plan keeps its own copies, so the caller may change or free them
 *     after the build returns.
 *   heads_q must be a multiple of heads_k (GQA: Q head h reads K/V head
 *   h / (heads_q / heads_k)).
 */
typedef struct {
  int32_t layout;
  int32_t batch;
  int32_t seqlen_q;
  int32_t seqlen_k;
  int32_t total_q;
  int32_t total_k;
  const int32_t* cu_seqlens_q; /* device, THD only */
  const int32_t* cu_seqlens_k; /* device, THD only */
  int32_t heads_q;
  int32_t heads_k;
  int32_t head_dim;            /* 64 or 128 */
  int32_t dtype;               /* FA_DTYPE_BF16 */
} fa_geometry;

/*
 * Optional allocator for plan and workspace memory.  alloc returns device
 * memory of at least `bytes` usable in stream order on `stream` (NULL on
 * failure); free releases it in stream order.  Pass NULL to use the
 * library's own stream-ordered pool (cudaMallocAsync-style).
 */
typedef struct {
  void* (*alloc)(size_t bytes, void* stream, void* ctx);
  void (*free)(void* ptr, size_t bytes, void* stream, void* ctx);
  void* ctx;
} fa_allocator;

/*
 * Build a plan from per-row interval endpoints ("Flex Attention Mask Plan
 * Design" §2 Public Mask Representation, §4.2-§4.6, §4.8, §5).
 *   mask_func: device int32 [Hmask, nfunc, total_q] (BSHD: total_q =
 *     batch*seqlen_q, rows batch-major).  Row q's visible keys are
 *     [0,F0) U [F1,F2) U ... with sample-local key positions and
 *     0 <= F0 <= ... <= F(nfunc-1) <= k_len of the row's sample.
 *   Hmask: 1 (one mask for every Q head) or heads_q.  nfunc: odd, >= 1.
 * The build validates every endpoint and (THD) prefix on the GPU, reads an
 * 8-value header back once (the only host/device synchronisation), then
 * allocates exact-size outputs.  Malformed endpoints return
 * FA_ERR_INVALID_MASK, malformed prefixes FA_ERR_INVALID_SEQLENS; no plan
 * is produced.  Geometries with more than 2^26 Q tiles (batch x
 * ceil(seqlen_q / 128)), or whose Q tiles times Hmask or times heads_q
 * reach 2^31, return FA_ERR_UNSUPPORTED.  The caller owns mask_func and may
 * reuse it after return.
 * On success *out receives a plan the caller must release with fa_plan_free.
 */
int fa_plan_build_intervals(const fa_geometry* geom, const int32_t* mask_func,
                            int32_t Hmask, int32_t nfunc, const fa_allocator* allocator,
                            void* stream, fa_plan** out);

/*
 * Same as fa_plan_build_intervals with build flags.  FA_PLAN_BACKWARD also
 * builds the backward views of "Flex Attention Mask Plan Design" §4.4 and
 * §4.7 for the training consumers (§6.3): the K2Q view (for every K plan
 * row, i.e. mask head x sample x 128-key tile, independent ascending CSR
 * lists of the partial and full 128-row Q tiles), its key-major packed
 * predicate, and the dQ write order.  The backward consumers use the
 * forward's tile geometry, so the dQ consumer reads the forward Q2K view.
 * The header then reads {fwd Q rows, fwd partial nnz, fwd full nnz, bwd Q
 * rows, bwd K rows, bwd partial nnz, bwd full nnz, error}.  Unknown flags
 * return FA_ERR_INVALID_ARG.
 */
#define FA_PLAN_BACKWARD 1u
/*
 * FA_PLAN_QUADRANT_PAYLOAD (block plans only): when block_q, block_kv,
 * seqlen_q and seqlen_k are all multiples of 64, every 64x64 quadrant of a
 * 128x128 tile is wholly visible or wholly masked, so the per-entry
 * quadrant bits describe the partial tiles exactly.  The plan then keeps
 * only those bits (a block-granular payload: "Decoupling Logical Masks from
 * GPU Execution for Dynamic Block-Sparse Attention", launch preparation
 * derives only the metadata the selected plan needs) and not the 2 KB of
 * predicate words per partial entry; the planner neither writes nor
 * allocates them.  Such a plan runs the Direct 64x64 forward only: fa_fwd
 * with score mods or FA_FWD_COARSENED returns FA_ERR_UNSUPPORTED, and
 * fa_plan_info_get reports payload_bytes = 0.  For plans that are not
 * quadrant-exact, and together with FA_PLAN_BACKWARD (whose key-major view
 * is built from the words), the flag has no effect.
 */
#define FA_PLAN_QUADRANT_PAYLOAD 2u
int fa_plan_build_intervals_ex(const fa_geometry* geom, const int32_t* mask_func, int32_t Hmask,
                               int32_t nfunc, uint32_t flags, const fa_allocator* allocator, void* stream,
                               fa_plan** out);

/*
 * Build a plan from a logical block-pair mask ("Decoupling Logical Masks
 * from GPU Execution for Dynamic Block-Sparse Attention" §2: mask M with
 * logical geometry B = (block_q, block_kv), effective set E(M); physical
 * tiles T = 128 x 128 are chosen independently of B).
 *   block_mask: device uint8 [Hmask, ceil(seqlen_q/block_q),
 *     ceil(seqlen_k/block_kv)]; nonzero = active block pair.  Token pair
 *     (q, k) is visible iff its block pair is active and q < seqlen_q,
 *     k < seqlen_k.  Fixed-length (BSHD) geometry only; the same mask is
 *     applied to every sample.
 * Errors and ownership as for fa_plan_build_intervals.
 */
int fa_plan_build_blocks(const fa_geometry* geom, const uint8_t* block_mask, int32_t Hmask,
                         int32_t block_q, int32_t block_kv, const fa_allocator* allocator,
                         void* stream, fa_plan** out);
/* Same with build flags (FA_PLAN_BACKWARD: see fa_plan_build_intervals_ex). */
int fa_plan_build_blocks_ex(const fa_geometry* geom, const uint8_t* block_mask, int32_t Hmask,
                            int32_t block_q, int32_t block_kv, uint32_t flags, const fa_allocator* allocator,
                            void* stream, fa_plan** out);

/*
 * Release a plan ("Flex Attention Mask Plan Design" §8 Ownership: the plan
 * owns every buffer it holds, including its cu_seqlens clones, and releases
 * them itself).  NULL is accepted.  Device memory is returned in stream
 * order on `stream` (through the plan's allocator when one was given): the
 * caller must make sure no work that reads the plan is still pending on any
 * other stream.
 */
int fa_plan_free(fa_plan* plan, void* stream);

/* Score modifications applied after scaling (FlexAttention score_mod):
 *   FA_MOD_SOFTCAP: s <- softcap * tanh(s / softcap)
 *   FA_MOD_ALIBI:   s <- s + alibi_slopes[h] * (k - q)   (sample-local k, q)
 * applied in that order.  alibi_slopes is a host array of heads_q floats,
 * read during the call.  flags may also hold the plan choices FA_FWD_*
 * (fa_fwd only). */
typedef struct {
  int32_t flags;
  float softcap;
  const float* alibi_slopes;
} fa_mods;

/*
 * Masked attention forward ("Flex Attention Mask Plan Design" §6.1):
 * for every (sample, Q head, Q tile) task of the plan, partial tiles are
 * computed with the packed predicate, full tiles without, empty tiles are
 * skipped; rows without a visible key get O = 0 and LSE = -inf.
 *   q, k, v: device bf16 in the geometry's layout; o: device bf16, same
 *   layout as q; lse: device float32 [heads_q, total_q] (natural log), may
 *   be NULL.  scale (> 0, finite) multiplies Q K^T before the mods.  mods
 *   may be NULL.
 * Every base pointer must be 16-byte aligned.  The geometry must equal the
 * one the plan was built for (FA_ERR_PLAN_MISMATCH otherwise).  The call
 * is asynchronous on `stream` and issues exactly one kernel launch: the
 * kernel schedules its tasks on the device (one CTA per task, running CTAs
 * take over CTAs that have not started, through the GPU's cluster launch
 * control), so a call keeps no state between launches.  One plan may be
 * used concurrently on several streams and captured into graphs.
 */
int fa_fwd(const fa_plan* plan, const void* q, const void* k, const void* v, void* o,
           float* lse, const fa_geometry* geom, float scale, const fa_mods* mods,
           void* stream);

/*
 * Masked attention backward ("Flex Attention Mask Plan Design" §6.3) for a
 * plan built with FA_PLAN_BACKWARD (FA_ERR_PLAN_MISMATCH otherwise): the
 * gradients of FlexAttention Eq. 1 with the same mods as the forward.  A
 * Q-major kernel walks the forward Q2K view and writes dQ; a K-major kernel
 * walks the K2Q view and writes dK and dV, summing the Q heads of each K/V
 * head's group; partial tiles use their packed predicate, full tiles none.
 * Scores are recomputed from q and k; P = exp(mod(scale QK^T) - lse).
 *   q, k, v, o, dout: device bf16 in the geometry's layout (o and lse are
 *   the forward's outputs for these q, k, v); lse: device float32
 *   [heads_q, total_q]; dq (like q), dk, dv (like k): device bf16, written
 *   in full (rows and keys without a visible pair get 0).
 * head_dim 128 only (FA_ERR_UNSUPPORTED otherwise).  A [heads_q, total_q]
 * float32 workspace comes from the plan's allocator (or the library's
 * pool) and is returned in stream order.  Asynchronous on `stream`: three
 * kernel launches (Delta = rowsum(dout * o), dQ, dK/dV).  Pointers must be
 * 16-byte aligned.
 */
int fa_bwd(const fa_plan* plan, const void* q, const void* k, const void* v, const void* o,
           const void* dout, const float* lse, void* dq, void* dk, void* dv, const fa_geometry* geom,
           float scale, const fa_mods* mods, void* stream);

/*
 * Decoding over a paged KV cache ("FlexAttention: A Programming Model for
 * Generating Optimized Attention Kernels", summary page, §3.4 Paged
 * Attention Integration and Modification Conversion for Inference).
 *
 * The plan is an interval plan whose geometry is THD with one query row per
 * sequence (max_seqlen_q = 1, total_q = batch) and the sequences' logical
 * key counts (cu_seqlens_k); the endpoints of each query row are those of
 * its absolute position offset = k_len - 1 (the mask converted for
 * inference).  Key j of sequence b is read from page page_table[b][j /
 * page_size], row j % page_size: before the attention kernel, one small
 * kernel converts every K tile of the plan's lists into the physical rows
 * of its pages (the page table becomes part of the index lists; the
 * attention loop sees physical rows only).  The attention kernel runs one
 * persistent CTA per SM; the K tiles of all sequences and K/V heads are cut
 * into equal ranges, one per CTA (Split-K: a sequence's list may be split
 * over several CTAs); a last kernel merges the pieces of each query row.
 *   q: device bf16 [batch, heads_q, 128]; k_cache, v_cache: device bf16
 *   [num_pages, page_size, heads_k, 128]; page_table: device int32
 *   [batch, pages_per_seq] (entries for pages past a sequence's k_len are
 *   never read); o: device bf16 like q; lse: device float32 [heads_q, batch]
 *   (natural log), may be NULL.  page_size: a power of two >= 16.
 * A page number outside [0, num_pages) for a key that is needed sets bit 3
 * of the device error flags (fa_device_error_flags) and reads zeros.
 * One mask for every head (Hmask = 1, any GQA group up to 64 query heads
 * per K/V head), or per-head masks without GQA (FA_ERR_UNSUPPORTED
 * otherwise).  mods (may be NULL) as for fa_fwd, converted for inference:
 * the ALiBi bias is alibi_slopes[h] * (k - (k_len - 1)), the query's
 * absolute position.  A workspace (index conversion, row
 * prefix, per-piece O, max and sum) comes from the plan's allocator or the
 * library's pool and is returned in stream order.  Asynchronous on
 * `stream`: three kernel launches.  Pointers must be 16-byte aligned.
 */
int fa_decode_paged(const fa_plan* plan, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* page_table, int32_t pages_per_seq, int32_t page_size,
                    int64_t num_pages, void* o, float* lse, const fa_geometry* geom, float scale,
                    const fa_mods* mods, void* stream);

/* Plan statistics and layout sizes (Tessera-style mask statistics). */
typedef struct {
  int64_t header[8];      /* fwd Q rows, partial nnz, full nnz, 0, 0, 0, 0, error flags */
  int32_t tile_q, tile_k;
  int32_t mask_heads;     /* Hmask */
  int32_t batch;
  int32_t heads_q, heads_k, head_dim, layout;
  int64_t num_tasks;      /* fwd Q rows * heads_q */
  int64_t payload_bytes;  /* partial nnz * 128 * 4 * 4 */
  int64_t plan_bytes;     /* device bytes owned by the plan */
  int64_t visible_pairs;  /* visible (q,k) pairs summed over mask heads; -1 unless requested */
  uint64_t signature;     /* consumer signature (§7); equal plans share it */
  double build_us;        /* host wall time of the build call */
} fa_plan_info;

/*
 * Fill `info`.  With count_visible != 0 the visible pairs are counted on
 * the GPU (stream-synchronous); otherwise info->visible_pairs = -1.
 */
int fa_plan_info_get(const fa_plan* plan, int32_t count_visible, void* stream,
                     fa_plan_info* info);

/*
 * Debug snapshot ("Flex Attention Mask Plan Design" §8 debug_snapshot):
 * copy the plan's arrays to caller-owned host buffers (each may be NULL to
 * skip).  Sizes, with R = header[0], P = header[1], F = header[2],
 * Hm = mask_heads, T = num_tasks:
 *   cu_q_rows [batch+1], sequence_desc [batch*8]
 *   (q_offset, k_offset, q_len, k_len, row begin, row count, K tiles, 0),
 *   partial_offset / full_offset [Hm*R+1] (row-major over (mask head, row)),
 *   partial_idx [P], full_idx [F] (sample-local K tile indices, ascending
 *   per row), payload [P*128*4] (entry e, tile row r, word w: bit l keeps
 *   column 32*w+l), work_desc [T*4] (m_block, head, batch, q_valid_rows) in
 *   execution order, halves [P] (bit s: some element of key columns
 *   64s..64s+63 of the partial tile is visible), quads [P] (quadrant
 *   (a, s) = tile rows 64a..64a+63 x key columns 64s..64s+63: bit 2a+s set
 *   if one of its elements is visible, bit 4+2a+s if all are), lpt [T] (the
 *   positions of work_desc ordered by task cost -- partial + full entries of
 *   the task's row -- descending, ties in work_desc order, zero-cost tasks
 *   last: the longest-first order in which a consumer with few tasks per SM
 *   takes the tasks; block-mask plans carry no such order on the device and
 *   export the identity, work_desc's own section order, which their
 *   forwards keep for L2 reuse; "Flex Attention Mask Plan Design" §4.8
 *   leaves the consumer's traversal of the task list open).  Synchronous.
 */
typedef struct {
  int32_t* cu_q_rows;
  int32_t* sequence_desc;
  int32_t* partial_offset;
  int32_t* partial_idx;
  int32_t* full_offset;
  int32_t* full_idx;
  uint32_t* payload;
  int32_t* work_desc;
  uint8_t* halves;
  uint8_t* quads;
  int32_t* lpt;
} fa_plan_host_view;

int fa_plan_export(const fa_plan* plan, fa_plan_host_view* dst);

/*
 * Debug snapshot of the backward views ("Flex Attention Mask Plan Design"
 * §4.7) of a plan built with FA_PLAN_BACKWARD (FA_ERR_INVALID_ARG
 * otherwise).  Sizes, with KR = header[4], KP = header[5], KF = header[6]:
 *   cu_k_rows [batch+1] (K plan rows per sample: ceil(k_len / 128)),
 *   partial_offset / full_offset [Hm*KR+1] (row-major over (mask head,
 *   K row)), partial_idx [KP], full_idx [KF] (sample-local Q tiles,
 *   ascending per K row), payload [KP*128*4] (entry e, key column c, word w:
 *   bit l = query row 32*w+l of the tile is visible for key c),
 *   dq_write_order [KP], dq_write_order_full [KF] (parallel to the lists:
 *   rank of the entry's K tile among its Q tile's non-empty K tiles in
 *   ascending order, a legal order for accumulating dQ).  Synchronous.
 */
typedef struct {
  int32_t* cu_k_rows;
  int32_t* partial_offset;
  int32_t* partial_idx;
  int32_t* full_offset;
  int32_t* full_idx;
  uint32_t* payload;
  int32_t* dq_write_order;
  int32_t* dq_write_order_full;
} fa_plan_bwd_host_view;

int fa_plan_export_backward(const fa_plan* plan, fa_plan_bwd_host_view* dst);

/*
 * Error bits written by the library's kernels on the current device (bit 0:
 * a bounded in-kernel wait ran out and the kernel stopped early, so its
 * output is incomplete; bit 1: dynamic shared memory was not aligned as
 * the kernel requires, so it did no work; bit 2, only in the bounds-checked
 * debug build libbsm_fa_checked.so: a planner, forward or backward kernel
 * computed a plan-derived global index outside the plan's exact sizes, and
 * the access was redirected or skipped; bit 3: fa_decode_paged met a page
 * number outside the cache for a key it needed, and read zeros instead).  Synchronises `stream`, returns
 * the bits in *flags and clears them.
 */
int fa_device_error_flags(void* stream, uint32_t* flags);

/*
 * Diagnostic of the bounded in-kernel waits: launches one small kernel on
 * `stream` whose mbarrier wait can never complete.  Each wait gives up after
 * timeout_ns (1 us .. 100 ms), bit 0 of the device error flags is set and
 * the kernel ends normally, so the CUDA context stays usable; read the bit
 * with fa_device_error_flags.  Nothing faults, traps or hangs.
 */
int fa_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * Debug only (the bounds-checked build libbsm_fa_checked.so; the release
 * build returns FA_ERR_UNSUPPORTED and changes nothing): overwrites field
 * `field` (0 Q tile, 1 head, 2 sample, 3 valid rows) of task `task` of the
 * plan's work_desc with `value`, synchronously on `stream`.  It breaks the
 * plan's immutability on purpose, so that tests can check that an
 * out-of-range head or sample is caught by the kernels' index checks (bit
 * 2 of the device error flags) instead of being used.  FA_ERR_INVALID_ARG
 * when the task or field is out of range.
 */
int fa_debug_set_work_desc(fa_plan* plan, int64_t task, int32_t field, int32_t value, void* stream);

/*
 * Allocation-free sizing of an interval plan.  The paper has no counterpart
 * of this entry point; it exists for callers that cannot allocate device
 * memory, neither themselves nor through this library: for example code
 * running inside a memory manager that owns all device memory and must not
 * re-enter cudaMalloc, or a loop with a strict latency budget where
 * allocation calls (which may synchronise the device) are not allowed.
 *
 * It runs the geometry and classification stage of fa_plan_build_intervals
 * (which also totals the entries) and writes the same 8-value header (fwd Q rows,
 * partial nnz, full nnz, 0, 0, 0, 0, error flags) to `header_out`, a
 * caller-owned device int64[8].  Nothing else is produced and nothing is
 * read back: the call is asynchronous on `stream`, and a malformed mask or
 * prefix shows up as a nonzero header_out[7] (bit 0: endpoints, bit 1:
 * cu_seqlens) instead of an error code.  Arguments are those of
 * fa_plan_build_intervals.
 *
 * The planner's scratch lives in one fixed 4 MiB array per device, held by
 * every device that loads the library until the process exits.  No
 * cudaMalloc, cudaFree or other allocating routine is called.  Masks whose
 * scratch (about 8 bytes per (mask head, Q tile, 32 K tiles) plus small
 * per-sample arrays) exceeds 4 MiB are rejected with FA_ERR_UNSUPPORTED.
 * The first call on each device looks up the array's device address; make
 * that first call before any stream capture.  Later calls outside capture
 * look it up again (so a cudaDeviceReset or a new context on the device is
 * picked up); calls during capture reuse the address of the last call made
 * outside capture on that device.  All calls on a device share
 * the array and it keeps the previous call's contents (the call clears what
 * must start at zero), so calls whose GPU work overlaps (e.g. on unordered
 * streams) race on it and give wrong results: order them.
 */
int fa_plan_header_noalloc(const fa_geometry* geom, const int32_t* mask_func, int32_t Hmask,
                           int32_t nfunc, int64_t* header_out, void* stream);

/* Message of the last error on the calling thread ("" if none). */
const char* fa_last_error(void);

/* Library version string. */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BSM_FA_H */
