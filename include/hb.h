/*
 * hb.h -- C ABI of the hybrid-batch paged-attention library (libhb.so).
 *
 * One call sequence runs one attention layer of a hybrid batch: many decode
 * rows (one new token each, over a long cached context) plus prefill chunks
 * (q_len > 1 new tokens that attend causally to themselves and re-read the
 * KV of the earlier chunks of their prompt), all over a paged KV cache.
 *
 *   hb_kv_append  scatter the batch's new K/V rows into their pages
 *   hb_plan       (host) split the batch into work items; upload the plan
 *   hb_attention  attention of every new token over its sequence's pages
 *
 * The operation follows "Sarathi-Serve：以 chunked-prefills 与 stall-free batching
 * 驯服 LLM 推理的吞吐—延迟权衡", §GPU / 系统数据路径 ③ (a batch of decode tokens
 * plus prefill chunks within a token budget) and ⑤ (attention reads and
 * writes the KV cache through the page table; a chunk appends its KV, decodes
 * read all earlier KV, chunk i re-reads chunks 1..i-1), and "In-flight
 * Batching", §KV Cache 管理的协同优化 (16-token pages, a block table mapping
 * logical pages to non-contiguous physical ones) and §Batch 内的异构执行
 * (different lengths handled inside the kernel, no padding).
 *
 * Conventions shared by every call
 *  - Pointers are borrowed: the library allocates no device memory and keeps
 *    no pointer after the call returns (work already queued on `stream` uses
 *    them until it completes).  The caller owns all memory and streams.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *  - Argument errors are detected on the host and returned synchronously;
 *    nothing is launched then.  Device-side index errors (a block-table entry
 *    outside [0, num_pages)) set a device error word and skip the access;
 *    hb_check() turns it into HB_ERR_DEVICE_INDEX.  A device wait that runs
 *    out of time sets HB_ERR_TIMEOUT the same way.  No C++ exception crosses
 *    this boundary.  hb_last_error() gives a message for the last failure of
 *    the calling thread.
 *  - All calls are asynchronous on `stream` unless stated otherwise; append
 *    must be ordered before attention on the same stream.
 *  - The kernels are launched with programmatic stream serialization: a
 *    kernel of this library may start under the tail of the kernel before
 *    it and waits for that kernel before it depends on it.  When the
 *    library's previous launch on the stream is hb_kv_append of the same
 *    batch (same descriptors and pools), hb_attention waits for it only
 *    before reading the cache pages that hold the batch's new tokens and
 *    reads every other page at once; after anything else it waits first.
 *    Work of other libraries is complete before a kernel of this library
 *    starts (it does not release it early).
 *
 * Data layout (bf16 = IEEE bfloat16 stored as uint16)
 *  - q      [total_q, num_q_heads,  head_dim] bf16, rows in batch order
 *  - k_new  [total_q, num_kv_heads, head_dim] bf16 (same for v_new)
 *  - cache  [num_pages, page_size, num_kv_heads, head_dim] bf16, separate
 *           K and V pools ("NHD" pages)
 *  - out    [total_q, num_q_heads,  head_dim] bf16
 *  - Rows of sequence s are q rows cu_q_len[s] .. cu_q_len[s+1]-1.  Its new
 *    token j sits at logical position p = context_len[s] - q_len[s] + j in
 *    physical page block_table[s*max_pages_per_seq + p/page_size], slot
 *    p % page_size, and attends to logical keys 0..p (causal, aligned to the
 *    absolute position).  Query head h reads kv head h / (Hq/Hkv).
 *
 * Supported shapes: page_size 16, head_dim 64 or 128, Hq a multiple of Hkv
 * with group size Hq/Hkv <= 16, 1 <= q_len <= context_len per sequence.
 */
#ifndef HB_H_
#define HB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum hb_status {
  HB_OK = 0,
  HB_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, misaligned pointer   */
  HB_ERR_SHAPE = 2,         /* inconsistent sizes or a row breaking          */
                            /* 1 <= q_len <= context_len                      */
  HB_ERR_UNSUPPORTED = 3,   /* valid but not built (page size, head_dim ...) */
  HB_ERR_WORKSPACE = 4,     /* plan or workspace buffer too small / stale    */
  HB_ERR_CUDA = 5,          /* a CUDA runtime/driver call failed             */
  HB_ERR_DEVICE_INDEX = 6,  /* a kernel met an out-of-range page index       */
  HB_ERR_TIMEOUT = 7,       /* a kernel wait gave up                         */
  HB_ERR_OUT_OF_PAGES = 8   /* batch builder: no free page for a decode      */
} hb_status;

/* Message for the last failed call on this thread ("" if none).  The string
 * is owned by the library and valid until the next call on this thread. */
const char* hb_last_error(void);

/* Name of a status code (static string). */
const char* hb_status_string(hb_status s);

/* Descriptor of one hybrid batch.  The three arrays are DEVICE pointers.
 *
 * sliding_window: 0 for full causal attention; W > 0 restricts the query at
 * absolute position p to the keys p-W+1 .. p (W keys, itself included).  The
 * pages name sliding-window model variants ("Sarathi-Serve: Chunked Prefills
 * for Stall-Free LLM Inference", §Results and evidence) without a size, so W
 * is a parameter.  With W > 0 the kernels never read the block-table entry
 * of a page that holds no key inside any of its row's windows (such entries
 * may be stale). */
typedef struct hb_batch {
  int32_t num_seqs;            /* sequences (rows of the batch), >= 0         */
  int32_t total_q;             /* sum of q_len = rows of q / k_new / out      */
  int32_t max_pages_per_seq;   /* row stride of block_table                   */
  int32_t num_pages;           /* physical pages in each cache pool           */
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;           /* tokens per page; must be 16                 */
  int32_t sliding_window;      /* 0: none; W > 0: keys p-W+1 .. p (above)     */
  int32_t reserved;            /* must be 0                                   */
  const int32_t* cu_q_len;     /* [num_seqs+1] prefix sums of q_len, [0] = 0  */
  const int32_t* context_len;  /* [num_seqs] tokens in cache AFTER append     */
  const int32_t* block_table;  /* [num_seqs * max_pages_per_seq] page ids     */
} hb_batch;

/*
 * KV append (scatter).  For every new token j of sequence s, copy row
 * cu_q_len[s]+j of k_new / v_new ([num_kv_heads*head_dim] contiguous bf16)
 * to its page slot in k_cache / v_cache (see the layout above).  The copy is
 * bit-exact; no other slot is written.  Cited passage: the first page,
 * §GPU / 系统数据路径 ⑤ ("a prefill chunk appends new KV").
 *   k_new, v_new     device, [total_q, Hkv, D] bf16, 16-byte aligned
 *   k_cache, v_cache device, [num_pages, 16, Hkv, D] bf16, 16-byte aligned
 * Errors: HB_ERR_INVALID_ARG / HB_ERR_SHAPE / HB_ERR_UNSUPPORTED on the host;
 * a page id outside [0, num_pages) is skipped and reported by hb_check().
 */
hb_status hb_kv_append(const hb_batch* batch, const void* k_new,
                       const void* v_new, void* k_cache, void* v_cache,
                       void* stream);

/*
 * Plan (host).  Cuts the batch into work items for hb_attention: decode rows
 * (q_len == 1) become split-KV items over page ranges, chunk rows (q_len > 1)
 * become (kv head, query tile) items; both lists are ordered longest first.
 * Needs HOST copies of q_len and context_len (the same values the device
 * arrays of `batch` hold) and the number of SMs of the device.
 *   h_q_len, h_context_len  host, [num_seqs] int32
 *   h_plan                  host buffer for the plan, or NULL
 *   plan_bytes              in: size of h_plan; out: bytes needed
 *   d_workspace             device buffer (256-byte aligned), or NULL
 *   workspace_bytes         in: size of d_workspace; out: bytes needed
 * The sizes are always reported.  With h_plan == NULL nothing else happens;
 * otherwise the plan is written into h_plan, and if d_workspace is not NULL
 * it is also copied into d_workspace and the workspace counters are cleared,
 * asynchronously on `stream` (only this step makes CUDA calls): h_plan must
 * stay unchanged until that copy has completed, and a workspace must not be
 * shared by attention calls in flight at once.  From pageable memory the
 * CUDA driver may wait for `stream` before it stages the copy: a caller
 * whose host should run ahead of the kernels passes a stream without the
 * previous step's kernels on it (for example its input-copy stream, ordered
 * before the kernels by an event).
 * The plan stays valid for any later hb_attention on a batch with the same
 * q_len / context_len / head geometry (block tables and tensors may change).
 * Errors: HB_ERR_SHAPE for rows outside 1 <= q_len <= context_len, or
 * context_len > max_pages_per_seq*page_size; HB_ERR_WORKSPACE if a buffer is
 * too small.
 */
hb_status hb_plan(const hb_batch* batch, const int32_t* h_q_len,
                  const int32_t* h_context_len, int32_t num_sms, void* h_plan,
                  size_t* plan_bytes, void* d_workspace,
                  size_t* workspace_bytes, void* stream);

/*
 * Attention.  out[row, h, :] = sum_t softmax_t(scale * <q[row,h], K[t]>) V[t]
 * over keys t = 0..p of the row's sequence (p its absolute position), K/V of
 * kv head h/(Hq/Hkv) read through the block table from the caches as they
 * stand after hb_kv_append.  fp32 accumulation, one bf16 rounding at the
 * store.  One kernel launch does all of it: decode rows are streamed as equal
 * page ranges per CTA (a row that straddles ranges leaves partial softmax
 * states, merged by the last piece to finish) and chunk rows are tiled for
 * the tensor cores, the two kinds of CTAs running side by side.
 * Cited passages: the first page, §GPU / 系统数据路径 ③-⑤, and §核心机制 3
 * (chunk i re-reads the KV of chunks 1..i-1; same computation as unchunked).
 *   h_plan      host plan written by hb_plan for this batch
 *   q, out      device, [total_q, Hq, D] bf16, 16-byte aligned
 *   k_cache, v_cache device pools as in hb_kv_append
 *   d_workspace the workspace hb_plan prepared
 * Errors: HB_ERR_WORKSPACE if h_plan does not match the batch; argument
 * errors as above; launch failures as HB_ERR_CUDA.
 */
hb_status hb_attention(const hb_batch* batch, const void* h_plan,
                       const void* q, const void* k_cache,
                       const void* v_cache, float softmax_scale, void* out,
                       void* d_workspace, void* stream);

/*
 * hb_attention, with the batch's new K/V rows also given as k_new / v_new
 * (the arrays passed to hb_kv_append for this batch, [total_q, Hkv, D] bf16,
 * 16-byte aligned).  The result is the same; the chunk rows read the pages
 * that hold only their sequence's new tokens from k_new / v_new instead of
 * from the caches, so they do not wait for the append kernel that writes
 * those pages (the one page holding a chunk's first token, when that token
 * does not start a page, and the decode rows' last pages are still read
 * from the caches after the append).  The caches must receive the new rows
 * by hb_kv_append as usual, queued before this call on the same stream.
 * Same passages as hb_attention.  Errors: as hb_attention;
 * HB_ERR_INVALID_ARG for a NULL or misaligned k_new / v_new.
 */
hb_status hb_attention_new_kv(const hb_batch* batch, const void* h_plan, const void* q,
                              const void* k_new, const void* v_new, const void* k_cache,
                              const void* v_cache, float softmax_scale, void* out,
                              void* d_workspace, void* stream);

/*
 * Decode attention without a workspace, for callers that cannot allocate
 * device memory.  (The pages have no counterpart of this call: it exists for
 * callers such as a serving engine that gives nearly all free HBM to its
 * KV-cache pool at start-up and allows no device allocation afterwards, or a
 * plugin that is handed raw tensor pointers but no allocator.)
 *
 * Same result as hb_plan + hb_attention on a batch whose rows are all decode
 * rows (q_len == 1), using the same split-KV kernel, but its scratch (work
 * items, counters, split partial states) is a fixed device array of
 * HB_NOALLOC_SCRATCH_BYTES inside the library, which every device that loads
 * the library holds until the process exits.  The call makes no cudaMalloc /
 * cudaFree and no other allocating call; its host-side plan also uses static
 * storage.  The caller still owns and passes q, the caches and out (layouts as
 * in hb_attention) plus host copies of q_len and context_len.
 *   - The first call on a device looks up that device's copy of the array
 *     (with the device current); make that first call before any stream
 *     capture.
 *   - All calls share the array and it keeps the last call's contents: each
 *     call clears the counters it needs; calls that overlap on the GPU (other
 *     streams or host threads) race and must be serialised by the caller.
 *     Host calls are serialised by a lock inside the library.
 *   - The plan's items are copied from pageable host memory, so the call
 *     returns after the copy is staged.  That storage is the library's own
 *     and the next call overwrites it, so a call on a stream that is being
 *     captured into a CUDA graph is refused with HB_ERR_UNSUPPORTED (a
 *     replayed copy would read a later call's items).
 *   - The work is spread over fewer CTAs when the partial states would not
 *     fit the array; a batch that needs more than 4096 work items (about
 *     num_seqs times ceil(Hkv / 8), plus one per SM) is rejected with
 *     HB_ERR_WORKSPACE.  Rows with q_len != 1 give HB_ERR_UNSUPPORTED.  Other
 *     errors as hb_attention.
 */
#define HB_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

hb_status hb_decode_attention_noalloc(const hb_batch* batch,
                                      const int32_t* h_q_len,
                                      const int32_t* h_context_len,
                                      const void* q, const void* k_cache,
                                      const void* v_cache, float softmax_scale,
                                      void* out, void* stream);

/* ---------------------------------------------------------------------------
 * One step from host memory.  For a serving loop that keeps a few steps in
 * flight: the step's inputs cross the host link as one packed block, the
 * plan goes up ahead of them on the input-copy stream, hb_kv_append and
 * hb_attention run on the compute stream, the output comes back on the
 * output-copy stream, and the step's slot (CUDA events and a device flag)
 * orders the three streams against the previous step that used the same
 * buffers.  The input copy is followed by a write of the step's sequence
 * number to the slot's flag, which the append kernel polls before it reads
 * its inputs (so the compute stream carries no wait between two steps and
 * each step's append launches under the previous attention's tail).  The
 * host does not wait, so one step's copies overlap the neighbouring steps'
 * kernels.  The operation is that of hb_kv_append then hb_attention (same
 * citations); only the copies and their ordering are added.
 *
 * Packed input block (host and device alike): q [total_q, Hq, D] bf16 |
 * k_new | v_new [total_q, Hkv, D] bf16 | cu_q_len [num_seqs+1] | context_len
 * [num_seqs] | block_table [num_seqs, max_pages_per_seq] int32, each section
 * starting on a 256-byte boundary.  hb_step_layout writes the six section
 * offsets and the block's size; it checks only the sizes it reads.
 * ------------------------------------------------------------------------- */
#define HB_STEP_SECTIONS 6

hb_status hb_step_layout(const hb_batch* shape, size_t offsets[HB_STEP_SECTIONS],
                         size_t* in_bytes);

/* Events and a 4-byte device flag of one set of staging buffers, on the
 * current device (creating a slot allocates the flag; destroying it frees
 * it, which synchronises the device). */
typedef struct hb_step_slot hb_step_slot;
hb_status hb_step_slot_create(hb_step_slot** out);
void hb_step_slot_destroy(hb_step_slot* slot);
/* Blocks until the slot's last step has completed (inputs consumed, output on
 * the host): call it before refilling the slot's host inputs or reading its
 * output. */
hb_status hb_step_slot_sync(hb_step_slot* slot);

typedef struct hb_step_buffers {
  const void* h_in;        /* host packed inputs (page-locked, for the copy to overlap) */
  void* d_in;              /* device packed inputs, 256-byte aligned                      */
  void* h_out;             /* host output [total_q, Hq, D] bf16                           */
  void* d_out;             /* device output, 16-byte aligned                              */
  void* h_plan;            /* host plan buffer (hb_plan's plan_bytes; page-locked makes   */
                           /* its upload asynchronous like the inputs')                    */
  size_t plan_bytes;
  void* d_workspace;       /* device workspace (hb_plan's workspace_bytes), 256-aligned   */
  size_t workspace_bytes;
} hb_step_buffers;

/*
 * The step.  `shape` gives the sizes (its three device pointers are ignored:
 * the descriptors are read from d_in); h_q_len / h_context_len are the host
 * copies hb_plan needs.  On copy_in_stream: wait for the slot's last kernels,
 * plan + upload (hb_plan), copy h_in -> d_in, raise the slot's flag.  On
 * stream: wait for the slot's last output copy if it is still pending when
 * the step is issued, hb_kv_append (which waits for the flag on the device,
 * bounded: a flag that does not come within about a second is reported as
 * HB_ERR_TIMEOUT by hb_check and the step's output is undefined),
 * hb_attention.  On copy_out_stream: wait for the kernels, copy d_out ->
 * h_out.  The buffers
 * belong to the slot until hb_step_slot_sync says its step is over; a slot's
 * buffers must not be shared with another slot.  The host blocks only if the
 * slot's previous input copy has not yet run (its plan buffer is rewritten
 * here).  Errors: as hb_plan, hb_kv_append and hb_attention;
 * HB_ERR_INVALID_ARG for NULL or misaligned buffers or a slot of another
 * device; HB_ERR_CUDA if an event or copy call fails.
 */
hb_status hb_step(const hb_batch* shape, const int32_t* h_q_len,
                  const int32_t* h_context_len, int32_t num_sms, hb_step_slot* slot,
                  const hb_step_buffers* buf, void* k_cache, void* v_cache,
                  float softmax_scale, void* copy_in_stream, void* stream,
                  void* copy_out_stream);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device: HB_OK, HB_ERR_DEVICE_INDEX or HB_ERR_TIMEOUT (or
 * HB_ERR_CUDA if the stream itself failed).  Blocking.
 */
hb_status hb_check(void* stream);

/*
 * Self-test of the failure path: launches one CTA that waits on a barrier
 * nothing arrives at, using the bounded wait every kernel of the library
 * uses.  After the wait's time limit (about one second) the kernel records a
 * timeout in the device error word and returns; hb_check() then gives
 * HB_ERR_TIMEOUT and the CUDA context stays usable.  No fault or hang.
 */
hb_status hb_selftest_wait_timeout(void* stream);

/*
 * The same for the flag wait of hb_step's append kernel (a device counter
 * that the input-copy stream raises): one CTA of two warps waits for a
 * device word that nothing raises; after the time limit each warp gives up,
 * the kernel records a timeout and returns, and hb_check() gives
 * HB_ERR_TIMEOUT.  No fault or hang.
 */
hb_status hb_selftest_flag_timeout(void* stream);

/* ---------------------------------------------------------------------------
 * Linear layer of a hybrid batch on the tensor cores: y = x W^T.  Cited
 * passage: the first page, §问题背景 (两阶段天然不对称) -- every token of the
 * batch also passes through the model's linear layers, which take most of
 * the iteration (compute-bound for prefill tokens, weight-read-bound for
 * decodes).  One persistent launch.
 *   x        device, [M, K] bf16 row-major (one row per token), 16-byte aligned
 *   w        device, [N, K] bf16 row-major (row n: weights of output n)
 *   M        rows (tokens), >= 0 (0: nothing to do)
 *   K        multiple of 64
 *   epilogue HB_LINEAR_STORE: y = x W^T, N a multiple of 256, its columns
 *              split over out->y[0..2] (out->cols[i] consecutive columns to
 *              y[i], each a multiple of 256 or 0, summing to N; y[i] is
 *              [M, cols[i]] row-major) -- e.g. q, k and v of a fused QKV
 *              projection;
 *            HB_LINEAR_GATED: w = [W_gate; W_up] with N = 2F rows (F a
 *              multiple of 128); y[0] [M, F] receives silu(x W_gate^T) *
 *              (x W_up^T), silu(g) = g / (1 + e^-g); cols[0] = F;
 *            HB_LINEAR_RESIDUAL: as STORE but y[i] += (its columns of)
 *              x W^T, in place (a residual connection).
 * Ownership: all pointers borrowed; nothing is allocated.  Errors:
 * HB_ERR_INVALID_ARG (NULL or misaligned pointer, unknown epilogue),
 * HB_ERR_SHAPE (sizes breaking the rules above); a wait that gives up is
 * reported by hb_check as HB_ERR_TIMEOUT.
 * ------------------------------------------------------------------------- */
typedef enum hb_linear_epilogue {
  HB_LINEAR_STORE = 0,
  HB_LINEAR_GATED = 1,
  HB_LINEAR_RESIDUAL = 2
} hb_linear_epilogue;

typedef struct hb_linear_out {
  void* y[3];          /* device, bf16; unused entries NULL                     */
  int32_t cols[3];     /* columns per destination (0 = unused)                 */
} hb_linear_out;

hb_status hb_linear(const void* x, const void* w, int32_t M, int32_t N, int32_t K,
                    int32_t epilogue, const hb_linear_out* out, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Workspace that hb_linear can use for this problem on a device with num_sms
 * SMs (0: it needs none).  When the output tiles are too few to occupy the
 * SMs (few tokens), hb_linear splits each tile's K range over several CTAs;
 * the pieces meet in `workspace` (device, 256-byte aligned, ZERO-FILLED before
 * its first use; every call leaves it ready for the next, whatever its shape,
 * so one workspace of the largest size serves all problems).  With a NULL or
 * smaller workspace hb_linear runs unsplit.  Calls sharing a workspace must
 * not overlap on the GPU. */
size_t hb_linear_workspace_size(int32_t M, int32_t N, int32_t K, int32_t epilogue,
                                int32_t num_sms);

/* ---------------------------------------------------------------------------
 * Instrumentation.  When enabled, every kernel launch of this library is
 * bracketed by CUDA events recorded on its launch stream.
 *   kernel ids: 0 = kv append, 1 = attention (decode and chunk work in one
 *   launch), 2 = linear layer
 * ------------------------------------------------------------------------- */
#define HB_NUM_KERNEL_IDS 3

/* enable = 1: start recording, clearing earlier records; 2: resume
 * recording, keeping them (to time a sample of the launches); 0: stop (the
 * records stay readable).  Other values: HB_ERR_INVALID_ARG.  Not
 * thread-safe with concurrent launches from other threads. */
hb_status hb_timing_enable(int32_t enable);

/* Synchronise the recorded events and return, per kernel id, the summed
 * duration in milliseconds and the number of launches recorded.  Both arrays
 * have HB_NUM_KERNEL_IDS entries. */
hb_status hb_timing_read(double* total_ms, int32_t* launches);

/* Durations in milliseconds of the recorded launches of one kernel id, in
 * launch order: up to `max` of them go to ms[], *n receives how many were
 * recorded (which may exceed max).  Synchronises the events it reads. */
hb_status hb_timing_durations(int32_t kernel, float* ms, int32_t max, int32_t* n);

/* Number of kernels this library has launched in this process so far. */
int64_t hb_launch_count(void);

/* ---------------------------------------------------------------------------
 * Stall-free batch builder (host only, no CUDA).  Each step forms the next
 * hybrid batch: (1) one decode token of every request past its prefill,
 * (2) a chunk of every unfinished prefill, (3) first chunks of waiting
 * requests, first come first served, while the token budget lasts; then the
 * caller runs the batch and calls hb_builder_complete, which advances every
 * request and retires finished ones, returning their pages.  Cited passages:
 * the first page, §核心机制 2 (the four steps; decodes always in the batch,
 * at most B tokens per iteration); "In-flight Batching", §调度状态机 (waiting
 * -> prefill (chunked) -> decode -> completed).  Readings where the pages
 * are silent: chunk = min(prompt left, budget left); ongoing chunks shrink to
 * the pages available; admission stops at the first request whose first
 * chunk's pages cannot be allocated; pages come from the front of a FIFO free
 * list and return to its back; no preemption (a decode that finds no page
 * fails with HB_ERR_OUT_OF_PAGES); decodes that alone exceed the budget are
 * all kept and flagged over_budget.
 * ------------------------------------------------------------------------- */
typedef struct hb_builder hb_builder;

/* page_order: NULL for 0..num_pages-1, else a host permutation of it that
 * seeds the free list.  *out receives a new builder. */
hb_status hb_builder_create(int32_t budget, int32_t page_size,
                            int32_t num_pages, int32_t max_pages_per_seq,
                            const int32_t* page_order, hb_builder** out);
void hb_builder_destroy(hb_builder* b);

/* Queue a request (arrival order = call order).  HB_ERR_SHAPE if
 * prompt_len < 1, max_new < 1 or the request cannot fit max_pages_per_seq;
 * HB_ERR_INVALID_ARG for a duplicate id. */
hb_status hb_builder_add_request(hb_builder* b, int64_t id, int32_t prompt_len,
                                 int32_t max_new);

/* Form the next batch into caller-owned host arrays with room for max_rows
 * rows: q_len, context_len [max_rows], block_table [max_rows *
 * max_pages_per_seq] (unused entries -1), row_ids [max_rows], row_kind
 * [max_rows] (0 decode, 1 prefill).  *num_rows = 0 means nothing to run.
 * HB_ERR_WORKSPACE if max_rows is too small, HB_ERR_OUT_OF_PAGES if a
 * decode finds no free page; after any error the builder is unchanged.
 * A step costs what its rows and their pages cost, whatever the pool size.
 * Call hb_builder_complete before the next step. */
hb_status hb_builder_step(hb_builder* b, int32_t max_rows, int32_t* num_rows,
                          int32_t* q_len, int32_t* context_len,
                          int32_t* block_table, int64_t* row_ids,
                          int32_t* row_kind, int32_t* over_budget);

/* The batch of the last step ran.  Writes up to max_finished ids of the
 * requests that finished (in batch order) and their count. */
hb_status hb_builder_complete(hb_builder* b, int32_t max_finished,
                              int32_t* num_finished, int64_t* finished_ids);

/* Message for the last failed hb_builder_* call on this thread. */
const char* hb_builder_last_error(void);

/* Counts: waiting requests, running requests, free pages. */
hb_status hb_builder_counts(const hb_builder* b, int32_t* waiting,
                            int32_t* running, int32_t* free_pages);

/* The free list, front first (up to max entries; *n receives its length). */
hb_status hb_builder_free_list(const hb_builder* b, int32_t max, int32_t* n,
                               int32_t* pages);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* HB_H_ */
