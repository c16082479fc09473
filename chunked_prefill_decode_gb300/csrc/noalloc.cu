// noalloc.cu -- decode-row attention for callers that cannot allocate.
//
// hb_attention needs a caller-provided device workspace (work items, counters
// and the split-KV partial softmax states).  Some callers have no way to get
// one: a serving engine that hands nearly all free HBM to its KV-cache pool
// at start-up and forbids device allocations afterwards, or a plugin that
// receives raw tensor pointers but no allocator.  hb_decode_attention_noalloc
// serves them: it runs the same attention kernel (decode CTAs only) with its
// scratch in a
// fixed array of HB_NOALLOC_SCRATCH_BYTES that lives in this file and is
// created when the library is loaded (every device that loads the library
// holds it until the process exits).  It makes no cudaMalloc / cudaFree call
// and uses no allocating library routine; the host-side plan goes into static
// host storage as well.
//
// Consequences of the shared array: all calls on a device use the same
// scratch, so calls whose work overlaps on the GPU (two streams, two host
// threads) race and must be serialised by the caller; each call clears the
// counters it needs, everything else is overwritten before it is read.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "decode_plan.h"
#include "hb.h"
#include "hb_internal.h"

namespace hb {
cudaError_t launch_attention(const DecodeParams& dec, int decode_grid, const ChunkParams& chk,
                             int head_dim, const CUtensorMap& dec_k, const CUtensorMap& dec_v,
                             const CUtensorMap& chunk_q, const CUtensorMap& chunk_k,
                             const CUtensorMap& chunk_v, const CUtensorMap& chunk_knew,
                             const CUtensorMap& chunk_vnew, const void* k_cache,
                             const void* v_cache, cudaStream_t stream, bool early,
                             int pairs_mode);
hb_status internal_fail(hb_status s, const char* msg);
hb_status internal_ok();
hb_status internal_check_batch(const hb_batch* b);
hb_status internal_device(int** err, int* num_sms);
hb_status internal_decode_maps(const hb_batch* b, int kvhb, const void* k_cache,
                               const void* v_cache, CUtensorMap* kmap, CUtensorMap* vmap);
void internal_count_launch();
void internal_note_other_launch(void* stream);
}  // namespace hb

using namespace hb;

// The scratch: [items | CTA offsets | counters | partial o | partial (m, l)].
static __device__ __align__(256) unsigned char g_noalloc_scratch[HB_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxItems = 4096;
constexpr int kMaxMerges = 4096;
constexpr int kMaxGrid = 1024;
constexpr size_t kItemsBytes = (size_t)kMaxItems * sizeof(DecodeItem);
constexpr size_t kOffsetsOff = kItemsBytes;
constexpr size_t kCountersOff = kOffsetsOff + (size_t)(kMaxGrid + 1) * 4;
constexpr size_t kCountersBytes = (size_t)(kCounterMerge0 + kMaxMerges) * 4;
constexpr size_t kPartialOff = (kCountersOff + kCountersBytes + 255) / 256 * 256;
static_assert(kPartialOff < HB_NOALLOC_SCRATCH_BYTES, "scratch layout");

std::mutex g_mu;
void* g_scratch[64] = {};     // device address of the array, per device
DecodeItem g_items[kMaxItems];  // host-side plan (static: nothing is allocated)
int32_t g_offsets[kMaxGrid + 1];

// Address of this device's copy of the array; looked up on the first call on
// each device (the device must be current).
hb_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return internal_fail(HB_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= 64) return internal_fail(HB_ERR_UNSUPPORTED, "device index out of range");
  if (!g_scratch[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return internal_fail(HB_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return HB_OK;
}

}  // namespace

extern "C" hb_status hb_decode_attention_noalloc(const hb_batch* batch, const int32_t* h_q_len,
                                                 const int32_t* h_context_len, const void* q,
                                                 const void* k_cache, const void* v_cache,
                                                 float softmax_scale, void* out, void* stream) {
  try {
    std::lock_guard<std::mutex> lk(g_mu);
    hb_status s = internal_check_batch(batch);
    if (s != HB_OK) return s;
    const int S = batch->num_seqs;
    if (S == 0) return internal_ok();
    if (!h_q_len || !h_context_len)
      return internal_fail(HB_ERR_INVALID_ARG, "h_q_len and h_context_len must be non-NULL");
    for (const void* ptr : {q, k_cache, v_cache, static_cast<const void*>(out)})
      if (!ptr || (reinterpret_cast<uintptr_t>(ptr) & 15u))
        return internal_fail(HB_ERR_INVALID_ARG, "q, k_cache, v_cache and out must be non-NULL and 16-byte aligned");
    const int Hq = batch->num_q_heads, Hkv = batch->num_kv_heads, D = batch->head_dim;
    const int64_t max_ctx = (int64_t)batch->max_pages_per_seq * kPageSize;
    for (int i = 0; i < S; ++i) {
      if (h_q_len[i] != 1)
        return internal_fail(HB_ERR_UNSUPPORTED, "hb_decode_attention_noalloc takes decode rows only (q_len == 1)");
      if (h_context_len[i] < 1 || h_context_len[i] > max_ctx)
        return internal_fail(HB_ERR_SHAPE, "context_len outside 1 .. max_pages_per_seq * 16");
    }
    if (batch->total_q != S) return internal_fail(HB_ERR_SHAPE, "total_q must equal num_seqs");
    const int g = Hq / Hkv;
    // The work list below is copied from this file's static host storage
    // when the call is made.  A captured copy would read that storage again
    // at every replay, after later calls have overwritten it, so a call on a
    // stream that is being captured is refused.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap) != cudaSuccess)
      return internal_fail(HB_ERR_CUDA, "cudaStreamIsCapturing failed");
    if (cap != cudaStreamCaptureStatusNone)
      return internal_fail(HB_ERR_UNSUPPORTED,
                           "hb_decode_attention_noalloc cannot be called on a stream that is "
                           "being captured (its work list is copied from host memory at the call)");

    // ---- plan into static host storage: the decode partition over at most
    // one CTA per SM; fewer, longer ranges until the partial states fit
    const int kvhb = std::min(Hkv, kDecodeKvhBlock);
    const int n_blocks = Hkv / kvhb;
    int* err = nullptr;
    int num_sms = 0;
    if ((s = internal_device(&err, &num_sms)) != HB_OK) return s;
    const size_t slot_bytes = (size_t)Hq * D * 4 + (size_t)Hq * 8;
    const size_t partial_room = HB_NOALLOC_SCRATCH_BYTES - kPartialOff;
    int max_grid = std::min(num_sms, kMaxGrid);
    DecodePartition part;
    for (;;) {
      if (!partition_decode(S, h_q_len, h_context_len, n_blocks, kvhb, num_sms, 4, g_items,
                            kMaxItems, g_offsets, max_grid, &part, batch->sliding_window))
        return internal_fail(HB_ERR_WORKSPACE,
                             "batch needs more work items than the static scratch holds "
                             "(at most 4096 = num_seqs * ceil(Hkv / 8) plus one per SM)");
      if (part.n_merge <= kMaxMerges && (size_t)part.n_slots * slot_bytes <= partial_room) break;
      if (max_grid == 1)
        return internal_fail(HB_ERR_WORKSPACE, "partial states do not fit the static scratch");
      max_grid = std::max(1, max_grid / 2);
    }
    const int k = part.n_items;
    const int n_slots = part.n_slots, n_merge = part.n_merge;

    void* scratch = nullptr;
    if ((s = scratch_address(&scratch)) != HB_OK) return s;
    uint8_t* base = static_cast<uint8_t*>(scratch);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(base, g_items, (size_t)k * sizeof(DecodeItem),
                                    cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return internal_fail(HB_ERR_CUDA, "copy of the work items failed");
    e = cudaMemcpyAsync(base + kOffsetsOff, g_offsets, (size_t)(part.grid + 1) * 4,
                        cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return internal_fail(HB_ERR_CUDA, "copy of the CTA offsets failed");
    e = cudaMemsetAsync(base + kCountersOff, 0, (size_t)(kCounterMerge0 + n_merge) * 4, st);
    if (e != cudaSuccess) return internal_fail(HB_ERR_CUDA, "clearing the counters failed");

    CUtensorMap kmap, vmap;
    if ((s = internal_decode_maps(batch, kvhb, k_cache, v_cache, &kmap, &vmap)) != HB_OK) return s;
    DecodeParams p{};
    p.items = reinterpret_cast<const DecodeItem*>(base);
    p.cta_offsets = reinterpret_cast<const int32_t*>(base + kOffsetsOff);
    p.num_static = part.grid;
    p.num_dynamic = 0;
    p.num_items = k;
    p.counters = reinterpret_cast<int32_t*>(base + kCountersOff);
    p.part_o = reinterpret_cast<float*>(base + kPartialOff);
    p.part_ml = reinterpret_cast<float*>(base + kPartialOff + (size_t)n_slots * Hq * D * 4);
    p.cu_q_len = batch->cu_q_len;
    p.context_len = batch->context_len;
    p.block_table = batch->block_table;
    p.max_pages_per_seq = batch->max_pages_per_seq;
    p.num_pages = batch->num_pages;
    p.q = static_cast<const uint16_t*>(q);
    p.out = static_cast<uint16_t*>(out);
    p.num_q_heads = Hq;
    p.num_kv_heads = Hkv;
    p.group = g;
    p.kvh_block = kvhb;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.dev_error = err;
    p.window = batch->sliding_window;
    ChunkParams none{};
    none.group = g;
    CUtensorMap unused;
    std::memset(&unused, 0, sizeof(unused));
    e = launch_attention(p, part.grid, none, D, kmap, vmap, unused, unused, unused, unused,
                         unused, k_cache, v_cache, st, /*early=*/false, /*pairs_mode=*/0);
    if (e != cudaSuccess) return internal_fail(HB_ERR_CUDA, "decode launch failed");
    internal_note_other_launch(stream);
    internal_count_launch();
    return internal_ok();
  } catch (...) {
    return internal_fail(HB_ERR_CUDA, "unexpected exception in hb_decode_attention_noalloc");
  }
}
