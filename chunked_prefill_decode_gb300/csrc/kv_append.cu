// kv_append.cu -- scatter the batch's new K/V rows into their cache pages.
//
// "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §GPU / 系统数据路径 ⑤: a prefill chunk appends its new KV (and a
// decode its one new token) into the paged cache before attention reads it.
//
// With NHD pages ([page][slot][kv_head][head_dim]) one token's K row
// (Hkv * D bf16 = 2 KB at Hkv 8, D 128) is contiguous both in k_new and in
// its page slot, so the scatter is a set of contiguous row copies.  The
// kernel is bound by HBM: 2 * T * Hkv * D * 2 bytes read + the same written.
//
// One warp moves one segment of up to 2 KB of one row (4 x 16 bytes per
// lane), so every segment is in flight at once: the grid is one warp per
// segment; with <= 64 registers per thread two 512-thread CTAs share an SM,
// so a batch of up to 152 x 2 x 16 segments (19 MB of K and V at 2 KB rows)
// runs in a single wave, and the CTA size shrinks with the batch so that a
// small batch still spreads over many SMs.  A warp issues its data loads
// first; the row -> sequence search (over a shared-memory copy of
// cu_q_len), the context length and the block-table entry are looked up
// while the data is on its way, so the dependent index chain overlaps the
// copy instead of preceding it.
#include <cuda_runtime.h>

#include <algorithm>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// cu_q_len and context_len are staged in shared memory for batches up to this
// many sequences (at most 48 KB, the dynamic shared memory a launch gets
// without opting in)
constexpr int kAppendSmemSeqs = 6143;
constexpr int kAppendMaxWarps = 16;             // warps per CTA (at most)
constexpr int kSegVecsPerLane = 4;              // 16-byte vectors per lane
constexpr int kSegVecs = 32 * kSegVecsPerLane;  // vectors per segment (2 KB)

__global__ void __launch_bounds__(32 * kAppendMaxWarps, 2) kv_append_kernel(AppendParams p) {
  extern __shared__ int32_t s_cu[];
  // k_new / v_new may come from the kernel before this one, and the pages
  // written here may be read by it: wait for it first
  griddep_wait();
  if (p.ready_flag) {
    // the inputs come from a copy on another stream, which then raises the
    // flag; the next kernel (which reads more of what that stream copied)
    // is let in only after it.  One lane per warp polls; the CTA goes on
    // only if every warp saw the flag (a barrier reduction, so the CTA
    // decides as one and no shared memory is taken from the staging).  The
    // wait is bounded: a flag that never comes is reported as a timeout and
    // the batch is left unwritten.
    if (!__syncthreads_and(warp_wait_flag(p.ready_flag, p.ready_value, p.dev_error))) {
      griddep_launch_dependents();
      return;
    }
  }
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int spr = (p.row_vec16 + kSegVecs - 1) / kSegVecs;   // segments per row
  const int64_t n_k = (int64_t)p.total_q * spr;              // segments of the K rows
  const int64_t seg = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const bool live = seg < 2 * n_k;
  const bool is_v = seg >= n_k;
  const int64_t sk = is_v ? seg - n_k : seg;
  const int tok = (int)(sk / spr);
  const int v_begin = (int)(sk % spr) * kSegVecs;
  const int v_end = min(p.row_vec16, v_begin + kSegVecs);
  const size_t row_vecs = (size_t)p.row_vec16;
  uint4 buf[kSegVecsPerLane];
  if (live) {
    const uint4* src = reinterpret_cast<const uint4*>(is_v ? p.v_new : p.k_new) +
                       (size_t)tok * row_vecs;
#pragma unroll
    for (int i = 0; i < kSegVecsPerLane; ++i) {
      const int v = v_begin + lane + 32 * i;
      if (v < v_end) buf[i] = ld_stream(src + v);
    }
  }
  // cu_q_len and context_len are staged together (their loads overlap), so
  // the only dependent global load left after the search is the page id
  const bool staged = p.num_seqs <= kAppendSmemSeqs;
  int32_t* s_ctx = s_cu + p.num_seqs + 1;
  if (staged) {
    for (int i = threadIdx.x; i <= p.num_seqs; i += blockDim.x) s_cu[i] = __ldg(&p.cu_q_len[i]);
    for (int i = threadIdx.x; i < p.num_seqs; i += blockDim.x) s_ctx[i] = __ldg(&p.context_len[i]);
  }
  __syncthreads();
  if (!live) return;
  const int32_t* cu = staged ? s_cu : p.cu_q_len;
  const int32_t* ctx = staged ? s_ctx : p.context_len;
  // sequence owning this token: the largest s with cu_q_len[s] <= tok
  int lo = 0, hi = p.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  const int q0 = cu[s];
  const int q_len = cu[s + 1] - q0;
  const int pos = ctx[s] - q_len + (tok - q0);
  const int lp = pos / kPageSize;
  int page = -1;
  if (pos >= 0 && lp < p.max_pages_per_seq)
    page = __ldg(&p.block_table[(size_t)s * p.max_pages_per_seq + lp]);
  if (page < 0 || page >= p.num_pages) {
    if (lane == 0) report_error(p.dev_error, HB_DEVERR_INDEX);
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(is_v ? p.v_cache : p.k_cache) +
               ((size_t)page * kPageSize + (pos % kPageSize)) * row_vecs;
#pragma unroll
  for (int i = 0; i < kSegVecsPerLane; ++i) {
    const int v = v_begin + lane + 32 * i;
    if (v < v_end) dst[v] = buf[i];
  }
}

cudaError_t launch_kv_append(const AppendParams& p, int num_sms, cudaStream_t stream) {
  if (p.total_q == 0) return cudaSuccess;
  const int64_t spr = (p.row_vec16 + kSegVecs - 1) / kSegVecs;
  const int64_t segs = 2LL * p.total_q * spr;
  // CTAs of 4 to 16 warps: about two per SM when the batch is large (few
  // CTAs to schedule, one wave), smaller ones spread a small batch over more
  // SMs
  int64_t warps = (segs + 2LL * num_sms - 1) / (2LL * num_sms);
  warps = std::min<int64_t>(kAppendMaxWarps, std::max<int64_t>(4, warps));
  const int64_t blocks = (segs + warps - 1) / warps;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = p.num_seqs <= kAppendSmemSeqs ? (size_t)(2 * p.num_seqs + 1) * 4 : 0;
  return launch_serialized(kv_append_kernel, (unsigned)blocks, (unsigned)(32 * warps), smem,
                           stream, p);
}

}  // namespace hb
