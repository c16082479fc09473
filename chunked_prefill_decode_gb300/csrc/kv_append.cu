// kv_append.cu -- scatter the batch's new K/V rows into their cache pages.
//
// "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §GPU / 系统数据路径 ⑤: a prefill chunk appends its new KV (and a
// decode its one new token) into the paged cache before attention reads it.
//
// With NHD pages ([page][slot][kv_head][head_dim]) one token's K row
// (Hkv * D bf16 = 2 KB at Hkv 8, D 128) is contiguous both in k_new and in
// its page slot, so the scatter is a set of contiguous row copies: one warp
// per (token, K|V) row moves it with 16-byte loads/stores, fully coalesced.
// The kernel is bound by HBM: 2 * T * Hkv * D * 2 bytes read + the same
// written.
#include <cuda_runtime.h>

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

// cu_q_len is staged in shared memory for batches up to this many sequences
constexpr int kAppendSmemSeqs = 8191;
// 16-byte vectors per lane held in registers (rows up to 32 x 8 x 16 B = 4 KB)
constexpr int kAppendVecsPerLane = 8;

__global__ void __launch_bounds__(256) kv_append_kernel(AppendParams p) {
  extern __shared__ int32_t s_cu[];
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  // the row -> sequence search runs on a shared-memory copy of cu_q_len (one
  // coalesced load per CTA instead of a chain of dependent global loads)
  const bool staged = p.num_seqs <= kAppendSmemSeqs;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int n_rows = 2 * p.total_q;
  const size_t row_vecs = (size_t)p.row_vec16;
  // a row's data does not depend on where it goes: its loads are issued
  // before the sequence / page lookups (for the first row, even before the
  // staging of cu_q_len) and overlap them
  uint4 buf[kAppendVecsPerLane];
  auto load_row = [&](int r) {
    const uint4* src = reinterpret_cast<const uint4*>((r & 1) ? p.v_new : p.k_new) +
                       (size_t)(r >> 1) * row_vecs;
#pragma unroll
    for (int i = 0; i < kAppendVecsPerLane; ++i) {
      const int v = lane + 32 * i;
      if (v < p.row_vec16) buf[i] = ld_stream(src + v);
    }
  };
  int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (r < n_rows) load_row(r);
  if (staged)
    for (int i = threadIdx.x; i <= p.num_seqs; i += blockDim.x) s_cu[i] = __ldg(&p.cu_q_len[i]);
  __syncthreads();
  const int32_t* cu = staged ? s_cu : p.cu_q_len;
  for (bool first = true; r < n_rows; r += warps_total, first = false) {
    const int tok = r >> 1;
    const bool is_v = (r & 1) != 0;
    if (!first) load_row(r);
    const uint4* src = reinterpret_cast<const uint4*>(is_v ? p.v_new : p.k_new) +
                       (size_t)tok * row_vecs;
    // sequence owning this token: the largest s with cu_q_len[s] <= tok
    int lo = 0, hi = p.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu[mid] <= tok) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int q0 = cu[s];
    const int q_len = cu[s + 1] - q0;
    const int pos = __ldg(&p.context_len[s]) - q_len + (tok - q0);
    const int lp = pos / kPageSize;
    int page = -1;
    if (pos >= 0 && lp < p.max_pages_per_seq)
      page = __ldg(&p.block_table[(size_t)s * p.max_pages_per_seq + lp]);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) report_error(p.dev_error, HB_DEVERR_INDEX);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(is_v ? p.v_cache : p.k_cache) +
                 ((size_t)page * kPageSize + (pos % kPageSize)) * row_vecs;
#pragma unroll
    for (int i = 0; i < kAppendVecsPerLane; ++i) {
      const int v = lane + 32 * i;
      if (v < p.row_vec16) dst[v] = buf[i];
    }
    // rows of more than 4 KB (Hkv * D > 2048) copy the rest directly
    for (int v = lane + 32 * kAppendVecsPerLane; v < p.row_vec16; v += 32) dst[v] = ld_stream(src + v);
  }
}

cudaError_t launch_kv_append(const AppendParams& p, int num_sms,
                             cudaStream_t stream) {
  if (p.total_q == 0) return cudaSuccess;
  const int warps_per_block = 8;
  long blocks = (2L * p.total_q + warps_per_block - 1) / warps_per_block;
  const long cap = 16L * num_sms;
  if (blocks > cap) blocks = cap;
  const size_t smem = p.num_seqs <= kAppendSmemSeqs ? (size_t)(p.num_seqs + 1) * 4 : 0;
  return launch_serialized(kv_append_kernel, (unsigned)blocks, 32 * warps_per_block, smem, stream, p);
}

}  // namespace hb
