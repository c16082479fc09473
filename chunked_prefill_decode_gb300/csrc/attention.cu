// attention.cu -- the single attention launch of a hybrid batch.
//
// "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §GPU / 系统数据路径 ③: one iteration's batch holds decode tokens and
// prefill chunks together; "In-flight Batching", §Batch 内的异构执行: the
// different lengths are handled inside one kernel launch.
//
// One grid serves both kinds of work.  CTAs 0 .. decode_grid-1 each stream
// one equal range of the decode rows' pages (decode_body.cuh, HBM-bound);
// every later CTA takes one chunk work item, longest first
// (chunk_body.cuh, tensor-core-bound).  Every CTA uses ~220 KB of shared
// memory, so one CTA runs per SM and the hardware hands out CTAs in index
// order as SMs free up: the first wave runs decode ranges and chunk items
// side by side, and SMs that finish their decode range go on to the
// remaining chunk items.  The host plan picks decode_grid so that both kinds
// of work end together.  No CTA waits for another.
#include <cuda_runtime.h>

#include <atomic>

#include "chunk_body.cuh"
#include "decode_body.cuh"
#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

constexpr int kAttnThreads = 384;

struct AttnParams {
  DecodeParams dec;
  DecodeLayout dl;
  ChunkParams chk;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  int32_t decode_grid;
  // 1: the grid before this one is the append of this batch, which writes
  // only the pages with new tokens -- read every other page before it ends
  int32_t early;
};

template <int D, bool kPairs, bool kFew>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_kernel(const AttnParams p, const __grid_constant__ CUtensorMap dec_k,
                     const __grid_constant__ CUtensorMap dec_v,
                     const __grid_constant__ CUtensorMap chunk_q,
                     const __grid_constant__ CUtensorMap chunk_k,
                     const __grid_constant__ CUtensorMap chunk_v,
                     const __grid_constant__ CUtensorMap chunk_knew,
                     const __grid_constant__ CUtensorMap chunk_vnew) {
  extern __shared__ uint8_t smem_raw[];
  // the next kernel may be scheduled now (it waits for this one to finish).
  // After the append of this batch the previous grid is waited for only
  // before the pages that hold new tokens (decode_body.cuh, chunk_body.cuh
  // producers); after anything else, first.
  if (!p.early) griddep_wait();
  griddep_launch_dependents();
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  if ((int)blockIdx.x < p.decode_grid)
    decode_cta<D>(p.dec, p.dl, dec_k, dec_v, smem, blockIdx.x);
  else
    chunk_cta<D, kPairs, kFew>(p.chk, chunk_q, chunk_k, chunk_v, chunk_knew, chunk_vnew, p.k_cache,
                         p.v_cache, smem, blockIdx.x - p.decode_grid);
}

// Dynamic shared memory of the attention kernel for this geometry.
int attention_smem_bytes(int head_dim, int kvh_block, int group) {
  const DecodeLayout L = decode_layout(head_dim, kvh_block, group);
  const int c = head_dim == 128 ? ChunkCfg<128>::kSmemBytes : ChunkCfg<64>::kSmemBytes;
  return L.smem_bytes > c ? L.smem_bytes : c;
}

// Launch decode_grid decode CTAs followed by one CTA per chunk item.  Either
// part may be empty (dec.num_items == 0: no decode CTA).  dec.kvh_block and
// dec.group must be set in every case (they size the shared memory).
// chunk_knew / chunk_vnew map k_new / v_new when chk.has_new (else any map).
// pairs_mode bit 0: every chunk item is an unsplit pair of query tiles, and
// the kernel instantiation without the single-tile and split paths runs (the
// pair loop compiles to faster code on its own); bit 1: some item's first
// row sees few keys (its P is written in two terms), and the instantiation
// that can do so runs.
cudaError_t launch_attention(const DecodeParams& dec, int decode_grid, const ChunkParams& chk,
                             int head_dim, const CUtensorMap& dec_k, const CUtensorMap& dec_v,
                             const CUtensorMap& chunk_q, const CUtensorMap& chunk_k,
                             const CUtensorMap& chunk_v, const CUtensorMap& chunk_knew,
                             const CUtensorMap& chunk_vnew, const void* k_cache,
                             const void* v_cache, cudaStream_t stream, bool early,
                             int pairs_mode) {
  AttnParams p{};
  p.early = early ? 1 : 0;
  p.dec = dec;
  p.chk = chk;
  p.decode_grid = dec.num_items > 0 ? decode_grid : 0;
  p.dl = decode_layout(head_dim, dec.kvh_block, dec.group);
  if (p.decode_grid > 0 && p.dl.n_stages < 2) return cudaErrorInvalidConfiguration;
  p.k_cache = static_cast<const uint16_t*>(k_cache);
  p.v_cache = static_cast<const uint16_t*>(v_cache);
  const int grid = p.decode_grid + chk.num_items;
  if (grid == 0) return cudaSuccess;
  const int smem = attention_smem_bytes(head_dim, dec.kvh_block, dec.group);
  using Kernel = void (*)(const AttnParams, const __grid_constant__ CUtensorMap,
                          const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                          const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                          const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap);
  if (pairs_mode < 0 || pairs_mode > 3) return cudaErrorInvalidValue;
  const int which = (head_dim == 128 ? 4 : 0) + pairs_mode;
  const Kernel kernels[8] = {attention_kernel<64, false, false>,  attention_kernel<64, true, false>,
                             attention_kernel<64, false, true>,   attention_kernel<64, true, true>,
                             attention_kernel<128, false, false>, attention_kernel<128, true, false>,
                             attention_kernel<128, false, true>,  attention_kernel<128, true, true>};
  const Kernel kernel = kernels[which];
  // setmaxnreg.inc waits until the block's register pool holds what it asks
  // for; the chunk CTAs' split assumes the launch allocation of
  // kChunkLaunchRegs per thread, so a build that allocated fewer is refused
  // here instead of launched
  {
    static std::atomic<int> regs[8] = {};   // registers per instantiation, once known
    int n = regs[which].load(std::memory_order_relaxed);
    if (n == 0) {
      cudaFuncAttributes fa{};
      const cudaError_t ea = cudaFuncGetAttributes(&fa, kernel);
      if (ea != cudaSuccess) return ea;
      n = fa.numRegs;
      regs[which].store(n, std::memory_order_relaxed);
    }
    if (n < kChunkLaunchRegs) return cudaErrorInvalidConfiguration;
  }
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_serialized(kernel, grid, kAttnThreads, smem, stream, p, dec_k, dec_v, chunk_q,
                           chunk_k, chunk_v, chunk_knew, chunk_vnew);
}

}  // namespace hb
