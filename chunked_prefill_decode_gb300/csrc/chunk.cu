// chunk.cu -- attention of prefill chunks on the tcgen05 tensor cores.
//
// "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §核心机制 3 and §GPU / 系统数据路径 ⑤: chunk i of a prompt attends
// causally to itself and re-reads the KV of chunks 1..i-1 through the page
// table; the computation equals that of the unchunked prefill.  "In-flight
// Batching", §LLM 推理的两阶段计算特征: prefill is compute-bound, so QK^T and PV
// run as the dense contractions they are, on the tensor cores.
//
// One CTA takes one work item: a 128-row query tile made of (token, q head)
// pairs of one kv head's GQA group (tokens_per_tile = 128 / g tokens times
// the g heads, so one K/V tile in shared memory serves the whole group), and
// walks the 128-key tiles 0 .. (last position in the tile) of its sequence.
//
// Warp roles (192 threads):
//   warp 0     TMA producer: the Q tile once (3-D map over q, box
//              64 x g x tokens), then per KV tile eight 16-token pages of K
//              and of V (3-D map over the pools, one box per page and
//              64-wide head-dim chunk, coordinates from the block table;
//              pages past the context are fetched out of range, i.e. zeros);
//   warp 1     TMEM owner and MMA issuer: S_j = Q K_j^T (M 128, N 128, K D)
//              into one of two S buffers, then O += P_j V_j (M 128, N D,
//              K 128) with V read MN-major straight from its page layout;
//   warps 2-5  softmax: thread = query row = TMEM lane; S row to registers
//              (tcgen05.ld), causal mask on tiles that cross the diagonal,
//              exp2 with the scale * log2 e folded in, P as bf16 into a
//              128-byte-swizzled K-major shared tile (the A operand of PV),
//              row sum from the same rounded P; O in TMEM is rescaled only
//              when a row maximum grows by more than 2^8 (the stale maximum is
//              exact as long as it bounds P, and P <= 2^8 is safe); epilogue
//              O / l to bf16.
// TMEM: S0 columns 0-127, S1 128-255, O 256-(256+D).
#include <cuda_runtime.h>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

constexpr int kChunkThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct ChunkCfg {
  static constexpr int CH = D / 64;                    // 128-byte K chunks
  static constexpr int NS = (D == 128) ? 2 : 3;         // KV stages
  static constexpr int kTileBytes = CH * 16384;         // 128 rows x D bf16
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kTileBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;    // K tile + V tile
  static constexpr int kPOff = kKVOff + NS * kStageBytes;
  static constexpr int kPBytes = 2 * 16384;             // 128 x 128 bf16
  static constexpr int kBarOff = kPOff + 2 * kPBytes;
  static constexpr int kNumBars = 1 + 2 * NS + 2 + 2 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 256;
};

template <int D>
__global__ void __launch_bounds__(kChunkThreads, 1)
    chunk_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap) {
  using C = ChunkCfg<D>;
  constexpr int CH = C::CH;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sKV = smem + C::kKVOff;
  uint8_t* sP = smem + C::kPOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + NS;
  uint64_t* s_full = kv_empty + NS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* mma_done = o_full + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  int* abort_i = reinterpret_cast<int*>(smem + C::kMiscOff + 16);
  volatile int* abort_flag = abort_i;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const ChunkItem it = p.items[blockIdx.x];
  const int g = p.group;
  const int tpt = p.tokens_per_tile;
  const int q0 = __ldg(&p.cu_q_len[it.seq]);
  const int q_len = __ldg(&p.cu_q_len[it.seq + 1]) - q0;
  const int ctx = __ldg(&p.context_len[it.seq]);
  const int off = ctx - q_len;            // tokens cached before this chunk
  const int n_tiles = it.kv_tiles;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 128);
    }
    mbar_init(o_full, 1);
    mbar_init(mma_done, 1);
    *abort_i = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      mbar_arrive_expect_tx(q_full, (uint32_t)(CH * g * tpt * 128));
#pragma unroll
      for (int c = 0; c < CH; ++c)
        tma_load_3d(sQ + c * 16384, &qmap, q_full, c * 64, it.kv_head * g,
                    q0 + it.tok0);
      const int n_pages = (ctx + kPageSize - 1) / kPageSize;
      bool issued[NS];
      uint32_t last_par[NS];
      for (int s = 0; s < NS; ++s) {
        issued[s] = false;
        last_par[s] = 0;
      }
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % NS;
        const uint32_t ph = (uint32_t)(j / NS) & 1u;
        if (!mbar_wait(&kv_empty[s], ph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(&kv_full[s], (uint32_t)C::kStageBytes);
        uint8_t* sK = sKV + s * C::kStageBytes;
        uint8_t* sV = sK + C::kTileBytes;
#pragma unroll 1
        for (int pp = 0; pp < kChunkKeys / kPageSize; ++pp) {
          const int lp = j * (kChunkKeys / kPageSize) + pp;
          int phys = p.num_pages;  // out of range: the copy fills zeros
          if (lp < n_pages) {
            phys = (lp < p.max_pages_per_seq)
                       ? __ldg(&p.block_table[(size_t)it.seq * p.max_pages_per_seq + lp])
                       : -1;
            if (phys < 0 || phys >= p.num_pages) {
              report_error(p.dev_error, HB_DEVERR_INDEX);
              phys = p.num_pages;
            }
          }
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            tma_load_3d(sK + c * 16384 + pp * 2048, &kmap, &kv_full[s], c * 64,
                        it.kv_head, phys * kPageSize);
            tma_load_3d(sV + c * 16384 + pp * 2048, &vmap, &kv_full[s], c * 64,
                        it.kv_head, phys * kPageSize);
          }
        }
        issued[s] = true;
        last_par[s] = ph;
      }
      // copies in flight must land before the CTA exits
      drain_wait(q_full, 0u, abort_flag);
      for (int s = 0; s < NS; ++s)
        if (issued[s]) drain_wait(&kv_full[s], last_par[s], abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, kChunkKeys, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      const uint32_t aQ = smem_u32(sQ);
      const uint32_t aP = smem_u32(sP);
      const uint32_t aKV = smem_u32(sKV);
      bool ok = mbar_wait(q_full, 0u, abort_flag);
      auto issue_pv = [&](int i) -> bool {
        const int pb = i & 1;
        if (!mbar_wait(&p_full[pb], (uint32_t)(i >> 1) & 1u, abort_flag)) return false;
        tc_fence_after_sync();
        const int s = i % NS;
        const uint32_t aV = aKV + s * C::kStageBytes + C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kChunkKeys / 16; ++kk) {
          const uint64_t a = sdesc_sw128(aP + pb * C::kPBytes + (kk >> 2) * 16384 + (kk & 3) * 32,
                                         16, 1024);
          const uint64_t b = sdesc_sw128(aV + kk * 2048, 16384, 1024);
          tc_mma_bf16(tmem + C::kOCol, a, b, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&kv_empty[s]);
        tc_commit(o_full);
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j % NS;
        if (!mbar_wait(&kv_full[s], (uint32_t)(j / NS) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int sb = j & 1;
        const uint32_t aK = aKV + s * C::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(aQ + koff, 16, 1024);
          const uint64_t b = sdesc_sw128(aK + koff, 16, 1024);
          tc_mma_bf16(tmem + sb * kChunkKeys, a, b, idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[sb]);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(n_tiles - 1);
      // every MMA issued must complete before TMEM is freed
      tc_commit(mma_done);
      drain_wait(mma_done, 0u, abort_flag);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const int tok_local = row / g;
    const bool valid_row = (row < g * tpt) && (tok_local < it.ntok);
    const int tok_rel = it.tok0 + tok_local;
    const int pos = valid_row ? off + tok_rel : ctx - 1;  // absolute position
    const int min_pos = off + it.tok0;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    uint8_t* prow_base = sP + row * 128;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (uint32_t)(j >> 1) & 1u, abort_flag)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t sr[kChunkKeys];
#pragma unroll
      for (int q = 0; q < kChunkKeys / 32; ++q)
        tmem_ld32(t_lane + sb * kChunkKeys + q * 32, &sr[q * 32]);
      tmem_ld_wait();
      const int kbase = j * kChunkKeys;
      const bool need_mask = kbase + kChunkKeys - 1 > min_pos;
      float alpha = 1.f;
      bool resc = false;
      uint8_t* prow = prow_base + sb * C::kPBytes;
      if (valid_row) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < kChunkKeys; ++i) {
          float x = __uint_as_float(sr[i]) * sl2;
          if (need_mask && kbase + i > pos) x = -INFINITY;
          sr[i] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
        const float m_new = fmaxf(m_run, mx);
        if (m_new > m_run + kRescaleThreshold) {
          alpha = fast_exp2(m_run - m_new);
          m_run = m_new;
          resc = true;
        }
        float lsum = 0.f;
#pragma unroll
        for (int u = 0; u < kChunkKeys / 8; ++u) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a0 = fast_exp2(__uint_as_float(sr[u * 8 + 2 * e]) - m_run);
            const float a1 = fast_exp2(__uint_as_float(sr[u * 8 + 2 * e + 1]) - m_run);
            pk[e] = pack_bf16x2(a0, a1);
            lsum += bf16lo_to_f32(pk[e]) + bf16hi_to_f32(pk[e]);
          }
          const int c = u >> 3, uu = u & 7;
          *reinterpret_cast<uint4*>(prow + c * 16384 + ((uu ^ (row & 7)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        l_run = l_run * alpha + lsum;
      } else {
#pragma unroll
        for (int u = 0; u < kChunkKeys / 8; ++u) {
          const int c = u >> 3, uu = u & 7;
          *reinterpret_cast<uint4*>(prow + c * 16384 + ((uu ^ (row & 7)) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (j == n_tiles - 1) {
        // keys past the context in the last page were never written: clear
        // their V rows so that P = 0 never multiplies a NaN
        const int s = j % NS;
        const int first_bad = ctx - kbase;
        const int end_bad = min(kChunkKeys, ((ctx + kPageSize - 1) / kPageSize) * kPageSize - kbase);
        if (first_bad < end_bad) {
          if (!mbar_wait(&kv_full[s], (uint32_t)(j / NS) & 1u, abort_flag)) { ok = false; break; }
          uint8_t* sV = sKV + s * C::kStageBytes + C::kTileBytes;
          const int n_units = (end_bad - first_bad) * CH * 8;
          for (int e = row; e < n_units; e += 128) {
            const int key = first_bad + e / (CH * 8);
            const int rem = e % (CH * 8);
            *reinterpret_cast<uint4*>(sV + (rem >> 3) * 16384 + key * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      if (j >= 1) {
        // PV(j-1) must be complete before O is rescaled (and, one tile later,
        // before P buffer (j+1)&1 is overwritten)
        if (!mbar_wait(o_full, (uint32_t)(j - 1) & 1u, abort_flag)) { ok = false; break; }
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, resc)) {
          const float f = resc ? alpha : 1.f;
#pragma unroll 1
          for (int q = 0; q < D / 32; ++q) {
            uint32_t orow[32];
            tmem_ld32(t_lane + C::kOCol + q * 32, orow);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              orow[i] = __float_as_uint(__uint_as_float(orow[i]) * f);
            tmem_st32(t_lane + C::kOCol + q * 32, orow);
          }
          tmem_st_wait();
        }
      }
      fence_async_shared();
      tc_fence_before_sync();
      mbar_arrive(&p_full[sb]);
    }
    // epilogue: O / l -> bf16
    if (ok && mbar_wait(o_full, (uint32_t)(n_tiles - 1) & 1u, abort_flag)) {
      tc_fence_after_sync();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      uint16_t* dst = p.out + ((size_t)(q0 + tok_rel) * p.num_q_heads +
                               (size_t)it.kv_head * g + (row % g)) * D;
#pragma unroll 1
      for (int q = 0; q < D / 32; ++q) {
        uint32_t orow[32];
        tmem_ld32(t_lane + C::kOCol + q * 32, orow);
        tmem_ld_wait();
        if (valid_row) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(orow[v * 8 + 0]) * inv, __uint_as_float(orow[v * 8 + 1]) * inv);
            pk.y = pack_bf16x2(__uint_as_float(orow[v * 8 + 2]) * inv, __uint_as_float(orow[v * 8 + 3]) * inv);
            pk.z = pack_bf16x2(__uint_as_float(orow[v * 8 + 4]) * inv, __uint_as_float(orow[v * 8 + 5]) * inv);
            pk.w = pack_bf16x2(__uint_as_float(orow[v * 8 + 6]) * inv, __uint_as_float(orow[v * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + q * 32 + v * 8) = pk;
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) report_error(p.dev_error, HB_DEVERR_TIMEOUT);
}

cudaError_t launch_chunk(const ChunkParams& p, int head_dim,
                         const CUtensorMap& qmap, const CUtensorMap& kmap,
                         const CUtensorMap& vmap, cudaStream_t stream) {
  if (p.num_items == 0) return cudaSuccess;
  cudaError_t e;
  if (head_dim == 128) {
    constexpr int smem = ChunkCfg<128>::kSmemBytes;
    e = cudaFuncSetAttribute(chunk_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_kernel<128><<<p.num_items, kChunkThreads, smem, stream>>>(p, qmap, kmap, vmap);
  } else {
    constexpr int smem = ChunkCfg<64>::kSmemBytes;
    e = cudaFuncSetAttribute(chunk_kernel<64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_kernel<64><<<p.num_items, kChunkThreads, smem, stream>>>(p, qmap, kmap, vmap);
  }
  return cudaGetLastError();
}

}  // namespace hb
