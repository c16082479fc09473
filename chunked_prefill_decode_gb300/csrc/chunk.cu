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
//              64 x g x tokens), then K and V tiles into two separate rings
//              (K runs one tile ahead of V, since QK_j comes a softmax earlier
//              than PV_j); a tile is eight 16-token pages, one box per page
//              and 64-wide head-dim chunk, coordinates from the block table
//              (prefetched 32 pages at a time by the whole warp); pages past
//              the context are fetched out of range, i.e. as zeros;
//   warp 1     TMEM owner and MMA issuer: S_j = Q K_j^T (M 128, N 128, K D,
//              both operands K-major in shared memory) into one of two S
//              buffers, then O += P_j V_j (M 128, N D, K 128) with P read from
//              TMEM and V read MN-major straight from its page layout;
//   warps 2-5  softmax: thread = query row = TMEM lane; S row to registers
//              (tcgen05.ld), causal mask only on tiles that cross the
//              diagonal, p = 2^(s * scale * log2 e - m) as one FFMA + EX2, P
//              as bf16 into TMEM (tcgen05.st), row sum from the same rounded
//              P; O is rescaled in TMEM only when a row maximum grows by more
//              than 2^8 (a stale maximum stays exact while it bounds P, and
//              P <= 2^8 is safe in bf16 and fp32); epilogue O / l to bf16.
// TMEM (512 columns): S0 0-127, S1 128-255, O 256-(256+D), P0 384-447,
// P1 448-511 (P is 128 bf16 per row = 64 columns).
#include <cuda_runtime.h>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

constexpr int kChunkThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct ChunkCfg {
  static constexpr int CH = D / 64;                    // 128-byte K chunks
  static constexpr int kTileBytes = CH * 16384;         // 128 rows x D bf16
  static constexpr int NK = (D == 128) ? 3 : 4;         // K stages
  static constexpr int NV = (D == 128) ? 3 : 4;         // V stages
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTileBytes;
  static constexpr int kVOff = kKOff + NK * kTileBytes;
  static constexpr int kBarOff = kVOff + NV * kTileBytes;
  static constexpr int kNumBars = 1 + 2 * NK + 2 * NV + 2 + 2 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 256;
  static constexpr uint32_t kPCol = 384;
};
static_assert(ChunkCfg<128>::kSmemBytes <= 227 * 1024, "chunk smem (D=128)");
static_assert(ChunkCfg<64>::kSmemBytes <= 227 * 1024, "chunk smem (D=64)");

template <int D>
__global__ void __launch_bounds__(kChunkThreads, 1)
    chunk_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap) {
  using C = ChunkCfg<D>;
  constexpr int CH = C::CH;
  constexpr int NK = C::NK;
  constexpr int NV = C::NV;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;
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
  const int q0 = it.q0;
  const int ctx = it.ctx;
  const int off = ctx - it.q_len;         // tokens cached before this chunk
  const int n_tiles = it.kv_tiles;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
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
    constexpr int kPagesPerTile = kChunkKeys / kPageSize;
    const int n_pages = (ctx + kPageSize - 1) / kPageSize;
    const int32_t* bt_row = p.block_table + (size_t)it.seq * p.max_pages_per_seq;
    auto load_window = [&](int base) -> int {
      const int lp = base + lane;
      int phys = p.num_pages;  // out of range: the copy fills zeros
      if (lp < n_pages) {
        phys = (lp < p.max_pages_per_seq) ? __ldg(&bt_row[lp]) : -1;
        if (phys < 0 || phys >= p.num_pages) {
          report_error(p.dev_error, HB_DEVERR_INDEX);
          phys = p.num_pages;
        }
      }
      return phys;
    };
    // block-table windows of 32 pages (4 tiles each), one window ahead
    int win_k = load_window(0), win_k_next = load_window(32);
    int win_v = win_k, win_v_next = win_k_next;
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      mbar_arrive_expect_tx(q_full, (uint32_t)(CH * g * tpt * 128));
#pragma unroll
      for (int c = 0; c < CH; ++c)
        tma_load_3d(sQ + c * 16384, &qmap, q_full, c * 64, it.kv_head * g,
                    q0 + it.tok0);
    }
    uint32_t k_issued = 0, k_par = 0, v_issued = 0, v_par = 0;
    bool ok = true;
    auto issue_tile = [&](bool is_v, int j, int win) -> bool {
      const int s = is_v ? j % NV : j % NK;
      const uint32_t ph = (uint32_t)(is_v ? j / NV : j / NK) & 1u;
      const int w = j & 3;
      int phys[kPagesPerTile];
#pragma unroll
      for (int pp = 0; pp < kPagesPerTile; ++pp)
        phys[pp] = __shfl_sync(0xffffffffu, win, w * kPagesPerTile + pp);
      bool good = true;
      if (lane == 0) {
        uint64_t* empty = is_v ? &v_empty[s] : &k_empty[s];
        uint64_t* full = is_v ? &v_full[s] : &k_full[s];
        good = mbar_wait(empty, ph ^ 1u, abort_flag);
        if (good) {
          mbar_arrive_expect_tx(full, (uint32_t)C::kTileBytes);
          uint8_t* dst = (is_v ? sV : sK) + s * C::kTileBytes;
          const CUtensorMap* map = is_v ? &vmap : &kmap;
#pragma unroll
          for (int pp = 0; pp < kPagesPerTile; ++pp)
#pragma unroll
            for (int c = 0; c < CH; ++c)
              tma_load_3d(dst + c * 16384 + pp * 2048, map, full, c * 64,
                          it.kv_head, phys[pp] * kPageSize);
          if (is_v) {
            v_issued |= 1u << s;
            v_par = (v_par & ~(1u << s)) | (ph << s);
          } else {
            k_issued |= 1u << s;
            k_par = (k_par & ~(1u << s)) | (ph << s);
          }
        }
      }
      return __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
    };
    // issue K_j (j < n_tiles) and V_{j-1} (j >= 1): K runs one tile ahead
    for (int j = 0; ok && j <= n_tiles; ++j) {
      if (j < n_tiles) {
        if ((j & 3) == 0 && j > 0) {
          win_k = win_k_next;
          win_k_next = load_window((j + 4) * kPagesPerTile);
        }
        ok = issue_tile(false, j, win_k);
      }
      if (ok && j >= 1) {
        const int jv = j - 1;
        if ((jv & 3) == 0 && jv > 0) {
          win_v = win_v_next;
          win_v_next = load_window((jv + 4) * kPagesPerTile);
        }
        ok = issue_tile(true, jv, win_v);
      }
    }
    if (lane == 0) {
      // copies in flight must land before the CTA exits
      drain_wait(q_full, 0u, abort_flag);
      for (int s = 0; s < NK; ++s)
        if (k_issued & (1u << s)) drain_wait(&k_full[s], (k_par >> s) & 1u, abort_flag);
      for (int s = 0; s < NV; ++s)
        if (v_issued & (1u << s)) drain_wait(&v_full[s], (v_par >> s) & 1u, abort_flag);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(128, kChunkKeys, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      const uint32_t aQ = smem_u32(sQ);
      const uint32_t aK = smem_u32(sK);
      const uint32_t aV = smem_u32(sV);
      bool ok = mbar_wait(q_full, 0u, abort_flag);
      auto issue_pv = [&](int i) -> bool {
        const int pb = i & 1;
        if (!mbar_wait(&p_full[pb], (uint32_t)(i >> 1) & 1u, abort_flag)) return false;
        const int s = i % NV;
        if (!mbar_wait(&v_full[s], (uint32_t)(i / NV) & 1u, abort_flag)) return false;
        tc_fence_after_sync();
        const uint32_t vb = aV + s * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kChunkKeys / 16; ++kk) {
          const uint64_t b = sdesc_sw128(vb + kk * 2048, 16384, 1024);
          tc_mma_bf16_ts(tmem + C::kOCol, tmem + C::kPCol + pb * 64 + kk * 8, b, idesc_pv,
                         (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&v_empty[s]);
        tc_commit(o_full);
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j % NK;
        if (!mbar_wait(&k_full[s], (uint32_t)(j / NK) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int sb = j & 1;
        const uint32_t kb = aK + s * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(aQ + koff, 16, 1024);
          const uint64_t b = sdesc_sw128(kb + koff, 16, 1024);
          tc_mma_bf16(tmem + sb * kChunkKeys, a, b, idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[sb]);
        tc_commit(&k_empty[s]);
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
    float m_run = -INFINITY;   // running maximum, in scaled log2 units
    float l_run = 0.f;
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
      float alpha = 1.f;
      bool resc = false;
      uint32_t pk[kChunkKeys / 2];
      if (valid_row) {
        float mx = -INFINITY;
        if (kbase + kChunkKeys - 1 > min_pos) {
          const int lim = pos - kbase;   // keys 0..lim of this tile are visible
#pragma unroll
          for (int i = 0; i < kChunkKeys; ++i) {
            if (i > lim) sr[i] = __float_as_uint(-INFINITY);
            mx = fmaxf(mx, __uint_as_float(sr[i]));
          }
        } else {
#pragma unroll
          for (int i = 0; i < kChunkKeys; ++i) mx = fmaxf(mx, __uint_as_float(sr[i]));
        }
        const float m_new = fmaxf(m_run, mx * sl2);
        if (m_new > m_run + kRescaleThreshold) {
          alpha = fast_exp2(m_run - m_new);
          m_run = m_new;
          resc = true;
        }
        float lsum = 0.f;
#pragma unroll
        for (int i = 0; i < kChunkKeys / 2; ++i) {
          const float a0 = fast_exp2(fmaf(__uint_as_float(sr[2 * i]), sl2, -m_run));
          const float a1 = fast_exp2(fmaf(__uint_as_float(sr[2 * i + 1]), sl2, -m_run));
          pk[i] = pack_bf16x2(a0, a1);
          lsum += bf16lo_to_f32(pk[i]) + bf16hi_to_f32(pk[i]);
        }
        l_run = l_run * alpha + lsum;
      } else {
#pragma unroll
        for (int i = 0; i < kChunkKeys / 2; ++i) pk[i] = 0u;
      }
      // P_j into TMEM buffer j&1 (its previous reader, PV_{j-2}, completed:
      // this thread saw o_full for it one tile ago)
      tmem_st32(t_lane + C::kPCol + sb * 64, pk);
      tmem_st32(t_lane + C::kPCol + sb * 64 + 32, pk + 32);
      if (j == n_tiles - 1) {
        // keys past the context in the last page were never written: clear
        // their V rows so that P = 0 never multiplies a NaN
        const int s = j % NV;
        const int first_bad = ctx - kbase;
        const int end_bad = min(kChunkKeys, ((ctx + kPageSize - 1) / kPageSize) * kPageSize - kbase);
        if (first_bad < end_bad) {
          if (!mbar_wait(&v_full[s], (uint32_t)(j / NV) & 1u, abort_flag)) { ok = false; break; }
          uint8_t* vt = sV + s * C::kTileBytes;
          const int n_units = (end_bad - first_bad) * CH * 8;
          for (int e = row; e < n_units; e += 128) {
            const int key = first_bad + e / (CH * 8);
            const int rem = e % (CH * 8);
            *reinterpret_cast<uint4*>(vt + (rem >> 3) * 16384 + key * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_async_shared();
        }
      }
      if (j >= 1) {
        // PV_{j-1} must be complete before O is rescaled
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
        }
      }
      tmem_st_wait();
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
            uint4 pk4;
            pk4.x = pack_bf16x2(__uint_as_float(orow[v * 8 + 0]) * inv, __uint_as_float(orow[v * 8 + 1]) * inv);
            pk4.y = pack_bf16x2(__uint_as_float(orow[v * 8 + 2]) * inv, __uint_as_float(orow[v * 8 + 3]) * inv);
            pk4.z = pack_bf16x2(__uint_as_float(orow[v * 8 + 4]) * inv, __uint_as_float(orow[v * 8 + 5]) * inv);
            pk4.w = pack_bf16x2(__uint_as_float(orow[v * 8 + 6]) * inv, __uint_as_float(orow[v * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + q * 32 + v * 8) = pk4;
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
