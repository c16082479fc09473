// chunk_body.cuh -- attention of prefill chunks on the tcgen05 tensor cores:
// the per-CTA body that the attention kernel (attention.cu) runs for chunk
// items.
//
// "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §核心机制 3 and §GPU / 系统数据路径 ⑤: chunk i of a prompt attends
// causally to itself and re-reads the KV of chunks 1..i-1 through the page
// table; the computation equals that of the unchunked prefill.  "In-flight
// Batching", §LLM 推理的两阶段计算特征: prefill is compute-bound, so QK^T and PV
// run as the dense contractions they are, on the tensor cores.
//
// A query tile is 128 rows of (token, q head) pairs of one kv head's GQA
// group: tokens_per_tile = 128 / g tokens times the g heads, so a K/V tile in
// shared memory serves the whole group.  One CTA takes one work item: two
// consecutive query tiles, A and B (B may be short or absent), which share
// every 128-key K/V tile; the CTA walks the key tiles 0 .. (last position of
// B) of its sequence, A stopping at its own last position.
//
// Warp roles (384 threads):
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: thread = query
//              row = TMEM lane (warp w owns lanes 32 (w % 4) ..).  Per key
//              tile, pass 1 reads S in 32-column pieces (tcgen05.ld) for the
//              row maximum, with the causal mask only on tiles that cross the
//              diagonal; pass 2 re-reads them, forms p = 2^(s c - m) with one
//              FFMA + EX2 (c = scale * log2 e), rounds to bf16 and writes P
//              into the S columns it has already consumed (tcgen05.st); the
//              row sum uses the same rounded P.  O is rescaled in TMEM only
//              when a row maximum grows by more than 2^8 (a stale maximum
//              stays exact while it bounds P, and P <= 2^8 is safe); epilogue
//              O / l to bf16.
//   warp 8     TMEM owner and MMA issuer (one thread): Q tiles by TMA (3-D map
//              over q, box 64 x g x tokens); then, ping-ponging the two tiles,
//              PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1), ... so that the tensor
//              cores work on one tile while the other tile's softmax runs.
//              S = Q K^T (M 128, N 128, K D, both operands K-major in shared
//              memory); O += P V (M 128, N D, K 128) with P read from TMEM and
//              V read MN-major.  QK_t(j) is issued after PV_t(j-1), and the
//              tensor pipe runs one thread's MMAs in order, so "S_t(j) ready"
//              also means PV_t(j-1) is done: the softmax may then rescale O_t
//              and P_t may live in the S_t columns.
//   warps 9-11 producers: fetch each 128-key K or V tile as its eight
//              16-token pages, one TMA box per page and 64-column head-dim
//              chunk (2 KB), coordinates from the block table; each warp's
//              lane 0 issues the boxes of its pages, so three threads share
//              the per-box issue cost.  Pages past the context are fetched out
//              of range (zeros); the unwritten tail slots of the last page
//              are zeroed in V by the softmax group that reads that tile
//              first.  K runs one tile ahead of V.
// TMEM (512 columns): S_A 0-127, S_B 128-255, O_A 256-(256+D), O_B after it.
#pragma once

#include <cuda_runtime.h>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

constexpr int kMmaWarp = 8;
constexpr int kProducerWarp0 = 9;
constexpr int kProducerWarps = 3;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kSoftmaxRegs = 176;   // per thread, softmax warpgroups (warps 0-7)
constexpr int kLightRegs = 152;     // per thread, MMA + producer warpgroup (8-11)

template <int D>
struct ChunkCfg {
  static constexpr int CH = D / 64;                    // 128-byte K chunks
  static constexpr int kTileBytes = CH * 16384;         // 128 rows x D bf16
  static constexpr int NK = (D == 128) ? 3 : 4;         // K stages
  static constexpr int NV = (D == 128) ? 2 : 4;         // V stages
  static constexpr int kQOff = 0;                       // Q_A, then Q_B
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + NK * kTileBytes;
  static constexpr int kBarOff = kVOff + NV * kTileBytes;
  static constexpr int kNumBars = 1 + 2 * NK + 2 * NV + 2 + 2 + 2 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 256;                // O_A; O_B at kOCol + D
  static constexpr int kUnits = D / 8;                  // 16-byte units per token row
  static constexpr int kRowsPerInstr = 32 / kUnits;     // token rows per warp access
  static constexpr int kInstrPerTile = kChunkKeys / kRowsPerInstr;  // warp accesses per tile
};
static_assert(ChunkCfg<128>::kSmemBytes <= 227 * 1024, "chunk smem (D=128)");
static_assert(ChunkCfg<64>::kSmemBytes <= 227 * 1024, "chunk smem (D=64)");

// Body of one chunk CTA working on item `item`; `smem` is the 1024-byte-
// aligned dynamic shared memory.
template <int D>
__device__ __forceinline__ void chunk_cta(const ChunkParams& p, const CUtensorMap& qmap,
                                          const CUtensorMap& kmap, const CUtensorMap& vmap,
                                          const uint16_t* __restrict__ k_cache,
                                          const uint16_t* __restrict__ v_cache,
                                          uint8_t* smem, int item) {
  using C = ChunkCfg<D>;
  constexpr int CH = C::CH;
  constexpr int NK = C::NK;
  constexpr int NV = C::NV;
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;   // [A, B]
  uint64_t* p_full = s_full + 2;     // [A, B]
  uint64_t* o_done = p_full + 2;     // [A, B]
  uint64_t* mma_done = o_done + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  int* abort_i = reinterpret_cast<int*>(smem + C::kMiscOff + 16);
  volatile int* abort_flag = abort_i;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const ChunkItem it = p.items[item];
  const int g = p.group;
  const int tpt = p.tokens_per_tile;
  const int q0 = it.q0;
  const int ctx = it.ctx;
  const int off = ctx - it.q_len;         // tokens cached before this chunk
  const int ntokA = min(tpt, it.ntok);
  const int ntokB = it.ntok - ntokA;
  const bool hasB = ntokB > 0;
  const int T = it.kv_tiles;              // key tiles of the later tile
  const int TA = (off + it.tok0 + ntokA + kChunkKeys - 1) / kChunkKeys;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], kProducerWarps);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], kProducerWarps);
      mbar_init(&v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(mma_done, 1);
    *abort_i = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_holder;
  // registers move from the MMA / producer warpgroup (warps 8-11) to the two
  // softmax warpgroups, which hold a whole S row: 2 x 128 x 176 + 128 x 152 =
  // 384 x 168, the CTA's launch allocation
  if (warp >= kMmaWarp) setmaxnreg_dec<kLightRegs>();
  else setmaxnreg_inc<kSoftmaxRegs>();

  if (warp >= kProducerWarp0) {
    // ------------------------------------------------------------ producers
    // Each of the three producer warps owns pages pw, pw + 3, pw + 6 of every
    // tile and its lane 0 issues their TMA boxes (one 16-token x 64-column box
    // per page and head-dim chunk, 2 KB each): spreading the issue over three
    // threads hides the per-box issue latency.  Lane l < 8 holds the physical
    // page of page l of a tile; pages past the context are fetched out of
    // range, i.e. as zeros.
    const int pw = warp - kProducerWarp0;
    const int n_pages = (ctx + kPageSize - 1) / kPageSize;
    const int32_t* bt_row = p.block_table + (size_t)it.seq * p.max_pages_per_seq;
    auto page_of = [&](int j) -> int {   // lane l: page l of tile j
      const int lp = j * (kChunkKeys / kPageSize) + (lane & 7);
      int phys = p.num_pages;
      if (lp < n_pages) {
        phys = (lp < p.max_pages_per_seq) ? __ldg(&bt_row[lp]) : -1;
        if (phys < 0 || phys >= p.num_pages) {
          if (lane < 8) report_error(p.dev_error, HB_DEVERR_INDEX);
          phys = p.num_pages;
        }
      }
      return phys;
    };
    constexpr int kMyPages = (kChunkKeys / kPageSize + kProducerWarps - 1) / kProducerWarps;
    int my_pages = 0;
    for (int pp = pw; pp < kChunkKeys / kPageSize; pp += kProducerWarps) ++my_pages;
    uint32_t issued = 0, par = 0;   // bit s: stage s (K in 0..NK-1, V from NK)
    auto tma_tile = [&](const CUtensorMap* map, uint8_t* stage, uint64_t* full, int pages,
                        int bit, uint32_t ph) {
      int phys[kMyPages];
#pragma unroll
      for (int pi = 0; pi < kMyPages; ++pi)
        phys[pi] = __shfl_sync(0xffffffffu, pages, (pw + pi * kProducerWarps) & 7);
      if (lane == 0) {
        mbar_arrive_expect_tx(full, (uint32_t)(my_pages * CH * 2048));
#pragma unroll
        for (int pi = 0; pi < kMyPages; ++pi) {
          const int pp = pw + pi * kProducerWarps;
          if (pp >= kChunkKeys / kPageSize) break;
#pragma unroll
          for (int c = 0; c < CH; ++c)
            tma_load_3d(stage + c * 16384 + pp * 2048, map, full, c * 64, it.kv_head,
                        phys[pi] * kPageSize);
        }
        issued |= 1u << bit;
        par = (par & ~(1u << bit)) | (ph << bit);
      }
    };
    int pg_prev = p.num_pages, pg_cur = page_of(0), pg_next = page_of(1);
    bool ok = true;
    for (int j = 0; ok && j <= T; ++j) {
      if (j < T) {
        const int s = j % NK;
        const uint32_t ph = (uint32_t)(j / NK) & 1u;
        ok = lane != 0 || mbar_wait(&k_empty[s], ph ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        tma_tile(&kmap, sK + s * C::kTileBytes, &k_full[s], pg_cur, s, ph);
      }
      if (j >= 1) {
        const int jv = j - 1;
        const int s = jv % NV;
        const uint32_t ph = (uint32_t)(jv / NV) & 1u;
        ok = lane != 0 || mbar_wait(&v_empty[s], ph ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        tma_tile(&vmap, sV + s * C::kTileBytes, &v_full[s], pg_prev, NK + s, ph);
      }
      pg_prev = pg_cur;
      pg_cur = pg_next;
      pg_next = page_of(j + 2);
    }
    if (lane == 0) {
      // copies in flight must land before the CTA exits
      for (int b = 0; b < NK + NV; ++b)
        if (issued & (1u << b))
          drain_wait(b < NK ? &k_full[b] : &v_full[b - NK], (par >> b) & 1u, abort_flag);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      mbar_arrive_expect_tx(q_full, (uint32_t)(CH * g * tpt * 128 * (hasB ? 2 : 1)));
#pragma unroll
      for (int c = 0; c < CH; ++c)
        tma_load_3d(sQ + c * 16384, &qmap, q_full, c * 64, it.kv_head * g, q0 + it.tok0);
      if (hasB) {
#pragma unroll
        for (int c = 0; c < CH; ++c)
          tma_load_3d(sQ + C::kTileBytes + c * 16384, &qmap, q_full, c * 64, it.kv_head * g,
                      q0 + it.tok0 + tpt);
      }
      const uint32_t idesc_qk = idesc_bf16_f32(128, kChunkKeys, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
      const uint32_t aQ = smem_u32(sQ);
      const uint32_t aK = smem_u32(sK);
      const uint32_t aV = smem_u32(sV);
      auto qk = [&](int t, int j) {
        const uint32_t kb = aK + (j % NK) * C::kTileBytes;
        const uint32_t qb = aQ + t * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          tc_mma_bf16(tmem + t * kChunkKeys, sdesc_sw128(qb + koff, 16, 1024),
                      sdesc_sw128(kb + koff, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[t]);
      };
      auto pv = [&](int t, int j) {
        const uint32_t vb = aV + (j % NV) * C::kTileBytes;
        const uint32_t ocol = C::kOCol + t * D;
#pragma unroll
        for (int kk = 0; kk < kChunkKeys / 16; ++kk)
          tc_mma_bf16_ts(tmem + ocol, tmem + t * kChunkKeys + kk * 8,
                         sdesc_sw128(vb + kk * 2048, 16384, 1024), idesc_pv,
                         (j > 0 || kk > 0) ? 1u : 0u);
      };
      auto wait_k = [&](int j) -> bool {
        if (!mbar_wait(&k_full[j % NK], (uint32_t)(j / NK) & 1u, abort_flag)) return false;
        fence_async_shared();   // gathered K (generic proxy) -> tensor core
        tc_fence_after_sync();
        return true;
      };
      auto wait_v = [&](int j) -> bool {
        if (!mbar_wait(&v_full[j % NV], (uint32_t)(j / NV) & 1u, abort_flag)) return false;
        fence_async_shared();
        tc_fence_after_sync();
        return true;
      };
      bool ok = mbar_wait(q_full, 0u, abort_flag) && wait_k(0);
      if (ok) {
        qk(0, 0);
        if (hasB) qk(1, 0);
        tc_commit(&k_empty[0]);
      }
      for (int j = 0; ok && j < T; ++j) {
        bool k_next_ready = false, v_ready = false;
        if (j < TA) {
          if (!mbar_wait(&p_full[0], (uint32_t)j & 1u, abort_flag) || !wait_v(j)) { ok = false; break; }
          v_ready = true;
          pv(0, j);
          if (j == TA - 1) tc_commit(&o_done[0]);
          if (j + 1 < TA) {
            if (!wait_k(j + 1)) { ok = false; break; }
            k_next_ready = true;
            qk(0, j + 1);
          }
        }
        if (hasB) {
          if (!mbar_wait(&p_full[1], (uint32_t)j & 1u, abort_flag)) { ok = false; break; }
          if (!v_ready && !wait_v(j)) { ok = false; break; }
          tc_fence_after_sync();
          pv(1, j);
          if (j == T - 1) tc_commit(&o_done[1]);
        }
        tc_commit(&v_empty[j % NV]);
        if (j + 1 < T) {
          if (!k_next_ready && !wait_k(j + 1)) { ok = false; break; }
          if (hasB) qk(1, j + 1);
          tc_commit(&k_empty[(j + 1) % NK]);
        }
      }
      // every MMA issued must complete before TMEM is freed
      tc_commit(mma_done);
      drain_wait(mma_done, 0u, abort_flag);
      drain_wait(q_full, 0u, abort_flag);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;               // 0: tile A, 1: tile B
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const int ntok_t = t ? ntokB : ntokA;
    const int T_t = t ? (hasB ? T : 0) : TA;
    const int tok0_t = it.tok0 + t * tpt;
    const int tok_local = row / g;
    const bool valid_row = (row < g * tpt) && (tok_local < ntok_t);
    const int tok_rel = tok0_t + tok_local;
    const int pos = valid_row ? off + tok_rel : ctx - 1;  // absolute position
    const int min_pos = off + tok0_t;
    const float sl2 = p.scale_log2;
    const uint32_t s_col = t_lane + t * kChunkKeys;
    const uint32_t o_col = t_lane + C::kOCol + t * D;
    float m_run = -INFINITY;   // running maximum, in scaled log2 units
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < T_t; ++j) {
      if (!mbar_wait(&s_full[t], (uint32_t)j & 1u, abort_flag)) { ok = false; break; }
      tc_fence_after_sync();
      const int kbase = j * kChunkKeys;
      const bool masked = kbase + kChunkKeys - 1 > min_pos;
      const int lim = pos - kbase;   // keys 0..lim of this tile are visible
      float alpha = 1.f;
      bool resc = false;
      // tcgen05.ld / tcgen05.st are warp-collective: every lane executes each
      // of them; rows that hold no query only change the arithmetic (P = 0).
      // The whole 128-column S row comes in with one wait.
      uint32_t sr[kChunkKeys];
#pragma unroll
      for (int q = 0; q < kChunkKeys / 32; ++q) tmem_ld32(s_col + q * 32, sr + q * 32);
      tmem_ld_wait();
      if (masked) {
#pragma unroll
        for (int i = 0; i < kChunkKeys; ++i)
          if (i > lim) sr[i] = __float_as_uint(-INFINITY);
      }
      float mxp[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mxp[u] = -INFINITY;
#pragma unroll
      for (int i = 0; i < kChunkKeys; i += 16) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          mxp[u] = fmax3(mxp[u], __uint_as_float(sr[i + 2 * u]), __uint_as_float(sr[i + 2 * u + 1]));
      }
      if (valid_row) {
        const float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                               fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
        const float m_new = fmaxf(m_run, mx * sl2);
        if (m_new > m_run + kRescaleThreshold) {
          alpha = fast_exp2(m_run - m_new);
          m_run = m_new;
          resc = true;
        }
      }
      // P = 2^(s c - m) as bf16, written over the S columns (all of S is in
      // registers by now)
      const float neg_m = valid_row ? -m_run : -INFINITY;   // dead rows: P = 0
      const uint64_t c2 = pack_f32x2(sl2, sl2);
      const uint64_t nm2 = pack_f32x2(neg_m, neg_m);
      uint64_t lsum2[2] = {pack_f32x2(0.f, 0.f), pack_f32x2(0.f, 0.f)};
#pragma unroll
      for (int q = 0; q < kChunkKeys / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(sr[q * 32 + 2 * i]),
                                            __uint_as_float(sr[q * 32 + 2 * i + 1])),
                                 c2, nm2), x0, x1);
          pk[i] = pack_bf16x2(fast_exp2(x0), fast_exp2(x1));
          lsum2[i & 1] = add_f32x2(lsum2[i & 1], bf16x2_to_f32x2(pk[i]));
        }
        tmem_st16(s_col + q * 16, pk);
      }
      float lsp[4];
      unpack_f32x2(lsum2[0], lsp[0], lsp[1]);
      unpack_f32x2(lsum2[1], lsp[2], lsp[3]);
      if (valid_row) l_run = l_run * alpha + ((lsp[0] + lsp[1]) + (lsp[2] + lsp[3]));
      if (j == T - 1 && t == (TA == T ? 0 : 1)) {
        // the last page's slots past the context were never written (its TMA
        // box brings them in as they are): clear those V rows before the
        // first PV that reads this tile, so that P = 0 never meets a NaN
        const int kb = j * kChunkKeys;
        const int first_bad = ctx - kb;
        const int end_bad = min(kChunkKeys, ((ctx + kPageSize - 1) / kPageSize) * kPageSize - kb);
        if (first_bad < end_bad) {
          const int s = j % NV;
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
      // O_t is stable here (PV_t(j-1) completed before S_t(j) was ready)
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        const float f = resc ? alpha : 1.f;
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t orow[32];
          tmem_ld32(o_col + q * 32, orow);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) orow[i] = __float_as_uint(__uint_as_float(orow[i]) * f);
          tmem_st32(o_col + q * 32, orow);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&p_full[t]);
    }
    // epilogue: O / l -> bf16
    if (T_t > 0 && ok && mbar_wait(&o_done[t], 0u, abort_flag)) {
      tc_fence_after_sync();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      uint16_t* dst = p.out + ((size_t)(q0 + tok_rel) * p.num_q_heads +
                               (size_t)it.kv_head * g + (row % g)) * D;
#pragma unroll 1
      for (int q = 0; q < D / 32; ++q) {
        uint32_t orow[32];
        tmem_ld32(o_col + q * 32, orow);
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
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) report_error(p.dev_error, HB_DEVERR_TIMEOUT);
}

}  // namespace hb
