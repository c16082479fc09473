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
// shared memory serves the whole group.  One CTA takes one work item over key
// tiles kv_begin .. kv_tiles-1 of its sequence, in one of two modes:
//   pair:        two consecutive query tiles, A and B (B may be short), that
//                share every 128-key K/V tile; A stops at its own last
//                position.  Used when there are enough tiles to fill the SMs.
//   interleaved: one query tile; the even key tiles go to half 0 (S_0, O_0,
//                softmax warps 0-3) and the odd ones to half 1 (S_1, O_1,
//                warps 4-7), so one half's softmax overlaps the other half's
//                MMAs; at the end warps 0-3 merge the two partial softmax
//                states.  A tile whose key range is split over several CTAs
//                (split-KV) publishes its state to the workspace instead,
//                and the last piece to finish merges all pieces.
//
// Warp roles (384 threads):
//   warps 0-3, 4-7  softmax of half 0 and half 1 (tile A and tile B in pair
//              mode): thread = query row = TMEM lane (warp w owns lanes
//              32 (w % 4) ..).  Per key tile the whole 128-column S row is
//              read with one wait (tcgen05.ld), masked causally only on tiles
//              that cross the diagonal, reduced to its maximum, and turned
//              into p = 2^(s c - m) with one FFMA + EX2 (c = scale * log2 e),
//              rounded to bf16 and written over the S columns (tcgen05.st);
//              the row sum adds p in fp32.  An item whose first row
//              sees at most 256 keys (a prompt's first tokens, short windows)
//              also writes the bf16 remainder of P into the S columns P
//              leaves free, and its PV runs a second pass over it (P to
//              ~2^-17; write_p32).  O is rescaled in TMEM
//              only when a row maximum grows by more than 2^8 (a stale
//              maximum stays exact while it bounds P, and P <= 2^8 is safe);
//              epilogue O / l to bf16.  These warps hold 176 registers (the
//              MMA / producer warpgroup gives up 16 with setmaxnreg).
//   warp 8     TMEM owner and MMA issuer (one thread): Q tiles by TMA (3-D map
//              over q, box 64 x g x tokens); S = Q K^T (M 128, N 128, K D,
//              both operands K-major in shared memory); O += P V (M 128, N D,
//              K 128) with P read from TMEM and V read MN-major.  A half's
//              next QK is issued after its PV, and the tensor pipe runs one
//              thread's MMAs in order, so "S ready" also means that half's
//              previous PV is done: the softmax may then rescale O and P may
//              live in the S columns.
//   warps 9-11 producers: fetch each 128-key K or V tile as its eight
//              16-token pages, one TMA box per page and 64-column head-dim
//              chunk (2 KB), coordinates from the block table (read a
//              batch of four key tiles ahead); the lanes of the three warps
//              issue the boxes side by side.  Pages past the context are
//              fetched out of range (zeros); the unwritten tail slots of the
//              last page are zeroed in V by the softmax group that reads that
//              tile first.  K runs one tile ahead of V.
// TMEM (512 columns): S_0 0-127, S_1 128-255, O_0 256-(256+D), O_1 after it.
#pragma once

#include <cuda_runtime.h>

#include <climits>
#include <type_traits>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

constexpr int kMmaWarp = 8;
constexpr int kProducerWarp0 = 9;
constexpr int kProducerWarps = 3;
constexpr int kProducerThreads = 32 * kProducerWarps;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// (kChunkFewKeys, hb_internal.h: an item whose first query row sees at most
// that many keys carries P as two bf16 terms, see write_p32: with few keys a
// row's output leans on a few weights, whose bf16 rounding alone, 2^-9
// relative, can move it by more than half a bf16 step of an output near 2.)
constexpr int kSoftmaxRegs = 176;   // per thread, softmax warpgroups (warps 0-7)
constexpr int kLightRegs = 152;     // per thread, MMA + producer warpgroup (8-11)
constexpr int kChunkLaunchRegs = 168;   // per thread at launch: 65536 / 384, rounded down
static_assert(256 * kSoftmaxRegs + 128 * kLightRegs <= 384 * kChunkLaunchRegs,
              "register split exceeds the launch allocation");

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

// The last piece of a split key range merges the pieces' partial states of
// one query row: o = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k over the
// ns pieces (M their largest m), for head-dim columns c0 .. c0 + nc - 1, and
// stores the row (if it holds a query) as bf16 at out_row.  o0 / ml0 point at
// this row in the first piece's slot of part_o ([slot][D][128 rows]) and
// part_ml ([slot][2][128 rows]).  A piece that saw no key of the row has
// m = -inf and weight 0 (its O is not read).  The partial states were
// written by other CTAs: read through L2.  Each piece's block of BW columns
// is loaded in one round (BW loads in flight per thread), so the merge costs
// about one L2 round trip per piece and block.
template <int D, int BW>
__device__ __forceinline__ void merge_pieces(const float* o0, const float* ml0, int ns, int c0,
                                             int nc, bool valid_row, uint16_t* out_row) {
  static_assert(BW % 8 == 0 && BW <= 64, "merge block width");
  float mk[kMaxChunkSplits];
  float mmax = -INFINITY;
#pragma unroll
  for (int k = 0; k < kMaxChunkSplits; ++k) {
    mk[k] = k < ns ? __ldcg(ml0 + (size_t)k * 2 * kChunkRows) : -INFINITY;
    mmax = fmaxf(mmax, mk[k]);
  }
  float lsum = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxChunkSplits; ++k) {
    mk[k] = (mk[k] == -INFINITY) ? 0.f : fast_exp2(mk[k] - mmax);   // now the weight
    if (mk[k] != 0.f) lsum += mk[k] * __ldcg(ml0 + (size_t)k * 2 * kChunkRows + kChunkRows);
  }
  const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
  for (int cb = c0; cb < c0 + nc; cb += BW) {
    float acc[BW];
#pragma unroll
    for (int i = 0; i < BW; ++i) acc[i] = 0.f;
#pragma unroll 1
    for (int k = 0; k < ns; ++k) {
      float wk = 0.f;
#pragma unroll
      for (int x = 0; x < kMaxChunkSplits; ++x)
        if (x == k) wk = mk[x];
      if (wk == 0.f) continue;
      const float* src = o0 + ((size_t)k * D + cb) * kChunkRows;
      float v[BW];
#pragma unroll
      for (int i = 0; i < BW; ++i) v[i] = __ldcg(src + (size_t)i * kChunkRows);
#pragma unroll
      for (int i = 0; i < BW; ++i) acc[i] += wk * v[i];
    }
    if (valid_row) {
#pragma unroll
      for (int i = 0; i < BW; i += 8) {
        uint4 pk4;
        pk4.x = pack_bf16x2(acc[i + 0] * inv, acc[i + 1] * inv);
        pk4.y = pack_bf16x2(acc[i + 2] * inv, acc[i + 3] * inv);
        pk4.z = pack_bf16x2(acc[i + 4] * inv, acc[i + 5] * inv);
        pk4.w = pack_bf16x2(acc[i + 6] * inv, acc[i + 7] * inv);
        *reinterpret_cast<uint4*>(out_row + cb + i) = pk4;
      }
    }
  }
}

// p = 2^(s c - m) for 32 keys of one row (s = sr[0..31]; c2 / nm2 hold c
// and -m twice), written as 16 columns of bf16 pairs at TMEM address `col`.
// With kSplit the remainder p - bf16(p), rounded to bf16, goes to the 16
// columns at col + 32 as well, and the PV runs over both terms, so P enters
// the products to about 2^-17 relative; otherwise P is the bf16 value alone.
// lsum2 receives p in fp32 (two lanes, alternating): what the two passes
// read, to 2^-17; with bf16 P alone it differs from the rounded weights by
// 2^-9 relative, which a row over many keys averages away (the few-key rows
// that it would not are the ones that take the split).
template <bool kSplit>
__device__ __forceinline__ void write_p32(const uint32_t* sr, uint64_t c2, uint64_t nm2,
                                          uint32_t col, uint64_t (&lsum2)[2]) {
  if constexpr (kSplit) {
    // 16 keys at a time, so that the two terms of only 8 pairs are live
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t ph[8], pl[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = 16 * h + 2 * i;
        float x0, x1;
        unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2, nm2),
                     x0, x1);
        const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
        ph[i] = pack_bf16x2(e0, e1);
        pl[i] = pack_bf16x2(e0 - bf16lo_to_f32(ph[i]), e1 - bf16hi_to_f32(ph[i]));
        lsum2[i & 1] = add_f32x2(lsum2[i & 1], pack_f32x2(e0, e1));
      }
      tmem_st8(col + 8 * h, ph);
      tmem_st8(col + 32 + 8 * h, pl);
    }
  } else {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float x0, x1;
      unpack_f32x2(fma_f32x2(pack_f32x2(__uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1])),
                             c2, nm2), x0, x1);
      const float e0 = fast_exp2(x0), e1 = fast_exp2(x1);
      pk[i] = pack_bf16x2(e0, e1);
      lsum2[i & 1] = add_f32x2(lsum2[i & 1], pack_f32x2(e0, e1));
    }
    tmem_st16(col, pk);
  }
}

// Body of one chunk CTA working on item `item`; `smem` is the 1024-byte-
// aligned dynamic shared memory.  kPairs: the launch holds only unsplit
// pairs of query tiles (the plan says so), and the single-tile and split
// paths are left out of this instantiation.  kFew: items whose first row sees
// at most kChunkFewKeys keys may occur (their P is written in two terms; the
// plan says so).
template <int D, bool kPairs, bool kFew>
__device__ __forceinline__ void chunk_cta(const ChunkParams& p, const CUtensorMap& qmap,
                                          const CUtensorMap& kmap, const CUtensorMap& vmap,
                                          const CUtensorMap& knewmap, const CUtensorMap& vnewmap,
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
  // key tiles jb .. T-1 of this item; tile A ends at TA.  Stage and phase
  // counters below run over r = j - jb.
  const int jb = it.kv_begin;
  const int T = it.kv_tiles;
  const int TA = min(T, (off + it.tok0 + ntokA + kChunkKeys - 1) / kChunkKeys);
  const int n_all = T - jb;
  const int nA = TA - jb;
  // one query tile: the two softmax groups take alternate key tiles of it
  // (even: S_0/O_0, odd: S_1/O_1) and merge their states at the end
  const bool inter = !kPairs && !hasB;
  // the item's first row sees the fewest keys (P in two terms, write_p32;
  // kFew: the launch may hold such items, which the plan says)
  const bool few = kFew && (p.window > 0 ? min(p.window, off + it.tok0 + 1)
                                         : off + it.tok0 + 1) <= kChunkFewKeys;

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
      mbar_init(&p_full[t], 4);   // softmax warps per S tile (one arrival each)
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
    // tile; its lanes issue their TMA boxes side by side, one box each (a
    // 16-token x 64-column box per page and head-dim chunk, 2 KB).
    const int pw = warp - kProducerWarp0;
    const int n_pages = (ctx + kPageSize - 1) / kPageSize;
    const int32_t* bt_row = p.block_table + (size_t)it.seq * p.max_pages_per_seq;
    constexpr int kPagesPerTile = kChunkKeys / kPageSize;
    constexpr int kTilesPerBatch = 32 / kPagesPerTile;
    // Block-table entries arrive 32 at a time, one batch of key tiles ahead
    // of their use: lane l holds the entry of page l of the batch (raw; it is
    // checked where it is used, so no instruction waits on the load before
    // then).  Pages past the context are marked and fetched out of range,
    // i.e. as zeros.
    constexpr int kPastContext = INT_MIN;
    // with a sliding window, pages that end at or below the item's lowest
    // visible key are never looked up either (their entries may be stale)
    const int lowest_key = p.window > 0 ? off + it.tok0 - p.window + 1 : 0;
    auto load_batch = [&](int b) -> int {
      const int lp = (jb + b * kTilesPerBatch) * kPagesPerTile + lane;
      if (lp >= n_pages || (lp + 1) * kPageSize <= lowest_key) return kPastContext;
      return lp < p.max_pages_per_seq ? __ldg(&bt_row[lp]) : -1;
    };
    auto phys_of = [&](int raw) -> int {
      if (raw == kPastContext) return p.num_pages;
      if ((unsigned)raw >= (unsigned)p.num_pages) {
        report_error(p.dev_error, HB_DEVERR_INDEX);
        return p.num_pages;
      }
      return raw;
    };
    int my_pages = 0;
    for (int pp = pw; pp < kPagesPerTile; pp += kProducerWarps) ++my_pages;
    // lane l < my_pages * CH issues one box: page pw + 3 (l / CH), chunk l % CH
    const int pp_l = pw + (lane / CH) * kProducerWarps;
    const int c_l = lane % CH;
    const bool issuer = lane < my_pages * CH;
    uint32_t issued = 0, par = 0;   // bit s: stage s (K in 0..NK-1, V from NK)
    // The chunk's own tokens (positions off .. ctx-1) are written into their
    // pages by the append before this launch.  With the append's inputs at
    // hand (p.has_new), the pages from the first page boundary at or after
    // off on are read from k_new / v_new instead (token q0 + position - off)
    // and need no wait; what is left for after griddep_wait is the one page
    // that holds position off when off is not page-aligned -- and, without
    // k_new / v_new, every page from off on.
    const int new_from = p.has_new ? (off + kPageSize - 1) / kPageSize * kPageSize : INT_MAX;
    bool dep_done = false;
    auto tma_tile = [&](const CUtensorMap* map, const CUtensorMap* new_map, uint8_t* stage,
                        uint64_t* full, int batch_reg, int jt, int bit, uint32_t ph) {
      const int tpos = (jb + jt) * kChunkKeys;
      const bool needs_append = p.has_new ? (off % kPageSize != 0 && tpos <= off &&
                                             off < tpos + kChunkKeys)
                                          : tpos + kChunkKeys - 1 >= off;
      if (!dep_done && needs_append) {
        griddep_wait();
        fence_proxy_async_global();
        dep_done = true;
      }
      const int raw = __shfl_sync(0xffffffffu, batch_reg,
                                  ((jt % kTilesPerBatch) * kPagesPerTile + (pp_l & 7)) & 31);
      if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)(my_pages * CH * 2048));
      __syncwarp();
      if (issuer) {
        const int page_pos = tpos + pp_l * kPageSize;
        if (page_pos >= new_from && page_pos < ctx)
          tma_load_3d(stage + c_l * 16384 + pp_l * 2048, new_map, full, c_l * 64, it.kv_head,
                      q0 + (page_pos - off));
        else
          tma_load_3d(stage + c_l * 16384 + pp_l * 2048, map, full, c_l * 64, it.kv_head,
                      phys_of(raw) * kPageSize);
      }
      if (lane == 0) {
        issued |= 1u << bit;
        par = (par & ~(1u << bit)) | (ph << bit);
      }
    };
    int bt_prev = kPastContext, bt_cur = load_batch(0), bt_next = load_batch(1);
    bool ok = true;
    for (int j = 0; ok && j <= n_all; ++j) {   // j: tile jb + j
      if (j > 0 && j % kTilesPerBatch == 0) {
        bt_prev = bt_cur;
        bt_cur = bt_next;
        bt_next = load_batch(j / kTilesPerBatch + 1);
      }
      if (j < n_all) {
        const int s = j % NK;
        const uint32_t ph = (uint32_t)(j / NK) & 1u;
        ok = lane != 0 || mbar_wait(&k_empty[s], ph ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        tma_tile(&kmap, &knewmap, sK + s * C::kTileBytes, &k_full[s], bt_cur, j, s, ph);
      }
      if (j >= 1) {
        const int jv = j - 1;
        const int s = jv % NV;
        const uint32_t ph = (uint32_t)(jv / NV) & 1u;
        ok = lane != 0 || mbar_wait(&v_empty[s], ph ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        const int breg = (jv / kTilesPerBatch == j / kTilesPerBatch) ? bt_cur : bt_prev;
        tma_tile(&vmap, &vnewmap, sV + s * C::kTileBytes, &v_full[s], breg, jv, NK + s, ph);
      }
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
      // S_t = Q_qt K(j)^T
      auto qk = [&](int t, int qt, int j) {
        const uint32_t kb = aK + (j % NK) * C::kTileBytes;
        const uint32_t qb = aQ + qt * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          tc_mma_bf16(tmem + t * kChunkKeys, sdesc_sw128(qb + koff, 16, 1024),
                      sdesc_sw128(kb + koff, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[t]);
      };
      // O_t (+)= P_t V(j); `first` starts O_t.  With P in two terms a
      // second pass adds the remainder (S columns 32-63 and 96-127).
      auto pv = [&](int t, int j, bool first) {
        const uint32_t vb = aV + (j % NV) * C::kTileBytes;
        const uint32_t ocol = C::kOCol + t * D;
#pragma unroll
        for (int kk = 0; kk < kChunkKeys / 16; ++kk)
          tc_mma_bf16_ts(tmem + ocol, tmem + t * kChunkKeys + (kk >> 2) * 64 + (kk & 3) * 8,
                         sdesc_sw128(vb + kk * 2048, 16384, 1024), idesc_pv,
                         (!first || kk > 0) ? 1u : 0u);
        if (few) {
#pragma unroll
          for (int kk = 0; kk < kChunkKeys / 16; ++kk)
            tc_mma_bf16_ts(tmem + ocol, tmem + t * kChunkKeys + (kk >> 2) * 64 + 32 + (kk & 3) * 8,
                           sdesc_sw128(vb + kk * 2048, 16384, 1024), idesc_pv, 1u);
        }
      };
      // K and V arrive by TMA (async proxy, made visible by the barrier's
      // transaction count); the V rows the softmax zeroes by generic stores
      // are fenced to the async proxy by their writers before p_full
      auto wait_k = [&](int j) -> bool {
        if (!mbar_wait(&k_full[j % NK], (uint32_t)(j / NK) & 1u, abort_flag)) return false;
        tc_fence_after_sync();
        return true;
      };
      auto wait_v = [&](int j) -> bool {
        if (!mbar_wait(&v_full[j % NV], (uint32_t)(j / NV) & 1u, abort_flag)) return false;
        tc_fence_after_sync();
        return true;
      };
      bool ok = mbar_wait(q_full, 0u, abort_flag) && wait_k(0);
      if (inter) {
        // one query tile, key tiles alternating between S_0/O_0 (even) and
        // S_1/O_1 (odd): QK of tile j + 2 follows PV of tile j on the same
        // half, so each half's softmax overlaps the other half's MMAs
        if (ok) {
          qk(0, 0, 0);
          tc_commit(&k_empty[0]);
        }
        if (ok && n_all > 1) {
          ok = wait_k(1);
          if (ok) {
            qk(1, 0, 1);
            tc_commit(&k_empty[1 % NK]);
          }
        }
        for (int j = 0; ok && j < n_all; ++j) {   // j: tile jb + j, half j & 1
          const int t = j & 1;
          if (!mbar_wait(&p_full[t], (uint32_t)(j >> 1) & 1u, abort_flag) || !wait_v(j)) { ok = false; break; }
          pv(t, j, j < 2);
          if (j + 2 >= n_all) tc_commit(&o_done[t]);
          tc_commit(&v_empty[j % NV]);
          if (j + 2 < n_all) {
            if (!wait_k(j + 2)) { ok = false; break; }
            qk(t, 0, j + 2);
            tc_commit(&k_empty[(j + 2) % NK]);
          }
        }
      } else {
        if (ok) {
          qk(0, 0, 0);
          qk(1, 1, 0);
          tc_commit(&k_empty[0]);
        }
        for (int j = 0; ok && j < n_all; ++j) {   // j: tile jb + j
          bool k_next_ready = false, v_ready = false;
          if (j < nA) {
            if (!mbar_wait(&p_full[0], (uint32_t)j & 1u, abort_flag) || !wait_v(j)) { ok = false; break; }
            v_ready = true;
            pv(0, j, j == 0);
            if (j == nA - 1) tc_commit(&o_done[0]);
            if (j + 1 < nA) {
              if (!wait_k(j + 1)) { ok = false; break; }
              k_next_ready = true;
              qk(0, 0, j + 1);
            }
          }
          if (!mbar_wait(&p_full[1], (uint32_t)j & 1u, abort_flag)) { ok = false; break; }
          if (!v_ready && !wait_v(j)) { ok = false; break; }
          tc_fence_after_sync();
          pv(1, j, j == 0);
          if (j == n_all - 1) tc_commit(&o_done[1]);
          tc_commit(&v_empty[j % NV]);
          if (j + 1 < n_all) {
            if (!k_next_ready && !wait_k(j + 1)) { ok = false; break; }
            qk(1, 1, j + 1);
            tc_commit(&k_empty[(j + 1) % NK]);
          }
        }
      }
      // every MMA issued must complete before TMEM is freed
      tc_commit(mma_done);
      drain_wait(mma_done, 0u, abort_flag);
      drain_wait(q_full, 0u, abort_flag);
    }
  } else if (!inter) {
    // ------------------------------------------------------------ softmax (pair)
    // Warps 4t .. 4t+3 own tile t (A or B): thread = query row = TMEM lane,
    // the whole 128-column S row in registers.  P of keys 0-63 goes to S
    // columns 0-31 and of keys 64-127 to columns 64-95.
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const int n_t = t ? n_all : nA;
    const int tok0_t = it.tok0 + t * tpt;
    const int tok_local = row / g;
    const bool valid_row = (row < g * tpt) && (tok_local < (t ? ntokB : ntokA));
    const int tok_rel = tok0_t + tok_local;
    const int pos = valid_row ? off + tok_rel : ctx - 1;   // absolute position
    const int min_pos = off + tok0_t;
    // sliding window: row sees keys pos - W + 1 .. pos; a key tile below the
    // window edge of the tile's last row needs the lower mask
    const int max_pos = off + tok0_t + (t ? ntokB : ntokA) - 1;
    const int win_lo = p.window > 0 ? pos - p.window + 1 : INT_MIN;
    const int tile_lo = p.window > 0 ? max_pos - p.window + 1 : INT_MIN;
    const float sl2 = p.scale_log2;
    const uint32_t s_col = t_lane + t * kChunkKeys;
    const uint32_t o_col = t_lane + C::kOCol + t * D;
    const int zero_t = (TA == T) ? 0 : 1;    // the tile whose PV reads V(T-1) first
    float m_run = -INFINITY;   // running maximum, scaled log2 units
    float l_run = 0.f;
    bool ok = true;
    // the loop once per way of writing P (write_p32), so that the
    // common one keeps its own register allocation
    auto pair_loop = [&](auto split_c) {
      constexpr bool kSplit = decltype(split_c)::value;
      for (int j = 0; j < n_t; ++j) {   // key tile jb + j
        // waits are made warp-uniform: a lane that gave up must not leave its
        // warp's collective TMEM accesses
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t], (uint32_t)j & 1u, abort_flag))) { ok = false; break; }
        tc_fence_after_sync();
        const int kbase = (jb + j) * kChunkKeys;
        const bool masked = kbase + kChunkKeys - 1 > min_pos || kbase < tile_lo;
        const int lim = pos - kbase;   // keys 0..lim of this tile are visible
        const int lo_lim = win_lo == INT_MIN ? INT_MIN : win_lo - kbase;   // .. and lo_lim..
        uint32_t sr[kChunkKeys];
#pragma unroll
        for (int q = 0; q < kChunkKeys / 32; ++q) tmem_ld32(s_col + q * 32, sr + q * 32);
        tmem_ld_wait();
        if (masked) {
#pragma unroll
          for (int i = 0; i < kChunkKeys; ++i)
            if (i > lim || i < lo_lim) sr[i] = __float_as_uint(-INFINITY);
        }
        float mxp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mxp[e] = -INFINITY;
#pragma unroll
        for (int i = 0; i < kChunkKeys; i += 16) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            mxp[e] = fmax3(mxp[e], __uint_as_float(sr[i + 2 * e]), __uint_as_float(sr[i + 2 * e + 1]));
        }
        float alpha = 1.f;
        bool resc = false;
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
        // P = 2^(s c - m) as bf16; dead rows and rows that have seen no key
        // yet get P = 0
        const float neg_m = (valid_row && m_run != -INFINITY) ? -m_run : -INFINITY;
        const uint64_t c2 = pack_f32x2(sl2, sl2);
        const uint64_t nm2 = pack_f32x2(neg_m, neg_m);
        uint64_t lsum2[2] = {pack_f32x2(0.f, 0.f), pack_f32x2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < kChunkKeys / 32; ++q)
          write_p32<kSplit>(sr + q * 32, c2, nm2, s_col + (q >> 1) * 64 + (q & 1) * 16, lsum2);
        float lsp[4];
        unpack_f32x2(lsum2[0], lsp[0], lsp[1]);
        unpack_f32x2(lsum2[1], lsp[2], lsp[3]);
        if (valid_row) l_run = l_run * alpha + ((lsp[0] + lsp[1]) + (lsp[2] + lsp[3]));
        if (jb + j == T - 1 && t == zero_t) {
          // the last page's slots past the context were never written (its TMA
          // box brings them in as they are): clear those V rows before the
          // first PV that reads this tile, so that P = 0 never meets a NaN
          const int first_bad = ctx - kbase;
          const int end_bad = min(kChunkKeys, ((ctx + kPageSize - 1) / kPageSize) * kPageSize - kbase);
          if (first_bad < end_bad) {
            const int s = j % NV;
            if (!__all_sync(0xffffffffu, mbar_wait(&v_full[s], (uint32_t)(j / NV) & 1u, abort_flag))) { ok = false; break; }
            uint8_t* vt = sV + s * C::kTileBytes;
            const int n_units = (end_bad - first_bad) * CH * 8;
            for (int e = row; e < n_units; e += kChunkRows) {
              const int key = first_bad + e / (CH * 8);
              const int rem = e % (CH * 8);
              *reinterpret_cast<uint4*>(vt + (rem >> 3) * 16384 + key * 128 + (rem & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_async_shared();
          }
        }
        // O_t is stable here (PV_t of the previous key tile completed before
        // S_t was ready)
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
        // one arrival per warp: the barrier completes after 4 (pair) or 8
        // (interleaved) arrivals instead of one per thread
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[t]);
      }
    };
    if (few) pair_loop(std::true_type{});
    else pair_loop(std::false_type{});
    // epilogue.  t_ok: this tile's waits held (a tile with no key tile in
    // this item -- tile A of a split piece past its own last key -- has
    // nothing to wait for); have_o: its O is complete
    const bool t_ok =
        __all_sync(0xffffffffu, ok && (n_t <= 0 || mbar_wait(&o_done[t], 0u, abort_flag)));
    const bool have_o = t_ok && n_t > 0;
    if (have_o) tc_fence_after_sync();
    if (kPairs || it.n_splits == 1) {
      // O / l -> bf16
      if (have_o) {
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
    } else {
      // one piece of a split key range of the pair: each tile publishes its
      // unnormalised O and (m, l) to its own slot (tile A's pieces first,
      // then tile B's; a tile with no key tile here publishes m = -inf), and
      // the last piece to arrive merges every piece of both tiles,
      // o = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k
      const int ns = it.n_splits;
      const size_t tile_slot0 = (size_t)it.slot + (size_t)t * ns;
      const size_t slot = tile_slot0 + it.split;
      float* po = p.part_o + slot * D * kChunkRows + row;
      float* pml = p.part_ml + slot * 2 * kChunkRows + row;
      if (have_o) {
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t orow[32];
          tmem_ld32(o_col + q * 32, orow);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) po[(size_t)(q * 32 + i) * kChunkRows] = __uint_as_float(orow[i]);
        }
        pml[0] = m_run;
        pml[kChunkRows] = l_run;
      } else {
        pml[0] = -INFINITY;
        pml[kChunkRows] = 0.f;
      }
      __threadfence();
      // all 256 softmax threads reach these barriers; a piece whose waits
      // gave up does not arrive (the error word reports it)
      volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 32);
      if (named_bar_and(2, 2 * kChunkRows, t_ok)) {
        if (threadIdx.x == 0) {
          __threadfence();
          const int old = atomicAdd(&p.counters[it.merge_id], 1);
          __threadfence();
          *last_flag = (old == ns - 1) ? 1 : 0;
        }
        named_bar_sync(2, 2 * kChunkRows);
        if (*last_flag) {
          __threadfence();
          const float* o0 = p.part_o + tile_slot0 * D * kChunkRows + row;
          const float* ml0 = p.part_ml + tile_slot0 * 2 * kChunkRows + row;
          merge_pieces<D, 32>(o0, ml0, ns, 0, D, valid_row,
                          p.out + ((size_t)(q0 + tok_rel) * p.num_q_heads +
                                   (size_t)it.kv_head * g + (row % g)) * D);
          if (threadIdx.x == 0) p.counters[it.merge_id] = 0;   // ready for the next launch
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax (interleaved)
    // One query tile; its key tiles alternate between two slots: the even
    // ones go to S_0/O_0 and warps 0-3, the odd ones to S_1/O_1 and warps
    // 4-7, so the two slots' softmaxes run side by side while the tensor
    // cores work on the other slot.  As in pair mode, thread = query row =
    // TMEM lane and one thread holds the whole 128-column S row (one TMEM
    // load wait per key tile); each slot keeps its own running maximum and
    // row sum.  At the end warps w and w + 4 exchange their slots' (m, l)
    // through shared memory and each writes half the head-dim columns of the
    // merged O.  P of keys 0-63 goes to S columns 0-31 and of keys 64-127 to
    // columns 64-95.
    const int t = warp >> 2;                          // slot (and head-dim half at the end)
    const int h = t;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t bar_pair = 4u + (uint32_t)wq;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const float sl2 = p.scale_log2;
    const int o_c0 = h * (D / 2);                     // head-dim columns written at the end
    constexpr int o_nc = D / 2;
    const int tok_local = row / g;
    const bool valid_row = (row < g * tpt) && (tok_local < ntokA);
    const int tok_rel = it.tok0 + tok_local;
    const int pos = valid_row ? off + tok_rel : ctx - 1;   // absolute position
    const int min_pos = off + it.tok0;
    // sliding window: row sees keys pos - W + 1 .. pos
    const int win_lo = p.window > 0 ? pos - p.window + 1 : INT_MIN;
    const int tile_lo = p.window > 0 ? off + it.tok0 + ntokA - p.window : INT_MIN;
    const uint32_t s_col = t_lane + t * kChunkKeys;
    const uint32_t o_col = t_lane + C::kOCol + t * D;
    float m_run = -INFINITY;   // this slot's running maximum, scaled log2 units
    float l_run = 0.f;
    bool ok = true;
    // the loop once per way of writing P (write_p32), so that the
    // common one keeps its own register allocation
    auto slot_loop = [&](auto split_c) {
      constexpr bool kSplit = decltype(split_c)::value;
      for (int j = t; j < n_all; j += 2) {   // key tile jb + j, this slot's u-th
        const uint32_t u = (uint32_t)j >> 1;
        // waits are made warp-uniform: a lane that gave up must not leave its
        // warp's collective TMEM accesses
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t], u & 1u, abort_flag))) { ok = false; break; }
        tc_fence_after_sync();
        const int kbase = (jb + j) * kChunkKeys;
        const bool masked = kbase + kChunkKeys - 1 > min_pos || kbase < tile_lo;
        const int lim = pos - kbase;   // keys 0..lim of this tile are visible
        const int lo_lim = win_lo == INT_MIN ? INT_MIN : win_lo - kbase;   // .. and lo_lim..
        uint32_t sr[kChunkKeys];
#pragma unroll
        for (int q = 0; q < kChunkKeys / 32; ++q) tmem_ld32(s_col + q * 32, sr + q * 32);
        tmem_ld_wait();
        if (masked) {
#pragma unroll
          for (int i = 0; i < kChunkKeys; ++i)
            if (i > lim || i < lo_lim) sr[i] = __float_as_uint(-INFINITY);
        }
        float mxp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mxp[e] = -INFINITY;
#pragma unroll
        for (int i = 0; i < kChunkKeys; i += 16) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            mxp[e] = fmax3(mxp[e], __uint_as_float(sr[i + 2 * e]), __uint_as_float(sr[i + 2 * e + 1]));
        }
        float alpha = 1.f;
        bool resc = false;
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
        // P = 2^(s c - m) as bf16; dead rows and rows that have seen no key
        // yet get P = 0
        const float neg_m = (valid_row && m_run != -INFINITY) ? -m_run : -INFINITY;
        const uint64_t c2 = pack_f32x2(sl2, sl2);
        const uint64_t nm2 = pack_f32x2(neg_m, neg_m);
        uint64_t lsum2[2] = {pack_f32x2(0.f, 0.f), pack_f32x2(0.f, 0.f)};
#pragma unroll
        for (int q = 0; q < kChunkKeys / 32; ++q)
          write_p32<kSplit>(sr + q * 32, c2, nm2, s_col + (q >> 1) * 64 + (q & 1) * 16, lsum2);
        float lsp[4];
        unpack_f32x2(lsum2[0], lsp[0], lsp[1]);
        unpack_f32x2(lsum2[1], lsp[2], lsp[3]);
        if (valid_row) l_run = l_run * alpha + ((lsp[0] + lsp[1]) + (lsp[2] + lsp[3]));
        if (jb + j == T - 1) {
          // the last page's slots past the context were never written (its
          // TMA box brings them in as they are): clear those V rows before
          // the first PV that reads this tile, so that P = 0 never meets a NaN
          const int first_bad = ctx - kbase;
          const int end_bad = min(kChunkKeys, ((ctx + kPageSize - 1) / kPageSize) * kPageSize - kbase);
          if (first_bad < end_bad) {
            const int s = j % NV;
            if (!__all_sync(0xffffffffu, mbar_wait(&v_full[s], (uint32_t)(j / NV) & 1u, abort_flag))) { ok = false; break; }
            uint8_t* vt = sV + s * C::kTileBytes;
            const int n_units = (end_bad - first_bad) * CH * 8;
            for (int e = row; e < n_units; e += kChunkRows) {
              const int key = first_bad + e / (CH * 8);
              const int rem = e % (CH * 8);
              *reinterpret_cast<uint4*>(vt + (rem >> 3) * 16384 + key * 128 + (rem & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_async_shared();
          }
        }
        // O_t is stable here (slot t's previous PV completed before its S was
        // ready)
        if (u > 0 && __any_sync(0xffffffffu, resc)) {
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
        // one arrival per warp: the barrier completes after the slot's 4
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[t]);
      }
    };
    if (few) slot_loop(std::true_type{});
    else slot_loop(std::false_type{});
    // ---- epilogue: every MMA is complete once both slots' last PV is (slot
    // 1 is empty with one key tile)
    bool have_o = ok && mbar_wait(&o_done[0], 0u, abort_flag);
    if (n_all > 1) have_o = have_o && mbar_wait(&o_done[1], 0u, abort_flag);
    tc_fence_after_sync();
    // the slots' (m, l) of every row, through the second Q tile's room
    // (unused with one query tile)
    float* xl = reinterpret_cast<float*>(sQ + C::kTileBytes);
    xl[(t * 2 + 0) * kChunkRows + row] = m_run;
    xl[(t * 2 + 1) * kChunkRows + row] = l_run;
    have_o = named_bar_and(bar_pair, 64, have_o);
    const float m0 = xl[0 * kChunkRows + row], l0 = xl[1 * kChunkRows + row];
    const float m1 = xl[2 * kChunkRows + row], l1 = xl[3 * kChunkRows + row];
    // the two slots merge: O = w0 O_0 + w1 O_1 relative to 2^m_fin, l_fin
    // likewise
    const bool merge_slots = n_all > 1;
    float m_fin = m0, l_fin = l0, w0 = 1.f, w1 = 0.f;
    if (merge_slots) {
      m_fin = fmaxf(m0, m1);
      w0 = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - m_fin);
      w1 = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - m_fin);
      l_fin = w0 * l0 + w1 * l1;
    }
    // 32 head-dim columns c0 .. c0 + 31 of the final O (warp-collective)
    auto load_o = [&](int c0, uint32_t (&o)[32]) {
      tmem_ld32(t_lane + C::kOCol + c0, o);
      if (merge_slots) {
        uint32_t o1[32];
        tmem_ld32(t_lane + C::kOCol + D + c0, o1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          o[i] = __float_as_uint(w0 * __uint_as_float(o[i]) + w1 * __uint_as_float(o1[i]));
      } else {
        tmem_ld_wait();
      }
    };
    if (it.n_splits == 1) {
      // O / l -> bf16, this half's columns
      if (have_o) {
        const float inv = (l_fin > 0.f) ? 1.f / l_fin : 0.f;
        uint16_t* dst = p.out + ((size_t)(q0 + tok_rel) * p.num_q_heads +
                                 (size_t)it.kv_head * g + (row % g)) * D + o_c0;
#pragma unroll 1
        for (int q = 0; q < o_nc / 32; ++q) {
          uint32_t orow[32];
          load_o(o_c0 + q * 32, orow);
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
    } else {
      // one piece of a split key range (an interleaved tile): publish the
      // unnormalised O and (m, l) of every row; the last piece to arrive
      // merges all pieces, o = sum_k 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k
      const size_t slot = (size_t)(it.slot + it.split);
      float* po = p.part_o + slot * D * kChunkRows + row;
      float* pml = p.part_ml + slot * 2 * kChunkRows + row;
      if (have_o) {
#pragma unroll 1
        for (int q = 0; q < o_nc / 32; ++q) {
          uint32_t orow[32];
          load_o(o_c0 + q * 32, orow);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            po[(size_t)(o_c0 + q * 32 + i) * kChunkRows] = __uint_as_float(orow[i]);
        }
        if (h == 0) {
          pml[0] = m_fin;
          pml[kChunkRows] = l_fin;
        }
        __threadfence();
      }
      // all 256 softmax threads reach these barriers; a piece whose waits
      // gave up does not arrive (the error word reports it)
      volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 32);
      if (named_bar_and(2, 2 * kChunkRows, have_o)) {
        if (threadIdx.x == 0) {
          __threadfence();
          const int old = atomicAdd(&p.counters[it.merge_id], 1);
          __threadfence();
          *last_flag = (old == it.n_splits - 1) ? 1 : 0;
        }
        named_bar_sync(2, 2 * kChunkRows);
        if (*last_flag) {
          __threadfence();
          const int ns = it.n_splits;
          const float* o0 = p.part_o + (size_t)it.slot * D * kChunkRows + row;
          const float* ml0 = p.part_ml + (size_t)it.slot * 2 * kChunkRows + row;
          merge_pieces<D, 32>(o0, ml0, ns, o_c0, o_nc, valid_row,
                          p.out + ((size_t)(q0 + tok_rel) * p.num_q_heads +
                                   (size_t)it.kv_head * g + (row % g)) * D);
          if (threadIdx.x == 0) p.counters[it.merge_id] = 0;   // ready for the next launch
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
