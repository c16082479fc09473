// decode_body.cuh -- attention of decode rows (one new token over a long
// cached context), split over the keys, read through the block table: the
// per-CTA body that the attention kernel (attention.cu) runs for decode CTAs.
//
// "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §GPU / 系统数据路径 ⑤: a decode reads all earlier KV of its
// sequence every step; "In-flight Batching", §LLM 推理的两阶段计算特征: decode is
// memory-bound (every step reads the whole KV cache).  So this kernel is
// built to stream KV pages at HBM speed:
//
//  * persistent and balanced: the host plan lays the decode rows' pages end
//    to end and gives each CTA (at most one per SM) an equal contiguous
//    range of them (optionally only ~90 %, the rest as short intervals that
//    CTAs claim from a counter when their own range is done; the plan
//    leaves this off, it measured slower); every range is cut at row
//    boundaries into work items (a page range of one row and one block of
//    <= 8 kv heads);
//  * one producer warp streams whole pages (all kv heads of the block, K and
//    V) into a ring of shared-memory stages with 4-D TMA copies laid out as
//    [kv head][slot][64 head-dim] rows with the 128-byte swizzle, so the
//    consumer's ldmatrix reads are bank-conflict free; the q row of each item
//    arrives by a bulk copy into a two-slot ring;
//  * eight consumer warps, one per kv head, with warp MMAs taken transposed
//    (S^T = K Q^T, O^T += V^T P^T) so the group's g <= 16 q heads sit on
//    the MMA's N side and each K/V element read from shared memory serves
//    all g heads; a stage is handed back as soon as its K and V are in
//    registers; online softmax in registers with the exp2 form (scale *
//    log2 e folded in);
//  * a row that straddles ranges leaves one partial state (m, l,
//    unnormalised o) per piece in the workspace; the last piece of a
//    (row, kv block) to finish, found with an atomic counter, merges them:
//    m = max m_i, l = sum 2^(m_i - m) l_i, o = sum 2^(m_i - m) o_i / l.
//    Nobody waits on another CTA.
//
// Bytes per decode row: 2 * context * Hkv * D * 2 (K and V read once).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

constexpr int kDecConsumerWarps = 8;   // warps 0-7; warp 8 is the producer
constexpr int kDecMaxStages = 8;
constexpr float kDecRescaleThreshold = 8.0f;   // log2 units
constexpr int kHdrFirst = 1, kHdrLast = 2, kHdrEnd = 4;

struct StageHeader {
  DecodeItem item;
  int32_t lpage;
  int32_t flags;
  int32_t qslot;
  int32_t pad;
};
static_assert(sizeof(StageHeader) == 64, "stage header size");

struct DecodeLayout {
  int32_t n_stages;
  int32_t chunk_bytes;   // one 64-wide head-dim chunk of one page, all heads
  int32_t half_bytes;    // K (or V) part of a stage
  int32_t stage_bytes;
  int32_t qslot_bytes;
  int32_t smem_bytes;    // dynamic shared memory to request (with alignment)
};

inline __host__ DecodeLayout decode_layout(int head_dim, int kvh_block, int group) {
  DecodeLayout L{};
  const int ch = head_dim / 64;
  L.chunk_bytes = kvh_block * kPageSize * 128;
  L.half_bytes = ch * L.chunk_bytes;
  L.stage_bytes = 2 * L.half_bytes;
  L.qslot_bytes = ((kvh_block * group * head_dim * 2) + 1023) / 1024 * 1024;
  const int fixed = 1024 /*align*/ + 2 * L.qslot_bytes +
                    kDecMaxStages * (int)sizeof(StageHeader) +
                    (2 * kDecMaxStages + 4) * 8 + 64;
  const int budget = 227 * 1024;
  int s = (budget - fixed) / L.stage_bytes;
  if (s > kDecMaxStages) s = kDecMaxStages;
  L.n_stages = s;
  L.smem_bytes = fixed + s * L.stage_bytes;
  return L;
}

// Body of one decode CTA (index `cta` among the decode CTAs); `smem` is the
// 1024-byte-aligned dynamic shared memory.  Warps 0-7 consume, warp 8
// produces, any further warps of the block only join the barriers.
template <int D>
__device__ __forceinline__ void decode_cta(const DecodeParams& p, const DecodeLayout& L,
                                           const CUtensorMap& kmap, const CUtensorMap& vmap,
                                           uint8_t* smem, int cta) {
  constexpr int CH = D / 64;

  const int S = L.n_stages;
  uint8_t* stages = smem;
  uint8_t* qbuf = smem + S * L.stage_bytes;
  StageHeader* hdr = reinterpret_cast<StageHeader*>(qbuf + 2 * L.qslot_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(hdr + kDecMaxStages);
  uint64_t* empty = full + kDecMaxStages;
  uint64_t* qfull = empty + kDecMaxStages;
  uint64_t* qempty = qfull + 2;
  int* flags = reinterpret_cast<int*>(qempty + 2);  // [0] abort, [1] merge
  volatile int* abort_flag = flags;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = p.group;
  const int kvhb = p.kvh_block;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfull[i], 1);
      mbar_init(&qempty[i], kDecConsumerWarps);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDecConsumerWarps) {
    // ------------------------------------------------------------ producer
    // This CTA streams its own contiguous range of pages (items
    // cta_offsets[b] .. cta_offsets[b+1], cut at row boundaries).  The whole
    // warp runs the loop: each lane holds one block-table entry of a 32-page
    // window (one coalesced load, fetched a window ahead; the next item's
    // first window is fetched while the current item starts) and lane 0
    // issues the barrier operations and copies.
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    int st = 0;
    uint32_t ph = 0;
    int qslot = 0;
    uint32_t qph[2] = {0u, 0u};
    uint32_t issued_mask = 0, last_par_mask = 0;
    bool dep_done = false;   // griddep_wait done (before the first page with a new token)
    const uint32_t page_tx = 2u * (uint32_t)L.half_bytes;
    const uint32_t qbytes = (uint32_t)(kvhb * g * D * 2);
    // lane l: block-table entry of page base + l of item x, unchecked -- it is
    // checked where it is used, so no instruction waits on the load earlier
    auto window = [&](const DecodeItem& x, int base) -> int {
      const int lp = base + lane;
      if (lp >= x.page_end) return -1;
      return (lp < p.max_pages_per_seq)
                 ? __ldg(&p.block_table[(size_t)x.seq * p.max_pages_per_seq + lp])
                 : -1;
    };
    // Items: the CTA's own static interval, then dynamic intervals claimed
    // from the shared counter (lane 0 claims, the warp learns the result by
    // shuffle).  The item after the current one is found (and its first
    // block-table window fetched) while the current one streams.
    auto claim = [&](int& ni, int& ne) -> bool {
      int c = 0x7fffffff;
      if (lane == 0 && p.num_dynamic > 0) c = atomicAdd(&p.counters[kCounterWork], 1);
      c = __shfl_sync(0xffffffffu, c, 0);
      if (c >= p.num_dynamic) return false;
      ni = p.cta_offsets[p.num_static + c];
      ne = p.cta_offsets[p.num_static + c + 1];
      return true;
    };
    auto next_item = [&](int i, int e, int& ni, int& ne) -> bool {
      if (i + 1 < e) {
        ni = i + 1;
        ne = e;
        return true;
      }
      while (claim(ni, ne))
        if (ni < ne) return true;
      return false;
    };
    int cur_i = p.cta_offsets[cta], cur_e = p.cta_offsets[cta + 1];
    bool have = cur_i < cur_e || next_item(cur_i, cur_i, cur_i, cur_e);
    bool ok = true;
    DecodeItem it{}, nxt{};
    int win = 0, win_next = 0, nxt_win = 0;
    if (have) {
      it = p.items[cur_i];
      win = window(it, it.page_begin);
      win_next = window(it, it.page_begin + 32);
    }
    while (ok && have) {
      int ni = 0, ne = 0;
      bool has_next = false;
      if (lane == 0) {
        ok = mbar_wait(&qempty[qslot], qph[qslot] ^ 1u, abort_flag);
        if (ok) {
          mbar_arrive_expect_tx(&qfull[qslot], qbytes);
          bulk_load(qbuf + qslot * L.qslot_bytes,
                    p.q + ((size_t)it.tok * p.num_q_heads + (size_t)it.kvh0 * g) * D,
                    qbytes, &qfull[qslot]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      qph[qslot] ^= 1u;
      for (int lp = it.page_begin; ok && lp < it.page_end; ++lp) {
        const int k = (lp - it.page_begin) & 31;
        if (k == 0 && lp != it.page_begin) {
          win = win_next;
          win_next = window(it, lp + 32);
        }
        int phys = __shfl_sync(0xffffffffu, win, k);
        if (phys < 0 || phys >= p.num_pages) {
          // out of range: reported, and fetched out of bounds (zeros)
          if (lane == 0) report_error(p.dev_error, HB_DEVERR_INDEX);
          phys = p.num_pages;
        }
        if (lane == 0) {
          ok = mbar_wait(&empty[st], ph ^ 1u, abort_flag);
          if (ok) {
            StageHeader& h = hdr[st];
            h.item = it;
            h.lpage = lp;
            h.flags = (lp == it.page_begin ? kHdrFirst : 0) |
                      (lp == it.page_end - 1 ? kHdrLast : 0);
            h.qslot = qslot;
            // a decode row's new token (position ctx - 1, written by the
            // append before this launch) is on its last page
            if (!dep_done && lp >= (it.ctx - 1) / kPageSize) {
              griddep_wait();
              fence_proxy_async_global();
              dep_done = true;
            }
            mbar_arrive_expect_tx(&full[st], page_tx);
            uint8_t* kd = stages + st * L.stage_bytes;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
              tma_load_4d(kd + c * L.chunk_bytes, &kmap, &full[st], c * 64, 0,
                          it.kvh0, phys);
              tma_load_4d(kd + L.half_bytes + c * L.chunk_bytes, &vmap, &full[st],
                          c * 64, 0, it.kvh0, phys);
            }
            issued_mask |= 1u << st;
            last_par_mask = (last_par_mask & ~(1u << st)) | (ph << st);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (++st == S) {
          st = 0;
          ph ^= 1u;
        }
        if (lp == it.page_begin) {
          // with the item's first page in flight: find the next item (a
          // claim of a dynamic interval waits on its atomic) and start its
          // first block-table window
          has_next = next_item(cur_i, cur_e, ni, ne);
          if (has_next) {
            nxt = p.items[ni];
            nxt_win = window(nxt, nxt.page_begin);
          }
        }
      }
      qslot ^= 1;
      if (!has_next) break;
      cur_i = ni;
      cur_e = ne;
      it = nxt;
      win = nxt_win;
      win_next = window(it, it.page_begin + 32);
    }
    if (lane == 0) {
      if (ok && mbar_wait(&empty[st], ph ^ 1u, abort_flag)) {
        hdr[st].flags = kHdrEnd;
        issued_mask &= ~(1u << st);  // its earlier copy was consumed
        mbar_arrive(&full[st]);
      }
      for (int s2 = 0; s2 < S; ++s2)
        if (issued_mask & (1u << s2))
          drain_wait(&full[s2], (last_par_mask >> s2) & 1u, abort_flag);
      if (p.num_dynamic > 0) {
        // this CTA claims no more intervals; the last decode CTA to get here
        // resets both counters for the next launch
        __threadfence();
        if (atomicAdd(&p.counters[kCounterDone], 1) == p.num_static - 1) {
          p.counters[kCounterWork] = 0;
          p.counters[kCounterDone] = 0;
        }
      }
    }
  } else if (warp < kDecConsumerWarps) {
    // ------------------------------------------------------------ consumers
    // One warp per kv head of the block.  The products are taken transposed,
    // so the g <= 16 q heads of the group sit on the MMA's narrow N side
    // (8 per column tile) instead of padding its 16 rows:
    //   S^T [16 keys x 8 NQ heads]  = K [16 keys x D] Q^T          (A = K)
    //   O^T [D x 8 NQ heads]       += V^T [D x 16 keys] P^T         (A = V^T)
    // which takes D / 8 MMAs per column tile and page instead of D / 4.
    // P^T leaves the S^T accumulator layout (key = lane / 4) and enters the
    // B operand layout (key = 2 (lane % 4) ..): one movmatrix.trans per
    // 8 x 8 quadrant.  The running maximum is raised (and O, l rescaled)
    // only when it grows by more than 2^8; a stale maximum still bounds
    // P <= 2^8, which bf16 and the fp32 sums carry exactly as well.
    auto consume = [&](auto nq_const) {
      constexpr int NQ = decltype(nq_const)::value;   // 8-head column tiles
      const int w = warp;                  // local kv head of this warp
      const bool active = w < kvhb;
      const int r = lane >> 2;             // accumulator row: key r, r + 8 / dim r, r + 8
      const int c = lane & 3;              // accumulator columns 2c, 2c + 1 (heads)
      const int mi = lane >> 3, r8 = lane & 7;   // ldmatrix: matrix, row
      uint32_t qb[D / 16][NQ][2];          // B operand Q^T (k = head dim, n = head)
      float o[D / 16][NQ][4];              // O^T: dims 16 jj + r (+8), heads 2c, 2c + 1
      float m_run[NQ][2], l_part[NQ][2];   // head 8 nq + 2c + e; l summed over this lane's keys
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq) qb[kk][nq][0] = qb[kk][nq][1] = 0u;
#pragma unroll
      for (int jj = 0; jj < D / 16; ++jj)
#pragma unroll
        for (int nq = 0; nq < NQ; ++nq) o[jj][nq][0] = o[jj][nq][1] = o[jj][nq][2] = o[jj][nq][3] = 0.f;
#pragma unroll
      for (int nq = 0; nq < NQ; ++nq) {
        m_run[nq][0] = m_run[nq][1] = -INFINITY;
        l_part[nq][0] = l_part[nq][1] = 0.f;
      }

      int st = 0;
      uint32_t ph = 0;
      uint32_t qph[2] = {0u, 0u};
      while (true) {
        if (!mbar_wait(&full[st], ph, abort_flag)) break;
        const StageHeader h = hdr[st];
        if (h.flags & kHdrEnd) break;
        if (h.flags & kHdrFirst) {
          if (!mbar_wait(&qfull[h.qslot], qph[h.qslot], abort_flag)) break;
          qph[h.qslot] ^= 1u;
          if (active) {
            const uint16_t* qs =
                reinterpret_cast<const uint16_t*>(qbuf + h.qslot * L.qslot_bytes) +
                (size_t)w * g * D;
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) {
              const int head = nq * 8 + r;
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const int d0 = kk * 16 + c * 2;
                qb[kk][nq][0] = (head < g) ? *reinterpret_cast<const uint32_t*>(qs + head * D + d0) : 0u;
                qb[kk][nq][1] = (head < g) ? *reinterpret_cast<const uint32_t*>(qs + head * D + d0 + 8) : 0u;
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&qempty[h.qslot]);
#pragma unroll
          for (int jj = 0; jj < D / 16; ++jj)
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) o[jj][nq][0] = o[jj][nq][1] = o[jj][nq][2] = o[jj][nq][3] = 0.f;
#pragma unroll
          for (int nq = 0; nq < NQ; ++nq) {
            m_run[nq][0] = m_run[nq][1] = -INFINITY;
            l_part[nq][0] = l_part[nq][1] = 0.f;
          }
        }

        if (active) {
          uint8_t* kst = stages + st * L.stage_bytes;
          uint8_t* vst = kst + L.half_bytes;
          const uint32_t kbase = smem_u32(kst);
          const uint32_t vbase = smem_u32(vst);
          const int valid = min(kPageSize, h.item.ctx - h.lpage * kPageSize);
          // with a sliding window the row sees keys ctx - W .. ctx - 1 only
          const int lo_valid = p.window > 0 ? h.item.ctx - p.window - h.lpage * kPageSize : 0;
          if (valid < kPageSize) {
            // Slots past the context were never written: clear this kv head's
            // V rows there so that P = 0 never meets a NaN in the PV product.
            const int nrow = kPageSize - valid;
            for (int e = lane; e < nrow * CH * 8; e += 32) {
              const int row = valid + e / (CH * 8);
              const int rem = e % (CH * 8);
              const int cc = rem / 8, u = rem % 8;
              uint4* dst = reinterpret_cast<uint4*>(vst + cc * L.chunk_bytes +
                                                    (w * kPageSize + row) * 128 + u * 16);
              *dst = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_async_shared();
            __syncwarp();
          }
          // S^T = K Q^T: every K fragment is loaded before the first MMA;
          // head-dim step kk accumulates into set kk % kQk, so kQk short
          // MMA chains run side by side instead of one long one
          constexpr int kQk = NQ == 1 ? 4 : 2;
          float s[kQk][NQ][4];
#pragma unroll
          for (int x = 0; x < kQk; ++x)
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq) s[x][nq][0] = s[x][nq][1] = s[x][nq][2] = s[x][nq][3] = 0.f;
          {
            // matrix mi: keys 8 (mi & 1) .., head dims 8 (mi >> 1) .. of the step
            const int tokr = ((mi & 1) << 3) + r8;
            const uint32_t rowaddr = kbase + (uint32_t)((w * kPageSize + tokr) * 128);
            uint32_t ka[D / 16][4];
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int unit = ((kk & 3) << 1) + (mi >> 1);
              ldsm_x4(rowaddr + (uint32_t)((kk >> 2) * L.chunk_bytes) +
                          (uint32_t)((unit ^ (tokr & 7)) << 4),
                      ka[kk][0], ka[kk][1], ka[kk][2], ka[kk][3]);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
              for (int nq = 0; nq < NQ; ++nq)
                mma_bf16_16816(s[kk % kQk][nq], ka[kk], qb[kk][nq][0], qb[kk][nq][1]);
          }
          // V^T fragments, loaded while the softmax runs; matrix mi: keys
          // 8 (mi >> 1) .., head dims 8 (mi & 1) .. of the 16-dim block
          uint32_t va[D / 16][4];
          {
            const int tokr = ((mi >> 1) << 3) + r8;
            const uint32_t rowaddr = vbase + (uint32_t)((w * kPageSize + tokr) * 128);
#pragma unroll
            for (int jj = 0; jj < D / 16; ++jj) {
              const int u = 2 * jj + (mi & 1);   // 8-wide head-dim block
              ldsm_x4_trans(rowaddr + (uint32_t)((u >> 3) * L.chunk_bytes) +
                                (uint32_t)((((u & 7) ^ (tokr & 7)) << 4)),
                            va[jj][0], va[jj][1], va[jj][2], va[jj][3]);
            }
          }
          // K and V of the page are in registers: the stage goes back to the
          // producer now, a softmax and a PV ahead of the end of the page
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
          // softmax over the keys of each head column: keys r and r + 8 here,
          // the other 14 in the lanes of the same c.  The column maxima are
          // reduced (xor 4, 8, 16) only when some key of the page exceeds a
          // running maximum by more than the threshold -- after the first
          // pages of an item, almost never.
          const bool ok0 = r < valid && r >= lo_valid;
          const bool ok1 = r + 8 < valid && r + 8 >= lo_valid;
          float x0[NQ][2], x1[NQ][2], alpha[NQ][2];
          bool need = false;
#pragma unroll
          for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float a0 = s[0][nq][e], a1 = s[0][nq][2 + e];
#pragma unroll
              for (int x = 1; x < kQk; ++x) {
                a0 += s[x][nq][e];
                a1 += s[x][nq][2 + e];
              }
              x0[nq][e] = ok0 ? a0 * p.scale_log2 : -INFINITY;
              x1[nq][e] = ok1 ? a1 * p.scale_log2 : -INFINITY;
              need |= fmaxf(x0[nq][e], x1[nq][e]) > m_run[nq][e] + kDecRescaleThreshold;
              alpha[nq][e] = 1.f;
            }
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float mx = fmaxf(x0[nq][e], x1[nq][e]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                if (mx > m_run[nq][e] + kDecRescaleThreshold) {
                  alpha[nq][e] = fast_exp2(m_run[nq][e] - mx);
                  m_run[nq][e] = mx;
                }
              }
#pragma unroll
            for (int jj = 0; jj < D / 16; ++jj)
#pragma unroll
              for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
                for (int x = 0; x < 4; ++x) o[jj][nq][x] *= alpha[nq][x & 1];
          }
          uint32_t pb[NQ][2];
#pragma unroll
          for (int nq = 0; nq < NQ; ++nq) {
            float p0[2], p1[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              // no key seen yet: every x is -inf and so is P's exponent
              const float mu = m_run[nq][e] == -INFINITY ? 0.f : m_run[nq][e];
              p0[e] = fast_exp2(x0[nq][e] - mu);
              p1[e] = fast_exp2(x1[nq][e] - mu);
            }
            const uint32_t lo = pack_bf16x2(p0[0], p0[1]);   // keys r, heads 2c, 2c + 1
            const uint32_t hi = pack_bf16x2(p1[0], p1[1]);   // keys r + 8
            // the row sums use the same bf16-rounded P that feeds the MMA
            l_part[nq][0] = l_part[nq][0] * alpha[nq][0] + (bf16lo_to_f32(lo) + bf16lo_to_f32(hi));
            l_part[nq][1] = l_part[nq][1] * alpha[nq][1] + (bf16hi_to_f32(lo) + bf16hi_to_f32(hi));
            pb[nq][0] = movmatrix_trans(lo);   // B: keys 2c, 2c + 1 of head r
            pb[nq][1] = movmatrix_trans(hi);   // keys 8 + 2c ..
          }
          // O^T += V^T P^T
#pragma unroll
          for (int jj = 0; jj < D / 16; ++jj)
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq)
              mma_bf16_16816(o[jj][nq], va[jj], pb[nq][0], pb[nq][1]);
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
        }

        if (h.flags & kHdrLast) {
          const DecodeItem& it = h.item;
          const int Hq = p.num_q_heads;
          if (active) {
            float l_tot[NQ][2];
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                float t = l_part[nq][e];
                t += __shfl_xor_sync(0xffffffffu, t, 4);
                t += __shfl_xor_sync(0xffffffffu, t, 8);
                t += __shfl_xor_sync(0xffffffffu, t, 16);
                l_tot[nq][e] = t;
              }
            const int head0 = (it.kvh0 + w) * g;
#pragma unroll
            for (int nq = 0; nq < NQ; ++nq)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int head = nq * 8 + 2 * c + e;
                if (head >= g) continue;
                if (it.n_splits == 1) {
                  const float inv = 1.f / l_tot[nq][e];
                  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(
                      p.out + ((size_t)it.tok * Hq + head0 + head) * D + r);
#pragma unroll
                  for (int jj = 0; jj < D / 16; ++jj) {
                    dst[jj * 16] = __float2bfloat16_rn(o[jj][nq][e] * inv);
                    dst[jj * 16 + 8] = __float2bfloat16_rn(o[jj][nq][2 + e] * inv);
                  }
                } else {
                  const size_t slot = (size_t)(it.slot + it.split);
                  float* dst = p.part_o + (slot * Hq + head0 + head) * D + r;
#pragma unroll
                  for (int jj = 0; jj < D / 16; ++jj) {
                    dst[jj * 16] = o[jj][nq][e];
                    dst[jj * 16 + 8] = o[jj][nq][2 + e];
                  }
                  if (r == 0) {
                    float2* ml = reinterpret_cast<float2*>(p.part_ml) + slot * Hq + head0 + head;
                    *ml = make_float2(m_run[nq][e], l_tot[nq][e]);
                  }
                }
              }
          }
          if (it.n_splits > 1) {
            // publish this split's partial state: the CTA barrier orders every
            // consumer's stores before thread 0's device-scope fence + atomic
            named_bar_sync(1, 32 * kDecConsumerWarps);
            if (threadIdx.x == 0) {
              __threadfence();
              const int old = atomicAdd(&p.counters[kCounterMerge0 + it.merge_id], 1);
              __threadfence();  // acquire: the other splits' states are visible
              flags[1] = (old == it.n_splits - 1) ? 1 : 0;
            }
            named_bar_sync(1, 32 * kDecConsumerWarps);
            if (flags[1]) {
              __threadfence();
              // one warp per head of the block; each lane owns D/32 head-dim
              // elements; every split's (m, l) is read once per head
              constexpr int E = D / 32;
              const float2* ml = reinterpret_cast<const float2*>(p.part_ml);
              const int nh = kvhb * g;
              for (int hl = warp; hl < nh; hl += kDecConsumerWarps) {
                const int hh = it.kvh0 * g + hl;
                float mmax = -INFINITY;
                for (int i = 0; i < it.n_splits; ++i)
                  mmax = fmaxf(mmax, __ldcg(&ml[(size_t)(it.slot + i) * Hq + hh]).x);
                float acc[E];
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = 0.f;
                float lsum = 0.f;
#pragma unroll 4
                for (int i = 0; i < it.n_splits; ++i) {
                  const size_t slot = (size_t)(it.slot + i);
                  const float2 st2 = __ldcg(&ml[slot * Hq + hh]);
                  const float wgt = fast_exp2(st2.x - mmax);
                  lsum += wgt * st2.y;
                  const float* po = p.part_o + (slot * Hq + hh) * D + lane * E;
                  if constexpr (E == 4) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(po));
                    acc[0] += wgt * v.x; acc[1] += wgt * v.y;
                    acc[2] += wgt * v.z; acc[3] += wgt * v.w;
                  } else {
                    const float2 v = __ldcg(reinterpret_cast<const float2*>(po));
                    acc[0] += wgt * v.x; acc[1] += wgt * v.y;
                  }
                }
                const float inv = 1.f / lsum;
                uint32_t* dst = reinterpret_cast<uint32_t*>(
                    p.out + ((size_t)h.item.tok * Hq + hh) * D + lane * E);
#pragma unroll
                for (int e = 0; e < E; e += 2) dst[e / 2] = pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
              }
              if (threadIdx.x == 0) p.counters[kCounterMerge0 + it.merge_id] = 0;
            }
          }
        }
        if (++st == S) {
          st = 0;
          ph ^= 1u;
        }
      }
    };
    if (g <= 8) consume(std::integral_constant<int, 1>{});
    else consume(std::integral_constant<int, 2>{});
  }
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) report_error(p.dev_error, HB_DEVERR_TIMEOUT);
}

}  // namespace hb
