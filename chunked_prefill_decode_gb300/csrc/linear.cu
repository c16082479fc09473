// linear.cu -- the linear layers around the attention step, on the tcgen05
// tensor cores.
//
// "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §问题背景 (两阶段天然不对称): every token of a hybrid batch goes
// through the model's linear layers, which take most of the iteration --
// compute-bound for prefill tokens, bound by the weight read for decodes.
//
// y = x W^T with x [M, K] (one row per token) and W [N, K], bf16 in, fp32
// accumulation in tensor memory, bf16 out.  A persistent kernel of CTA pairs
// (clusters of two CTAs on two SMs): each pair walks output tiles of 256 rows
// x 256 columns (m fastest, so pairs that run together share the weight tile
// through L2) and computes each with tcgen05.mma.cta_group::2 M256 N256 K16.
// Each CTA stages its own 128 rows of x and 128 of the tile's 256 weight rows
// -- per 64-wide K block 32 KB by TMA into a 6-stage ring -- and keeps its
// 128 output rows in its own TMEM.  The odd CTA's copies complete on the even
// CTA's barrier (TMA .cta_group::2), which counts both CTAs' bytes: a thread
// relaying each landing with a remote mbarrier arrive (release at cluster
// scope) measured ~1 us per stage on GB300 and held the pair to a third of
// its MMA rate.  Against one CTA per 128 x 256 tile (x 16
// KB + W 32 KB per K block and SM) this moves a third less through shared
// memory per FLOP, which is what bounds an SS MMA at this size (the TMA
// writes and the tensor cores' operand reads share the SM's shared-memory
// bandwidth).  The accumulator is double-buffered in TMEM (2 x 256 columns),
// so the epilogue of one tile overlaps the main loop of the next.
//
// Warp roles (192 threads per CTA): warp 0 TMA producer (one thread); warp 1
// TMEM owner, and in the even CTA (rank 0) the MMA issuer (one thread); warps
// 2-5 epilogue (thread = output row = TMEM lane; warp w reads lanes 32 (w % 4)
// ..).
//
// Epilogues: store (columns split over up to three destinations, e.g. q, k
// and v of a fused QKV projection), gated (W = [W_gate; W_up] with 2F rows:
// the even CTA stages 128 gate rows and the odd CTA the matching 128 up rows,
// so accumulator columns 0-127 hold x W_gate^T and 128-255 x W_up^T; output
// silu(g) * u), residual (y += x W^T).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

constexpr int kLinBM = 128;                               // output rows per CTA
constexpr int kLinPairBM = 2 * kLinBM;                    // output rows per tile (pair)
constexpr int kLinBN = 256;                               // output columns per tile
constexpr int kLinBK = 64;
constexpr int kLinStages = 6;
constexpr int kLinThreads = 192;
constexpr int kLinABytes = kLinBM * kLinBK * 2;          // 16 KB: this CTA's x rows
constexpr int kLinBBytes = (kLinBN / 2) * kLinBK * 2;    // 16 KB: this CTA's W rows
constexpr int kLinStageBytes = kLinABytes + kLinBBytes;
constexpr int kLinBarOff = kLinStages * kLinStageBytes;
constexpr int kLinNumBars = 2 * kLinStages + 2 + 2 + 1;
constexpr int kLinMiscOff = kLinBarOff + kLinNumBars * 8;
constexpr int kLinSmemBytes = kLinMiscOff + 64 + 1024;    // + alignment slack
constexpr uint32_t kLinTmemCols = 2 * kLinBN;
static_assert(kLinSmemBytes <= 227 * 1024, "linear smem");
// epilogue warps of both CTAs release an accumulator, one arrival per warp
constexpr uint32_t kLinAccEmptyArrivals = 2 * 4;

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kLinThreads, 1)
    linear_kernel(const LinearParams p, const __grid_constant__ CUtensorMap xmap,
                  const __grid_constant__ CUtensorMap wmap) {
  extern __shared__ uint8_t smem_raw[];
  griddep_wait();
  griddep_launch_dependents();
  // the same offset in both CTAs: the leader's MMAs address the peer's
  // stages at this CTA's offsets
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kLinBarOff);
  uint64_t* full = bars;                       // [stages] leader: both CTAs' TMA bytes
  uint64_t* empty = full + kLinStages;         // [stages] leader's MMAs done with it
  uint64_t* acc_full = empty + kLinStages;     // [2]
  uint64_t* acc_empty = acc_full + 2;          // [2] leader: both epilogues drained it
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kLinMiscOff);
  int* abort_i = reinterpret_cast<int*>(smem + kLinMiscOff + 16);
  volatile int* abort_flag = abort_i;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();     // 0: leader (issues the MMAs)
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  const bool gated = p.epilogue == 1;
  const int m_tiles = (p.M + kLinPairBM - 1) / kLinPairBM;
  const int n_tiles = gated ? p.F / (kLinBN / 2) : p.N / kLinBN;
  const int tiles = m_tiles * n_tiles;
  const int n_units = tiles * p.split;    // (tile, K piece) pairs
  const int k_blocks = p.K / kLinBK;
  // K blocks of work unit u: [kb_lo, kb_hi)
  auto k_range = [&](int u, int& kb_lo, int& kb_hi) {
    const int piece = u / tiles;
    kb_lo = piece * p.kb_per_piece;
    kb_hi = min(k_blocks, kb_lo + p.kb_per_piece);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLinStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kLinAccEmptyArrivals);
    }
    mbar_init(mma_done, 1);
    *abort_i = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, kLinTmemCols);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before either touches the other's
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&xmap);
      tma_prefetch_desc(&wmap);
      uint32_t g = 0;                  // k-blocks issued by this CTA so far
      bool ok = true;
      for (int u = pair; ok && u < n_units; u += n_pairs) {
        const int t = u % tiles;
        const int m = t % m_tiles, n = t / m_tiles;
        int kb_lo, kb_hi;
        k_range(u, kb_lo, kb_hi);
        // this CTA's 128 rows of x and 128 weight rows of the tile
        const int x_row = m * kLinPairBM + (int)rank * kLinBM;
        const int w_row = gated ? (int)rank * p.F + n * (kLinBN / 2)
                                : n * kLinBN + (int)rank * (kLinBN / 2);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++g) {
          const int s = (int)(g % kLinStages);
          const uint32_t ph = (g / kLinStages) & 1u;
          if (!mbar_wait_cluster(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
          uint8_t* st = smem + s * kLinStageBytes;
          if (rank == 0) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * kLinStageBytes));
            tma_load_2d(st, &xmap, &full[s], kb * kLinBK, x_row);
            tma_load_2d(st + kLinABytes, &wmap, &full[s], kb * kLinBK, w_row);
          } else {
            const uint32_t bar0 = mapa_shared(smem_u32(&full[s]), 0);
            tma_load_2d_to_leader(st, &xmap, bar0, kb * kLinBK, x_row);
            tma_load_2d_to_leader(st + kLinABytes, &wmap, bar0, kb * kLinBK, w_row);
          }
        }
      }
      // before the CTA exits: the leader's releases of every stage
      // (multicast arrivals on this CTA's barriers) have arrived, so the
      // leader's MMAs have read the stage and its copies have landed
      for (int s = 0; s < kLinStages && (uint32_t)s < g; ++s) {
        const uint32_t last = (g - 1 - (uint32_t)s) / kLinStages;   // last round of stage s
        if (rank == 0) drain_wait(&full[s], last & 1u, abort_flag);
        drain_wait_cluster(&empty[s], last & 1u, abort_flag);
      }
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_bf16_f32(kLinPairBM, kLinBN, false);
      uint32_t g = 0;
      int i = 0;                       // tiles of this pair so far
      bool ok = true;
      for (int u = pair; ok && u < n_units; u += n_pairs, ++i) {
        const int buf = i & 1;
        const uint32_t use = (uint32_t)(i >> 1);
        // both CTAs' epilogues have drained this accumulator (first use: free)
        if (!mbar_wait_cluster(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag)) break;
        tc_fence_after_sync();
        const uint32_t acc = tmem + (uint32_t)(buf * kLinBN);
        int kb_lo, kb_hi;
        k_range(u, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++g) {
          const int s = (int)(g % kLinStages);
          const uint32_t ph = (g / kLinStages) & 1u;
          if (!mbar_wait_cluster(&full[s], ph, abort_flag)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a = smem_u32(smem + s * kLinStageBytes);
          const uint32_t b = a + kLinABytes;
#pragma unroll
          for (int kk = 0; kk < kLinBK / 16; ++kk)
            tc_mma_bf16_pair(acc, sdesc_sw128(a + kk * 32, 16, 1024),
                             sdesc_sw128(b + kk * 32, 16, 1024), idesc,
                             (kb > kb_lo || kk > 0) ? 1u : 0u);
          // the stage is free in both CTAs once these MMAs are done
          tc_commit_pair_mc(&empty[s], 0x3);
        }
        if (ok) tc_commit_pair_mc(&acc_full[buf], 0x3);
      }
      // every MMA issued must complete before TMEM is freed
      tc_commit_pair(mma_done);
      drain_wait(mma_done, 0u, abort_flag);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int etid = threadIdx.x - 64;          // 0..127 over the epilogue warps
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t acc_empty0 = mapa_shared(smem_u32(acc_empty), 0);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + kLinMiscOff + 32);
    // y columns of 32 accumulator columns c0 .. c0 + 31 of tile (m, n) for
    // this thread's row; gated: g / u are the gate and up sums
    auto out_row = [&](int m) { return m * kLinPairBM + (int)rank * kLinBM + row; };
    auto store_plain = [&](int m, int n, int c0, const float* v) {
      const int r = out_row(m);
      if (r >= p.M) return;
      const int col0 = n * kLinBN;
      int seg = 0, seg_start = 0;
      while (seg < 2 && col0 >= seg_start + p.seg_cols[seg]) {
        seg_start += p.seg_cols[seg];
        ++seg;
      }
      uint16_t* dst = p.y[seg] + (size_t)r * p.seg_cols[seg] + (col0 - seg_start) + c0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + q * 8);
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = v[q * 8 + e];
        if (p.epilogue == 2) {
          const uint4 old = *d4;
          const uint32_t o[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            f[2 * e] += bf16lo_to_f32(o[e]);
            f[2 * e + 1] += bf16hi_to_f32(o[e]);
          }
        }
        *d4 = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                         pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
      }
    };
    auto store_gated = [&](int m, int n, int c0, const float* gv, const float* uv) {
      const int r = out_row(m);
      if (r >= p.M) return;
      uint16_t* dst = p.y[0] + (size_t)r * p.seg_cols[0] + n * (kLinBN / 2) + c0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = q * 8 + e * 2;
          w4[e] = pack_bf16x2(silu_f(gv[k]) * uv[k], silu_f(gv[k + 1]) * uv[k + 1]);
        }
        *reinterpret_cast<uint4*>(dst + q * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    };
    // this warp is done reading accumulator buf: one arrival on the leader's
    // barrier
    auto release = [&](int buf) {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + (uint32_t)buf * 8u);
    };
    int i = 0;
    for (int u = pair; u < n_units; u += n_pairs, ++i) {
      const int t = u % tiles;
      const int m = t % m_tiles, n = t / m_tiles;
      const int buf = i & 1;
      const uint32_t use = (uint32_t)(i >> 1);
      bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&acc_full[buf], use & 1u, abort_flag));
      // with split-K the four epilogue warps meet at barriers below, so they
      // leave together
      if (p.split > 1) got = named_bar_and(3, 128, got);
      if (!got) break;
      tc_fence_after_sync();
      const uint32_t acc = t_lane + (uint32_t)(buf * kLinBN);
      if (p.split == 1) {
        if (gated) {
#pragma unroll 1
          for (int c = 0; c < kLinBN / 2 / 32; ++c) {
            uint32_t gr[32], ur[32];
            tmem_ld32(acc + c * 32, gr);
            tmem_ld32(acc + kLinBN / 2 + c * 32, ur);
            tmem_ld_wait();
            store_gated(m, n, c * 32, reinterpret_cast<const float*>(gr),
                        reinterpret_cast<const float*>(ur));
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < kLinBN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(acc + c * 32, r);
            tmem_ld_wait();
            store_plain(m, n, c * 32, reinterpret_cast<const float*>(r));
          }
        }
        // this accumulator may be overwritten now
        release(buf);
        continue;
      }
      // split-K: publish this CTA's half of the piece's fp32 tile as 64
      // groups of 4 columns, each group [128 rows][4] (a thread stores and
      // later loads its row's 4 columns as one float4; a warp's accesses to a
      // group are contiguous), release the accumulator
      float4* part = reinterpret_cast<float4*>(p.partial + ((size_t)u * 2 + rank) * kLinBN * kLinBM) + row;
#pragma unroll 1
      for (int c = 0; c < kLinBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(acc + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4)
          __stcg(part + (size_t)(c * 8 + g4) * kLinBM,
                 make_float4(__uint_as_float(r[4 * g4]), __uint_as_float(r[4 * g4 + 1]),
                             __uint_as_float(r[4 * g4 + 2]), __uint_as_float(r[4 * g4 + 3])));
      }
      release(buf);
      __threadfence();
      // the last piece of the tile half to get here sums all pieces (the 128
      // epilogue threads all reach these barriers)
      named_bar_sync(2, 128);
      const int counter = t * 2 + (int)rank;
      if (etid == 0) {
        __threadfence();
        const int old = atomicAdd(&p.tile_counters[counter], 1);
        __threadfence();
        *last_flag = (old == p.split - 1) ? 1 : 0;
      }
      named_bar_sync(2, 128);
      if (*last_flag) {
        __threadfence();
        // four rounds of 16 groups (plain: 64 columns; gated: 32 gate and
        // the matching 32 up columns), two pieces' loads in flight at once:
        // each round costs about one L2 round trip per two pieces
        const float4* src0 =
            reinterpret_cast<const float4*>(p.partial + ((size_t)t * 2 + rank) * kLinBN * kLinBM) + row;
        const size_t piece_stride = (size_t)tiles * 2 * kLinBN * kLinBM / 4;   // float4s
#pragma unroll 1
        for (int rd = 0; rd < 4; ++rd) {
          float v[64];
#pragma unroll
          for (int e = 0; e < 64; ++e) v[e] = 0.f;
#pragma unroll 1
          for (int pc = 0; pc < p.split; pc += 2) {
            const bool two = pc + 1 < p.split;
            float4 a4[16], b4[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int grp = gated ? (i < 8 ? 8 * rd + i : 32 + 8 * rd + (i - 8)) : 16 * rd + i;
              a4[i] = __ldcg(src0 + (size_t)pc * piece_stride + (size_t)grp * kLinBM);
              b4[i] = two ? __ldcg(src0 + (size_t)(pc + 1) * piece_stride + (size_t)grp * kLinBM)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              v[4 * i] += a4[i].x + b4[i].x;
              v[4 * i + 1] += a4[i].y + b4[i].y;
              v[4 * i + 2] += a4[i].z + b4[i].z;
              v[4 * i + 3] += a4[i].w + b4[i].w;
            }
          }
          if (gated) {
            store_gated(m, n, 32 * rd, v, v + 32);
          } else {
            store_plain(m, n, 64 * rd, v);
            store_plain(m, n, 64 * rd + 32, v + 32);
          }
        }
        if (etid == 0) p.tile_counters[counter] = 0;   // ready for the next launch
      }
    }
  }
  if (rank == 1 && threadIdx.x == 0 && *abort_flag) {
    // after an abort the odd CTA cannot see its own copies land (they
    // complete on the leader's barrier): give any in flight time to land
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 20000ull) {}
  }
  // neither CTA leaves while the other may still arrive on its barriers or
  // (the leader's MMAs) read its shared memory and write its TMEM
  tc_fence_before_sync();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kLinTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) report_error(p.dev_error, HB_DEVERR_TIMEOUT);
}

// Split-K for few tiles: when the 256 x 256 tiles cannot fill half the CTA
// pairs, each tile's K range is cut into up to 16 pieces of at least four
// 64-wide blocks, so that tiles x pieces ~ pairs.  Returns the pieces (1: no
// split) and the K blocks per piece.
int linear_split(int M, int N, int K, int epilogue, int num_sms, int* kb_per_piece) {
  const int pairs = num_sms / 2;
  const int m_tiles = (M + kLinPairBM - 1) / kLinPairBM;
  const int n_tiles = epilogue == 1 ? (N / 2) / (kLinBN / 2) : N / kLinBN;
  const long long tiles = (long long)m_tiles * n_tiles;
  const int k_blocks = K / kLinBK;
  *kb_per_piece = k_blocks;
  if (tiles == 0 || 2 * tiles > pairs) return 1;
  int s = (int)std::min<long long>(16, std::min<long long>(pairs / tiles, k_blocks / 4));
  if (s < 2) return 1;
  const int kbp = (k_blocks + s - 1) / s;
  *kb_per_piece = kbp;
  return (k_blocks + kbp - 1) / kbp;
}

// Workspace of the split-K path: a fixed region of kLinCounterBytes for the
// per-tile-half counters at the start (the same place for every problem, so
// that a workspace shared by calls of different shapes keeps zeroed counters
// -- split-K runs with at most num_sms / 4 tiles), then the fp32 partial
// tiles, two 128-row halves per tile and piece.
constexpr size_t kLinCounterBytes = 4096;

size_t linear_workspace_bytes(int M, int N, int K, int epilogue, int num_sms) {
  int kbp = 0;
  const int split = linear_split(M, N, K, epilogue, num_sms, &kbp);
  if (split == 1) return 0;
  const long long tiles = (long long)((M + kLinPairBM - 1) / kLinPairBM) * (N / kLinBN);
  if (tiles * 2 * 4 > (long long)kLinCounterBytes) return 0;
  return kLinCounterBytes + (size_t)split * tiles * 2 * kLinBN * kLinBM * 4;
}

size_t linear_counter_bytes() { return kLinCounterBytes; }

// Rows of the weight tensor map's box: the weight rows one CTA stages.
int linear_w_box_rows() { return kLinBN / 2; }

// Persistent launch: CTA pairs, at most as many as can be resident at once
// (and at most one per tile).
cudaError_t launch_linear(const LinearParams& p, const CUtensorMap& xmap, const CUtensorMap& wmap,
                          int num_sms, cudaStream_t stream) {
  const int m_tiles = (p.M + kLinPairBM - 1) / kLinPairBM;
  const int n_tiles = p.epilogue == 1 ? p.F / (kLinBN / 2) : p.N / kLinBN;
  const int units = m_tiles * n_tiles * p.split;
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kLinSmemBytes);
  if (e != cudaSuccess) return e;
  // resident pairs, found once per SM count
  static std::mutex mu;
  static int cached_sms = -1, max_pairs = 1;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (cached_sms != num_sms) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (num_sms / 2));
      cfg.blockDim = dim3(kLinThreads);
      cfg.dynamicSmemBytes = kLinSmemBytes;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, linear_kernel, &cfg);
      if (e != cudaSuccess) return e;
      max_pairs = std::max(1, std::min(n, num_sms / 2));
      cached_sms = num_sms;
    }
  }
  const int pairs = std::min(units, max_pairs);
  return launch_serialized(linear_kernel, 2 * pairs, kLinThreads, kLinSmemBytes, stream, p, xmap,
                           wmap);
}

}  // namespace hb
