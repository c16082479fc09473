// linear.cu -- the linear layers around the attention step, on the tcgen05
// tensor cores.
//
// "Sarathi-Serve：以 chunked-prefills 与 stall-free batching 驯服 LLM 推理的吞吐—
// 延迟权衡", §问题背景 (两阶段天然不对称): every token of a hybrid batch goes
// through the model's linear layers, which take most of the iteration --
// compute-bound for prefill tokens, bound by the weight read for decodes.
//
// y = x W^T with x [M, K] (one row per token) and W [N, K], bf16 in, fp32
// accumulation in tensor memory, bf16 out.  A persistent kernel: one CTA per
// SM walks output tiles of 128 rows x BN columns (m fastest, so CTAs that
// run together share the weight tile through L2; BN = 256); per
// tile, 64-wide slices of K stream through a 4-stage ring of shared memory by
// TMA (128-byte swizzle) and feed tcgen05.mma M128 N(BN) K16; the accumulator
// is double-buffered in TMEM (2 x BN columns), so the epilogue of one tile
// overlaps the main loop of the next.
//
// Warp roles (192 threads): warp 0 TMA producer (one thread), warp 1 TMEM
// owner and MMA issuer (one thread), warps 2-5 epilogue (thread = output
// row = TMEM lane; warp w reads lanes 32 (w % 4) ..).
//
// Epilogues: store (columns split over up to three destinations, e.g. q, k
// and v of a fused QKV projection), gated (W = [W_gate; W_up] with 2F rows:
// per tile two N(BN/2) accumulators, output silu(g) * u), residual
// (y += x W^T).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

constexpr int kLinBM = 128;
constexpr int kLinBK = 64;
constexpr int kLinStages = 4;
constexpr int kLinThreads = 192;
constexpr int kLinABytes = kLinBM * kLinBK * 2;          // 16 KB

// Tile width BN (output columns per tile); the kernel is built for 256.
template <int BN>
struct LinCfg {
  static constexpr int kBBytes = BN * kLinBK * 2;
  static constexpr int kStageBytes = kLinABytes + kBBytes;
  static constexpr int kBarOff = kLinStages * kStageBytes;
  static constexpr int kNumBars = 2 * kLinStages + 4 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;   // + alignment slack
  static constexpr uint32_t kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
};
static_assert(LinCfg<256>::kSmemBytes <= 227 * 1024, "linear smem");

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

template <int BN>
__global__ void __launch_bounds__(kLinThreads, 1)
    linear_kernel(const LinearParams p, const __grid_constant__ CUtensorMap xmap,
                  const __grid_constant__ CUtensorMap wmap) {
  using C = LinCfg<BN>;
  constexpr int kLinBN = BN;
  constexpr int kLinBBytes = C::kBBytes;
  constexpr int kLinStageBytes = C::kStageBytes;
  constexpr int kLinBarOff = C::kBarOff;
  constexpr int kLinMiscOff = C::kMiscOff;
  extern __shared__ uint8_t smem_raw[];
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kLinBarOff);
  uint64_t* full = bars;                       // [stages]
  uint64_t* empty = full + kLinStages;         // [stages]
  uint64_t* acc_full = empty + kLinStages;     // [2]
  uint64_t* acc_empty = acc_full + 2;          // [2]
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kLinMiscOff);
  int* abort_i = reinterpret_cast<int*>(smem + kLinMiscOff + 16);
  volatile int* abort_flag = abort_i;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool gated = p.epilogue == 1;
  const int m_tiles = (p.M + kLinBM - 1) / kLinBM;
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
      mbar_init(&acc_empty[b], 4 * 32);
    }
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
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&xmap);
      tma_prefetch_desc(&wmap);
      uint32_t g = 0;                  // k-blocks issued by this CTA so far
      uint32_t issued = 0, par = 0;    // per stage: issued at all / last phase
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const int t = u % tiles;
        const int m = t % m_tiles, n = t / m_tiles;
        int kb_lo, kb_hi;
        k_range(u, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++g) {
          const int s = (int)(g % kLinStages);
          const uint32_t ph = (g / kLinStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
          uint8_t* st = smem + s * kLinStageBytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kLinStageBytes);
          tma_load_2d(st, &xmap, &full[s], kb * kLinBK, m * kLinBM);
          if (gated) {
            tma_load_2d(st + kLinABytes, &wmap, &full[s], kb * kLinBK, n * (kLinBN / 2));
            tma_load_2d(st + kLinABytes + kLinBBytes / 2, &wmap, &full[s], kb * kLinBK,
                        p.F + n * (kLinBN / 2));
          } else {
            tma_load_2d(st + kLinABytes, &wmap, &full[s], kb * kLinBK, n * kLinBN);
          }
          issued |= 1u << s;
          par = (par & ~(1u << s)) | (ph << s);
        }
      }
      // copies in flight land before the CTA exits
      for (int s = 0; s < kLinStages; ++s)
        if (issued & (1u << s)) drain_wait(&full[s], (par >> s) & 1u, abort_flag);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = gated ? idesc_bf16_f32(kLinBM, kLinBN / 2, false)
                                   : idesc_bf16_f32(kLinBM, kLinBN, false);
      uint32_t g = 0;
      int i = 0;                       // tiles of this CTA so far
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x, ++i) {
        const int buf = i & 1;
        const uint32_t use = (uint32_t)(i >> 1);
        // the epilogue has drained this accumulator (first use: free)
        if (!mbar_wait(&acc_empty[buf], (use & 1u) ^ 1u, abort_flag)) break;
        tc_fence_after_sync();
        const uint32_t acc = tmem + (uint32_t)(buf * kLinBN);
        int kb_lo, kb_hi;
        k_range(u, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++g) {
          const int s = (int)(g % kLinStages);
          if (!mbar_wait(&full[s], (g / kLinStages) & 1u, abort_flag)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a = smem_u32(smem + s * kLinStageBytes);
          const uint32_t b = a + kLinABytes;
#pragma unroll
          for (int kk = 0; kk < kLinBK / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(a + kk * 32, 16, 1024);
            const uint32_t accum = (kb > kb_lo || kk > 0) ? 1u : 0u;
            if (gated) {
              tc_mma_bf16(acc, ad, sdesc_sw128(b + kk * 32, 16, 1024), idesc, accum);
              tc_mma_bf16(acc + kLinBN / 2, ad,
                          sdesc_sw128(b + kLinBBytes / 2 + kk * 32, 16, 1024), idesc, accum);
            } else {
              tc_mma_bf16(acc, ad, sdesc_sw128(b + kk * 32, 16, 1024), idesc, accum);
            }
          }
          tc_commit(&empty[s]);         // the stage is free once these MMAs are done
        }
        if (ok) tc_commit(&acc_full[buf]);
      }
      // every MMA issued must complete before TMEM is freed
      tc_commit(mma_done);
      drain_wait(mma_done, 0u, abort_flag);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int etid = threadIdx.x - 64;          // 0..127 over the epilogue warps
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + kLinMiscOff + 32);
    // y columns of 32 accumulator columns c0 .. c0 + 31 of tile (m, n) for
    // this thread's row; gated: g / u are the gate and up sums
    auto store_plain = [&](int m, int n, int c0, const float* v) {
      const int gm = m * kLinBM + row;
      if (gm >= p.M) return;
      const int col0 = n * kLinBN;
      int seg = 0, seg_start = 0;
      while (seg < 2 && col0 >= seg_start + p.seg_cols[seg]) {
        seg_start += p.seg_cols[seg];
        ++seg;
      }
      uint16_t* dst = p.y[seg] + (size_t)gm * p.seg_cols[seg] + (col0 - seg_start) + c0;
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
      const int gm = m * kLinBM + row;
      if (gm >= p.M) return;
      uint16_t* dst = p.y[0] + (size_t)gm * p.seg_cols[0] + n * (kLinBN / 2) + c0;
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
    int i = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++i) {
      const int t = u % tiles;
      const int m = t % m_tiles, n = t / m_tiles;
      const int buf = i & 1;
      const uint32_t use = (uint32_t)(i >> 1);
      bool got = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], use & 1u, abort_flag));
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
        tc_fence_before_sync();
        mbar_arrive(&acc_empty[buf]);
        continue;
      }
      // split-K: publish this piece's fp32 tile, release the accumulator
      float* part = p.partial + (size_t)u * kLinBN * kLinBM + row;
#pragma unroll 1
      for (int c = 0; c < kLinBN / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(acc + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) part[(size_t)(c * 32 + e) * kLinBM] = __uint_as_float(r[e]);
      }
      tc_fence_before_sync();
      mbar_arrive(&acc_empty[buf]);
      __threadfence();
      // the last piece of the tile to get here sums all pieces (the 128
      // epilogue threads all reach these barriers)
      named_bar_sync(2, 128);
      if (etid == 0) {
        __threadfence();
        const int old = atomicAdd(&p.tile_counters[t], 1);
        __threadfence();
        *last_flag = (old == p.split - 1) ? 1 : 0;
      }
      named_bar_sync(2, 128);
      if (*last_flag) {
        __threadfence();
        const float* src0 = p.partial + (size_t)t * kLinBN * kLinBM + row;   // piece 0
        const size_t piece_stride = (size_t)tiles * kLinBN * kLinBM;
        auto sum_cols = [&](int c0, float* v) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
          for (int pc = 0; pc < p.split; ++pc) {
            const float* src = src0 + pc * piece_stride + (size_t)c0 * kLinBM;
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] += __ldcg(src + (size_t)e * kLinBM);
          }
        };
        if (gated) {
#pragma unroll 1
          for (int c = 0; c < kLinBN / 2 / 32; ++c) {
            float gv[32], uv[32];
            sum_cols(c * 32, gv);
            sum_cols(kLinBN / 2 + c * 32, uv);
            store_gated(m, n, c * 32, gv, uv);
          }
        } else {
#pragma unroll 1
          for (int c = 0; c < kLinBN / 32; ++c) {
            float v[32];
            sum_cols(c * 32, v);
            store_plain(m, n, c * 32, v);
          }
        }
        if (etid == 0) p.tile_counters[t] = 0;   // ready for the next launch
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

// Tile width for a problem.  Measured on GB300 (Mistral-7B projections at
// 512 tokens): 256-column tiles beat 128- and 64-column ones even when they
// leave SMs idle -- a narrower MMA re-reads its 16 KB activation tile for
// fewer output columns and becomes bound by shared memory -- so 256 is used.
int linear_tile_n(int M, int N, int epilogue, int num_sms) {
  (void)M;
  (void)N;
  (void)epilogue;
  (void)num_sms;
  return 256;
}

// Split-K for few tiles: when the 128 x 256 tiles cannot fill half the SMs,
// each tile's K range is cut into up to 16 pieces of at least four 64-wide
// blocks, so that tiles x pieces ~ SMs.  Returns the pieces (1: no split)
// and the K blocks per piece.
int linear_split(int M, int N, int K, int epilogue, int num_sms, int* kb_per_piece) {
  const int m_tiles = (M + kLinBM - 1) / kLinBM;
  const int n_tiles = epilogue == 1 ? (N / 2) / 128 : N / 256;
  const long long tiles = (long long)m_tiles * n_tiles;
  const int k_blocks = K / kLinBK;
  *kb_per_piece = k_blocks;
  if (tiles == 0 || 2 * tiles > num_sms) return 1;
  int s = (int)std::min<long long>(16, std::min<long long>(num_sms / tiles, k_blocks / 4));
  if (s < 2) return 1;
  const int kbp = (k_blocks + s - 1) / s;
  *kb_per_piece = kbp;
  return (k_blocks + kbp - 1) / kbp;
}

// Workspace of the split-K path: a fixed region of kLinCounterBytes for the
// per-tile counters at the start (the same place for every problem, so that
// a workspace shared by calls of different shapes keeps zeroed counters --
// split-K runs with at most num_sms / 2 tiles), then the fp32 partial tiles.
constexpr size_t kLinCounterBytes = 4096;

size_t linear_workspace_bytes(int M, int N, int K, int epilogue, int num_sms) {
  int kbp = 0;
  const int split = linear_split(M, N, K, epilogue, num_sms, &kbp);
  if (split == 1) return 0;
  const long long tiles = (long long)((M + kLinBM - 1) / kLinBM) * (N / 256);   // gated: F / 128
  if (tiles * 4 > (long long)kLinCounterBytes) return 0;
  return kLinCounterBytes + (size_t)split * tiles * 256 * kLinBM * 4;
}

size_t linear_counter_bytes() { return kLinCounterBytes; }

template <int BN>
static cudaError_t launch_bn(const LinearParams& p, const CUtensorMap& xmap,
                             const CUtensorMap& wmap, int num_sms, cudaStream_t stream) {
  const int m_tiles = (p.M + kLinBM - 1) / kLinBM;
  const int n_tiles = p.epilogue == 1 ? p.F / (BN / 2) : p.N / BN;
  const int units = m_tiles * n_tiles * p.split;
  if (units == 0) return cudaSuccess;
  const int grid = units < num_sms ? units : num_sms;
  cudaError_t e = cudaFuncSetAttribute(linear_kernel<BN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       LinCfg<BN>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_serialized(linear_kernel<BN>, grid, kLinThreads, LinCfg<BN>::kSmemBytes, stream, p,
                           xmap, wmap);
}

// Persistent launch: one CTA per SM (at most one per tile).  `bn` is the
// tile width the weight map's box was made for (linear_tile_n).
cudaError_t launch_linear(const LinearParams& p, const CUtensorMap& xmap, const CUtensorMap& wmap,
                          int bn, int num_sms, cudaStream_t stream) {
  if (bn != 256) return cudaErrorInvalidValue;
  return launch_bn<256>(p, xmap, wmap, num_sms, stream);
}

}  // namespace hb
