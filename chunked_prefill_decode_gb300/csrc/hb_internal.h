// hb_internal.h -- plan layout, work items and kernel parameter blocks shared
// by the host side of libhb (api.cu) and its kernels.  Not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#define HB_DEVERR_INDEX 1
#define HB_DEVERR_TIMEOUT 2

#if defined(__CUDACC__)
#define HB_HD __host__ __device__
#else
#define HB_HD
#endif

namespace hb {

constexpr int kPageSize = 16;
constexpr int kChunkRows = 128;        // M of the tensor-core query tile
constexpr int kChunkKeys = 128;        // keys per tensor-core KV tile
constexpr int kDecodeKvhBlock = 8;     // kv heads per decode work item (max)
constexpr int kMaxGroup = 16;          // max q heads per kv head
constexpr uint32_t kPlanMagic = 0x31504248u;  // "HBP1"
constexpr uint32_t kPlanVersion = 4;
constexpr int kMaxChunkSplits = 16;    // key-range pieces of one query tile (max)
// A chunk item whose first query row sees at most this many keys carries its
// softmax weights P as two bf16 terms (chunk_body.cuh, write_p32), and a
// launch holding one runs the general kernel instantiation.
constexpr int kChunkFewKeys = 256;

// One decode work item: a range of logical pages of one decode row, for one
// block of kv heads.  Rows of the same (sequence, kv block) with n_splits > 1
// leave partial softmax states in slots slot .. slot+n_splits-1; the last
// split to finish merges them.
struct DecodeItem {
  int32_t seq;
  int32_t kvh0;         // first kv head of the block
  int32_t page_begin;   // first logical page
  int32_t page_end;     // one past the last logical page
  int32_t split;        // index of this split within its (seq, block)
  int32_t n_splits;
  int32_t slot;         // first partial slot of its (seq, block)
  int32_t merge_id;     // index of the (seq, block) merge counter
  int32_t ctx;          // context_len of the row (copied from the plan input)
  int32_t tok;          // its q / out row (cu_q_len of the sequence)
  int32_t pad0, pad1;
};
static_assert(sizeof(DecodeItem) == 48, "decode item size");

// One tensor-core work item: query tokens tok0 .. tok0+ntok-1 (relative to
// the sequence's first new token) of one kv head, all q heads of its group,
// as two query tiles of tokens_per_tile tokens (the second may be short or
// empty), over key tiles kv_begin .. kv_tiles-1 (kv_tiles covers the later
// tile).  A single-tile item may be one of n_splits > 1 pieces of its tile's
// key range (split-KV): each piece leaves a partial softmax state in slot
// slot + split, and the last piece to finish merges them.
struct ChunkItem {
  int32_t seq;
  int32_t kv_head;
  int32_t tok0;
  int32_t ntok;
  int32_t kv_tiles;     // one past the last 128-key tile visited
  int32_t q0;           // first q row of the sequence (cu_q_len[seq])
  int32_t q_len;
  int32_t ctx;          // context_len of the sequence
  int32_t kv_begin;     // first 128-key tile visited
  int32_t split;        // index of this piece within its tile's key range
  int32_t n_splits;     // 1: the item covers the whole key range
  int32_t slot;         // first partial slot of the tile (n_splits > 1)
  int32_t merge_id;     // the tile's merge counter (n_splits > 1)
  int32_t pad0, pad1, pad2;
};
static_assert(sizeof(ChunkItem) == 64, "chunk item size");

// Host plan = header, then DecodeItem[num_decode_items] (in CTA order), then
// ChunkItem[num_chunk_items], then int32 decode CTA offsets[decode_grid + 1].
// That body is copied verbatim to the start of the device workspace; the
// header records where everything else lives.
struct PlanHeader {
  uint32_t magic;
  uint32_t version;
  int32_t num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, page_size;
  int32_t max_pages_per_seq;
  int32_t num_sms;
  int32_t num_decode_items;
  int32_t num_chunk_items;
  int32_t num_partial_slots;
  int32_t num_merge_counters;
  int32_t decode_grid;
  int32_t decode_kvh_block;
  int32_t chunk_tokens_per_tile;
  int32_t num_chunk_slots;     // partial states of split chunk tiles
  int32_t num_chunk_merges;    // split chunk tiles
  int32_t sliding_window;      // the batch's window (the plan depends on it)
  int32_t num_decode_dynamic;  // claimable decode intervals after the static ones
  int32_t chunk_pairs_only;    // bit 0: chunk items exist and all are unsplit
                               // pairs; bit 1: some item's first row sees at
                               // most kChunkFewKeys keys
  uint64_t ws_decode_offsets;  // device offset of the per-CTA item offsets
  uint64_t items_bytes;     // bytes of the item arrays (host and device)
  uint64_t ws_counters;     // device offsets (bytes from workspace start)
  uint64_t ws_partial_o;
  uint64_t ws_partial_ml;
  uint64_t ws_total;
  uint64_t plan_bytes;
  uint64_t ws_chunk_counters;   // [num_chunk_merges] arrivals per split tile
  uint64_t ws_chunk_o;          // [num_chunk_slots, D, 128] fp32
  uint64_t ws_chunk_ml;         // [num_chunk_slots, 2, 128] fp32: (m in log2 units, l)
  uint64_t pad1;
};
static_assert(sizeof(PlanHeader) == 176, "header size");
static_assert(sizeof(PlanHeader) % 16 == 0, "header alignment");

// Workspace counters: [0] decode dynamic intervals claimed, [1] decode CTAs
// done (the last one resets both for the next launch),
// [2 .. 2+num_merge_counters) per-(sequence, kv block) split arrivals.
constexpr int kCounterWork = 0;
constexpr int kCounterDone = 1;
constexpr int kCounterMerge0 = 2;

struct DecodeParams {
  const DecodeItem* items;      // in interval order
  // [grid + num_dynamic + 1]: interval k holds items [offsets[k], offsets[k+1]);
  // CTA b works through interval b, then claims intervals grid + c for
  // c = counters[kCounterWork]++ while c < num_dynamic
  const int32_t* cta_offsets;
  int32_t num_static;           // static intervals = decode CTAs
  int32_t num_dynamic;
  int32_t num_items;
  int32_t* counters;
  float* part_o;          // [slots, Hq, D]
  float* part_ml;         // [slots, Hq, 2]: (m in log2 units, l)
  const int32_t* cu_q_len;
  const int32_t* context_len;
  const int32_t* block_table;
  int32_t max_pages_per_seq;
  int32_t num_pages;
  const uint16_t* q;
  uint16_t* out;
  int32_t num_q_heads, num_kv_heads, group, kvh_block;
  float scale_log2;       // softmax scale * log2(e)
  int* dev_error;         // device error word
  int32_t window;         // sliding window in tokens, 0 = none
};

struct ChunkParams {
  const ChunkItem* items;
  int32_t num_items;
  const int32_t* cu_q_len;
  const int32_t* context_len;
  const int32_t* block_table;
  int32_t max_pages_per_seq;
  int32_t num_pages;
  uint16_t* out;
  int32_t num_q_heads, num_kv_heads, group, tokens_per_tile;
  float scale_log2;
  int* dev_error;
  int32_t* counters;      // [merges]: arrivals of the pieces of a split tile
  float* part_o;          // [slots, D, 128]: unnormalised O, row fastest
  float* part_ml;         // [slots, 2, 128]: row maximum (log2 units), row sum
  int32_t window;         // sliding window in tokens, 0 = none
  // 1: the batch's new K/V rows are also given as k_new / v_new (the append's
  // inputs, [total_q, Hkv, D]): pages that hold only new tokens are read from
  // there, so the chunk does not wait for the append that writes them
  int32_t has_new;
};

// Linear layer y = x W^T (linear.cu).  epilogue: 0 store, 1 gated (W has
// 2F rows [gate; up], y[0] receives silu(g) * u, F columns), 2 residual
// (y += x W^T).  Output columns are split over up to three destinations:
// y[i] receives seg_cols[i] consecutive columns with row stride seg_cols[i].
struct LinearParams {
  int32_t M, N, K;
  int32_t epilogue;
  int32_t F;
  uint16_t* y[3];
  int32_t seg_cols[3];
  int* dev_error;
  // split-K: each output tile's K range is cut into `split` pieces of
  // `kb_per_piece` 64-wide blocks (the last may be shorter); every piece
  // writes its fp32 partial tile to `partial` ([unit][column][row], unit =
  // piece * tiles + tile) and the last piece of a tile (counter per tile in
  // `tile_counters`, reset by that piece) sums them and runs the epilogue.
  int32_t split;
  int32_t kb_per_piece;
  float* partial;
  int32_t* tile_counters;
};

struct AppendParams {
  const int32_t* cu_q_len;
  const int32_t* context_len;
  const int32_t* block_table;
  int32_t num_seqs, total_q, max_pages_per_seq, num_pages;
  int32_t row_vec16;      // 16-byte vectors per token row (Hkv * D * 2 / 16)
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_cache;
  uint16_t* v_cache;
  int* dev_error;
  // optional: k_new / v_new (and the next kernel's inputs) are copied in on
  // another stream, which then writes ready_value (or later) to *ready_flag;
  // the kernel reads nothing and starts the next kernel only after that
  const uint32_t* ready_flag;
  uint32_t ready_value;
};

}  // namespace hb
