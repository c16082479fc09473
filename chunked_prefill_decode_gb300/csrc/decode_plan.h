// decode_plan.h -- host-side partition of decode rows into per-CTA work.
//
// Decode is a pure stream over the rows' KV pages (every page is read once),
// so the work is balanced exactly: the pages of all decode rows (and kv-head
// blocks), laid end to end, are cut into `grid` contiguous ranges of equal
// length, one per CTA of the persistent decode kernel.  A range is cut again
// at row boundaries; each piece is a work item.  A row that lies in one range
// is finished by that CTA; a row that straddles ranges leaves one partial
// softmax state per piece, and the last piece to finish merges them.
//
// The function writes into caller-provided arrays and allocates nothing.
#pragma once

#include <algorithm>
#include <cstdint>

#include "hb_internal.h"

namespace hb {

struct DecodePartition {
  int n_items = 0;
  int n_slots = 0;   // partial-state slots (pieces of straddling rows)
  int n_merge = 0;   // rows (x kv blocks) with more than one piece
  int grid = 0;      // CTAs
  int64_t pages_per_cta = 0;
};

// First logical page a decode row of context ctx reads: 0, or with a sliding
// window of W tokens the page of key ctx - W (the row sees keys ctx-W .. ctx-1).
inline int decode_first_page(int ctx, int window) {
  return window > 0 && ctx > window ? (ctx - window) / kPageSize : 0;
}

// rows: S sequences with q_len[i], ctx[i]; rows with q_len != 1 are skipped.
// Writes items (capacity max_items) in CTA order and cta_offsets[grid + 1].
// Returns false if max_items (or max_grid + 1 offsets) would overflow.
inline bool partition_decode(int S, const int32_t* q_len, const int32_t* ctx, int n_blocks,
                             int kvhb, int num_sms, int min_pages_per_cta,
                             DecodeItem* items, int max_items, int32_t* cta_offsets,
                             int max_grid, DecodePartition* out, int window = 0) {
  DecodePartition r;
  int64_t total = 0;
  int32_t tok = 0;
  for (int i = 0; i < S; ++i)
    if (q_len[i] == 1)
      total += (int64_t)((ctx[i] + kPageSize - 1) / kPageSize - decode_first_page(ctx[i], window)) *
               n_blocks;
  if (total == 0) {
    *out = r;
    return true;
  }
  int64_t grid = std::min<int64_t>(num_sms, (total + min_pages_per_cta - 1) / min_pages_per_cta);
  grid = std::max<int64_t>(1, std::min<int64_t>(grid, max_grid));
  const int64_t per = (total + grid - 1) / grid;
  grid = (total + per - 1) / per;
  r.grid = (int)grid;
  r.pages_per_cta = per;
  for (int64_t b = 0; b <= grid; ++b) cta_offsets[b] = 0;
  int64_t pos = 0;   // start of the current row in the concatenation
  int k = 0;
  for (int i = 0; i < S; ++i) {
    const int32_t this_tok = tok;
    tok += q_len[i];
    if (q_len[i] != 1) continue;
    const int first = decode_first_page(ctx[i], window);
    const int64_t np = (ctx[i] + kPageSize - 1) / kPageSize - first;
    for (int blk = 0; blk < n_blocks; ++blk) {
      const int64_t a = pos, e = pos + np;
      const int64_t first_cta = a / per, last_cta = (e - 1) / per;
      const int pieces = (int)(last_cta - first_cta + 1);
      const int slot = pieces > 1 ? r.n_slots : 0;
      const int merge_id = pieces > 1 ? r.n_merge : 0;
      if (pieces > 1) {
        r.n_slots += pieces;
        r.n_merge += 1;
      }
      for (int64_t c = first_cta; c <= last_cta; ++c) {
        if (k >= max_items) return false;
        DecodeItem& it = items[k++];
        it = DecodeItem{};
        it.seq = i;
        it.kvh0 = blk * kvhb;
        it.page_begin = first + (int32_t)(std::max(a, c * per) - a);
        it.page_end = first + (int32_t)(std::min(e, (c + 1) * per) - a);
        it.split = (int32_t)(c - first_cta);
        it.n_splits = pieces;
        it.slot = slot;
        it.merge_id = merge_id;
        it.ctx = ctx[i];
        it.tok = this_tok;
        cta_offsets[c + 1] = k;
      }
      pos = e;
    }
  }
  // CTAs whose range ended before a later CTA's first item keep the running
  // offset (every CTA has at least one page, so this only fills gaps)
  for (int64_t b = 1; b <= grid; ++b) cta_offsets[b] = std::max(cta_offsets[b], cta_offsets[b - 1]);
  r.n_items = k;
  *out = r;
  return true;
}

}  // namespace hb
