// decode_plan.h -- host-side partition of decode rows into per-CTA work.
//
// Decode is a pure stream over the rows' KV pages (every page is read once).
// The pages of all decode rows (and kv-head blocks), laid end to end, are cut
// into intervals: `grid` equal contiguous static ranges, one per CTA of the
// persistent decode kernel, and -- with a dynamic tail -- after them a number
// of short intervals that CTAs claim from a shared counter when they finish
// their static range (SMs stream at slightly different rates, so an equal
// static split alone ends with a ragged tail).  An interval is cut again at
// row boundaries; each piece is a work item.  A row that lies in one interval
// is finished by one CTA; a row that straddles intervals leaves one partial
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
  int n_slots = 0;     // partial-state slots (pieces of straddling rows)
  int n_merge = 0;     // rows (x kv blocks) with more than one piece
  int grid = 0;        // CTAs, one static interval each
  int n_dynamic = 0;   // claimable intervals after the static ones
  int64_t pages_per_cta = 0;
  int64_t pages_per_dynamic = 0;
};

// First logical page a decode row of context ctx reads: 0, or with a sliding
// window of W tokens the page of key ctx - W (the row sees keys ctx-W .. ctx-1).
inline int decode_first_page(int ctx, int window) {
  return window > 0 && ctx > window ? (ctx - window) / kPageSize : 0;
}

// Share of the pages left to the dynamic tail, and its intervals per CTA.
constexpr int kDynamicTailPercent = 10;
constexpr int kDynamicPerCta = 1;

// rows: S sequences with q_len[i], ctx[i]; rows with q_len != 1 are skipped.
// Writes items (capacity max_items) in interval order and the item offsets of
// the intervals, offsets[grid + n_dynamic + 1] (static ranges first).
// Returns false if max_items or max_intervals would overflow.
inline bool partition_decode(int S, const int32_t* q_len, const int32_t* ctx, int n_blocks,
                             int kvhb, int num_sms, int min_pages_per_cta,
                             DecodeItem* items, int max_items, int32_t* offsets,
                             int max_intervals, DecodePartition* out, int window = 0,
                             bool dynamic_tail = false) {
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
  grid = std::max<int64_t>(1, std::min<int64_t>(grid, max_intervals));
  int64_t per, static_end, q = 1, n_dyn = 0;
  if (dynamic_tail && total >= 16 * grid) {
    per = total * (100 - kDynamicTailPercent) / 100 / grid;
    static_end = per * grid;
    const int64_t rest = total - static_end;
    q = std::max<int64_t>(4, (rest + kDynamicPerCta * grid - 1) / (kDynamicPerCta * grid));
    n_dyn = (rest + q - 1) / q;
    if (grid + n_dyn > max_intervals) return false;
  } else {
    per = (total + grid - 1) / grid;
    grid = (total + per - 1) / per;
    static_end = total;
  }
  r.grid = (int)grid;
  r.n_dynamic = (int)n_dyn;
  r.pages_per_cta = per;
  r.pages_per_dynamic = n_dyn ? q : 0;
  const int64_t n_int = grid + n_dyn;
  auto ibegin = [&](int64_t c) { return c < grid ? c * per : static_end + (c - grid) * q; };
  auto iend = [&](int64_t c) {
    return std::min(total, c < grid ? (c + 1) * per : static_end + (c - grid + 1) * q);
  };
  for (int64_t b = 0; b <= n_int; ++b) offsets[b] = 0;
  int64_t pos = 0;   // start of the current row in the concatenation
  int64_t c_pos = 0;  // the interval holding pos (intervals are consecutive and ascending)
  int k = 0;
  for (int i = 0; i < S; ++i) {
    const int32_t this_tok = tok;
    tok += q_len[i];
    if (q_len[i] != 1) continue;
    const int first = decode_first_page(ctx[i], window);
    const int64_t np = (ctx[i] + kPageSize - 1) / kPageSize - first;
    for (int blk = 0; blk < n_blocks; ++blk) {
      const int64_t a = pos, e = pos + np;
      while (iend(c_pos) <= a) ++c_pos;
      int64_t c_last = c_pos;
      while (iend(c_last) < e) ++c_last;
      const int64_t c0 = c_pos, c1 = c_last;
      const int pieces = (int)(c1 - c0 + 1);
      const int slot = pieces > 1 ? r.n_slots : 0;
      const int merge_id = pieces > 1 ? r.n_merge : 0;
      if (pieces > 1) {
        r.n_slots += pieces;
        r.n_merge += 1;
      }
      for (int64_t c = c0; c <= c1; ++c) {
        if (k >= max_items) return false;
        DecodeItem& it = items[k++];
        it = DecodeItem{};
        it.seq = i;
        it.kvh0 = blk * kvhb;
        it.page_begin = first + (int32_t)(std::max(a, ibegin(c)) - a);
        it.page_end = first + (int32_t)(std::min(e, iend(c)) - a);
        it.split = (int32_t)(c - c0);
        it.n_splits = pieces;
        it.slot = slot;
        it.merge_id = merge_id;
        it.ctx = ctx[i];
        it.tok = this_tok;
        offsets[c + 1] = k;
      }
      pos = e;
    }
  }
  // intervals that ended before a later interval's first item keep the
  // running offset (every interval has at least one page, so this only fills
  // gaps)
  for (int64_t b = 1; b <= n_int; ++b) offsets[b] = std::max(offsets[b], offsets[b - 1]);
  r.n_items = k;
  *out = r;
  return true;
}

}  // namespace hb
