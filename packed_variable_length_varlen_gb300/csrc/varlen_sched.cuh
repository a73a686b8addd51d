// varlen_sched.cuh -- exact persistent tile scheduler for packed varlen work.
//
// The work of one launch is the list of tiles
//     (segment b, row-block m, head h),  m < ceil(len_b / TILE),
// ordered segment-major, then head, then row-block, so that the tiles of one
// (segment, head) -- which read the same K/V (forward) or Q/dO (backward)
// rows -- are adjacent and run concurrently on neighbouring CTAs, sharing
// those rows through L2.  There are exactly H * sum_b ceil(len_b / TILE)
// tiles: nothing is over-provisioned, so no CTA ever decodes a tile that does
// not exist (the failure described on the "[FA4][SM120] flash_attn_varlen_func
// ... illegal memory access at >=4 varlen segments" issue, sections
// "Interpretation" and "Practical workaround": a grid of 15840 blocks for
// 15680 valid tiles whose tail blocks read cu_seqlens past its end).
//
// CTA c of G visits global tiles c, c+G, c+2G, ...; since that sequence
// increases, each role of the CTA walks the segments with a forward-only
// cursor and reads cu_seqlens[b], cu_seqlens[b+1] for b < batch only.  Every
// cu_seqlens entry is clamped into [0, total] before use, so a malformed
// array cannot produce an out-of-range row.
//
// Segments are walked longest-processing-time first: every tile of a
// segment iterates over the other side's rows (a forward unit over the
// segment's keys, a backward kv tile over its queries), so its cost is
// ceil(len_other / 128) steps, and the segments are ordered by that cost,
// descending (ties by index).  The most expensive tiles then start first and
// the round-robin ends on the cheapest ones, which shortens the tail where
// some CTAs have finished and others still work.  Each CTA computes the
// order itself from cu_seqlens into a table in its shared memory at start
// (nothing is read on the host, nothing stored between launches); past the
// table's capacity the index order is kept.
#pragma once

#include <cstdint>

#include "varlen_internal.h"

namespace varlen {

constexpr int kLptRows = 128;  // rows of the other side per step of a tile's cost
constexpr int kLptCapWide = 4096;   // order-table entries (segments) where shared memory allows (8 KB)
constexpr int kLptCapNarrow = 256;  // ... in the backward kernels, whose tiles leave 0.5 KB free

struct SegCursor {
  int32_t k;        // walk position
  int32_t b;        // current segment (order[k])
  int64_t first;    // global index of segment b's first tile
  int32_t nb;       // row-blocks per head in segment b (on the scheduled side)
  int32_t r0, len;  // scheduled side: first row and length of segment b
  int32_t o0, olen; // other side: first row and length of segment b
};

__device__ __forceinline__ int32_t clamp_row(int32_t v, int32_t total) { return min(max(v, 0), total); }

// Segment bound b of a view: cu_seqlens[b], or b * uni for uniform segments.
// For uniform segments b <= batch and batch * uni <= total < 2^31, so the
// product does not overflow.
__device__ __forceinline__ int32_t cu_at(const CuView& cu, int32_t b) {
  return cu.ptr != nullptr ? __ldg(cu.ptr + b) : b * cu.uni;
}

template <int TILE>
__device__ __forceinline__ void cursor_load(SegCursor& c, const CuView& cu_s, const CuView& cu_o, int32_t total_s,
                                            int32_t total_o) {
  const int32_t a = clamp_row(cu_at(cu_s, c.b), total_s);
  const int32_t e = clamp_row(cu_at(cu_s, c.b + 1), total_s);
  c.r0 = a;
  c.len = max(e - a, 0);
  const int32_t ao = clamp_row(cu_at(cu_o, c.b), total_o);
  const int32_t eo = clamp_row(cu_at(cu_o, c.b + 1), total_o);
  c.o0 = ao;
  c.olen = max(eo - ao, 0);
  c.nb = (c.len + TILE - 1) / TILE;
}

// The walk order: a CTA's order table (built by build_lpt_order) when the
// launch has 2 .. cap segments, else the index order.  The table's address is
// a constant of the kernel, so the choice costs no live register.
struct WalkOrder {
  const uint16_t* table;  // null: always the index order
  int32_t cap;
};

__device__ __forceinline__ int32_t segment_at(const WalkOrder& o, int32_t batch, int32_t k) {
  return (o.table != nullptr && batch > 1 && batch <= o.cap) ? (int32_t)o.table[k] : k;
}

// Writes the walk order of the segments into o.table[0, batch): descending
// ceil(len_o / kLptRows) of the other side, ties by index.  Every thread of
// the CTA calls it (it computes each segment's rank by counting), and the
// CTA synchronises before any cursor uses the table.  Does nothing when the
// index order applies (segment_at).  Reads cu_o[0 .. batch] only.
__device__ __forceinline__ void build_lpt_order(const WalkOrder& o, const CuView& cu_o, int32_t batch,
                                                int32_t total_o) {
  if (o.table == nullptr || batch <= 1 || batch > o.cap) return;
  uint16_t* table = const_cast<uint16_t*>(o.table);
  auto cost = [&](int32_t b) {
    const int32_t a = clamp_row(cu_at(cu_o, b), total_o), e = clamp_row(cu_at(cu_o, b + 1), total_o);
    return (max(e - a, 0) + kLptRows - 1) / kLptRows;
  };
  for (int32_t i = threadIdx.x; i < batch; i += blockDim.x) {
    const int32_t ci = cost(i);
    int32_t rank = 0;
    for (int32_t j = 0; j < batch; ++j) {
      const int32_t cj = cost(j);
      rank += (cj > ci || (cj == ci && j < i)) ? 1 : 0;
    }
    table[rank] = (uint16_t)i;
  }
}

template <int TILE>
__device__ __forceinline__ void cursor_init(SegCursor& c, const CuView& cu_s, const CuView& cu_o, int32_t batch,
                                            int32_t total_s, int32_t total_o, const WalkOrder& order = WalkOrder{nullptr, 0}) {
  c.k = 0;
  c.b = 0;
  c.first = 0;
  c.nb = 0;
  c.r0 = c.len = c.o0 = c.olen = 0;
  if (batch > 0) {
    c.b = segment_at(order, batch, 0);
    cursor_load<TILE>(c, cu_s, cu_o, total_s, total_o);
  }
}

// Moves the cursor to the segment holding global tile t (t never decreases
// between calls; tiles are numbered along the walk order, the `order` given
// to cursor_init).  Returns false when t is past the last tile.
template <int TILE>
__device__ __forceinline__ bool cursor_seek(SegCursor& c, int64_t t, int32_t num_heads, const CuView& cu_s,
                                            const CuView& cu_o, int32_t batch, int32_t total_s, int32_t total_o,
                                            const WalkOrder& order = WalkOrder{nullptr, 0}) {
  while (c.k < batch) {
    const int64_t span = (int64_t)num_heads * c.nb;
    if (t < c.first + span) return true;
    c.first += span;
    ++c.k;
    if (c.k < batch) {
      c.b = segment_at(order, batch, c.k);
      cursor_load<TILE>(c, cu_s, cu_o, total_s, total_o);
    }
  }
  return false;
}

struct Tile {
  int32_t b, m, h;
};

__device__ __forceinline__ Tile cursor_tile(const SegCursor& c, int64_t t) {
  const int64_t local = t - c.first;
  Tile x;
  x.b = c.b;
  x.h = (int32_t)(local / c.nb);
  x.m = (int32_t)(local - (int64_t)x.h * c.nb);
  return x;
}

}  // namespace varlen
