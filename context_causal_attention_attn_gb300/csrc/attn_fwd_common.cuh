// Pieces of the forward attention kernel on the tensor cores (attn_tc.cu):
// tile sizes, the walk over an item's KV tiles, the task decode's search and
// the timeout record.
#pragma once

#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"

namespace cpattn {

namespace tc {
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int HD = 128;
constexpr uint32_t TILE_BYTES = BM * HD * 2;  // 32768
constexpr uint32_t BOX_BYTES = BM * 64 * 2;   // 16384: rows x 64 columns
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;
}  // namespace tc

// Key segment s of an item: seg[s], or for a chunk-list item (a whole ring
// in one launch) sequence chunk chunk[s].
__device__ __forceinline__ int item_nseg(const WorkItem& it) {
  return it.nchunk > 0 ? it.nchunk : it.nseg;
}
// kStriped: the kernel instance with strided rows (the only one that sees
// striped chunk lists, whose check the plain instance compiles away).
template <bool kStriped>
__device__ __forceinline__ void item_seg(const WorkItem& it, const AttnParams& p, int s,
                                         int64_t& mem_row, int64_t& pos, int& len, int& stripe) {
  if (kStriped && it.nchunk > 0 && p.ring_striped) {
    // stripe c in stripe indices; its keys trail the queries' by one
    // position when c comes after the query stripe
    const int c = it.chunk[s];
    mem_row = 0;
    pos = c > it.q_stripe ? 1 : 0;
    len = static_cast<int>(p.ring_C);
    stripe = c;
  } else if (it.nchunk > 0) {
    const int64_t c0 = static_cast<int64_t>(it.chunk[s]) * p.ring_C;
    mem_row = c0;
    pos = c0;
    len = static_cast<int>(min(p.ring_S - c0, p.ring_C));
    stripe = 0;
  } else {
    mem_row = it.seg[s].mem_row;
    pos = it.seg[s].pos;
    len = it.seg[s].len;
    stripe = it.seg[s].stripe;
  }
}

// KV tiles of a segment holding a key visible to a query at position
// qp_last (causal: a prefix of the segment's tiles; keys grow along it).
__device__ __forceinline__ int seg_visible_tiles(int64_t pos, int len, int64_t qp_last,
                                                 bool causal) {
  const int T = (len + tc::BN - 1) / tc::BN;
  if (!causal) return T;
  if (qp_last < pos) return 0;
  const int64_t v = (qp_last - pos) / tc::BN + 1;
  return v < T ? static_cast<int>(v) : T;
}

// Walks the KV tiles a query tile evaluates, in item order: every segment's
// visible prefix.  (For ring-step items the segments ascend, so this is a
// prefix of all tiles; for chunk-list items the diagonal chunk may come
// before earlier ones.)  Only the position in the walk is kept (three
// registers); a tile's keys are re-derived from the item when asked for.
template <bool kStriped>
struct TileCursor {
  int s, t, tv;  // segment, tile within it, visible tiles of the segment
  __device__ __forceinline__ void seek(const WorkItem& it, const AttnParams& p, int64_t qp_last,
                                       bool causal) {
    const int n = item_nseg(it);
    for (; s < n; ++s) {
      int64_t mem_row, pos;
      int len, stripe;
      item_seg<kStriped>(it, p, s, mem_row, pos, len, stripe);
      tv = seg_visible_tiles(pos, len, qp_last, causal);
      if (tv > 0) return;
    }
  }
  __device__ __forceinline__ void init(const WorkItem& it, const AttnParams& p, int64_t qp_last,
                                       bool causal) {
    s = 0;
    t = 0;
    tv = 0;
    seek(it, p, qp_last, causal);
  }
  __device__ __forceinline__ void next(const WorkItem& it, const AttnParams& p, int64_t qp_last,
                                       bool causal) {
    if (++t >= tv) {
      ++s;
      t = 0;
      seek(it, p, qp_last, causal);
    }
  }
  // the current tile: first key row in memory, first key position, keys,
  // stripe of the keys
  __device__ __forceinline__ void keys(const WorkItem& it, const AttnParams& p, int64_t& kmem,
                                       int64_t& kpos, int& nk, int& stripe) const {
    int len;
    item_seg<kStriped>(it, p, s, kmem, kpos, len, stripe);
    kmem += static_cast<int64_t>(t) * tc::BN;
    kpos += static_cast<int64_t>(t) * tc::BN;
    nk = min(tc::BN, len - t * tc::BN);
  }
};

// Number of KV tiles a query tile whose last row sits at qp_last evaluates.
template <bool kStriped>
__device__ __forceinline__ int visible_tiles(const WorkItem& it, const AttnParams& p,
                                             int64_t qp_last, bool causal) {
  if (it.nchunk > 0 && causal && !(kStriped && p.ring_striped)) {
    // every chunk but the query chunk lies before it
    const int64_t pos = static_cast<int64_t>(it.q_chunk) * p.ring_C;
    const int len = static_cast<int>(min(p.ring_S - pos, p.ring_C));
    return it.full_tiles + seg_visible_tiles(pos, len, qp_last, true);
  }
  int n = 0;
  const int ns = item_nseg(it);
  for (int s = 0; s < ns; ++s) {
    int64_t mem_row, pos;
    int len, stripe;
    item_seg<kStriped>(it, p, s, mem_row, pos, len, stripe);
    n += seg_visible_tiles(pos, len, qp_last, causal);
  }
  return n;
}

// The last index i < n with start[i] <= x (start ascending, start[0] <= x):
// the item of grid position x.  A binary search: the kernel parameters sit
// in the constant bank, where each dependent load of a linear search costs
// a cache round trip.
__device__ __forceinline__ int last_at_most(const int* start, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void record_timeout(int* dev_err, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(dev_err, 0, kDevErrTimeout);
}

}  // namespace cpattn
