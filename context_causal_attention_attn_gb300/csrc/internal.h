// Internal types shared by the host scheduler and the kernels of libcpattn.
//
// A launch of the attention kernels processes a list of work items.  One
// item is one block of the ring (or the whole block of cp_attn_block, or all
// Ulysses head groups at once via `batch`): a range of query rows against up
// to two key segments, with global positions for the causal mask.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace cpattn {

// ------------------------------------------------------- per-device set-up
// Host-side state that belongs to one device (a kernel's shared-memory
// attribute, a symbol's device address) is set up once per device, with
// that device current, and is safe to reach from several host threads.
constexpr int kMaxDevices = 64;

struct PerDeviceOnce {
  std::atomic<bool> done[kMaxDevices] = {};
  std::mutex mu;
};

// Runs fn() on the current device the first time this device reaches `o`;
// later calls return cudaSuccess without running it.  A failing fn() is
// retried on the next call.
template <class F>
cudaError_t once_per_device(PerDeviceOnce& o, F&& fn) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (o.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(o.mu);
  if (o.done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = fn();
  if (e == cudaSuccess) o.done[dev].store(true, std::memory_order_release);
  return e;
}

constexpr int kMaxItems = 32;   // 2 items per virtual rank per ring step
constexpr int kMaxSegs = 2;     // zigzag: a late query chunk sees 2 KV chunks
constexpr int kMaxRingChunks = 32;  // chunks of a zigzag ring of 16 ranks

// Item flags.
constexpr int kFlagMerge = 1;   // merge into the fp32 accumulator (read acc, lse)
constexpr int kFlagFinal = 2;   // write the normalised result to `out` in out_dt
                                // (otherwise to the fp32 accumulator)
constexpr int kFlagCausal = 4;  // apply the causal mask with global positions

// Rows of the q / k / v tensors are addressed as (stripe r, index i) =
// token r + stride * i, with stride = AttnParams::stripe (1 unless the ring
// runs in the striped layout, where stripe r is virtual rank r's shard).
struct KSeg {
  int64_t mem_row;  // first key index i in the K/V tensor (within stripe `stripe`)
  int64_t pos;      // position of that key for the causal mask
  int32_t len;      // keys in the segment
  int32_t stripe;   // stripe r of the keys (0 unless striped)
};

struct WorkItem {
  int64_t q_mem_row;  // first query index i in the Q tensor (within stripe q_stripe)
  int64_t q_pos;      // position of that query for the causal mask
  int64_t o_row;      // row of out / acc ([rows, H, D]) of query 0
  int64_t lse_col;    // column of lse ([H, ld_lse]) of query 0
  int32_t sq;         // query rows
  int32_t nseg;       // 0..2 key segments, ascending positions, disjoint
  int32_t flags;
  int32_t batch;      // independent instances (Ulysses head groups); >= 1
  int32_t q_stripe;   // stripe r of the queries (0 unless striped)
  int32_t o_stride;   // query i goes to out row o_row + i * o_stride (and lse column)
  // per-batch strides: rows of q / k / out, heads of lse
  int64_t b_q_rows, b_k_rows, b_o_rows, b_lse_heads;
  KSeg seg[kMaxSegs];
  // A whole ring walked in one launch (tensor-core path): when nchunk > 0
  // the key segments are the sequence chunks chunk[0..nchunk) in the order
  // the ring's steps reach them (chunk c = rows [c C, min(S, (c+1) C)) with
  // C = AttnParams::ring_C, S = AttnParams::ring_S), and seg / nseg are unused.
  // With AttnParams::ring_striped the chunks are stripes: chunk c is stripe
  // c (C = S / P keys, stripe index i = token c + P i), whose key i is
  // visible to query i' of stripe q_stripe when i + (c > q_stripe) <= i'.
  int32_t nchunk;
  uint8_t chunk[kMaxRingChunks];
  // chunk-list items: the query chunk (which the list holds once) and the
  // KV tiles of the list's other chunks, all earlier and so visible to
  // every query row -- a query tile's visible tiles without a walk
  int32_t q_chunk;
  int32_t full_tiles;
};

struct AttnParams {
  int H, Hkv, D;               // heads of the q / kv tensors as addressed
  int stripe;                  // token = r + stripe * i for q rows (see KSeg)
  int kv_stripe;               // the same for k / v rows
  int maps4d;                  // TMA maps are 4-D (d, head, r, i); else 3-D (d, head, row)
  int b_q_heads;               // KV head of (batch b, head h) is
  int kv_group;                //   (b * b_q_heads + h) / kv_group
  int out_dt;                  // 0 fp32, 1 bf16
  float scale_log2;            // softmax scale * log2(e)
  float scale;                 // softmax scale
  void* out;                   // [rows, H, D] out_dt
  float* acc;                  // [rows, H, D] fp32 accumulator (may equal out)
  float* lse;                  // [H, ld_lse] fp32
  int64_t ld_lse;
  int nitems;
  int cta_start[kMaxItems + 1];  // prefix sum of CTAs per item
  WorkItem items[kMaxItems];
  // raw pointers for the CUDA-core path (the tensor-core path uses TMA maps)
  const void* q;
  const void* k;
  const void* v;
  int64_t q_rows, k_rows;      // rows of the q / k tensors (bounds)
  int64_t ring_C, ring_S;      // chunk rows and sequence length of chunk-list items
  int ring_striped;            // chunk-list items name stripes (see WorkItem::chunk)
  // head_major: the grid runs head by head (all items' query tiles of head 0,
  // then head 1, ...), so the CTAs resident at one time read one head's K/V;
  // tile_start is the prefix sum of query tiles per item.  Only the tile
  // ranks [0, hm_long) of every head run that way; the remaining (shortest)
  // ranks follow, rank by rank across all heads, so that the grid ends on
  // short tiles.  Otherwise item by item (cta_start), query tiles fastest
  // within a head.
  int head_major;
  int hm_long;
  int tma_out;                 // out has a TMA map (bf16 [q_rows, H, D], plain rows)
  int tile_start[kMaxItems + 1];
};

// Status word written by kernels whose bounded wait expired.
constexpr int kDevErrTimeout = 1;

// Bounds-checked build (compiled with CP_DEBUG_BOUNDS, as libcpattn_debug.so):
// the kernels check that every tile or row they read or write lies inside
// its tensor; a failed check writes kDevErrBounds | site << 8 to the status
// word and the access is skipped.  Release builds compile the checks away.
constexpr int kDevErrBounds = 2;
enum BoundsSite : int {
  kSiteFwdTile = 1,  // tensor-core forward: a query tile's q rows, out / acc rows, lse columns
  kSiteFwdKV = 2,    // tensor-core forward: a K/V tile's rows
  kSiteFwdSimt = 3,  // CUDA-core forward: a query row or a key row
  kSiteBwdStat = 4,  // tensor-core backward: a stationary tile's rows and lse / delta columns
  kSiteBwdStr = 5,   // tensor-core backward: a streamed tile's rows or lse / delta columns
  kSiteBwdSimt = 6,  // CUDA-core backward: a stationary or streamed row
};
#ifdef CP_DEBUG_BOUNDS
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

#ifdef __CUDACC__
// `cond` in the bounds-checked build, recording `site` when it fails; always
// true (and compiled away) in release builds.
__device__ __forceinline__ bool bounds_ok(bool cond, int* dev_err, int site) {
  if (!kDebugBounds) return true;
  if (!cond) atomicCAS(dev_err, 0, kDevErrBounds | (site << 8));
  return cond;
}
#endif

}  // namespace cpattn

namespace cpattn {

// ------------------------------------------------------------ backward
// One backward work item: a stationary row range (queries for the dQ kernel,
// keys for the dK/dV kernel) against up to two streamed row ranges (keys /
// queries).  Row i of a segment is token stripe + stride * (row + i) of the
// tensors (stride = BwdParams::stride, 1 unless the ring is striped); the
// token is also the LSE / delta column of a query and the gradient row.
// `pos` is the position of row 0 for the causal mask.
struct BwdSeg {
  int64_t row;
  int64_t pos;
  int32_t len;
  int32_t stripe;
};

constexpr int kBwdAccumulate = 1;  // add into the fp32 gradient buffer (else write it)
constexpr int kBwdFinal = 2;       // write the finished gradient to the output in out_dt

struct BwdItem {
  BwdSeg stat;
  BwdSeg str[kMaxSegs];
  int32_t nstr;
  int32_t flags;
  // A whole ring in one launch: when nchunk > 0 the streamed segments are
  // the sequence chunks chunk[0..nchunk) in the order the ring's steps reach
  // them (chunk c = rows [c C, min(S, (c+1) C)) with C = BwdParams::ring_C,
  // S = BwdParams::ring_S), and str / nstr are unused.  With
  // BwdParams::ring_striped they are stripes (C = S / P rows of stripe c),
  // key i of stripe a visible to query i' of stripe b when i + (a > b) <= i'.
  int32_t nchunk;
  uint8_t chunk[kMaxRingChunks];
};

struct BwdParams {
  int H, Hkv, D;
  int out_dt;            // 0 fp32, 1 bf16 (gradient outputs)
  int causal;
  int stride;            // token = stripe + stride * row (4-D TMA maps when > 1)
  float scale, scale_log2;
  const float* lse;      // [H, ld] natural log, the forward's whole-row LSE
  const float* delta;    // [H, ld] rowsum(dO * O)
  int64_t ld;
  float* acc0;           // dQ kernel: dq fp32 [rows, H, D]; dK/dV kernel: dv [rows, Hkv, D]
  float* acc1;           //                                      dk [rows, Hkv, D]
  void* out0;            // finished gradients in out_dt (same layouts)
  void* out1;
  int nitems;
  int cta_start[kMaxItems + 1];
  BwdItem items[kMaxItems];
  int64_t ring_C, ring_S;  // chunk rows and sequence length of chunk-list items
  int64_t q_rows, k_rows;  // rows of the q / dout / dq and k / v / dk / dv tensors (bounds)
  int ring_striped;        // chunk-list items name stripes (see BwdItem::chunk)
};

}  // namespace cpattn
