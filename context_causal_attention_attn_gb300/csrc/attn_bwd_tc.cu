// Backward of causal block attention on the tcgen05 tensor cores, from the
// forward's saved whole-row LSE and delta = rowsum(dO * O):
//   p_ij = exp(s_ij - lse_i),  dv_j = sum_i p_ij do_i,  dp_ij = do_i . v_j,
//   ds_ij = p_ij (dp_ij - delta_i),  dq_i = scale sum_j ds_ij k_j,
//   dk_j = scale sum_i ds_ij q_i.
// (The chain rule of the forward definition -- [CP-handbook]
// "上下文并行：Ring Attention 与 Ulysses", section "哪些运算可以直接切", the
// attention helper -- written with the saved LSE; the pages time forward +
// backward steps, [CP-practice] section 4.2.)
//
// One template, two kernels:
//  * kDKDV = false (dQ): the CTA holds 128 query rows (Q, dO) and streams
//    K, V tiles:  S = Q K^T (TMEM X), dP = dO V^T (TMEM Y0 / Y1 by tile
//    parity), dS as bf16 over the dP buffer, dQ += dS K (TS form, K as an
//    MN-major operand).  TMEM: X [0,128), Y0 [128,256), Y1 [256,384),
//    dQ [384,512).
//  * kDKDV = true (dK, dV): the CTA holds 128 key rows (K, V) of one KV head
//    and streams Q, dO tiles of every query head of its group:
//    S^T = K Q^T and dP^T = V dO^T into the two 128-column buffers X and Y,
//    whose roles swap every tile (tile j: S^T in one, dP^T in the other);
//    P^T and dS^T as bf16 pairs over the S^T buffer (columns 0-31 | 64-95
//    and 32-63 | 96-127); dV += P^T dO and dK += dS^T Q (TS form, dO and Q
//    MN-major).  S^T(j+1) goes into tile j's dP^T buffer as soon as dP^T(j)
//    has been read, dP^T(j+1) into tile j's S^T buffer once dV(j) and dK(j)
//    are done.  TMEM: X [0,128), Y [128,256), dV [256,384), dK [384,512).
// Two kernels recompute S and dP but need no atomics and are deterministic.
//
// Warps 0-7: elementwise.  Warp w owns TMEM lanes 32 (w % 4) .. +31 (the
// stationary rows) and the streamed columns 64 (w / 4) .. +63.  Per tile:
// phase 1 reads S -> P (fp32, kept in registers; dQ: frees X, dK/dV: writes
// P^T back); phase 2 reads dP -> dS (dK/dV: frees the dP^T buffer first).
// Warp 8: TMA producer; warp 9: TMEM allocator + single-thread MMA issuer,
// which runs the next tile's S (and dP) while the elementwise warps work on
// this one.  Every wait is bounded as in the forward kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"
#include "sm100.cuh"

namespace cpattn {

using namespace sm100;

namespace bw {
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int HD = 128;
// Streamed tiles: ring A holds the first operand (dQ: K, dK/dV: Q), ring B
// the second (V, dO).  Both kernels hold their ring-A tile from the first
// MMA of a tile to the last (dQ: K_j from S(j) to dQ(j); dK/dV: Q_j from
// S^T(j) to dK(j)), about two tile periods, so ring A gets 3 slots: the next
// tile then reuses the slot of tile j-2, long free, and loads a full period
// ahead.
template <bool kDKDV>
struct Rings {
  static constexpr int NA = 3;
  static constexpr int NB = 2;
};
constexpr uint32_t TILE_BYTES = BM * HD * 2;
constexpr uint32_t BOX_BYTES = BM * 64 * 2;
constexpr int EW_WARPS = 8;
constexpr int EW_THREADS = EW_WARPS * 32;
constexpr int THREADS = EW_THREADS + 64;
constexpr int WARP_LOAD = EW_WARPS;
constexpr int WARP_MMA = EW_WARPS + 1;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;
constexpr uint32_t SMEM_LIMIT = 232448;  // dynamic shared memory per block (227 KB)
// epilogue staging of one accumulator: 128 rows of 132 floats (the pad keeps
// row-per-thread and row-per-half-warp accesses free of bank conflicts)
constexpr uint32_t STG_PITCH = 132;
constexpr uint32_t STG_BYTES = 128 * STG_PITCH * 4;

// barriers: FULL / EMPTY of ring A slots 0-2 and ring B slots 3-4
constexpr int MAX_SLOTS = 5;
constexpr int BAR_STAT = 0;
constexpr int BAR_FULL = 1;
constexpr int BAR_EMPTY = BAR_FULL + MAX_SLOTS;
constexpr int BAR_S = BAR_EMPTY + MAX_SLOTS;  // S (dK/dV: S^T) of a tile done
constexpr int BAR_DP = BAR_S + 1;             // dP of a tile: [2] (dQ: per Y buffer)
constexpr int BAR_XFREE = BAR_DP + 2;         // dQ: elementwise read S; dK/dV: read dP^T
constexpr int BAR_E1 = BAR_XFREE + 1;         // dK/dV: P^T in TMEM
constexpr int BAR_E2 = BAR_E1 + 1;            // dS in TMEM: [2] (dQ: per Y buffer)
constexpr int BAR_G2 = BAR_E2 + 2;            // dQ MMA / dK MMA done
constexpr int BAR_DONE = BAR_G2 + 1;          // every MMA of the CTA done
constexpr int BAR_DRAIN = BAR_DONE + 1;
constexpr int NUM_BARS = BAR_DRAIN + 1;

template <bool kDKDV>
struct Smem {
  static constexpr uint32_t STAT = 0;
  static constexpr uint32_t STR = 2 * TILE_BYTES;
  static constexpr uint32_t COLS = STR + (Rings<kDKDV>::NA + Rings<kDKDV>::NB) * TILE_BYTES;
  // COLS (dK/dV): [2 slots][-l2 | delta][BN]
  static constexpr uint32_t BARS = COLS + (kDKDV ? 2 * 2 * BN * 4 : 0);
  static constexpr uint32_t TMEM_SLOT = BARS + NUM_BARS * 8;
  static constexpr uint32_t ABORT = TMEM_SLOT + 4;
  static constexpr uint32_t USED = ABORT + 4;
  // up to 1 KB to align the base to the 1024-byte swizzle atom
  static constexpr uint32_t BYTES = USED + 1024 <= SMEM_LIMIT ? USED + 1024 : SMEM_LIMIT;
};
static_assert(Smem<true>::USED <= SMEM_LIMIT, "dK/dV shared memory");
static_assert(Smem<false>::STR + STG_BYTES <= Smem<false>::BARS, "dQ epilogue staging");
static_assert(Smem<true>::STR + STG_BYTES <= Smem<true>::COLS, "dK/dV epilogue staging");
static_assert(Smem<false>::USED <= SMEM_LIMIT, "dQ shared memory");
}  // namespace bw

__device__ __forceinline__ int bw_tiles(int len) { return (len + bw::BN - 1) / bw::BN; }

// Streamed segment s of an item: str[s], or for a chunk-list item (a whole
// ring in one launch) sequence chunk chunk[s].
__device__ __forceinline__ int bw_nstr(const BwdItem& it) {
  return it.nchunk > 0 ? it.nchunk : it.nstr;
}
template <bool kDKDV, bool kStriped>
__device__ __forceinline__ void bw_str(const BwdItem& it, const BwdParams& p, int s,
                                       int64_t& row, int64_t& pos, int& len, int& stripe) {
  if (kStriped && it.nchunk > 0 && p.ring_striped) {
    // stripe c in stripe indices (only kernels with strided rows see
    // these).  Key i of stripe a sees query i' of stripe b when
    // i + (a > b) <= i': streamed keys (dQ) sit one position later when
    // their stripe follows the queries'; streamed queries (dK/dV) one
    // position earlier when the keys' stripe follows theirs.
    const int c = it.chunk[s];
    row = 0;
    pos = kDKDV ? (it.stat.stripe > c ? -1 : 0) : (c > it.stat.stripe ? 1 : 0);
    len = static_cast<int>(p.ring_C);
    stripe = c;
  } else if (it.nchunk > 0) {
    const int64_t c0 = static_cast<int64_t>(it.chunk[s]) * p.ring_C;
    row = c0;
    pos = c0;
    len = static_cast<int>(min(p.ring_S - c0, p.ring_C));
    stripe = 0;
  } else {
    row = it.str[s].row;
    pos = it.str[s].pos;
    len = it.str[s].len;
    stripe = it.str[s].stripe;
  }
}

// Streamed tiles [t0, t1) of a segment the stationary tile uses.  kDKDV =
// false: key tiles visible to a query at lim_pos (a prefix).  kDKDV = true:
// query tiles with a query at or after the stationary key at lim_pos (a
// suffix).
template <bool kDKDV>
__device__ __forceinline__ void bw_vis(int64_t pos, int len, int64_t lim_pos, bool causal,
                                       int& t0, int& t1) {
  const int T = bw_tiles(len);
  t0 = 0;
  t1 = T;
  if (!causal) return;
  if (!kDKDV) {
    if (lim_pos < pos) {
      t1 = 0;
      return;
    }
    const int64_t v = (lim_pos - pos) / bw::BN + 1;
    if (v < T) t1 = static_cast<int>(v);
  } else {
    if (pos + len - 1 < lim_pos) {  // every query before the keys
      t1 = 0;
      return;
    }
    t0 = lim_pos > pos ? static_cast<int>((lim_pos - pos) / bw::BN) : 0;
  }
}

// Streamed tiles of an item per head (the dK/dV kernel runs them once per
// query head of its group).
template <bool kDKDV, bool kStriped>
__device__ __forceinline__ int bw_count(const BwdItem& it, const BwdParams& p, int64_t lim_pos,
                                        bool causal) {
  int n = 0;
  const int ns = bw_nstr(it);
  for (int s = 0; s < ns; ++s) {
    int64_t row, pos;
    int len, stripe, t0, t1;
    bw_str<kDKDV, kStriped>(it, p, s, row, pos, len, stripe);
    bw_vis<kDKDV>(pos, len, lim_pos, causal, t0, t1);
    n += t1 - t0;
  }
  return n;
}

// Walks the streamed tiles of an item in order -- segment by segment, and
// for the dK/dV kernel head by head of the query group -- keeping only its
// position (a tile's rows are re-derived from the item when asked for).
template <bool kDKDV, bool kStriped>
struct BwCursor {
  int s, t, tend;  // segment, tile within it, end of its used tiles
  int k, g;        // tile within the head, query head within the group
  __device__ __forceinline__ void seek(const BwdItem& it, const BwdParams& p, int64_t lim,
                                       bool causal) {
    const int ns = bw_nstr(it);
    for (; s < ns; ++s) {
      int64_t row, pos;
      int len, stripe, t0;
      bw_str<kDKDV, kStriped>(it, p, s, row, pos, len, stripe);
      bw_vis<kDKDV>(pos, len, lim, causal, t0, tend);
      if (t0 < tend) {
        t = t0;
        return;
      }
    }
  }
  __device__ __forceinline__ void init(const BwdItem& it, const BwdParams& p, int64_t lim,
                                       bool causal) {
    s = 0;
    t = 0;
    tend = 0;
    k = 0;
    g = 0;
    seek(it, p, lim, causal);
  }
  // to the next tile; nper = tiles per head
  __device__ __forceinline__ void next(const BwdItem& it, const BwdParams& p, int64_t lim,
                                       bool causal, int nper) {
    if (++k == nper) {  // the next query head of the group starts over
      k = 0;
      ++g;
      s = 0;
      seek(it, p, lim, causal);
      return;
    }
    if (++t >= tend) {
      ++s;
      seek(it, p, lim, causal);
    }
  }
  // the current tile: first row, first position, valid rows, stripe
  __device__ __forceinline__ void tile(const BwdItem& it, const BwdParams& p, int64_t& row,
                                       int64_t& pos, int& n, int& stripe) const {
    int len;
    bw_str<kDKDV, kStriped>(it, p, s, row, pos, len, stripe);
    row += static_cast<int64_t>(t) * bw::BN;
    pos += static_cast<int64_t>(t) * bw::BN;
    n = min(bw::BN, len - t * bw::BN);
  }
};

__device__ __forceinline__ void bw_timeout(int* dev_err, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicCAS(dev_err, 0, kDevErrTimeout);
}

// kStriped: tensor rows are stripes (4-D maps (d, head, stripe, row)).
template <bool kDKDV, bool kStriped>
__global__ void __launch_bounds__(bw::THREADS, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ BwdParams p, int* dev_err) {
  using L = bw::Smem<kDKDV>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad + L::USED > L::BYTES) {
    // the base is not aligned enough for the layout: report, do nothing
    if (threadIdx.x == 0) atomicCAS(dev_err, 0, kDevErrTimeout);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sStat = sbase + L::STAT;
  const uint32_t sStr = sbase + L::STR;
  float* cols = reinterpret_cast<float*>(smem + L::COLS);
  auto bar = [&](int i) -> uint32_t { return sbase + L::BARS + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------------------------------------------------- task decode
  int ii = 0;
  while (ii + 1 < p.nitems && static_cast<int>(blockIdx.x) >= p.cta_start[ii + 1]) ++ii;
  const BwdItem& it = p.items[ii];
  int local = static_cast<int>(blockIdx.x) - p.cta_start[ii];
  const int ntile = bw_tiles(it.stat.len);
  const int tix = local % ntile;  // stationary tiles fastest: CTAs share heads
  local /= ntile;
  const int grp = p.H / p.Hkv;
  // dQ: heavier (later) query tiles first; dK/dV: heavier (earlier) key tiles first
  const int stile = kDKDV ? tix : ntile - 1 - tix;
  const int shead = local;  // dQ: query head; dK/dV: KV head
  const bool causal = p.causal != 0;
  const int64_t srow0 = it.stat.row + static_cast<int64_t>(stile) * bw::BM;
  const int64_t spos0 = it.stat.pos + static_cast<int64_t>(stile) * bw::BM;
  const int nstat = min(bw::BM, it.stat.len - stile * bw::BM);
  // visibility limit: last query position (dQ) / first key position (dK/dV)
  const int64_t lim = kDKDV ? spos0 : spos0 + nstat - 1;
  const int nper = bw_count<kDKDV, kStriped>(it, p, lim, causal);
  const int nstr = kDKDV ? nper * grp : nper;
  const int kvh = kDKDV ? shead : shead / grp;
  const int64_t stride = kStriped ? p.stride : 1;
  // Bounds-checked build: the stationary tile's rows (which are also its
  // gradient rows and, for dQ, its lse / delta columns) lie inside their
  // tensors; a tile that fails is recorded and skips its global reads and
  // writes.
  bool in_bounds = true;
  if (kDebugBounds) {
    const int64_t t0 = it.stat.stripe + stride * srow0;
    const int64_t t1 = it.stat.stripe + stride * (srow0 + nstat - 1);
    in_bounds = nstat > 0 && srow0 >= 0 && it.stat.stripe >= 0 && it.stat.stripe < stride &&
                t1 < (kDKDV ? p.k_rows : p.q_rows) && shead < (kDKDV ? p.Hkv : p.H) &&
                (kDKDV || t1 < p.ld) && t0 >= 0;
    if (threadIdx.x == 0) bounds_ok(in_bounds, dev_err, kSiteBwdStat);
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(bw::BAR_STAT), 1);
    for (int s = 0; s < bw::MAX_SLOTS; ++s) {
      mbar_init(bar(bw::BAR_FULL + s), 1);
      mbar_init(bar(bw::BAR_EMPTY + s), 1);
    }
    mbar_init(bar(bw::BAR_S), 1);
    mbar_init(bar(bw::BAR_DP), 1);
    mbar_init(bar(bw::BAR_DP + 1), 1);
    mbar_init(bar(bw::BAR_XFREE), bw::EW_THREADS);
    mbar_init(bar(bw::BAR_E1), bw::EW_THREADS);
    mbar_init(bar(bw::BAR_E2), bw::EW_THREADS);
    mbar_init(bar(bw::BAR_E2 + 1), bw::EW_THREADS);
    mbar_init(bar(bw::BAR_G2), 1);
    mbar_init(bar(bw::BAR_DONE), 1);
    mbar_init(bar(bw::BAR_DRAIN), 1);
    fence_mbar_init();
  }
  if (warp == bw::WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), bw::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t COL_X = 0;
  constexpr uint32_t COL_Y = 128;                 // dQ: Y0; Y1 at 256
  constexpr uint32_t COL_A0 = kDKDV ? 256 : 384;  // dV or dQ
  constexpr uint32_t COL_A1 = 384;                // dK

  // streamed tile j, operand w (0: ring A, 1: ring B) -> slot, use count
  constexpr int NA = bw::Rings<kDKDV>::NA, NB = bw::Rings<kDKDV>::NB;
  auto slot_of = [](int j, int w) { return w == 0 ? j % NA : NA + j % NB; };
  auto use_of = [](int j, int w) { return w == 0 ? j / NA : j / NB; };
  // the cursor's tile -> (row, pos, rows, stripe, query head), then advance
  auto str_tile = [&](BwCursor<kDKDV, kStriped>& c, int64_t& row, int64_t& pos, int& n, int& stripe,
                      int& qh) {
    c.tile(it, p, row, pos, n, stripe);
    qh = kDKDV ? shead * grp + c.g : shead;
    c.next(it, p, lim, causal, nper);
  };
  auto load = [&](uint32_t dst, const CUtensorMap* tm, uint32_t b, int c0, int head, int stripe,
                  int64_t row, uint64_t pol) {
    if (kStriped)
      tma_load_4d(dst, tm, b, c0, head, stripe, static_cast<int>(row), pol);
    else
      tma_load_3d(dst, tm, b, c0, head, static_cast<int>(row), pol);
  };

  if (warp == bw::WARP_LOAD) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      const uint64_t pol_stat = policy_evict_first();
      const uint64_t pol_str = policy_evict_last();
      const CUtensorMap* st0 = kDKDV ? &tm_k : &tm_q;
      const CUtensorMap* st1 = kDKDV ? &tm_v : &tm_do;
      const int sh = kDKDV ? kvh : shead;
      mbar_arrive_expect_tx(bar(bw::BAR_STAT), 2 * bw::TILE_BYTES);
      for (int w = 0; w < 2; ++w)
        for (int hh = 0; hh < 2; ++hh)
          load(sStat + w * bw::TILE_BYTES + hh * bw::BOX_BYTES, w == 0 ? st0 : st1,
               bar(bw::BAR_STAT), hh * 64, sh, it.stat.stripe, srow0, pol_stat);
      int issued = 0;  // tiles whose loads were issued
      BwCursor<kDKDV, kStriped> pc;
      pc.init(it, p, lim, causal);
      for (int j = 0; j < nstr; ++j) {
        int64_t row, pos;
        int n, stripe, qh;
        str_tile(pc, row, pos, n, stripe, qh);
        // (a copy outside the tensor would only read the fill value)
        if (kDebugBounds)
          bounds_ok(n > 0 && row >= 0 && stripe >= 0 && stripe < stride &&
                        stripe + stride * (row + n - 1) < (kDKDV ? p.q_rows : p.k_rows) &&
                        qh < p.H,
                    dev_err, kSiteBwdStr);
        bool ok = true;
        for (int w = 0; w < 2; ++w) {
          const int st = slot_of(j, w);
          if (!mbar_wait(bar(bw::BAR_EMPTY + st), (use_of(j, w) & 1) ^ 1, bw::WAIT_LIMIT_NS,
                         abort_flag)) {
            bw_timeout(dev_err, abort_flag);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(bw::BAR_FULL + st), bw::TILE_BYTES);
          // dQ streams K then V; dK/dV streams Q then dO
          const CUtensorMap* tm = kDKDV ? (w == 0 ? &tm_q : &tm_do) : (w == 0 ? &tm_k : &tm_v);
          const int hd = kDKDV ? qh : kvh;
          for (int hh = 0; hh < 2; ++hh)
            load(sStr + st * bw::TILE_BYTES + hh * bw::BOX_BYTES, tm, bar(bw::BAR_FULL + st),
                 hh * 64, hd, stripe, row, pol_str);
          issued = 2 * j + w + 1;
        }
        if (!ok) break;
      }
      // no copy may be in flight when the CTA exits: wait for the last use
      // of every slot that was loaded
      mbar_wait(bar(bw::BAR_STAT), 0, bw::WAIT_LIMIT_NS, nullptr);
      for (int w = 0; w < 2; ++w) {
        const int nw = (issued + 1 - w) / 2;  // tiles whose operand w was loaded
        for (int j = max(0, nw - (w == 0 ? NA : NB)); j < nw; ++j)
          mbar_wait(bar(bw::BAR_FULL + slot_of(j, w)), use_of(j, w) & 1, bw::WAIT_LIMIT_NS,
                    nullptr);
      }
    }
  } else if (warp == bw::WARP_MMA) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_xy = idesc_bf16_f32(bw::BM, bw::BN, false);
      constexpr uint32_t idesc_g = idesc_bf16_f32(bw::BM, bw::HD, true);
      auto wait = [&](int b, uint32_t parity) {
        return mbar_wait(bar(b), parity, bw::WAIT_LIMIT_NS, abort_flag);
      };
      // operand nn = 2 j + w of the stream
      auto full = [&](int nn) {
        return wait(bw::BAR_FULL + slot_of(nn >> 1, nn & 1), use_of(nn >> 1, nn & 1) & 1);
      };
      auto stage = [&](int nn) { return sStr + slot_of(nn >> 1, nn & 1) * bw::TILE_BYTES; };
      auto release = [&](int nn) { mma_commit(bar(bw::BAR_EMPTY + slot_of(nn >> 1, nn & 1))); };
      // X = stat0 . first^T (S) and Y = stat1 . second^T (dP), both K-major
      auto mma_xy = [&](uint32_t dcol, uint32_t a_smem, uint32_t b_smem) {
#pragma unroll
        for (int kk = 0; kk < bw::HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * bw::BOX_BYTES + (kk & 3) * 32;
          mma_ss(tmem + dcol, sdesc_sw128(a_smem + off, 16, 1024),
                 sdesc_sw128(b_smem + off, 16, 1024), idesc_xy, kk > 0 ? 1u : 0u);
        }
      };
      // acc (+)= bf16 operand in TMEM (packed: streamed columns 0-63 in the
      // first 32 columns, 64-127 at +64) . B (MN-major streamed tile)
      auto mma_tmem_a = [&](uint32_t dcol, uint32_t acol, uint32_t b_smem, bool acc) {
#pragma unroll
        for (int kk = 0; kk < bw::BN / 16; ++kk)
          mma_ts(tmem + dcol, tmem + acol + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                 sdesc_sw128(b_smem + kk * 2048, bw::BOX_BYTES, 1024), idesc_g,
                 (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      if (nstr > 0) {
        ok = wait(bw::BAR_STAT, 0) && full(0) && full(1);
        tc_fence_after();
        if (ok) {
          mma_xy(COL_X, sStat, stage(0));
          mma_commit(bar(bw::BAR_S));
          mma_xy(COL_Y, sStat + bw::TILE_BYTES, stage(1));
          mma_commit(bar(bw::BAR_DP));
          if (!kDKDV) release(1);  // V_0 done
        }
      }
      for (int j = 0; ok && j < nstr; ++j) {
        const int n0 = 2 * j, n1 = 2 * j + 1;
        const bool next = j + 1 < nstr;
        if (!kDKDV) {
          // S(j+1) once X is read, dP(j+1) into the other Y buffer once
          // dQ(j-1) (which read it) is done, then dQ(j)
          if (next) {
            if (!(ok = wait(bw::BAR_XFREE, j & 1) && full(n0 + 2))) break;
            tc_fence_after();
            mma_xy(COL_X, sStat, stage(n0 + 2));
            mma_commit(bar(bw::BAR_S));
            if (j >= 1 && !(ok = wait(bw::BAR_G2, (j - 1) & 1))) break;
            if (!(ok = full(n1 + 2))) break;
            tc_fence_after();
            mma_xy(COL_Y + ((j + 1) & 1) * 128, sStat + bw::TILE_BYTES, stage(n1 + 2));
            mma_commit(bar(bw::BAR_DP + ((j + 1) & 1)));
            release(n1 + 2);  // V_{j+1} done
          }
          if (!(ok = wait(bw::BAR_E2 + (j & 1), (j >> 1) & 1))) break;
          tc_fence_after();
          mma_tmem_a(COL_A0, COL_Y + (j & 1) * 128, stage(n0), j > 0);
          mma_commit(bar(bw::BAR_G2));
          release(n0);  // K_j done
        } else {
          // tile j: S^T, P^T, dS^T in buffer cs(j), dP^T in the other one;
          // the roles swap every tile
          const uint32_t cs = (j & 1) ? COL_Y : COL_X, cd = (j & 1) ? COL_X : COL_Y;
          // dV += P^T dO_j, P^T packed in cs (columns 0-31 | 64-95)
          if (!(ok = wait(bw::BAR_E1, j & 1))) break;
          tc_fence_after();
          mma_tmem_a(COL_A0, cs, stage(n1), j > 0);
          release(n1);  // dO_j done (dP^T(j) read it earlier)
          // S^T(j+1) into cd once the elementwise warps have read dP^T(j)
          if (next) {
            if (!(ok = wait(bw::BAR_XFREE, j & 1) && full(n0 + 2))) break;
            tc_fence_after();
            mma_xy(cd, sStat, stage(n0 + 2));
            mma_commit(bar(bw::BAR_S));
          }
          // dK += dS^T Q_j, dS^T packed in cs (columns 32-63 | 96-127)
          if (!(ok = wait(bw::BAR_E2, j & 1))) break;
          tc_fence_after();
          mma_tmem_a(COL_A1, cs + 32, stage(n0), j > 0);
          mma_commit(bar(bw::BAR_G2));
          release(n0);  // Q_j done
          // dP^T(j+1) into cs once dV(j) and dK(j) (which read it) are done
          if (next) {
            if (!(ok = wait(bw::BAR_G2, j & 1) && full(n1 + 2))) break;
            tc_fence_after();
            mma_xy(cs, sStat + bw::TILE_BYTES, stage(n1 + 2));
            mma_commit(bar(bw::BAR_DP));
          }
        }
      }
      if (!ok) bw_timeout(dev_err, abort_flag);
      mma_commit(bar(bw::BAR_DONE));
      mma_commit(bar(bw::BAR_DRAIN));
      mbar_wait(bar(bw::BAR_DRAIN), 0, bw::WAIT_LIMIT_NS, nullptr);
    }
  } else {
    // ------------------------------------------------ elementwise + epilogue
    const int q4 = warp & 3;
    const int hf = warp >> 2;
    const int row = q4 * 32 + lane;  // stationary row = TMEM lane
    const int c0 = hf * 64;          // first streamed column of this warp
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int etid = threadIdx.x;    // 0 .. 255
    const float LOG2E = 1.4426950408889634f;
    const uint64_t sl2 = f2_pack(p.scale_log2, p.scale_log2);
    const int64_t my_pos = spos0 + row;
    const int64_t my_tok = it.stat.stripe + stride * (srow0 + row);  // gradient row, LSE column
    // dQ: this row's -LSE (log2) and delta; a row without keys gets -inf so
    // that every p = 2^(s - inf) = 0
    uint64_t nl2 = 0;
    float my_dl = 0.f;
    if (!kDKDV) {
      float l = -CUDART_INF_F;
      if (row < nstat && in_bounds) {
        const float v = p.lse[static_cast<int64_t>(shead) * p.ld + my_tok];
        l = v == -CUDART_INF_F ? -CUDART_INF_F : -v * LOG2E;
        my_dl = p.delta[static_cast<int64_t>(shead) * p.ld + my_tok];
      }
      nl2 = f2_pack(l, l);
    }
    const uint64_t ndl_row = f2_pack(-my_dl, -my_dl);
    bool ok = true;
    auto ewait = [&](int b, uint32_t parity) {
      if (!ok) return false;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(b), parity, bw::WAIT_LIMIT_NS, abort_flag));
      if (!ok) bw_timeout(dev_err, abort_flag);
      return ok;
    };
    // dK/dV: the per-column -LSE (log2) and delta of a streamed tile, one
    // value per elementwise thread (threads 0-127: -LSE of column t, 128-255:
    // delta of column t - 128), loaded one tile ahead
    const int ccol = etid & (bw::BN - 1);
    const bool is_l = etid < bw::BN;
    // cursors of the tile loop and of the column loads (one tile ahead)
    BwCursor<kDKDV, kStriped> cc, lc;
    cc.init(it, p, lim, causal);
    lc = cc;
    // the next tile's column value; called for tiles 0, 1, ... in order
    auto col_load = [&]() -> float {
      int64_t trow, tpos;
      int tn, tstripe, qh;
      str_tile(lc, trow, tpos, tn, tstripe, qh);
      if (ccol >= tn) return is_l ? CUDART_INF_F : 0.f;
      const int64_t tok = tstripe + stride * (trow + ccol);
      if (kDebugBounds && !bounds_ok(tok >= 0 && tok < p.ld && qh < p.H, dev_err, kSiteBwdStr))
        return is_l ? CUDART_INF_F : 0.f;
      return (is_l ? p.lse : p.delta)[static_cast<int64_t>(qh) * p.ld + tok];
    };
    float col_next = (kDKDV && nstr > 0) ? col_load() : 0.f;
    for (int j = 0; j < nstr; ++j) {
      int64_t trow, tpos;
      int tn, tstripe, qh;
      str_tile(cc, trow, tpos, tn, tstripe, qh);
      float* cnl = cols + (j & 1) * 2 * bw::BN;  // dK/dV: per-column -LSE (log2)
      float* cdl = cnl + bw::BN;                 //        and delta
      if (kDKDV) {
        // every elementwise thread passes this barrier on every tile; slot
        // j & 1 was last read in tile j - 2, before the barrier of tile j - 1
        const float x = col_next;
        (is_l ? cnl : cdl)[ccol] =
            is_l ? ((x == -CUDART_INF_F || x == CUDART_INF_F) ? -CUDART_INF_F : -x * LOG2E) : x;
        named_bar_sync(1, bw::EW_THREADS);
        if (j + 1 < nstr) col_next = col_load();
      }
      // visibility: key pos <= query pos, streamed index < tn; the visible
      // columns of this row are [c_lo, c_hi)
      const bool full =
          tn == bw::BN &&
          (!causal || (kDKDV ? spos0 + bw::BM - 1 <= tpos : tpos + bw::BN - 1 <= spos0));
      int c_lo = 0, c_hi = tn;
      if (causal && !full) {
        if (!kDKDV)
          c_hi = static_cast<int>(
              min(static_cast<int64_t>(tn), max(my_pos - tpos + 1, int64_t(0))));
        else
          c_lo = static_cast<int>(min(static_cast<int64_t>(tn), max(my_pos - tpos, int64_t(0))));
      }
      // ---- phase 1: P = 2^(s * scale * log2e - lse * log2e), masked
      uint64_t pv[32];  // P of columns c0 .. c0+63, packed pairs
      if (!ewait(bw::BAR_S, j & 1)) continue;
      tc_fence_after();
      // dK/dV: tile j's S^T (then P^T, dS^T) in cs, dP^T in cd, swapping
      // every tile; dQ: S in X, dP in Y0 / Y1
      const uint32_t cs = (kDKDV && (j & 1)) ? COL_Y : COL_X;
      {
        uint32_t sa[32], sb[32];
        tmem_ld32(tmem + lane_off + cs + c0, sa);
        tmem_ld32(tmem + lane_off + cs + c0 + 32, sb);
        tmem_wait_ld();
        reg_dep(sa);
        reg_dep(sb);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t* src = i < 16 ? sa : sb;
          const int k = (i & 15) * 2;
          const uint64_t s2 = f2_pack(__uint_as_float(src[k]), __uint_as_float(src[k + 1]));
          uint64_t nl = nl2;
          if (kDKDV) {
            const float4 x = *reinterpret_cast<const float4*>(cnl + c0 + 4 * (i >> 1));
            nl = (i & 1) ? f2_pack(x.z, x.w) : f2_pack(x.x, x.y);
          }
          float e0, e1;
          f2_unpack(f2_fma(s2, sl2, nl), e0, e1);
          e0 = ex2_approx(e0);
          e1 = ex2_approx(e1);
          if (!full) {
            const int cc = c0 + 2 * i;
            if (cc < c_lo || cc >= c_hi) e0 = 0.f;
            if (cc + 1 < c_lo || cc + 1 >= c_hi) e1 = 0.f;
          }
          pv[i] = f2_pack(e0, e1);
        }
      }
      if (!kDKDV) {
        tc_fence_before();
        mbar_arrive(bar(bw::BAR_XFREE));  // X read: S(j+1) may overwrite it
      } else {
        // P^T as bf16 pairs over the first 32 of this warp's (already read)
        // S^T columns of buffer cs; dV(j) takes it from there
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float a0, a1;
          f2_unpack(pv[i], a0, a1);
          pk[i] = pack_bf16x2(a0, a1);
        }
        __syncwarp();
        tmem_st32(tmem + lane_off + cs + (hf ? 64 : 0), pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(bw::BAR_E1));
      }
      // ---- phase 2: dS = P (dP - delta) as bf16: dQ over the dP buffer,
      // dK/dV over the other 32 S^T columns of X (Y is released once read)
      const int yb = kDKDV ? 0 : (j & 1);
      if (!ewait(bw::BAR_DP + yb, kDKDV ? (j & 1) : ((j >> 1) & 1))) continue;
      tc_fence_after();
      {
        const uint32_t ycol = kDKDV ? ((j & 1) ? COL_X : COL_Y) : COL_Y + yb * 128;
        uint32_t da[32], db[32];
        tmem_ld32(tmem + lane_off + ycol + c0, da);
        tmem_ld32(tmem + lane_off + ycol + c0 + 32, db);
        tmem_wait_ld();
        reg_dep(da);
        reg_dep(db);
        if (kDKDV) {
          tc_fence_before();
          mbar_arrive(bar(bw::BAR_XFREE));  // dP^T read: S^T(j+1) may overwrite it
        }
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t* src = i < 16 ? da : db;
          const int k = (i & 15) * 2;
          uint64_t nd = ndl_row;
          if (kDKDV) {
            const float4 x = *reinterpret_cast<const float4*>(cdl + c0 + 4 * (i >> 1));
            nd = (i & 1) ? f2_pack(-x.z, -x.w) : f2_pack(-x.x, -x.y);
          }
          const uint64_t d2 = f2_pack(__uint_as_float(src[k]), __uint_as_float(src[k + 1]));
          float g0, g1;
          f2_unpack(f2_mul(pv[i], f2_add(d2, nd)), g0, g1);
          pk[i] = pack_bf16x2(g0, g1);
        }
        __syncwarp();
        tmem_st32(tmem + lane_off + (kDKDV ? cs + 32 : ycol) + (hf ? 64 : 0), pk);
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(bar(bw::BAR_E2 + yb));
    }

    // ---------------------------------------------------- epilogue
    bool have = ok && nstr > 0;
    if (have) {
      have = ewait(bw::BAR_DONE, 0);
      tc_fence_after();
    }
    const bool accumulate = (it.flags & kBwdAccumulate) != 0;
    const bool final_out = (it.flags & kBwdFinal) != 0;
    const int nheads = kDKDV ? p.Hkv : p.H;
    if (ok && in_bounds) {
      // The accumulators pass through shared memory (the streamed rings,
      // idle once every MMA is done) so that global memory is read and
      // written 256 bytes of a row per half-warp instruction; thread = row
      // would touch 32 rows (32 cache lines) per instruction.  Warp (q4, hf)
      // owns rows 32 q4 .. +31, columns c0 .. +63 of the staging.
      constexpr int NACC = kDKDV ? 2 : 1;
      constexpr uint32_t PITCH = bw::STG_PITCH;
      const int wrow0 = q4 * 32;
      const int sub = lane >> 4;               // two rows per warp instruction
      const int cl = c0 + 4 * (lane & 15);     // this lane's four columns
      auto gel_of = [&](int rr) -> int64_t {   // stationary row -> gradient element
        const int64_t tok = it.stat.stripe + stride * (srow0 + rr);
        return (tok * nheads + shead) * static_cast<int64_t>(bw::HD);
      };
      float* stg = reinterpret_cast<float*>(smem + L::STR);
      // one accumulator at a time (dQ kernel: a = 0 dQ, scaled; dK/dV
      // kernel: a = 0 dV, a = 1 dK, scaled), through the same staging
#pragma unroll 1
      for (int a = 0; a < NACC; ++a) {
        const float mul = (!kDKDV || a == 1) ? p.scale : 1.f;
        const uint32_t acol = a == 0 ? COL_A0 : COL_A1;
        float* accb = a == 0 ? p.acc0 : p.acc1;
        void* outp = a == 0 ? p.out0 : p.out1;
        __syncwarp();  // the previous accumulator's rows are stored
        if (accumulate) {
          for (int i = 0; i < 16; ++i) {
            const int rr = wrow0 + 2 * i + sub;
            if (rr < nstat) cp_async16(smem_u32(stg + rr * PITCH + cl), accb + gel_of(rr) + cl);
          }
          cp_async_wait_all();
          __syncwarp();
        }
        // thread = row: the TMEM accumulator (scaled) (+ the staged one)
        float* srow = stg + row * PITCH + c0;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          __syncwarp();
          if (have) {
            tmem_ld32(tmem + lane_off + acol + c0 + 32 * c, o);
            tmem_wait_ld();
            reg_dep(o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4* d4 = reinterpret_cast<float4*>(srow + 32 * c + 4 * i);
            float4 r = make_float4(
                __uint_as_float(o[4 * i]) * mul, __uint_as_float(o[4 * i + 1]) * mul,
                __uint_as_float(o[4 * i + 2]) * mul, __uint_as_float(o[4 * i + 3]) * mul);
            if (accumulate) {
              const float4 x = *d4;
              r.x += x.x;
              r.y += x.y;
              r.z += x.z;
              r.w += x.w;
            }
            *d4 = r;
          }
        }
        __syncwarp();
        // rows back to the fp32 buffer, or finished to the output in out_dt;
        // eight rows' shared-memory reads ahead of their stores
#pragma unroll
        for (int i0 = 0; i0 < 16; i0 += 8) {
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            v[u] = *reinterpret_cast<const float4*>(stg + (wrow0 + 2 * (i0 + u) + sub) * PITCH +
                                                    cl);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int rr = wrow0 + 2 * (i0 + u) + sub;
            if (rr >= nstat) continue;
            const int64_t el = gel_of(rr) + cl;
            if (final_out && p.out_dt == 1)
              *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(outp) + el) =
                  make_uint2(pack_bf16x2(v[u].x, v[u].y), pack_bf16x2(v[u].z, v[u].w));
            else
              *reinterpret_cast<float4*>((final_out ? reinterpret_cast<float*>(outp) : accb) + el) =
                  v[u];
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == bw::WARP_MMA) tmem_dealloc(tmem, bw::TMEM_COLS);
}

// CTAs of one item: stationary tiles x heads (query heads for dQ, KV heads
// for dK/dV).
int attn_bwd_ctas(const BwdItem& it, int heads) {
  return (it.stat.len + bw::BM - 1) / bw::BM * heads;
}

template <bool kDKDV, bool kStriped>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                                int ctas, int* dev_err, cudaStream_t stream) {
  constexpr uint32_t bytes = bw::Smem<kDKDV>::BYTES;
  // the shared-memory attribute is a property of the function on each device
  static PerDeviceOnce attr_once;
  const cudaError_t e = once_per_device(attr_once, [] {
    return cudaFuncSetAttribute(attn_bwd_tc_kernel<kDKDV, kStriped>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes));
  });
  if (e != cudaSuccess) return e;
  attn_bwd_tc_kernel<kDKDV, kStriped><<<ctas, bw::THREADS, bytes, stream>>>(tq, tk, tv, tdo, p,
                                                                           dev_err);
  return cudaGetLastError();
}

// dkdv selects the kernel; maps are 4-D when p.stride > 1.
cudaError_t launch_attn_bwd(bool dkdv, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                            int ctas, int* dev_err, cudaStream_t stream) {
  const bool striped = p.stride > 1;
  if (dkdv)
    return striped ? launch_bwd_t<true, true>(tq, tk, tv, tdo, p, ctas, dev_err, stream)
                   : launch_bwd_t<true, false>(tq, tk, tv, tdo, p, ctas, dev_err, stream);
  return striped ? launch_bwd_t<false, true>(tq, tk, tv, tdo, p, ctas, dev_err, stream)
                 : launch_bwd_t<false, false>(tq, tk, tv, tdo, p, ctas, dev_err, stream);
}

}  // namespace cpattn
