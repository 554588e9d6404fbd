// Causal block attention with global offsets, per-row LSE and a fused LSE
// merge epilogue, on the sm_100-family tensor cores (tcgen05 + TMEM + TMA).
//
// What it computes ([CP-handbook] "上下文并行：Ring Attention 与 Ulysses",
// section "哪些运算可以直接切", the attention helper with offsets, and the
// merge from the self-test answers / section "Ring Attention：KV 沿环传一圈"):
// for each query row i of a work item and each head h,
//   s_j   = scale * q_i . k_j           over the item's key segments,
//   mask  k_pos(j) > q_pos(i)           (causal items),
//   lse_i = log sum_j e^{s_j},   o_i = sum_j e^{s_j - lse_i} v_j,
// then either writes (o_i, lse_i) or merges them into an accumulator with
//   lse = logaddexp(lse_acc, lse_i), o = o_acc e^{lse_acc-lse} + o_i e^{lse_i-lse}.
//
// Design (GB300-first, not the pages' FlashAttention/TE kernels):
//  * one CTA = one query tile of 128 rows of one head; two CTAs share each
//    SM, so one CTA's prologue and epilogue overlap the other's main loop and
//    the two CTAs' S -> softmax -> PV chains interleave on the tensor pipe;
//    BN = 128 keys per tile; D = 128.  (The code keeps a parameter NT for
//    query tiles per CTA; only NT = 1 is built: two tiles per CTA measured
//    slower, and the staged epilogue reuses the Q and K/V buffers that a
//    second tile could still be reading.)
//  * warp 4: TMA producer (Q once, then K_j, V_j through a ring of two 32 KB
//    stages, 128-byte swizzle, two 64-column boxes per tile).
//  * warp 5: TMEM allocator and single-thread tcgen05.mma issuer:
//      S = Q K_j^T   (SS form, both operands K-major in shared memory)
//      O += P V_j    (TS form: P read from TMEM, V MN-major in smem)
//  * warps 0-3: softmax; thread = one query row = one TMEM lane.  fp32
//    online softmax in the log2 domain with a lazy rescale: the running max
//    used for exponentiation only moves when the row max grows by more than
//    2^8, so O in TMEM is rarely touched; the final normalisation uses the
//    same max, so the result is exact.  P is written back as bf16 over the
//    first 64 columns of S.
//  * TMEM (256 columns): S at [0, 128), O at [128, 256).
//  * epilogue: each row's O/l (merged with the accumulator) is staged in
//    shared memory over the then idle Q and K/V buffers, so that the
//    accumulator is read and the result written a whole 512-byte row per
//    warp instruction rather than 32 rows (32 cache lines) per instruction.
//  * fully masked KV tiles are never loaded or computed; only tiles that
//    straddle the diagonal (or a ragged segment end) apply the element mask.
//  * every wait is bounded; on expiry the CTA records a status word, lets
//    in-flight copies and MMAs finish, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "attn_fwd_common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {

using namespace sm100;

namespace tc {
// NT query tiles per CTA (built: NT = 1, two CTAs per SM with 256 TMEM
// columns and a 2-stage ring each; NT = 2 would own the SM with 512 columns
// and a 4-stage ring).
template <int NT>
struct Cfg {
  static constexpr int STAGES = NT == 2 ? 4 : 2;
  static constexpr int THREADS = NT * 128 + 64;
  static constexpr int WARP_LOAD = NT * 4;
  static constexpr int WARP_MMA = NT * 4 + 1;
  static constexpr int MIN_BLOCKS = NT == 2 ? 1 : 2;
  static constexpr uint32_t TMEM_COLS = NT * 256;
  static constexpr uint32_t COL_O = NT * BN;  // O_X at COL_O + x * HD; S_X at x * BN
  // shared memory map (offsets from a 1024-byte aligned base)
  static constexpr uint32_t OFF_Q = 0;                              // NT tiles
  static constexpr uint32_t OFF_KV = OFF_Q + NT * TILE_BYTES;       // STAGES tiles
  static constexpr uint32_t OFF_BAR = OFF_KV + STAGES * TILE_BYTES;  // mbarriers
  static constexpr int BAR_Q = 0;
  static constexpr int BAR_KV_FULL = 1;  // + stage
  static constexpr int BAR_KV_EMPTY = BAR_KV_FULL + STAGES;
  static constexpr int BAR_S_FULL = BAR_KV_EMPTY + STAGES;  // + tile
  static constexpr int BAR_P_FULL = BAR_S_FULL + 2;
  static constexpr int BAR_O_DONE = BAR_P_FULL + 2;
  static constexpr int BAR_DRAIN = BAR_O_DONE + 2;
  static constexpr int NUM_BARS = BAR_DRAIN + 1;
  static constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;
  static constexpr uint32_t OFF_LSE = (OFF_ABORT + 4 + 15) / 16 * 16;  // 128 floats
  static constexpr uint32_t SMEM_USED = OFF_LSE + 128 * 4;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // alignment slack
  // Epilogue staging: 128 rows of 512 bytes over the Q buffer and K/V stage 0,
  // both free once the last S MMA is done (K_j always sits in stage 0), so
  // the merge's accumulator rows are fetched while the last PV runs.  16-byte
  // chunk c of row r sits at chunk c ^ (r & 7): the row-per-thread and the
  // row-per-warp accesses are both free of bank conflicts.
  static constexpr uint32_t STG_BYTES = 128 * 512;
  static_assert(OFF_Q == 0 && OFF_KV + TILE_BYTES == STG_BYTES && STAGES == 2,
                "staging = Q + K/V stage 0");
};
}  // namespace tc

// kStriped: rows are addressed as stripes (4-D maps, strided output rows);
// otherwise plain rows with 3-D maps, and those terms fold away.
template <bool kStriped, int NT>
__global__ void __launch_bounds__(tc::Cfg<NT>::THREADS, tc::Cfg<NT>::MIN_BLOCKS)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ AttnParams p, int* dev_err) {
  using C = tc::Cfg<NT>;
  // The staged epilogue reuses the Q and K/V buffers, which with two tiles
  // per CTA the other tile could still be reading.
  static_assert(NT == 1, "one query tile per CTA");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sKV = sbase + C::OFF_KV;
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The next ring step may be launched as a programmatic dependent: its CTAs
  // start as this grid's last ones run and wait for it only before their
  // epilogue (everything before reads only q, k, v).
  if (threadIdx.x == 0) grid_launch_dependents();

  // ---------------------------------------------------------- task decode
  int ii = 0, pair, local;
  const WorkItem* itp;
  if (p.head_major) {
    // tile rank r of a head: the items in order, later query tiles first.
    // Ranks [0, hm_long) head by head, then the rest rank by rank across
    // the heads (the grid is tiles x heads x batch CTAs).
    const int tiles = p.tile_start[p.nitems];
    const int nh = static_cast<int>(gridDim.x) / tiles;
    const int lead = p.hm_long * nh;
    const int g = static_cast<int>(blockIdx.x);
    int r;
    if (g < lead) {
      r = g % p.hm_long;
      local = g / p.hm_long;
    } else {
      r = p.hm_long + (g - lead) / nh;
      local = (g - lead) % nh;
    }
    ii = last_at_most(p.tile_start, p.nitems, r);
    itp = &p.items[ii];
    const int npairs = (itp->sq + NT * tc::BM - 1) / (NT * tc::BM);
    pair = npairs - 1 - (r - p.tile_start[ii]);
  } else {
    ii = last_at_most(p.cta_start, p.nitems, static_cast<int>(blockIdx.x));
    itp = &p.items[ii];
    local = static_cast<int>(blockIdx.x) - p.cta_start[ii];
    const int npairs = (itp->sq + NT * tc::BM - 1) / (NT * tc::BM);
    // query-tile groups vary fastest: the CTAs resident at one time share a
    // head (and its K/V), which then stays in L2
    pair = npairs - 1 - local % npairs;  // later query rows (more keys) first
    local /= npairs;
  }
  const WorkItem& it = *itp;
  const int head = local % p.H;
  const int b = local / p.H;
  const int row0 = pair * NT * tc::BM;
  const int kvh = (b * p.b_q_heads + head) / p.kv_group;
  const bool causal = (it.flags & kFlagCausal) != 0;
  const int64_t q_mem0 = it.q_mem_row + static_cast<int64_t>(b) * it.b_q_rows + row0;
  const int64_t q_pos0 = it.q_pos + row0;
  const int64_t k_boff = static_cast<int64_t>(b) * it.b_k_rows;
  const int nrows_a = min(tc::BM, it.sq - row0);
  const int nrows_b = NT == 2 ? max(0, min(tc::BM, it.sq - row0 - tc::BM)) : 0;
  const int n_a = visible_tiles<kStriped>(it, p, q_pos0 + nrows_a - 1, causal);
  const int n_b =
      nrows_b > 0 ? visible_tiles<kStriped>(it, p, q_pos0 + tc::BM + nrows_b - 1, causal) : 0;
  const int nkv = max(n_a, n_b);
  // Bounds-checked build: the tile's q rows, out / acc rows and lse columns
  // lie inside their tensors (out has the rows of q); a tile that fails is
  // recorded and skips its global reads and writes.
  bool in_bounds = true;
  if (kDebugBounds) {
    const int nr = nrows_a + nrows_b;
    const int64_t os = kStriped ? it.o_stride : 1;
    const int64_t o0 =
        it.o_row + static_cast<int64_t>(b) * it.b_o_rows + static_cast<int64_t>(row0) * os;
    const int64_t c0 = it.lse_col + static_cast<int64_t>(row0) * os;
    const int64_t lh = static_cast<int64_t>(head) + static_cast<int64_t>(b) * it.b_lse_heads;
    in_bounds = nr > 0 && q_mem0 >= 0 && q_mem0 + nr <= p.q_rows / p.stripe &&
                it.q_stripe >= 0 && it.q_stripe < p.stripe && kvh >= 0 && kvh < p.Hkv &&
                o0 >= 0 && o0 + (nr - 1) * os < p.q_rows &&
                lh < static_cast<int64_t>(p.H) * it.batch && c0 >= 0 &&
                c0 + (nr - 1) * os < p.ld_lse;
    if (threadIdx.x == 0) bounds_ok(in_bounds, dev_err, kSiteFwdTile);
  }

  // ---------------------------------------------------------------- setup
  // The producer thread initialises the barriers and starts the Q and first
  // K/V copies before the CTA-wide sync, so that they overlap the TMEM
  // allocation and the sync (the first K/V stages are empty: no wait).
  const bool producer = warp == C::WARP_LOAD && lane == 0;
  uint64_t pol_q = 0, pol_kv = 0;
  int issued = 0;  // producer: K/V copies issued
  TileCursor<kStriped> pcur;  // producer: the next tile to load
  // K_j and V_j into the next stages (n = 2 j + w), each once its stage is
  // released; false when a wait expired.  Called for j = 0, 1, ... in order.
  auto issue_kv = [&](int j) -> bool {
    int64_t kmem, kpos;
    int nk, kstripe;
    pcur.keys(it, p, kmem, kpos, nk, kstripe);
    pcur.next(it, p, q_pos0 + nrows_a - 1, causal);
    if (!kStriped) kstripe = 0;
    const int krow = static_cast<int>(kmem + k_boff);
    // (a copy outside the tensor would only read the fill value)
    if (kDebugBounds)
      bounds_ok(kmem + k_boff >= 0 && kmem + k_boff + nk <= p.k_rows / p.kv_stripe &&
                    kstripe >= 0 && kstripe < p.kv_stripe,
                dev_err, kSiteFwdKV);
    for (int w = 0; w < 2; ++w) {
      const int n = 2 * j + w;
      const int st = n % C::STAGES;
      const uint32_t ph = (n / C::STAGES) & 1;
      if (!mbar_wait(bar(C::BAR_KV_EMPTY + st), ph ^ 1, tc::WAIT_LIMIT_NS, abort_flag)) {
        record_timeout(dev_err, abort_flag);
        return false;
      }
      mbar_arrive_expect_tx(bar(C::BAR_KV_FULL + st), tc::TILE_BYTES);
      const CUtensorMap* tm = w == 0 ? &tm_k : &tm_v;
      for (int hh = 0; hh < 2; ++hh)
        if (kStriped)
          tma_load_4d(sKV + st * tc::TILE_BYTES + hh * tc::BOX_BYTES, tm, bar(C::BAR_KV_FULL + st),
                      hh * 64, kvh, kstripe, krow, pol_kv);
        else
          tma_load_3d(sKV + st * tc::TILE_BYTES + hh * tc::BOX_BYTES, tm, bar(C::BAR_KV_FULL + st),
                      hh * 64, kvh, krow, pol_kv);
      ++issued;
    }
    return true;
  };
  if (producer) {
    *abort_flag = 0;
    mbar_init(bar(C::BAR_Q), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::BAR_KV_FULL + s), 1);
      mbar_init(bar(C::BAR_KV_EMPTY + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::BAR_S_FULL + x), 1);
      mbar_init(bar(C::BAR_P_FULL + x), tc::BM);
      mbar_init(bar(C::BAR_O_DONE + x), 1);
    }
    mbar_init(bar(C::BAR_DRAIN), 1);
    fence_mbar_init();
    fence_proxy_async_smem();  // the copies below complete on these barriers
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    pol_q = policy_evict_first();
    pol_kv = policy_evict_last();
    pcur.init(it, p, q_pos0 + nrows_a - 1, causal);
    const int ntiles_q = nrows_b > 0 ? 2 : 1;
    mbar_arrive_expect_tx(bar(C::BAR_Q), ntiles_q * tc::TILE_BYTES);
    for (int x = 0; x < ntiles_q; ++x)
      for (int hh = 0; hh < 2; ++hh)
        if (kStriped)
          tma_load_4d(sQ + x * tc::TILE_BYTES + hh * tc::BOX_BYTES, &tm_q, bar(C::BAR_Q), hh * 64,
                      head, it.q_stripe, static_cast<int>(q_mem0 + x * tc::BM), pol_q);
        else
          tma_load_3d(sQ + x * tc::TILE_BYTES + hh * tc::BOX_BYTES, &tm_q, bar(C::BAR_Q), hh * 64,
                      head, static_cast<int>(q_mem0 + x * tc::BM), pol_q);
    if (nkv > 0) issue_kv(0);
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::WARP_LOAD) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      // The merge epilogue reads this task's accumulator rows and LSE: pull
      // them into L2 a few KV tiles before the end so the reads hit L2.
      const bool merge = (it.flags & kFlagMerge) != 0;
      const int prefetch_at = max(0, nkv - 4);
      const int64_t ostride = kStriped ? it.o_stride : 1;
      auto prefetch_acc = [&]() {
        const int nrows = nrows_a + nrows_b;
        const int64_t orow0 =
            it.o_row + static_cast<int64_t>(b) * it.b_o_rows + static_cast<int64_t>(row0) * ostride;
        for (int r = 0; r < nrows; ++r)
          prefetch_l2(p.acc + ((orow0 + static_cast<int64_t>(r) * ostride) * p.H + head) *
                                  static_cast<int64_t>(tc::HD),
                      tc::HD * 4);
        if (ostride == 1) {
          const float* l0 =
              p.lse +
              (static_cast<int64_t>(head) + static_cast<int64_t>(b) * it.b_lse_heads) * p.ld_lse +
              it.lse_col + row0;
          const uintptr_t a0 = reinterpret_cast<uintptr_t>(l0) & ~static_cast<uintptr_t>(15);
          const uintptr_t a1 =
              (reinterpret_cast<uintptr_t>(l0 + nrows) + 15) & ~static_cast<uintptr_t>(15);
          prefetch_l2(reinterpret_cast<const void*>(a0), static_cast<uint32_t>(a1 - a0));
        }
      };
      // tile 0 was issued before the sync
      if (merge && in_bounds && nkv > 0 && prefetch_at == 0) prefetch_acc();
      for (int j = 1; j < nkv; ++j) {
        if (merge && in_bounds && j == prefetch_at) prefetch_acc();
        if (!issue_kv(j)) break;
      }
      // let every copy this thread issued land before the CTA can exit
      mbar_wait(bar(C::BAR_Q), 0, tc::WAIT_LIMIT_NS, nullptr);
      for (int n = max(0, issued - C::STAGES); n < issued; ++n)
        mbar_wait(bar(C::BAR_KV_FULL + n % C::STAGES), (n / C::STAGES) & 1, tc::WAIT_LIMIT_NS,
                  nullptr);
    }
  } else if (warp == C::WARP_MMA) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(tc::BM, tc::BN, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(tc::BM, tc::HD, true);
      bool ok = mbar_wait(bar(C::BAR_Q), 0, tc::WAIT_LIMIT_NS, abort_flag);
      tc_fence_after();
      // S_X = Q_X K_j^T into the S columns of tile X
      auto issue_s = [&](int x, uint32_t k_s) {
        const uint32_t q_s = sQ + x * tc::TILE_BYTES;
        const uint32_t d_tm = tmem + x * tc::BN;  // S_X
#pragma unroll
        for (int kk = 0; kk < tc::HD / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * tc::BOX_BYTES + (kk & 3) * 32;
          mma_ss(d_tm, sdesc_sw128(q_s + koff, 16, 1024), sdesc_sw128(k_s + koff, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(C::BAR_S_FULL + x));
      };
      // O_X += P_X V_j, P_X read from TMEM, 16 keys = two 8-row groups of V
      auto issue_pv = [&](int x, uint32_t v_s, bool acc) {
        const uint32_t p_tm = tmem + x * tc::BN;
        const uint32_t o_tm = tmem + C::COL_O + x * tc::HD;
#pragma unroll
        for (int kk = 0; kk < tc::BN / 16; ++kk)
          mma_ts(o_tm, p_tm + kk * 8, sdesc_sw128(v_s + kk * 2048, tc::BOX_BYTES, 1024), idesc_o,
                 (acc || kk > 0) ? 1u : 0u);
        mma_commit(bar(C::BAR_O_DONE + x));
      };
      auto wait_stage = [&](int n) -> bool {
        if (!mbar_wait(bar(C::BAR_KV_FULL + n % C::STAGES), (n / C::STAGES) & 1,
                       tc::WAIT_LIMIT_NS, abort_flag))
          return false;
        tc_fence_after();
        return true;
      };
      if (ok && nkv > 0) {
        ok = wait_stage(0);
        if (ok) {
          if (n_a > 0) issue_s(0, sKV);
          if (n_b > 0) issue_s(1, sKV);
          mma_commit(bar(C::BAR_KV_EMPTY + 0));
        }
      }
      for (int j = 0; ok && j < nkv; ++j) {
        const int nv = 2 * j + 1, nk = 2 * j + 2;
        const uint32_t v_s = sKV + (nv % C::STAGES) * tc::TILE_BYTES;
        const uint32_t k_s = sKV + (nk % C::STAGES) * tc::TILE_BYTES;
        if (!(ok = wait_stage(nv))) break;
        bool k_ready = false;
        // both PVs back to back, then each S once its own PV has completed
        // (P_X lives in S_X's columns): the tensor pipe always holds the next
        // group while this thread waits
        for (int x = 0; x < NT && ok; ++x) {
          if (j >= (x == 0 ? n_a : n_b)) continue;
          if (!(ok = mbar_wait(bar(C::BAR_P_FULL + x), j & 1, tc::WAIT_LIMIT_NS, abort_flag)))
            break;
          tc_fence_after();
          issue_pv(x, v_s, j > 0);
        }
        for (int x = 0; x < NT && ok; ++x) {
          if (j + 1 >= (x == 0 ? n_a : n_b)) continue;
          if (!k_ready) {
            if (!(ok = wait_stage(nk))) break;
            k_ready = true;
          }
          if (!(ok = mbar_wait(bar(C::BAR_O_DONE + x), j & 1, tc::WAIT_LIMIT_NS, abort_flag)))
            break;
          tc_fence_after();
          issue_s(x, k_s);
        }
        if (!ok) break;
        mma_commit(bar(C::BAR_KV_EMPTY + nv % C::STAGES));
        if (j + 1 < nkv) {
          if (!k_ready && !(ok = wait_stage(nk))) break;  // K_{j+1} unused: release anyway
          mma_commit(bar(C::BAR_KV_EMPTY + nk % C::STAGES));
        }
      }
      if (!ok) record_timeout(dev_err, abort_flag);
      // no MMA may be in flight when TMEM is released
      mma_commit(bar(C::BAR_DRAIN));
      mbar_wait(bar(C::BAR_DRAIN), 0, tc::WAIT_LIMIT_NS, nullptr);
    }
  } else {
    // ------------------------------------------------ softmax + epilogue
    const int x = warp >> 2;       // query tile
    const int quad = warp & 3;     // TMEM lane quadrant
    const int row = quad * 32 + lane;
    const int nrows = x == 0 ? nrows_a : nrows_b;
    const int nx = x == 0 ? n_a : n_b;
    if (nrows > 0) {
      const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
      const uint32_t t_s = tmem + lane_off + x * tc::BN;
      const uint32_t t_o = tmem + lane_off + C::COL_O + x * tc::HD;
      const int64_t qp_first = q_pos0 + x * tc::BM;
      const int64_t qp = qp_first + row;
      const float sl2 = p.scale_log2;
      float m_used = -CUDART_INF_F;  // log2-domain max used as exponent base
      float l = 0.f;
      bool ok = true;
      const bool merge = (it.flags & kFlagMerge) != 0;
      const int64_t ostride = kStriped ? it.o_stride : 1;
      // element of acc / out of tile row 0 and the step between rows
      auto out_el0 = [&]() -> int64_t {
        return ((it.o_row + static_cast<int64_t>(b) * it.b_o_rows + (row0 + x * tc::BM) * ostride) *
                    p.H + head) * static_cast<int64_t>(tc::HD);
      };
      auto out_step = [&]() -> int64_t { return ostride * p.H * static_cast<int64_t>(tc::HD); };
      auto lse_addr = [&]() -> float* {  // this thread's row of lse (recomputed, not held)
        return p.lse +
               (static_cast<int64_t>(head) + static_cast<int64_t>(b) * it.b_lse_heads) * p.ld_lse +
               it.lse_col + (row0 + x * tc::BM + row) * ostride;
      };
      // The merge's reads, into shared memory: this warp's 32 accumulator
      // rows (a whole 512-byte row per warp instruction) and each thread's
      // LSE.  They may be written by the grid launched before this one (the
      // previous ring step), hence the wait.
      auto fetch_acc = [&]() {
        grid_wait_prerequisites();
        const int64_t el0 = out_el0(), stp = out_step();
        const int wrow0 = quad * 32;
        const int nw = min(32, nrows - wrow0);
        for (int i = 0; i < nw; ++i) {
          const int rr = wrow0 + i;
          cp_async16(sbase + C::OFF_Q + rr * 512 + ((lane ^ (rr & 7)) << 4),
                     p.acc + el0 + rr * stp + 4 * lane);
        }
        if (row < nrows) cp_async4(sbase + C::OFF_LSE + row * 4, lse_addr());
      };
      TileCursor<kStriped> cur;
      cur.init(it, p, qp_first + nrows - 1, causal);
      for (int j = 0; j < nx; ++j) {
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar(C::BAR_S_FULL + x), j & 1,
                                                           tc::WAIT_LIMIT_NS, abort_flag));
        if (!got) {
          record_timeout(dev_err, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, sr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_dep(sr[c]);
        float s[tc::BN];
#pragma unroll
        for (int c = 0; c < tc::BN; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);

        int64_t kmem, kpos;
        int nk, kstripe;
        cur.keys(it, p, kmem, kpos, nk, kstripe);
        cur.next(it, p, qp_first + nrows - 1, causal);
        const bool need_mask = nk < tc::BN || (causal && kpos + nk - 1 > qp_first);
        if (need_mask) {
          int64_t lim64 = causal ? min(static_cast<int64_t>(nk), qp - kpos + 1)
                                 : static_cast<int64_t>(nk);
          const int lim = static_cast<int>(max(lim64, static_cast<int64_t>(0)));
#pragma unroll
          for (int c = 0; c < tc::BN; ++c)
            if (c >= lim) s[c] = -CUDART_INF_F;
        }
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = s[i];
#pragma unroll
        for (int c = 8; c < tc::BN; ++c) m8[c & 7] = fmaxf(m8[c & 7], s[c]);
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        // the exponent base moves only when the row max grows by more than
        // the threshold; the rescale factor is derived after the
        // exponentials, so that only m_prev stays live across them
        const float m_new = fmaxf(m_used, mx * sl2);
        const float m_prev = m_used;
        if (m_new > m_used + tc::RESCALE_THRESHOLD) m_used = m_new;
        const float base = m_used == -CUDART_INF_F ? 0.f : m_used;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nbx2 = f2_pack(-base, -base);
        uint64_t rs2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
        __syncwarp();
        // P = 2^(s*scale_log2 - base) as bf16 pairs over the first 64 columns
        // of S, stored 32 keys at a time so the fp32 row dies as it goes;
        // the scale-subtract and the row sum run two keys per instruction
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), sl2x2, nbx2), x0,
                      x1);
            const float e0 = ex2_approx(x0);
            const float e1 = ex2_approx(x1);
            rs2[i & 1] = f2_add(rs2[i & 1], f2_pack(e0, e1));
            pk[i] = pack_bf16x2(e0, e1);
          }
          tmem_st16(t_s + 16 * c, pk);
        }
        float rs4[4];
        f2_unpack(rs2[0], rs4[0], rs4[1]);
        f2_unpack(rs2[1], rs4[2], rs4[3]);
        const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        const bool grow = m_used != m_prev;  // m_used is never NaN
        const float alpha = grow ? ex2_approx(m_prev - m_used) : 1.f;
        l = fmaf(l, alpha, rs);
        // rescale O_X (no MMA touches it now: PV_X(j-1) completed before S_X(j)
        // was issued, and PV_X(j) waits for the arrival below)
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(t_o + c * 32, o);
            tmem_wait_ld();
            reg_dep(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(t_o + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(C::BAR_P_FULL + x));
      }

      // ---------------------------------------------------- epilogue
      // the last S is done (Q and K/V stage 0 are free) while the last PV runs
      if (ok && in_bounds && merge && nx > 0) fetch_acc();
      bool have_o = ok && nx > 0;
      if (have_o) {
        const bool got = __all_sync(0xffffffffu, mbar_wait(bar(C::BAR_O_DONE + x), (nx - 1) & 1,
                                                           tc::WAIT_LIMIT_NS, abort_flag));
        if (!got) {
          record_timeout(dev_err, abort_flag);
          have_o = false;
          ok = false;
        }
        tc_fence_after();
      }
      if (!have_o) l = 0.f;
      // A tile without KV tiles never waited for its Q copy, whose buffer
      // the staging reuses; it fetches the merge's rows only now.
      if (ok && nx == 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::BAR_Q), 0, tc::WAIT_LIMIT_NS, abort_flag));
        if (!ok) record_timeout(dev_err, abort_flag);
        if (ok && in_bounds && merge) fetch_acc();
      }
      // out, acc and lse rows may be touched by the grid launched before
      // this one (a merge's fetch waited already; waiting again returns at
      // once, and every thread waits on every path)
      grid_wait_prerequisites();
      cp_async_wait_all();
      __syncwarp();
      const bool valid = ok && in_bounds && row < nrows;
      const float* lse_stg = reinterpret_cast<const float*>(smem + C::OFF_LSE);
      const float LOG2E = 1.4426950408889634f;
      const float LN2 = 0.6931471805599453f;
      // block result in log2 units; l == 0 exactly when no key was visible
      // (a NaN score leaves l NaN, which then reaches lse and out)
      const float lse_blk2 = l != 0.f ? m_used + __log2f(l) : -CUDART_INF_F;
      const bool final_out = (it.flags & kFlagFinal) != 0;
      float w_acc = 0.f, w_blk = 1.f, lse_new2 = lse_blk2;
      if (merge) {
        const float a2 = valid ? lse_stg[row] * LOG2E : -CUDART_INF_F;
        const float hi = fmaxf(a2, lse_blk2);
        if (a2 == -CUDART_INF_F && lse_blk2 == -CUDART_INF_F) {  // both empty (not NaN)
          w_acc = 0.f;
          w_blk = 0.f;
          lse_new2 = -CUDART_INF_F;
        } else {
          const float ea = ex2_approx(a2 - hi), eb = ex2_approx(lse_blk2 - hi);
          lse_new2 = hi + __log2f(ea + eb);
          w_acc = ex2_approx(a2 - lse_new2);
          w_blk = ex2_approx(lse_blk2 - lse_new2);
        }
      }
      const float c_blk = l != 0.f ? w_blk / l : 0.f;
      if (!kStriped && p.tma_out && final_out && !merge && nrows == tc::BM && in_bounds) {
        // A whole tile of bf16 result with nothing to merge: the rows are
        // staged in the output map's two boxes (64 columns, 128-byte
        // swizzle: 16-byte chunk j of row r at j ^ (r & 7)) and one thread
        // stores them with two TMA copies.  Every softmax thread takes this
        // branch (its condition is the CTA's), so all 128 reach the barrier.
        uint4* box = reinterpret_cast<uint4*>(smem + C::OFF_Q);
        const int sw = row & 7;
#pragma unroll 1
        for (int h2 = 0; h2 < 2 && ok; ++h2) {
          uint32_t o[2][32];
          __syncwarp();
          if (have_o) {
            tmem_ld32(t_o + h2 * 64, o[0]);
            tmem_ld32(t_o + h2 * 64 + 32, o[1]);
            tmem_wait_ld();
            reg_dep(o[0]);
            reg_dep(o[1]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[0][i] = o[1][i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            auto pk = [&](int e) {
              return pack_bf16x2(__uint_as_float(o[i >> 2][8 * (i & 3) + e]) * c_blk,
                                 __uint_as_float(o[i >> 2][8 * (i & 3) + e + 1]) * c_blk);
            };
            box[h2 * 1024 + row * 8 + (i ^ sw)] = make_uint4(pk(0), pk(2), pk(4), pk(6));
          }
        }
        fence_proxy_async_smem();  // the staged rows, to the copy engine
        named_bar_sync(1, 128);
        if (row == 0 && *abort_flag == 0) {
          const int orow0 =
              static_cast<int>(it.o_row + static_cast<int64_t>(b) * it.b_o_rows + row0);
          tma_store_3d(&tm_o, sbase + C::OFF_Q, 0, head, orow0);
          tma_store_3d(&tm_o, sbase + C::OFF_Q + 16384, 64, head, orow0);
          bulk_commit_group();
          bulk_wait_read_all();  // the boxes stay until the copies have read them
        }
      } else if (ok && in_bounds && final_out && p.out_dt == 1 && !merge) {
        // A bf16 result with nothing to merge: rows of 256 bytes staged in
        // bf16 over the Q buffer (16-byte chunk c of row r at c ^ (r & 7)),
        // half the shared-memory traffic of the fp32 staging below, which
        // the other CTA's MMAs on this SM compete for.
        uint4* stg16 = reinterpret_cast<uint4*>(smem + C::OFF_Q);
        uint4* srow16 = stg16 + row * 16;
        const int wrow0 = quad * 32;                // this warp's rows
        const int nwrows = min(32, nrows - wrow0);  // of them inside the tile
        const int sw = row & 7;
        // 64 columns per TMEM round trip (two loads, one wait)
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t o[2][32];
          __syncwarp();
          if (have_o) {
            tmem_ld32(t_o + h2 * 64, o[0]);
            tmem_ld32(t_o + h2 * 64 + 32, o[1]);
            tmem_wait_ld();
            reg_dep(o[0]);
            reg_dep(o[1]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[0][i] = o[1][i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            auto pk = [&](int e) {
              return pack_bf16x2(__uint_as_float(o[i >> 2][8 * (i & 3) + e]) * c_blk,
                                 __uint_as_float(o[i >> 2][8 * (i & 3) + e + 1]) * c_blk);
            };
            srow16[(h2 * 8 + i) ^ sw] = make_uint4(pk(0), pk(2), pk(4), pk(6));
          }
        }
        __syncwarp();
        // two rows per warp instruction (16 lanes x 16 bytes each), eight
        // instructions' shared-memory reads ahead of their stores
        const int sub = lane >> 4, l16 = lane & 15;
        __nv_bfloat16* dst16 = reinterpret_cast<__nv_bfloat16*>(p.out);
        const int64_t el0 = out_el0() + 8 * l16, stp = out_step();
#pragma unroll 1
        for (int i0 = 0; i0 < 32; i0 += 16) {
          uint4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int rr = wrow0 + i0 + 2 * u + sub;
            v[u] = stg16[rr * 16 + (l16 ^ (rr & 7))];
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int rr = i0 + 2 * u + sub;  // within this warp's rows
            if (rr < nwrows)
              *reinterpret_cast<uint4*>(dst16 + el0 + (wrow0 + rr) * stp) = v[u];
          }
        }
      } else if (ok && in_bounds) {
        float* stg = reinterpret_cast<float*>(smem + C::OFF_Q);
        const int wrow0 = quad * 32;                // this warp's rows
        const int nwrows = min(32, nrows - wrow0);  // of them inside the tile
        // thread = row: O * c_blk (+ staged acc * w_acc) back into the row
        float* srow = stg + row * 128;
        const int sw = row & 7;
#pragma unroll 1
        for (int h4 = 0; h4 < 4; ++h4) {
          uint32_t o[32];
          __syncwarp();
          if (have_o) {
            tmem_ld32(t_o + h4 * 32, o);
            tmem_wait_ld();
            reg_dep(o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4* d4 = reinterpret_cast<float4*>(srow + ((h4 * 8 + (i ^ sw)) << 2));
            float4 r = make_float4(__uint_as_float(o[4 * i]) * c_blk,
                                   __uint_as_float(o[4 * i + 1]) * c_blk,
                                   __uint_as_float(o[4 * i + 2]) * c_blk,
                                   __uint_as_float(o[4 * i + 3]) * c_blk);
            if (merge) {
              const float4 a = *d4;
              r.x = fmaf(a.x, w_acc, r.x);
              r.y = fmaf(a.y, w_acc, r.y);
              r.z = fmaf(a.z, w_acc, r.z);
              r.w = fmaf(a.w, w_acc, r.w);
            }
            *d4 = r;
          }
        }
        __syncwarp();
        // row per warp instruction, eight rows' shared-memory reads ahead of
        // their stores: the merged rows to out (bf16 / fp32) or acc
        const int64_t el0 = out_el0() + 4 * lane, stp = out_step();
        const bool to_bf16 = final_out && p.out_dt == 1;
        float* dst32 = final_out ? reinterpret_cast<float*>(p.out) : p.acc;
        __nv_bfloat16* dst16 = reinterpret_cast<__nv_bfloat16*>(p.out);
        auto put = [&](int rr, const float4& v) {
          const int64_t el = el0 + rr * stp;
          if (to_bf16)
            *reinterpret_cast<uint2*>(dst16 + el) = make_uint2(pack_bf16x2(v.x, v.y),
                                                               pack_bf16x2(v.z, v.w));
          else
            *reinterpret_cast<float4*>(dst32 + el) = v;
        };
        auto get = [&](int rr) -> float4 {
          return *reinterpret_cast<const float4*>(stg + rr * 128 + ((lane ^ (rr & 7)) << 2));
        };
        int i = 0;
        for (; i + 8 <= nwrows; i += 8) {
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = get(wrow0 + i + u);
#pragma unroll
          for (int u = 0; u < 8; ++u) put(wrow0 + i + u, v[u]);
        }
        for (; i < nwrows; ++i) put(wrow0 + i, get(wrow0 + i));
      }
      if (valid) *lse_addr() = lse_new2 == -CUDART_INF_F ? -CUDART_INF_F : lse_new2 * LN2;
    }
  }

  // --------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::WARP_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
}

// Query tiles per CTA of the launches below.
#ifndef CP_FWD_NT
#define CP_FWD_NT 1
#endif
constexpr int kNT = CP_FWD_NT;
static_assert(kNT == 1, "one query tile per CTA (two tiles per CTA measured slower)");

int attn_tc_smem_bytes() { return static_cast<int>(tc::Cfg<kNT>::SMEM_BYTES); }

cudaError_t launch_attn_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const AttnParams& p, int ctas, int* dev_err,
                           cudaStream_t stream, bool dependent) {
  using C = tc::Cfg<kNT>;
  // the shared-memory attribute is a property of the function on each device
  static PerDeviceOnce attr_once;
  cudaError_t e = once_per_device(attr_once, [] {
    cudaError_t r = cudaFuncSetAttribute(attn_fwd_tc_kernel<false, kNT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(C::SMEM_BYTES));
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(attn_fwd_tc_kernel<true, kNT>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(C::SMEM_BYTES));
    return r;
  });
  if (e != cudaSuccess) return e;
  // dependent: launched with programmatic stream serialisation, so that it
  // overlaps the tail of the previous kernel on the stream (which must be
  // this kernel, writing none of q, k, v)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  if (p.maps4d)
    return cudaLaunchKernelEx(&cfg, attn_fwd_tc_kernel<true, kNT>, tq, tk, tv, to, p, dev_err);
  return cudaLaunchKernelEx(&cfg, attn_fwd_tc_kernel<false, kNT>, tq, tk, tv, to, p, dev_err);
}

// Number of CTAs one item occupies (kNT x 128 query rows per CTA).
int attn_tc_ctas(const WorkItem& it, int H) {
  const int ngroups = (it.sq + kNT * tc::BM - 1) / (kNT * tc::BM);
  return ngroups * it.batch * H;
}

}  // namespace cpattn
