// C ABI of libcpattn: argument validation, the ring / Ulysses schedulers, TMA
// descriptor set-up and kernel launches.  See include/cpattn.h for the
// contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/cpattn.h"
#include "internal.h"

namespace cpattn {
cudaError_t launch_attn_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const AttnParams& p, int ctas, int* dev_err,
                           cudaStream_t stream, bool dependent);
int attn_tc_ctas(const WorkItem& it, int H);
cudaError_t launch_attn_simt(const AttnParams& p, int ctas, int* dev_err, cudaStream_t stream);
int attn_simt_ctas(const WorkItem& it, int H);
cudaError_t launch_lse_merge(float* out_acc, float* lse_acc, const float* out_blk,
                             const float* lse_blk, int64_t Sq, int H, int D, cudaStream_t s);
cudaError_t launch_permute(const void* src, void* dst, int64_t A, int64_t B, int64_t run_bytes,
                           cudaStream_t s);
cudaError_t launch_fill_empty(void* out, int out_bytes_per_el, int64_t n_out, float* lse,
                              int64_t n_lse, cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int* dev_err, cudaStream_t s);
int* device_status_ptr();
cudaError_t launch_attn_bwd(bool dkdv, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                            int ctas, int* dev_err, cudaStream_t stream);
int attn_bwd_ctas(const BwdItem& it, int heads);
int attn_bwd_simt_warps(const BwdItem& it, int heads);
cudaError_t launch_attn_bwd_simt(bool dkdv, const void* q, const void* k, const void* v,
                                 const void* dout, const BwdParams& p, int D, int warps,
                                 int* dev_err, cudaStream_t s);
cudaError_t launch_bwd_delta_f32(const void* out, const void* dout, float* delta, int64_t rows,
                                 int H, int D, int64_t ld, cudaStream_t s);
cudaError_t launch_bwd_delta(const void* out, const void* dout, float* delta, int64_t rows, int H,
                             int64_t ld, cudaStream_t s);
}  // namespace cpattn

using namespace cpattn;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return CP_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(CP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int elem_bytes(cp_dtype dt) { return dt == CP_BF16 ? 2 : 4; }

bool valid_dtype(int dt) { return dt == CP_F32 || dt == CP_BF16; }

// --------------------------------------------------------------- TMA maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor [rows, heads, 128] -> 4-D map (d, head, r, i) with token =
// r + stripe * i (stripe = 1: plain rows), box 64 x 1 x 1 x 128, 128-byte
// swizzle: one box = 128 tokens x 64 columns = 16 KB.  rows % stripe == 0.
// With dims4 = false a 3-D map (d, head, row) with box 64 x 1 x 128 is made
// instead (plain rows; stripe must be 1).
int make_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int stripe, bool dims4) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return fail(CP_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(heads) * 128 * 2;
  const cuuint64_t dims4v[4] = {128, static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(stripe),
                                static_cast<cuuint64_t>(rows / stripe)};
  const cuuint64_t strides4[3] = {128 * 2, row_bytes, row_bytes * static_cast<cuuint64_t>(stripe)};
  const cuuint32_t box4[4] = {64, 1, 1, 128};
  const cuuint64_t dims3v[3] = {128, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides3[2] = {128 * 2, row_bytes};
  const cuuint32_t box3[3] = {64, 1, 128};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dims4 ? 4 : 3, const_cast<void*>(base),
                   dims4 ? dims4v : dims3v, dims4 ? strides4 : strides3, dims4 ? box4 : box3, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CP_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return CP_OK;
}

// ---------------------------------------------------------------- launch
struct Launch {
  AttnParams p{};
  std::vector<WorkItem> items;
};

// Fill cta_start and launch the kernel for the input dtype.
// dependent: the launch may overlap the tail of the previous kernel on the
// stream, which must be an attention launch of the same ring (tensor-core
// path only; see launch_attn_tc).
int launch_items(Launch& L, cp_dtype in_dt, const void* q, int64_t q_rows, const void* k,
                 const void* v, int64_t k_rows, cudaStream_t stream, bool dependent = false) {
  AttnParams& p = L.p;
  if (L.items.empty()) return CP_OK;
  if (static_cast<int>(L.items.size()) > kMaxItems)
    return fail(CP_ERR_ARG, "too many work items (%d)", int(L.items.size()));
  p.nitems = static_cast<int>(L.items.size());
  int64_t total = 0, tiles = 0;
  for (int i = 0; i < p.nitems; ++i) {
    p.items[i] = L.items[i];
    if (p.items[i].o_stride == 0) p.items[i].o_stride = 1;  // plain rows by default
    p.cta_start[i] = static_cast<int>(total);
    p.tile_start[i] = static_cast<int>(tiles);
    total += in_dt == CP_BF16 ? attn_tc_ctas(L.items[i], p.H) : attn_simt_ctas(L.items[i], p.H);
    tiles += attn_tc_ctas(L.items[i], 1) / L.items[i].batch;
  }
  p.tile_start[p.nitems] = static_cast<int>(tiles);
  if (p.head_major) {
    if (p.hm_long < 0 || p.hm_long > tiles) p.hm_long = static_cast<int>(tiles);
    // the grid is tiles x (heads x batch): every item has the same batch
    bool uniform = in_dt == CP_BF16;
    for (int i = 1; i < p.nitems; ++i) uniform = uniform && p.items[i].batch == p.items[0].batch;
    if (!uniform || total != tiles * p.H * p.items[0].batch)
      return fail(CP_ERR_ARG, "head-major launch needs bf16 items of one batch size");
  }
  if (total > 0x7fffffff) return fail(CP_ERR_SHAPE, "grid too large");
  p.cta_start[p.nitems] = static_cast<int>(total);
  for (int i = p.nitems + 1; i <= kMaxItems; ++i) p.cta_start[i] = static_cast<int>(total);
  if (total == 0) return CP_OK;
  p.q = q;
  p.k = k;
  p.v = v;
  p.q_rows = q_rows;
  p.k_rows = k_rows;
  cudaError_t e;
  if (in_dt == CP_BF16) {
    CUtensorMap tq, tk, tv;
#ifdef CP_FORCE_4D
    p.maps4d = 1;
#else
    p.maps4d = (p.stripe != 1 || p.kv_stripe != 1) ? 1 : 0;
#endif
    int rc = make_map(&tq, q, q_rows, p.H, p.stripe, p.maps4d);
    if (rc == CP_OK) rc = make_map(&tk, k, k_rows, p.Hkv, p.kv_stripe, p.maps4d);
    if (rc == CP_OK) rc = make_map(&tv, v, k_rows, p.Hkv, p.kv_stripe, p.maps4d);
    // a bf16 out [q_rows, H, D] with plain rows is written by TMA stores
    // (whole tiles of unmerged results); otherwise the map is not used
    CUtensorMap to = tq;
    p.tma_out = 0;
    if (rc == CP_OK && !p.maps4d && p.out_dt == 1 && p.out != nullptr) {
      rc = make_map(&to, p.out, q_rows, p.H, 1, false);
      p.tma_out = 1;
    }
    if (rc != CP_OK) return rc;
    int* st = device_status_ptr();
    if (st == nullptr) return fail(CP_ERR_CUDA, "device status word unavailable");
    e = launch_attn_tc(tq, tk, tv, to, p, static_cast<int>(total), st, stream, dependent);
  } else {
    int* st = device_status_ptr();
    if (st == nullptr) return fail(CP_ERR_CUDA, "device status word unavailable");
    e = launch_attn_simt(p, static_cast<int>(total), st, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention kernel launch");
  return CP_OK;
}

void fill_common(AttnParams& p, int H, int Hkv, int D, float scale, cp_dtype out_dt, void* out,
                 float* acc, float* lse, int64_t ld_lse) {
  p.H = H;
  p.Hkv = Hkv;
  p.D = D;
  p.stripe = 1;
  p.kv_stripe = 1;
  p.b_q_heads = 0;
  p.kv_group = H / Hkv;
  p.out_dt = out_dt == CP_BF16 ? 1 : 0;
  const float sc = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D));
  p.scale = sc;
  p.scale_log2 = sc * 1.4426950408889634f;
  p.out = out;
  p.acc = acc;
  p.lse = lse;
  p.ld_lse = ld_lse;
}

int check_heads_dims(cp_dtype in_dt, int H, int Hkv, int D) {
  if (!valid_dtype(in_dt)) return fail(CP_ERR_DTYPE, "unknown input dtype %d", int(in_dt));
  if (H < 1 || Hkv < 1) return fail(CP_ERR_ARG, "H=%d and Hkv=%d must be >= 1", H, Hkv);
  if (H % Hkv != 0) return fail(CP_ERR_SHAPE, "H=%d is not a multiple of Hkv=%d", H, Hkv);
  if (in_dt == CP_BF16 && D != 128)
    return fail(CP_ERR_SHAPE, "bf16 inputs need D=128 (got %d)", D);
  if (in_dt == CP_F32 && D != 16 && D != 32 && D != 64 && D != 128)
    return fail(CP_ERR_SHAPE, "fp32 inputs need D in {16,32,64,128} (got %d)", D);
  return CP_OK;
}

// ------------------------------------------------------------ ring schedule
// Chunks held by rank r (queries, and KV initially).  In the striped layout
// a rank's "chunk" is its stripe (tokens r, r+P, ...), numbered r.
int rank_chunks(int P, cp_layout layout, int r, int out[2]) {
  if (layout == CP_CONTIGUOUS || layout == CP_STRIPED) {
    out[0] = r;
    return 1;
  }
  out[0] = r;
  out[1] = 2 * P - 1 - r;
  return 2;
}

struct StepItem {
  int rank, qc, nk, kc[2];
};

// Step t: rank r holds the KV of src = (r - t) mod P (the KV travels to
// rank + 1 after every step).  Per own query chunk, the held KV chunks not
// later than it, ascending.
std::vector<StepItem> step_items(int P, cp_layout layout, int t) {
  std::vector<StepItem> v;
  for (int r = 0; r < P; ++r) {
    const int src = ((r - t) % P + P) % P;
    int qcs[2], kcs[2];
    const int nq = rank_chunks(P, layout, r, qcs);
    const int nk = rank_chunks(P, layout, src, kcs);
    for (int a = 0; a < nq; ++a) {
      StepItem it{r, qcs[a], 0, {0, 0}};
      for (int b = 0; b < nk; ++b)  // striped: every held stripe has visible keys
        if (kcs[b] <= qcs[a] || layout == CP_STRIPED) it.kc[it.nk++] = kcs[b];
      if (it.nk == 2 && it.kc[0] > it.kc[1]) std::swap(it.kc[0], it.kc[1]);
      if (it.nk > 0) v.push_back(it);
    }
  }
  return v;
}

int check_ring(cp_dtype in_dt, int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
               cp_dtype out_dt) {
  int rc = check_heads_dims(in_dt, H, Hkv, D);
  if (rc != CP_OK) return rc;
  if (!valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown output dtype %d", int(out_dt));
  if (layout != CP_CONTIGUOUS && layout != CP_ZIGZAG && layout != CP_STRIPED)
    return fail(CP_ERR_ARG, "unknown layout %d", int(layout));
  if (P < 1 || P > CP_MAX_RANKS) return fail(CP_ERR_ARG, "P=%d outside [1,%d]", P, CP_MAX_RANKS);
  if (S < 1 || S >= (int64_t(1) << 31))
    return fail(CP_ERR_ARG, "S=%lld out of range", (long long)S);
  if (layout == CP_STRIPED && S % P != 0)
    return fail(CP_ERR_SHAPE, "striped layout: S=%lld is not a multiple of P=%d", (long long)S, P);
  return CP_OK;
}

// Where the ring's held KV lives at one step.  Without a view the virtual
// ranks read their held chunks in place in the natural-order k, v (a "send"
// is a change of row offset).  With a view (copy mode) rank r's held chunks
// sit, in slot order, at rows slot0 + r * R of the k / v buffers.
struct KvView {
  const void* k;
  const void* v;
  int64_t rows;   // rows of the buffers
  int64_t slot0;  // first row of this step's slots
  int64_t R;      // rows per rank slot
};

// A batch of independent sequences run through the ring together (the Pu
// head groups of USP): group b's rows start b_q_rows / b_k_rows / b_o_rows
// further (in row units of the tensors' addressing), its LSE rows b_lse_heads
// further, and its KV head is (b * b_q_heads + h) / kv_group.
struct RingBatch {
  int batch;
  int64_t b_q_rows, b_k_rows, b_o_rows;
  int b_lse_heads;
  int b_q_heads, kv_group;
  int64_t q_rows, k_rows;  // rows of the q and k tensors
};

// Rows per rank slot of a copy-mode buffer: all of a rank's chunks.
int64_t ring_rank_rows(int64_t S, int P, cp_layout layout) {
  if (layout == CP_STRIPED) return S / P;
  if (layout == CP_ZIGZAG) return 2 * ((S + 2 * P - 1) / (2 * P));
  return (S + P - 1) / P;
}

int ring_step_impl(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S, int H,
                   int Hkv, int D, int P, cp_layout layout, int t, void* out, cp_dtype out_dt,
                   float* lse, void* workspace, cudaStream_t stream,
                   const KvView* view = nullptr, const RingBatch* rb = nullptr,
                   bool dependent = false) {
  const void* kk = view ? view->k : k;
  const void* vv = view ? view->v : v;
  const int64_t k_rows = view ? view->rows : rb ? rb->k_rows : S;
  const int64_t q_rows = rb ? rb->q_rows : S;
  auto batched = [&](Launch& L) {
    if (!rb) return;
    L.p.b_q_heads = rb->b_q_heads;
    L.p.kv_group = rb->kv_group;
    for (WorkItem& w : L.items) {
      w.batch = rb->batch;
      w.b_q_rows = rb->b_q_rows;
      w.b_k_rows = rb->b_k_rows;
      w.b_o_rows = rb->b_o_rows;
      w.b_lse_heads = rb->b_lse_heads;
    }
  };
  const bool bf16_out = out_dt == CP_BF16;
  Launch L;
  fill_common(L.p, H, Hkv, D, 0.f, out_dt, out,
              bf16_out ? static_cast<float*>(workspace) : static_cast<float*>(out), lse, S);
  if (layout == CP_STRIPED) {
    // rank r's queries and held keys are stripes (token r + P*i); in stripe
    // indices the causal mask is j + (src > r) <= i
    const int64_t C = S / P;
    L.p.stripe = P;
    L.p.kv_stripe = view ? 1 : P;
    for (const StepItem& si : step_items(P, layout, t)) {
      WorkItem w{};
      w.q_stripe = si.rank;
      w.q_mem_row = 0;
      w.q_pos = 0;
      w.o_row = si.rank;
      w.o_stride = P;
      w.lse_col = si.rank;
      w.sq = static_cast<int32_t>(C);
      w.nseg = 1;
      w.batch = 1;
      w.flags = kFlagCausal;
      if (t > 0) w.flags |= kFlagMerge;
      if (!bf16_out || t == P - 1) w.flags |= kFlagFinal;
      w.seg[0].mem_row = view ? view->slot0 + si.rank * view->R : 0;
      w.seg[0].pos = si.kc[0] > si.rank ? 1 : 0;
      w.seg[0].len = static_cast<int32_t>(C);
      w.seg[0].stripe = view ? 0 : si.kc[0];
      L.items.push_back(w);
    }
    batched(L);
    return launch_items(L, in_dt, q, q_rows, kk, vv, k_rows, stream, dependent);
  }
  // contiguous / zigzag: n chunks of C = ceil(S / n) rows, the last ones
  // shorter (or empty) when n does not divide S -- the padding of a short
  // sequence, without padded rows
  const int64_t nchunks = layout == CP_ZIGZAG ? 2 * P : P;
  const int64_t C = (S + nchunks - 1) / nchunks;
  auto chunk_rows = [&](int c) -> int64_t {
    return std::max<int64_t>(0, std::min<int64_t>(S, (c + 1) * C) - c * C);
  };
  // last step at which each query chunk is evaluated
  std::vector<int> last(nchunks, -1);
  for (int s = 0; s < P; ++s)
    for (const StepItem& it : step_items(P, layout, s)) last[it.qc] = s;
  for (const StepItem& si : step_items(P, layout, t)) {
    if (chunk_rows(si.qc) == 0) continue;
    WorkItem w{};
    w.q_mem_row = si.qc * C;
    w.q_pos = si.qc * C;
    w.o_row = si.qc * C;
    w.lse_col = si.qc * C;
    w.sq = static_cast<int32_t>(chunk_rows(si.qc));
    w.batch = 1;
    w.flags = kFlagCausal;
    if (t > 0) w.flags |= kFlagMerge;  // every chunk is first evaluated at step 0
    if (!bf16_out || last[si.qc] == t) w.flags |= kFlagFinal;
    const int src = ((si.rank - t) % P + P) % P;
    for (int s = 0; s < si.nk; ++s) {
      if (chunk_rows(si.kc[s]) == 0) continue;
      KSeg& g = w.seg[w.nseg++];
      // slot order of a zigzag rank's chunks: src, then 2P-1-src
      g.mem_row = view ? view->slot0 + si.rank * view->R + (si.kc[s] == src ? 0 : C) : si.kc[s] * C;
      g.pos = si.kc[s] * C;
      g.len = static_cast<int32_t>(chunk_rows(si.kc[s]));
    }
    L.items.push_back(w);
  }
  // longest items first (the grid is scheduled roughly in order)
  std::stable_sort(L.items.begin(), L.items.end(), [](const WorkItem& a, const WorkItem& b) {
    int64_t ca = 0, cb = 0;
    for (int s = 0; s < a.nseg; ++s) ca += a.seg[s].len - (a.seg[s].pos == a.q_pos ? a.sq / 2 : 0);
    for (int s = 0; s < b.nseg; ++s) cb += b.seg[s].len - (b.seg[s].pos == b.q_pos ? b.sq / 2 : 0);
    return ca > cb;
  });
  batched(L);
  return launch_items(L, in_dt, q, q_rows, kk, vv, k_rows, stream, dependent);
}

// Head-major grid of the one-launch ring: how many of each head's tile ranks
// (the items in order, later query tiles first -- roughly longest first)
// run head by head before the rest runs rank by rank across the nh heads
// (heads x batch).  Run purely head by head, the grid ends with the last
// head's tiles: its longest CTA (Lmax KV tiles) starts about T_h = (the
// head's KV tiles) / (resident CTAs) before the other CTAs run out of work,
// so the launch ends on a tail of Lmax - T_h with most SMs idle (at 32K: 256
// against 108 tiles, 3.5% of the launch; none at 128K).  The shortest
// ranks of every head, together holding the work of that tail on every
// resident CTA, are moved to the end and run across the heads.
int head_major_lead(const std::vector<WorkItem>& items, int64_t C, int64_t S, bool striped, int nh,
                    int dev) {
  auto chunk_rows = [&](int64_t c) -> int64_t {
    return striped ? C : std::max<int64_t>(0, std::min<int64_t>(S, (c + 1) * C) - c * C);
  };
  std::vector<int64_t> w;  // KV tiles of each tile rank of one head
  for (const WorkItem& it : items) {
    const int nt = (it.sq + 127) / 128;
    for (int k = 0; k < nt; ++k) {
      const int t = nt - 1 - k;
      const int64_t qp_last = it.q_pos + std::min<int64_t>(it.sq, (t + 1) * 128) - 1;
      int64_t n = 0;
      for (int c = 0; c < it.nchunk; ++c) {
        const int64_t pos = striped ? (it.chunk[c] > it.q_stripe ? 1 : 0) : it.chunk[c] * C;
        const int64_t len = chunk_rows(it.chunk[c]);
        const int64_t vis = std::max<int64_t>(0, std::min<int64_t>(len, qp_last - pos + 1));
        n += (vis + 127) / 128;
      }
      w.push_back(n);
    }
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 0;
  const int64_t slots = 2 * static_cast<int64_t>(std::max(sms, 1));  // two CTAs per SM
  int64_t total = 0, lmax = 0;
  for (int64_t x : w) {
    total += x;
    lmax = std::max(lmax, x);
  }
  const int64_t tail = lmax - total / slots;  // KV tiles of one CTA
  if (tail <= 0 || nh < 1) return static_cast<int>(w.size());
  const int64_t need = (tail * slots + nh - 1) / nh;  // per head
  int64_t got = 0;
  size_t lead = w.size();
  while (lead > 0 && got < need) got += w[--lead];
  return static_cast<int>(lead);
}

// The ring in one launch (bf16 inputs): one work item per (virtual rank r,
// own query chunk qc; in the striped layout its stripe), whose key segments are
// the chunks rank r holds at steps t = 0, 1, ..., P-1 (src = (r - t) mod P,
// ascending within a step) that are not later than qc -- exactly the blocks
// the per-step ring evaluates for those rows, in the same order.  Each query
// tile carries its running max, sum and output in TMEM from one step to the
// next (the online-softmax form of the LSE merge) and writes the final
// result once, so no accumulator round trip, per-step epilogue or launch
// separates the steps.  With `rb` the launch covers a batch of independent
// sequences (the head groups of USP), each its own ring.
int ring_fused_impl(const void* q, const void* k, const void* v, int64_t S, int H, int Hkv,
                    int D, int P, cp_layout layout, void* out, cp_dtype out_dt, float* lse,
                    cudaStream_t stream, const RingBatch* rb = nullptr) {
  const int64_t q_rows = rb ? rb->q_rows : S, k_rows = rb ? rb->k_rows : S;
  const bool striped = layout == CP_STRIPED;
  const int64_t nchunks = layout == CP_ZIGZAG ? 2 * P : P;
  const int64_t C = (S + nchunks - 1) / nchunks;  // striped: S / P, the stripe length
  auto chunk_rows = [&](int64_t c) -> int64_t {
    return std::max<int64_t>(0, std::min<int64_t>(S, (c + 1) * C) - c * C);
  };
  Launch L;
  fill_common(L.p, H, Hkv, D, 0.f, out_dt, out,
              out_dt == CP_F32 ? static_cast<float*>(out) : nullptr, lse, S);
  L.p.ring_C = C;
  L.p.ring_S = S;
  if (striped) {
    // rank r's queries and every key it is handed are stripes (token
    // r + P i), addressed through 4-D maps
    L.p.stripe = P;
    L.p.kv_stripe = P;
    L.p.ring_striped = 1;
  }
  if (rb) {
    L.p.b_q_heads = rb->b_q_heads;
    L.p.kv_group = rb->kv_group;
  }
  // Every query tile walks its head's whole visible K/V.  When all heads' K/V
  // is more than L2 holds, run the grid head by head so that the CTAs
  // resident at one time share one head's K/V (at 32K, 512 MiB of K/V, this
  // cut DRAM reads from 4.8 GB to 0.83 GB per launch); otherwise keep the
  // items' longest-first order across all heads, which ends with a shorter
  // tail (4K, 64 MiB of K/V: 954 against 767 TFLOP/s head by head).
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
    l2 = 0;
  L.p.head_major = k_rows * Hkv * static_cast<int64_t>(D) * 2 * 2 > static_cast<int64_t>(l2);
  std::vector<int64_t> work;  // visible keys x rows, for the longest-first order
  for (int r = 0; r < P; ++r) {
    int qcs[2];
    const int nq = rank_chunks(P, layout, r, qcs);
    for (int a = 0; a < nq; ++a) {
      const int qc = qcs[a];
      if (striped) {
        // stripe r against the stripes src = r, r-1, ... the steps hand it;
        // every one holds keys visible to it (a causal prefix of each)
        WorkItem w{};
        w.q_stripe = r;
        w.o_row = r;
        w.o_stride = P;
        w.lse_col = r;
        w.sq = static_cast<int32_t>(C);
        w.batch = 1;
        if (rb) {
          w.batch = rb->batch;
          w.b_q_rows = rb->b_q_rows;
          w.b_k_rows = rb->b_k_rows;
          w.b_o_rows = rb->b_o_rows;
          w.b_lse_heads = rb->b_lse_heads;
        }
        w.flags = kFlagCausal | kFlagFinal;
        w.q_chunk = r;
        for (int t = 0; t < P; ++t)
          w.chunk[w.nchunk++] = static_cast<uint8_t>(((r - t) % P + P) % P);
        L.items.push_back(w);
        work.push_back(C * C * P);  // alike for every rank
        continue;
      }
      if (chunk_rows(qc) == 0) continue;
      WorkItem w{};
      w.q_mem_row = qc * C;
      w.q_pos = qc * C;
      w.o_row = qc * C;
      w.lse_col = qc * C;
      w.sq = static_cast<int32_t>(chunk_rows(qc));
      w.batch = 1;
      if (rb) {
        w.batch = rb->batch;
        w.b_q_rows = rb->b_q_rows;
        w.b_k_rows = rb->b_k_rows;
        w.b_o_rows = rb->b_o_rows;
        w.b_lse_heads = rb->b_lse_heads;
      }
      w.flags = kFlagCausal | kFlagFinal;
      w.q_chunk = qc;
      int64_t keys = 0;
      for (int t = 0; t < P; ++t) {
        const int src = ((r - t) % P + P) % P;
        int kcs[2];
        const int nk = rank_chunks(P, layout, src, kcs);
        for (int b = 0; b < nk; ++b) {
          if (kcs[b] > qc || chunk_rows(kcs[b]) == 0) continue;
          if (w.nchunk >= kMaxRingChunks) return fail(CP_ERR_ARG, "too many ring chunks");
          w.chunk[w.nchunk++] = static_cast<uint8_t>(kcs[b]);
          keys += kcs[b] == qc ? chunk_rows(qc) / 2 : chunk_rows(kcs[b]);
          if (kcs[b] != qc) w.full_tiles += static_cast<int32_t>((chunk_rows(kcs[b]) + 127) / 128);
        }
      }
      L.items.push_back(w);
      work.push_back(keys * w.sq);
    }
  }
  // longest items first (the grid is scheduled roughly in order)
  std::vector<size_t> order(L.items.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](size_t a, size_t b) { return work[a] > work[b]; });
  std::vector<WorkItem> sorted;
  for (size_t i : order) sorted.push_back(L.items[i]);
  L.items.swap(sorted);
  if (L.p.head_major)
    L.p.hm_long = head_major_lead(L.items, C, S, striped, H * (rb ? rb->batch : 1), dev);
  return launch_items(L, CP_BF16, q, q_rows, k, v, k_rows, stream);
}

// Copy-mode ring: one D2D copy per rank and tensor moves every rank's held
// KV into rank+1's other buffer on `copy_stream` while step t computes.
int ring_forward_copy_impl(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                           int H, int Hkv, int D, int P, cp_layout layout, void* out,
                           cp_dtype out_dt, float* lse, void* workspace, cudaStream_t cs,
                           cudaStream_t xs) {
  const int64_t e = elem_bytes(in_dt);
  const int64_t row_bytes = static_cast<int64_t>(Hkv) * D * e;
  const int64_t R = ring_rank_rows(S, P, layout);
  const int64_t acc_bytes = out_dt == CP_BF16 ? S * H * D * 4 : 0;
  const int64_t acc_pad = (acc_bytes + 255) / 256 * 256;
  const int64_t buf_bytes = 2 * P * R * row_bytes;
  char* ws = static_cast<char*>(workspace);
  char* kb = ws + acc_pad;
  char* vb = kb + (buf_bytes + 255) / 256 * 256;
  cudaEvent_t entry, comp[2], copied;
  cudaError_t err = cudaEventCreateWithFlags(&entry, cudaEventDisableTiming);
  for (int i = 0; i < 2 && err == cudaSuccess; ++i)
    err = cudaEventCreateWithFlags(&comp[i], cudaEventDisableTiming);
  if (err == cudaSuccess) err = cudaEventCreateWithFlags(&copied, cudaEventDisableTiming);
  if (err != cudaSuccess) return cuda_fail(err, "event create");
  int rc = CP_OK;
  auto check = [&](cudaError_t x, const char* what) {
    if (x != cudaSuccess && rc == CP_OK) rc = cuda_fail(x, what);
  };
  // Ragged chunks leave rows of a slot unused: they are masked (P = 0) but
  // must hold finite values, since 0 * NaN would reach O through the MMA.
  const int64_t nch = layout == CP_ZIGZAG ? 2 * P : P;
  if (layout != CP_STRIPED && S % nch != 0)
    check(cudaMemsetAsync(kb, 0, static_cast<size_t>(vb - kb) + buf_bytes, cs), "memset");
  // the copies read k, v (and the cleared buffers) from the compute stream
  check(cudaEventRecord(entry, cs), "event record");
  check(cudaStreamWaitEvent(xs, entry, 0), "stream wait");
  const int64_t nchunks = layout == CP_ZIGZAG ? 2 * P : P;
  const int64_t C = layout == CP_STRIPED ? S / P : (S + nchunks - 1) / nchunks;
  auto chunk_rows = [&](int64_t c) -> int64_t {
    return std::max<int64_t>(0, std::min<int64_t>(S, (c + 1) * C) - c * C);
  };
  for (int t = 0; t < P && rc == CP_OK; ++t) {
    // compute step t: step 0 reads every rank's own KV in place, later steps
    // the buffer filled by the copies of step t-1
    if (t > 0) check(cudaStreamWaitEvent(cs, copied, 0), "stream wait");
    if (rc != CP_OK) break;
    KvView view{kb, vb, 2 * P * R, (t % 2) * P * R, R};
    rc = ring_step_impl(q, k, v, in_dt, S, H, Hkv, D, P, layout, t, out, out_dt, lse, workspace,
                        cs, t == 0 ? nullptr : &view);
    if (rc != CP_OK) break;
    check(cudaEventRecord(comp[t % 2], cs), "event record");
    if (t == P - 1) break;
    // send: rank r's held KV -> rank r+1's slot of buffer (t+1) % 2, which
    // step t-1 read
    if (t > 0) check(cudaStreamWaitEvent(xs, comp[(t - 1) % 2], 0), "stream wait");
    const int64_t dst0 = ((t + 1) % 2) * P * R, src0 = (t % 2) * P * R;
    for (int r = 0; r < P && rc == CP_OK; ++r) {
      const int64_t dst_row = dst0 + ((r + 1) % P) * R;
      for (int w = 0; w < 2; ++w) {
        char* dst = (w == 0 ? kb : vb) + dst_row * row_bytes;
        const char* base = static_cast<const char*>(w == 0 ? k : v);
        if (t > 0) {
          const char* src = (w == 0 ? kb : vb) + (src0 + r * R) * row_bytes;
          check(cudaMemcpyAsync(dst, src, R * row_bytes, cudaMemcpyDeviceToDevice, xs), "copy");
        } else if (layout == CP_STRIPED) {
          check(cudaMemcpy2DAsync(dst, row_bytes, base + r * row_bytes, P * row_bytes, row_bytes,
                                  S / P, cudaMemcpyDeviceToDevice, xs),
                "copy");
        } else {
          // own chunks in slot order: r (and 2P-1-r for zigzag)
          int chunks[2] = {r, static_cast<int>(2 * P - 1 - r)};
          const int nc = layout == CP_ZIGZAG ? 2 : 1;
          for (int c = 0; c < nc; ++c) {
            const int64_t rows = chunk_rows(chunks[c]);
            if (rows > 0)
              check(cudaMemcpyAsync(dst + c * C * row_bytes, base + chunks[c] * C * row_bytes,
                                    rows * row_bytes, cudaMemcpyDeviceToDevice, xs),
                    "copy");
          }
        }
      }
    }
    check(cudaEventRecord(copied, xs), "event record");
  }
  cudaEventDestroy(entry);
  cudaEventDestroy(comp[0]);
  cudaEventDestroy(comp[1]);
  cudaEventDestroy(copied);
  return rc;
}


// ------------------------------------------------------------- backward
// One launch of a backward kernel: the dQ kernel (queries stationary) or the
// dK/dV kernel (keys stationary) over a list of items.  `chunk` names the
// gradient rows an item owns (a ring chunk or stripe) for the first / last
// touch flags.
struct BwdTask {
  bool dkdv;
  std::vector<BwdItem> items;
  std::vector<int> chunk;
  int64_t ring_C = 0, ring_S = 0;  // chunk geometry of chunk-list items
  bool striped = false;            // chunk-list items name stripes
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  int64_t q_rows, k_rows;  // rows of the q / dout and k / v tensors
  int H, Hkv, stride, causal;
  cp_dtype in_dt;  // bf16: tensor-core kernels (D = 128); fp32: CUDA-core kernels
  int D;
  float scale;
  const float* lse;
  const float* delta;
  int64_t ld;
  cp_dtype grad_dt;
  void* dq;
  void* dk;
  void* dv;
  float* acc_q;  // fp32 accumulators (the outputs themselves for fp32 gradients)
  float* acc_k;
  float* acc_v;
};

int run_bwd_task(const BwdArgs& a, const BwdTask& t, const CUtensorMap maps[4], cudaStream_t s) {
  if (t.items.empty()) return CP_OK;
  if (static_cast<int>(t.items.size()) > kMaxItems)
    return fail(CP_ERR_ARG, "too many backward items (%d)", int(t.items.size()));
  BwdParams p{};
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.D = 128;
  p.out_dt = a.grad_dt == CP_BF16 ? 1 : 0;
  p.causal = a.causal;
  p.stride = a.stride;
  p.scale = a.scale;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.lse = a.lse;
  p.delta = a.delta;
  p.ld = a.ld;
  p.ring_C = t.ring_C;
  p.ring_S = t.ring_S;
  p.ring_striped = t.striped ? 1 : 0;
  p.q_rows = a.q_rows;
  p.k_rows = a.k_rows;
  if (t.dkdv) {
    p.acc0 = a.acc_v;
    p.acc1 = a.acc_k;
    p.out0 = a.dv;
    p.out1 = a.dk;
  } else {
    p.acc0 = a.acc_q;
    p.acc1 = a.acc_q;
    p.out0 = a.dq;
    p.out1 = a.dq;
  }
  p.nitems = static_cast<int>(t.items.size());
  const bool f32 = a.in_dt == CP_F32;
  int64_t total = 0;  // CTAs (bf16) or warps (fp32)
  for (int i = 0; i < p.nitems; ++i) {
    p.items[i] = t.items[i];
    p.cta_start[i] = static_cast<int>(total);
    total += f32 ? attn_bwd_simt_warps(t.items[i], t.dkdv ? a.Hkv : a.H)
                 : attn_bwd_ctas(t.items[i], t.dkdv ? a.Hkv : a.H);
  }
  if (total > 0x7fffffff) return fail(CP_ERR_SHAPE, "grid too large");
  for (int i = p.nitems; i <= kMaxItems; ++i) p.cta_start[i] = static_cast<int>(total);
  if (total == 0) return CP_OK;
  int* st = device_status_ptr();
  if (st == nullptr) return fail(CP_ERR_CUDA, "device status word unavailable");
  if (f32) {
    cudaError_t e = launch_attn_bwd_simt(t.dkdv, a.q, a.k, a.v, a.dout, p, a.D,
                                         static_cast<int>(total), st, s);
    return e == cudaSuccess ? CP_OK : cuda_fail(e, "backward kernel launch");
  }
  cudaError_t e = launch_attn_bwd(t.dkdv, maps[0], maps[1], maps[2], maps[3], p,
                                  static_cast<int>(total), st, s);
  return e == cudaSuccess ? CP_OK : cuda_fail(e, "backward kernel launch");
}

// Set the accumulate / final flags from the first and last task touching
// each chunk, then run the tasks in order (only task `only` when >= 0).
int run_bwd_tasks(const BwdArgs& a, std::vector<BwdTask>& tasks, cudaStream_t s, int only = -1) {
  CUtensorMap maps[4];
  int rc = CP_OK;
  if (a.in_dt == CP_BF16) {
    const bool dims4 = a.stride > 1;
    rc = make_map(&maps[0], a.q, a.q_rows, a.H, a.stride, dims4);
    if (rc == CP_OK) rc = make_map(&maps[1], a.k, a.k_rows, a.Hkv, a.stride, dims4);
    if (rc == CP_OK) rc = make_map(&maps[2], a.v, a.k_rows, a.Hkv, a.stride, dims4);
    if (rc == CP_OK) rc = make_map(&maps[3], a.dout, a.q_rows, a.H, a.stride, dims4);
    if (rc != CP_OK) return rc;
  }
  for (int kind = 0; kind < 2; ++kind) {
    std::vector<int> first, last;
    auto at = [](std::vector<int>& v, int c) -> int& {
      if (static_cast<int>(v.size()) <= c) v.resize(c + 1, -1);
      return v[c];
    };
    for (int ti = 0; ti < static_cast<int>(tasks.size()); ++ti) {
      if (tasks[ti].dkdv != (kind == 1)) continue;
      for (int c : tasks[ti].chunk) {
        if (at(first, c) < 0) at(first, c) = ti;
        at(last, c) = ti;
      }
    }
    for (int ti = 0; ti < static_cast<int>(tasks.size()); ++ti) {
      if (tasks[ti].dkdv != (kind == 1)) continue;
      for (size_t i = 0; i < tasks[ti].items.size(); ++i) {
        const int c = tasks[ti].chunk[i];
        int f = 0;
        if (first[c] != ti) f |= kBwdAccumulate;
        if (a.grad_dt == CP_BF16 && last[c] == ti) f |= kBwdFinal;
        tasks[ti].items[i].flags = f;
      }
    }
  }
  for (int ti = 0; ti < static_cast<int>(tasks.size()); ++ti)
    if (only < 0 || only == ti)
      if ((rc = run_bwd_task(a, tasks[ti], maps, s)) != CP_OK) return rc;
  return CP_OK;
}

// The backward of the ring: per step the (query chunk, KV chunk) pairs of
// the forward; the dQ kernel runs one item per (rank, query chunk) against
// the held KV chunks, the dK/dV kernel one per (rank, held KV chunk) against
// the rank's query chunks that see it.
std::vector<BwdTask> ring_bwd_tasks(int64_t S, int P, cp_layout layout) {
  std::vector<BwdTask> tasks;
  if (layout == CP_STRIPED) {
    const int64_t C = S / P;
    for (int t = 0; t < P; ++t) {
      BwdTask tq{false, {}, {}}, tk{true, {}, {}};
      for (int r = 0; r < P; ++r) {
        const int src = ((r - t) % P + P) % P;
        const int64_t kpos = src > r ? 1 : 0;  // stripe-index mask j + (src > r) <= i
        BwdItem a{};
        a.stat = BwdSeg{0, 0, static_cast<int32_t>(C), r};
        a.str[0] = BwdSeg{0, kpos, static_cast<int32_t>(C), src};
        a.nstr = 1;
        tq.items.push_back(a);
        tq.chunk.push_back(r);
        BwdItem b{};
        b.stat = BwdSeg{0, kpos, static_cast<int32_t>(C), src};
        b.str[0] = BwdSeg{0, 0, static_cast<int32_t>(C), r};
        b.nstr = 1;
        tk.items.push_back(b);
        tk.chunk.push_back(src);
      }
      tasks.push_back(tk);
      tasks.push_back(tq);
    }
    return tasks;
  }
  const int64_t nchunks = layout == CP_ZIGZAG ? 2 * P : P;
  const int64_t C = (S + nchunks - 1) / nchunks;
  auto rows = [&](int c) -> int32_t {
    return static_cast<int32_t>(std::max<int64_t>(0, std::min<int64_t>(S, (c + 1) * C) - c * C));
  };
  auto seg = [&](int c) { return BwdSeg{c * C, c * C, rows(c), 0}; };
  for (int t = 0; t < P; ++t) {
    BwdTask tq{false, {}, {}}, tk{true, {}, {}};
    const std::vector<StepItem> items = step_items(P, layout, t);
    for (const StepItem& si : items) {
      if (rows(si.qc) == 0) continue;
      BwdItem a{};
      a.stat = seg(si.qc);
      for (int j = 0; j < si.nk; ++j)
        if (rows(si.kc[j]) > 0) a.str[a.nstr++] = seg(si.kc[j]);
      if (a.nstr == 0) continue;
      tq.items.push_back(a);
      tq.chunk.push_back(si.qc);
    }
    // transpose the step's pairs: per (rank, held KV chunk) the query chunks
    for (int r = 0; r < P; ++r) {
      const int src = ((r - t) % P + P) % P;
      int kcs[2], qcs[2];
      const int nk = rank_chunks(P, layout, src, kcs);
      const int nq = rank_chunks(P, layout, r, qcs);
      if (nq == 2 && qcs[0] > qcs[1]) std::swap(qcs[0], qcs[1]);
      for (int b = 0; b < nk; ++b) {
        if (rows(kcs[b]) == 0) continue;
        BwdItem it{};
        it.stat = seg(kcs[b]);
        for (int a = 0; a < nq; ++a)
          if (qcs[a] >= kcs[b] && rows(qcs[a]) > 0) it.str[it.nstr++] = seg(qcs[a]);
        if (it.nstr == 0) continue;
        tk.items.push_back(it);
        tk.chunk.push_back(kcs[b]);
      }
    }
    tasks.push_back(tk);
    tasks.push_back(tq);
  }
  return tasks;
}

// The ring's backward in two launches (bf16 inputs): the dK/dV
// kernel runs one item per KV chunk, streaming the query chunks that see it
// in the order the ring's steps bring them (at step t the chunk sits with
// rank owner + t, whose own query chunks not earlier than it are evaluated);
// the dQ kernel one item per (rank, own query chunk), streaming the KV chunks
// the rank holds at steps 0 .. P-1 not later than it -- the forward's walk.
// Each stationary tile keeps its gradient in TMEM across all steps and
// writes it once.
std::vector<BwdTask> ring_bwd_fused_tasks(int64_t S, int P, cp_layout layout) {
  if (layout == CP_STRIPED) {
    // every (key stripe, query stripe) pair has visible keys: the dK/dV item
    // of stripe c streams stripes c, c+1, ... (its holders at steps 0, 1,
    // ...), the dQ item of stripe r streams stripes r, r-1, ...
    const int64_t C = S / P;
    BwdTask tk{true, {}, {}, C, S, true}, tq{false, {}, {}, C, S, true};
    for (int c = 0; c < P; ++c) {
      BwdItem kt{}, qt{};
      kt.stat = BwdSeg{0, 0, static_cast<int32_t>(C), c};
      qt.stat = BwdSeg{0, 0, static_cast<int32_t>(C), c};
      for (int t = 0; t < P; ++t) {
        kt.chunk[kt.nchunk++] = static_cast<uint8_t>((c + t) % P);
        qt.chunk[qt.nchunk++] = static_cast<uint8_t>(((c - t) % P + P) % P);
      }
      tk.items.push_back(kt);
      tk.chunk.push_back(c);
      tq.items.push_back(qt);
      tq.chunk.push_back(c);
    }
    return {tk, tq};
  }
  const int64_t nchunks = layout == CP_ZIGZAG ? 2 * P : P;
  const int64_t C = (S + nchunks - 1) / nchunks;
  auto rows = [&](int c) -> int32_t {
    return static_cast<int32_t>(std::max<int64_t>(0, std::min<int64_t>(S, (c + 1) * C) - c * C));
  };
  auto seg = [&](int c) { return BwdSeg{c * C, c * C, rows(c), 0}; };
  auto owner = [&](int c) {
    return layout == CP_ZIGZAG && c >= P ? static_cast<int>(2 * P - 1 - c) : c;
  };
  BwdTask tk{true, {}, {}, C, S}, tq{false, {}, {}, C, S};
  std::vector<int64_t> wk, wq;  // streamed rows, for the longest-first order
  for (int kc = 0; kc < nchunks; ++kc) {
    if (rows(kc) == 0) continue;
    BwdItem it{};
    it.stat = seg(kc);
    int64_t w = 0;
    for (int t = 0; t < P; ++t) {
      int qcs[2];
      const int nq = rank_chunks(P, layout, (owner(kc) + t) % P, qcs);
      if (nq == 2 && qcs[0] > qcs[1]) std::swap(qcs[0], qcs[1]);
      for (int a = 0; a < nq; ++a)
        if (qcs[a] >= kc && rows(qcs[a]) > 0) {
          it.chunk[it.nchunk++] = static_cast<uint8_t>(qcs[a]);
          w += rows(qcs[a]);
        }
    }
    if (it.nchunk == 0) continue;
    tk.items.push_back(it);
    tk.chunk.push_back(kc);
    wk.push_back(w);
  }
  for (int r = 0; r < P; ++r) {
    int qcs[2];
    const int nq = rank_chunks(P, layout, r, qcs);
    for (int a = 0; a < nq; ++a) {
      const int qc = qcs[a];
      if (rows(qc) == 0) continue;
      BwdItem it{};
      it.stat = seg(qc);
      int64_t w = 0;
      for (int t = 0; t < P; ++t) {
        int kcs[2];
        const int nk = rank_chunks(P, layout, ((r - t) % P + P) % P, kcs);
        for (int b = 0; b < nk; ++b)
          if (kcs[b] <= qc && rows(kcs[b]) > 0) {
            it.chunk[it.nchunk++] = static_cast<uint8_t>(kcs[b]);
            w += rows(kcs[b]);
          }
      }
      tq.items.push_back(it);
      tq.chunk.push_back(qc);
      wq.push_back(w);
    }
  }
  // longest items first (the grid is scheduled roughly in order)
  auto sort_task = [](BwdTask& t, const std::vector<int64_t>& w) {
    std::vector<size_t> o(t.items.size());
    for (size_t i = 0; i < o.size(); ++i) o[i] = i;
    std::stable_sort(o.begin(), o.end(), [&](size_t a, size_t b) { return w[a] > w[b]; });
    BwdTask s{t.dkdv, {}, {}, t.ring_C, t.ring_S, t.striped};
    for (size_t i : o) {
      s.items.push_back(t.items[i]);
      s.chunk.push_back(t.chunk[i]);
    }
    t = s;
  };
  sort_task(tk, wk);
  sort_task(tq, wq);
  return {tk, tq};
}

int check_bwd_common(cp_dtype in_dt, int H, int Hkv, int D, cp_dtype grad_dt) {
  if (!valid_dtype(in_dt) || !valid_dtype(grad_dt)) return fail(CP_ERR_DTYPE, "unknown dtype");
  return check_heads_dims(in_dt, H, Hkv, D);
}

// delta = rowsum(dO * O) of the [rows, H, D] tensors into [H, ld]
cudaError_t launch_delta(cp_dtype in_dt, const void* out, const void* dout, float* delta,
                         int64_t rows, int H, int D, int64_t ld, cudaStream_t s) {
  return in_dt == CP_BF16 ? launch_bwd_delta(out, dout, delta, rows, H, ld, s)
                          : launch_bwd_delta_f32(out, dout, delta, rows, H, D, ld, s);
}

int64_t pad256(int64_t b) { return (b + 255) / 256 * 256; }

}  // namespace

namespace cpattn {
// Lets other translation units of the library report an error through
// cp_last_error() of the calling thread.
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

// Whether cp_ring_forward (and the host-buffer ring, Ulysses x ring) run all
// steps in one launch: bf16 inputs (tensor-core path), any layout.
bool ring_runs_fused(cp_dtype in_dt, cp_layout layout) {
  return in_dt == CP_BF16 &&
         (layout == CP_CONTIGUOUS || layout == CP_ZIGZAG || layout == CP_STRIPED);
}

// Whether cp_ring_backward runs in two launches over all steps: bf16 inputs,
// any layout.
bool ring_bwd_runs_fused(cp_dtype in_dt, cp_layout layout) {
  return ring_runs_fused(in_dt, layout);
}
}  // namespace cpattn

// =================================================================== C ABI
extern "C" {

const char* cp_last_error(void) { return g_last_error.c_str(); }

const char* cp_version(void) { return "cpattn 0.1 (sm_103a)"; }

int cp_attn_block(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t Sq,
                  int64_t Sk, int H, int Hkv, int D, int64_t q_offset, int64_t k_offset,
                  int causal, float scale, void* out, cp_dtype out_dt, float* lse,
                  cp_stream_t stream) {
  int rc = check_heads_dims(in_dt, H, Hkv, D);
  if (rc != CP_OK) return rc;
  if (!valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown output dtype %d", int(out_dt));
  if (Sq < 0 || Sk < 0 || Sq >= (int64_t(1) << 31) || Sk >= (int64_t(1) << 31))
    return fail(CP_ERR_ARG, "Sq=%lld / Sk=%lld out of range", (long long)Sq, (long long)Sk);
  if (std::llabs(q_offset) >= (int64_t(1) << 40) || std::llabs(k_offset) >= (int64_t(1) << 40))
    return fail(CP_ERR_ARG, "offsets out of range");
  if (Sq == 0) return ok();
  if (!q || !out || !lse || (Sk > 0 && (!k || !v)))
    return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(out) || (Sk > 0 && (!aligned16(k) || !aligned16(v))))
    return fail(CP_ERR_ALIGN, "q, k, v and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3) != 0)
    return fail(CP_ERR_ALIGN, "lse must be 4-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (Sk == 0) {
    cudaError_t e = launch_fill_empty(out, elem_bytes(out_dt), Sq * H * D, lse, Sq * H, s);
    return e == cudaSuccess ? ok() : cuda_fail(e, "fill launch");
  }
  Launch L;
  fill_common(L.p, H, Hkv, D, scale, out_dt, out, nullptr, lse, Sq);
  WorkItem w{};
  w.q_mem_row = 0;
  w.q_pos = q_offset;
  w.o_row = 0;
  w.lse_col = 0;
  w.sq = static_cast<int32_t>(Sq);
  w.nseg = 1;
  w.batch = 1;
  w.flags = kFlagFinal | (causal ? kFlagCausal : 0);
  w.seg[0].mem_row = 0;
  w.seg[0].pos = k_offset;
  w.seg[0].len = static_cast<int32_t>(Sk);
  L.items.push_back(w);
  rc = launch_items(L, in_dt, q, Sq, k, v, Sk, s);
  return rc == CP_OK ? ok() : rc;
}

int cp_lse_merge(float* out_acc, float* lse_acc, const float* out_blk, const float* lse_blk,
                 int64_t Sq, int H, int D, cp_stream_t stream) {
  if (Sq < 0 || H < 1 || D < 4)
    return fail(CP_ERR_ARG, "bad sizes Sq=%lld H=%d D=%d", (long long)Sq, H, D);
  const int d4 = D / 4;
  if (D % 4 != 0 || (d4 < 32 && (d4 & (d4 - 1)) != 0) || (d4 >= 32 && d4 % 32 != 0))
    return fail(CP_ERR_SHAPE,
                "D=%d: need D %% 4 == 0 and D/4 a power of two or a multiple of 32", D);
  if (Sq == 0) return ok();
  if (!out_acc || !lse_acc || !out_blk || !lse_blk)
    return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(out_acc) || !aligned16(out_blk))
    return fail(CP_ERR_ALIGN, "out buffers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse_acc) | reinterpret_cast<uintptr_t>(lse_blk)) & 3)
    return fail(CP_ERR_ALIGN, "lse buffers must be 4-byte aligned");
  cudaError_t e = launch_lse_merge(out_acc, lse_acc, out_blk, lse_blk, Sq, H, D,
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "merge launch");
}

int64_t cp_ring_workspace_size(int64_t S, int H, int D, cp_dtype out_dt) {
  if (S < 0 || H < 1 || D < 1) return fail(CP_ERR_ARG, "bad sizes");
  if (!valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown output dtype %d", int(out_dt));
  ok();
  return out_dt == CP_BF16 ? S * H * D * 4 : 0;
}

// One validated ring step; dependent: see launch_items (only for steps that
// directly follow the previous step of the same ring on the stream).
static int ring_step_checked(const void* q, const void* k, const void* v, cp_dtype in_dt,
                             int64_t S, int H, int Hkv, int D, int P, cp_layout layout, int step,
                             void* out, cp_dtype out_dt, float* lse, void* workspace,
                             cp_stream_t stream, bool dependent) {
  int rc = check_ring(in_dt, S, H, Hkv, D, P, layout, out_dt);
  if (rc != CP_OK) return rc;
  if (step < 0 || step >= P) return fail(CP_ERR_ARG, "step=%d outside [0,%d)", step, P);
  if (!q || !k || !v || !out || !lse) return fail(CP_ERR_ARG, "null pointer argument");
  if (out_dt == CP_BF16 && !workspace)
    return fail(CP_ERR_ARG, "bf16 output needs a workspace (cp_ring_workspace_size)");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (workspace && !aligned16(workspace)))
    return fail(CP_ERR_ALIGN, "q, k, v, out and workspace must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3) != 0)
    return fail(CP_ERR_ALIGN, "lse must be 4-byte aligned");
  rc = ring_step_impl(q, k, v, in_dt, S, H, Hkv, D, P, layout, step, out, out_dt, lse, workspace,
                      reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, dependent);
  return rc == CP_OK ? ok() : rc;
}

int cp_ring_step(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S, int H,
                 int Hkv, int D, int P, cp_layout layout, int step, void* out, cp_dtype out_dt,
                 float* lse, void* workspace, cp_stream_t stream) {
  return ring_step_checked(q, k, v, in_dt, S, H, Hkv, D, P, layout, step, out, out_dt, lse,
                           workspace, stream, false);
}

static int ring_fused_checked(const void* q, const void* k, const void* v, cp_dtype in_dt,
                              int64_t S, int H, int Hkv, int D, int P, cp_layout layout, void* out,
                              cp_dtype out_dt, float* lse, cp_stream_t stream) {
  int rc = check_ring(in_dt, S, H, Hkv, D, P, layout, out_dt);
  if (rc != CP_OK) return rc;
  if (in_dt != CP_BF16)
    return fail(CP_ERR_DTYPE, "the one-launch ring needs bf16 inputs (tensor-core path)");
  if (!q || !k || !v || !out || !lse) return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(CP_ERR_ALIGN, "q, k, v and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3) != 0)
    return fail(CP_ERR_ALIGN, "lse must be 4-byte aligned");
  rc = ring_fused_impl(q, k, v, S, H, Hkv, D, P, layout, out, out_dt, lse,
                       reinterpret_cast<cudaStream_t>(stream));
  return rc == CP_OK ? ok() : rc;
}

int cp_ring_forward_fused(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                          int H, int Hkv, int D, int P, cp_layout layout, void* out,
                          cp_dtype out_dt, float* lse, cp_stream_t stream) {
  return ring_fused_checked(q, k, v, in_dt, S, H, Hkv, D, P, layout, out, out_dt, lse, stream);
}

int cp_ring_forward_steps(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                          int H, int Hkv, int D, int P, cp_layout layout, void* out,
                          cp_dtype out_dt, float* lse, void* workspace, cp_stream_t stream) {
  int rc = check_ring(in_dt, S, H, Hkv, D, P, layout, out_dt);
  if (rc != CP_OK) return rc;
  for (int t = 0; t < P; ++t) {
    rc = ring_step_checked(q, k, v, in_dt, S, H, Hkv, D, P, layout, t, out, out_dt, lse,
                           workspace, stream, t > 0);
    if (rc != CP_OK) return rc;
  }
  return ok();
}

int cp_ring_forward(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S, int H,
                    int Hkv, int D, int P, cp_layout layout, void* out, cp_dtype out_dt,
                    float* lse, void* workspace, cp_stream_t stream) {
  int rc = check_ring(in_dt, S, H, Hkv, D, P, layout, out_dt);
  if (rc != CP_OK) return rc;
  // the tensor-core path runs the steps in one launch (measured faster at
  // every length: no per-step epilogue, accumulator round trip or launch)
  if (ring_runs_fused(in_dt, layout))
    return ring_fused_checked(q, k, v, in_dt, S, H, Hkv, D, P, layout, out, out_dt, lse, stream);
  for (int t = 0; t < P; ++t) {
    rc = ring_step_checked(q, k, v, in_dt, S, H, Hkv, D, P, layout, t, out, out_dt, lse,
                           workspace, stream, t > 0);
    if (rc != CP_OK) return rc;
  }
  return ok();
}

int64_t cp_ring_copy_workspace_size(int64_t S, int H, int Hkv, int D, int P, cp_layout layout,
                                    cp_dtype in_dt, cp_dtype out_dt) {
  if (S < 1 || H < 1 || Hkv < 1 || D < 1 || P < 1 || P > CP_MAX_RANKS)
    return fail(CP_ERR_ARG, "bad sizes");
  if (!valid_dtype(in_dt) || !valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown dtype");
  if (layout != CP_CONTIGUOUS && layout != CP_ZIGZAG && layout != CP_STRIPED)
    return fail(CP_ERR_ARG, "unknown layout");
  ok();
  const int64_t acc = out_dt == CP_BF16 ? S * H * D * 4 : 0;
  const int64_t buf = 2 * P * ring_rank_rows(S, P, layout) * Hkv * D * elem_bytes(in_dt);
  return (acc + 255) / 256 * 256 + 2 * ((buf + 255) / 256 * 256);
}

int cp_ring_forward_copy(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                         int H, int Hkv, int D, int P, cp_layout layout, void* out,
                         cp_dtype out_dt, float* lse, void* workspace, cp_stream_t compute_stream,
                         cp_stream_t copy_stream) {
  int rc = check_ring(in_dt, S, H, Hkv, D, P, layout, out_dt);
  if (rc != CP_OK) return rc;
  if (!q || !k || !v || !out || !lse || !workspace)
    return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(workspace))
    return fail(CP_ERR_ALIGN, "q, k, v, out and workspace must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3) != 0)
    return fail(CP_ERR_ALIGN, "lse must be 4-byte aligned");
  rc = ring_forward_copy_impl(q, k, v, in_dt, S, H, Hkv, D, P, layout, out, out_dt, lse, workspace,
                              reinterpret_cast<cudaStream_t>(compute_stream),
                              reinterpret_cast<cudaStream_t>(copy_stream));
  return rc == CP_OK ? ok() : rc;
}

// Ordering and copies of the host-buffer entry points.  G head groups:
// group g's inputs go in on the copy stream, its kernels run on the compute
// stream, its results come back on a third stream (created and destroyed
// here, so that device-to-host copies need not queue behind the remaining
// host-to-device ones); events (also created and destroyed here) keep each
// stream behind the others where it must be.  With one stream for compute
// and copies, everything simply runs in order on it.
class HostGroupPipeline {
 public:
  HostGroupPipeline(cudaStream_t cs, cudaStream_t xs, int groups)
      : cs_(cs), xs_(xs), os_(xs), G_(groups), overlap_(cs != xs),
        ev_(overlap_ ? 2 * groups + 3 : 0, nullptr) {
    // events: inputs of group g in (g), group g computed (G + g), all inputs
    // in (2G), all results out (2G + 1), earlier work on the compute stream
    // done (2G + 2)
    for (auto& e : ev_)
      if (!check(cudaEventCreateWithFlags(&e, cudaEventDisableTiming))) break;
    if (overlap_ && ok() && check(cudaStreamCreateWithFlags(&own_, cudaStreamNonBlocking)))
      os_ = own_;
    // the copies start after the work already enqueued on the compute
    // stream, which may still be using the staging area
    if (overlap_ && ok() && check(cudaEventRecord(ev_[2 * G_ + 2], cs_))) {
      check(cudaStreamWaitEvent(xs_, ev_[2 * G_ + 2], 0));
      check(cudaStreamWaitEvent(os_, ev_[2 * G_ + 2], 0));
    }
  }
  ~HostGroupPipeline() {
    // an early return (a failed launch) still joins the copy streams, so the
    // caller's host buffers are free once the compute stream has passed
    finish();
    // both are released once the device has passed them
    for (cudaEvent_t e : ev_)
      if (e) cudaEventDestroy(e);
    if (own_) cudaStreamDestroy(own_);
  }
  HostGroupPipeline(const HostGroupPipeline&) = delete;
  HostGroupPipeline& operator=(const HostGroupPipeline&) = delete;
  bool ok() const { return err_ == cudaSuccess; }
  cudaError_t error() const { return err_; }
  // `rows` rows of `width` bytes: host (row pitch `pitch`) -> compact device
  void in(char* dev, const void* host, size_t width, size_t pitch, size_t rows) {
    check(cudaMemcpy2DAsync(dev, width, host, pitch, width, rows, cudaMemcpyHostToDevice, xs_));
  }
  // compact device -> host (row pitch `pitch`)
  void out(void* host, const char* dev, size_t width, size_t pitch, size_t rows) {
    check(cudaMemcpy2DAsync(host, pitch, dev, width, width, rows, cudaMemcpyDeviceToHost, os_));
  }
  void inputs_done(int g) {
    if (overlap_) check(cudaEventRecord(ev_[g], xs_));
  }
  void compute_begin(int g) {
    if (overlap_) check(cudaStreamWaitEvent(cs_, ev_[g], 0));
  }
  void compute_end(int g) {
    if (overlap_ && check(cudaEventRecord(ev_[G_ + g], cs_)))
      check(cudaStreamWaitEvent(os_, ev_[G_ + g], 0));
  }
  // The compute stream waits for the last copy in each direction.  This
  // runs after an error too (then from the destructor), so that no copy the
  // call enqueued outlives the compute stream's later work.
  void finish() {
    if (!overlap_ || joined_) return;
    joined_ = true;
    join(xs_, ev_[2 * G_]);
    join(os_, ev_[2 * G_ + 1]);
  }

 private:
  void join(cudaStream_t from, cudaEvent_t e) {
    cudaError_t r = e ? cudaEventRecord(e, from) : cudaErrorInvalidResourceHandle;
    if (r == cudaSuccess) r = cudaStreamWaitEvent(cs_, e, 0);
    if (r != cudaSuccess) r = cudaStreamSynchronize(from);  // no event: wait on the host
    check(r);
  }
  bool check(cudaError_t e) {
    if (err_ == cudaSuccess) err_ = e;
    return err_ == cudaSuccess;
  }
  cudaStream_t cs_, xs_, os_;
  cudaStream_t own_ = nullptr;  // the device-to-host stream
  int G_;
  bool overlap_;
  std::vector<cudaEvent_t> ev_;
  cudaError_t err_ = cudaSuccess;
  bool joined_ = false;
};

// Device staging of cp_ring_forward_host: q, k, v, out, lse of every group
// (compact per group), then one group's fp32 accumulator.
struct HostStaging {
  int64_t q, k, v, out, lse, acc, total;
};

static HostStaging host_staging(int64_t S, int H, int Hkv, int D, int groups, cp_dtype in_dt,
                                cp_dtype out_dt) {
  const int64_t ei = elem_bytes(in_dt), eo = elem_bytes(out_dt);
  HostStaging h;
  h.q = 0;
  h.k = h.q + pad256(S * H * D * ei);
  h.v = h.k + pad256(S * Hkv * D * ei);
  h.out = h.v + pad256(S * Hkv * D * ei);
  h.lse = h.out + pad256(S * H * D * eo);
  h.acc = h.lse + pad256(S * H * 4);
  h.total = h.acc + (out_dt == CP_BF16 ? pad256(S * (H / groups) * D * 4) : 0);
  return h;
}

int64_t cp_ring_host_workspace_size(int64_t S, int H, int Hkv, int D, int groups,
                                    cp_dtype in_dt, cp_dtype out_dt) {
  if (S < 1 || H < 1 || Hkv < 1 || D < 1) return fail(CP_ERR_ARG, "bad sizes");
  if (!valid_dtype(in_dt) || !valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown dtype");
  if (groups < 1 || Hkv % groups != 0)
    return fail(CP_ERR_SHAPE, "groups=%d must divide Hkv=%d", groups, Hkv);
  ok();
  return host_staging(S, H, Hkv, D, groups, in_dt, out_dt).total;
}

int cp_ring_forward_host(const void* hq, const void* hk, const void* hv, cp_dtype in_dt,
                         int64_t S, int H, int Hkv, int D, int P, cp_layout layout, void* hout,
                         cp_dtype out_dt, float* hlse, int groups, void* workspace,
                         cp_stream_t stream, cp_stream_t copy_stream) {
  int rc = check_ring(in_dt, S, H, Hkv, D, P, layout, out_dt);
  if (rc != CP_OK) return rc;
  if (groups < 1 || Hkv % groups != 0)
    return fail(CP_ERR_SHAPE, "groups=%d must divide Hkv=%d", groups, Hkv);
  if (!hq || !hk || !hv || !hout || !hlse || !workspace)
    return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(workspace)) return fail(CP_ERR_ALIGN, "workspace must be 16-byte aligned");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t xs = reinterpret_cast<cudaStream_t>(copy_stream);
  const int G = groups, Hg = H / G, Hkg = Hkv / G;
  const size_t ei = elem_bytes(in_dt), eo = elem_bytes(out_dt);
  const HostStaging st = host_staging(S, H, Hkv, D, G, in_dt, out_dt);
  char* ws = static_cast<char*>(workspace);
  // group g's compact tensors inside the staging areas
  const size_t qg = static_cast<size_t>(S) * Hg * D * ei;
  const size_t kg = static_cast<size_t>(S) * Hkg * D * ei;
  const size_t og = static_cast<size_t>(S) * Hg * D * eo, lg = static_cast<size_t>(S) * Hg * 4;
  const size_t q_pitch = static_cast<size_t>(H) * D * ei;
  const size_t kv_pitch = static_cast<size_t>(Hkv) * D * ei;
  const size_t o_pitch = static_cast<size_t>(H) * D * eo;
  const size_t q_w = static_cast<size_t>(Hg) * D * ei, kv_w = static_cast<size_t>(Hkg) * D * ei;
  const size_t o_w = static_cast<size_t>(Hg) * D * eo;
  HostGroupPipeline pl(cs, xs, G);
  // inputs of every group, in group order, on the copy stream
  for (int g = 0; g < G && pl.ok(); ++g) {
    pl.in(ws + st.q + g * qg, static_cast<const char*>(hq) + g * q_w, q_w, q_pitch, S);
    pl.in(ws + st.k + g * kg, static_cast<const char*>(hk) + g * kv_w, kv_w, kv_pitch, S);
    pl.in(ws + st.v + g * kg, static_cast<const char*>(hv) + g * kv_w, kv_w, kv_pitch, S);
    pl.inputs_done(g);
  }
  // each group's ring on the compute stream, then its results out
  for (int g = 0; g < G && pl.ok(); ++g) {
    pl.compute_begin(g);
    char* dq = ws + st.q + g * qg;
    char* dk = ws + st.k + g * kg;
    char* dv = ws + st.v + g * kg;
    char* dout = ws + st.out + g * og;
    float* dlse = reinterpret_cast<float*>(ws + st.lse + g * lg);
    if (ring_runs_fused(in_dt, layout)) {
      rc = ring_fused_impl(dq, dk, dv, S, Hg, Hkg, D, P, layout, dout, out_dt, dlse, cs);
      if (rc != CP_OK) return rc;
    } else {
      for (int t = 0; t < P; ++t) {
        rc = ring_step_impl(dq, dk, dv, in_dt, S, Hg, Hkg, D, P, layout, t, dout, out_dt, dlse,
                            ws + st.acc, cs, nullptr, nullptr, t > 0);
        if (rc != CP_OK) return rc;
      }
    }
    pl.compute_end(g);
    pl.out(static_cast<char*>(hout) + g * o_w, dout, o_w, o_pitch, S);
    pl.out(hlse + static_cast<size_t>(g) * Hg * S, reinterpret_cast<const char*>(dlse), lg, lg, 1);
  }
  pl.finish();
  if (!pl.ok()) return cuda_fail(pl.error(), "host ring copies");
  return ok();
}

int cp_ring_step_blocks(int P, cp_layout layout, int step, int* blocks, int cap) {
  if (P < 1 || P > CP_MAX_RANKS) return fail(CP_ERR_ARG, "P=%d outside [1,%d]", P, CP_MAX_RANKS);
  if (layout != CP_CONTIGUOUS && layout != CP_ZIGZAG && layout != CP_STRIPED)
    return fail(CP_ERR_ARG, "unknown layout");
  if (step < 0 || step >= P) return fail(CP_ERR_ARG, "step out of range");
  if (cap < 0 || (cap > 0 && !blocks)) return fail(CP_ERR_ARG, "bad output buffer");
  int n = 0;
  for (const StepItem& it : step_items(P, layout, step))
    for (int s = 0; s < it.nk; ++s) {
      if (n < cap) {
        blocks[4 * n + 0] = it.rank;
        blocks[4 * n + 1] = it.qc;
        blocks[4 * n + 2] = it.kc[s];
        blocks[4 * n + 3] = it.kc[s] == it.qc ? 1 : 0;
      }
      ++n;
    }
  ok();
  return n;
}

static int check_perm(const void* a, const void* b, cp_dtype dt, int64_t S, int H, int D, int P) {
  if (!valid_dtype(dt)) return fail(CP_ERR_DTYPE, "unknown dtype %d", int(dt));
  if (S < 0 || H < 1 || D < 1 || P < 1) return fail(CP_ERR_ARG, "bad sizes");
  if (S % P != 0 || H % P != 0)
    return fail(CP_ERR_SHAPE, "S=%lld and H=%d must be multiples of P=%d", (long long)S, H, P);
  if (S > 0 && (!a || !b)) return fail(CP_ERR_ARG, "null pointer argument");
  return CP_OK;
}

int cp_seq_to_head(const void* x, void* y, cp_dtype dt, int64_t S, int H, int D, int P,
                   cp_stream_t stream) {
  int rc = check_perm(x, y, dt, S, H, D, P);
  if (rc != CP_OK) return rc;
  if (S == 0) return ok();
  const int64_t run = static_cast<int64_t>(H / P) * D * elem_bytes(dt);
  // x viewed as [S][P][run] -> y [P][S][run]
  cudaError_t e = launch_permute(x, y, S, P, run, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "permute launch");
}

int cp_head_to_seq(const void* y, void* x, cp_dtype dt, int64_t S, int H, int D, int P,
                   cp_stream_t stream) {
  int rc = check_perm(y, x, dt, S, H, D, P);
  if (rc != CP_OK) return rc;
  if (S == 0) return ok();
  const int64_t run = static_cast<int64_t>(H / P) * D * elem_bytes(dt);
  // y viewed as [P][S][run] -> x [S][P][run]
  cudaError_t e = launch_permute(y, x, P, S, run, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "permute launch");
}

int64_t cp_ulysses_workspace_size(int64_t S, int H, int Hkv, int D, cp_dtype in_dt,
                                  cp_dtype out_dt) {
  if (S < 0 || H < 1 || Hkv < 1 || D < 1) return fail(CP_ERR_ARG, "bad sizes");
  if (!valid_dtype(in_dt) || !valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown dtype");
  ok();
  const int64_t ei = elem_bytes(in_dt), eo = elem_bytes(out_dt);
  return pad256(S * H * D * ei) + 2 * pad256(S * Hkv * D * ei) + pad256(S * H * D * eo);
}

// stage -1: the whole forward; 0: seq_to_head of q, k, v; 1: the attention
// launch; 2: head_to_seq of the output.
static int ulysses_impl(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                        int H, int Hkv, int D, int P, void* out, cp_dtype out_dt, float* lse,
                        void* workspace, cp_stream_t stream, int stage) {
  int rc = check_heads_dims(in_dt, H, Hkv, D);
  if (rc != CP_OK) return rc;
  if (!valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown output dtype %d", int(out_dt));
  if (P < 1 || P > CP_MAX_RANKS) return fail(CP_ERR_ARG, "P=%d outside [1,%d]", P, CP_MAX_RANKS);
  if (S < 1 || S >= (int64_t(1) << 28))
    return fail(CP_ERR_ARG, "S=%lld out of range", (long long)S);
  if (S % P != 0) return fail(CP_ERR_SHAPE, "S=%lld is not a multiple of P=%d", (long long)S, P);
  // degree above the KV head count: each KV head serves P/Hkv ranks (read in
  // place, no copy); otherwise P must divide Hkv
  const bool replicate = P > Hkv && P % Hkv == 0;
  if (H % P != 0 || (!replicate && Hkv % P != 0))
    return fail(CP_ERR_SHAPE,
                "Ulysses degree P=%d must divide H=%d and either divide Hkv=%d or be a "
                "multiple of it",
                P, H, Hkv);
  if (!q || !k || !v || !out || !lse || !workspace)
    return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(workspace))
    return fail(CP_ERR_ALIGN, "q, k, v, out and workspace must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t ei = elem_bytes(in_dt), eo = elem_bytes(out_dt);
  char* ws = static_cast<char*>(workspace);
  void* qh = ws;
  void* kh = ws + pad256(S * H * D * ei);
  void* vh = static_cast<char*>(kh) + pad256(S * Hkv * D * ei);
  void* oh = static_cast<char*>(vh) + pad256(S * Hkv * D * ei);
  if (stage < 0 || stage == 0) {
    if ((rc = cp_seq_to_head(q, qh, in_dt, S, H, D, P, stream)) != CP_OK) return rc;
    if (!replicate) {
      if ((rc = cp_seq_to_head(k, kh, in_dt, S, Hkv, D, P, stream)) != CP_OK) return rc;
      if ((rc = cp_seq_to_head(v, vh, in_dt, S, Hkv, D, P, stream)) != CP_OK) return rc;
    }
  }
  if (stage == 2) return cp_head_to_seq(oh, out, out_dt, S, H, D, P, stream);
  if (stage == 0) return ok();
  // every rank's head group: full-sequence causal attention, one launch
  const int G = H / P, Gkv = replicate ? Hkv : Hkv / P;
  Launch L;
  fill_common(L.p, G, Gkv, D, 0.f, out_dt, oh, nullptr, lse, S);
  if (replicate) {
    // rank b's local query head h is global head b*G + h; its KV head is
    // (b*G + h) / (H/Hkv) in the unpermuted k, v
    L.p.b_q_heads = G;
    L.p.kv_group = H / Hkv;
  }
  WorkItem w{};
  w.q_mem_row = 0;
  w.q_pos = 0;
  w.o_row = 0;
  w.lse_col = 0;
  w.sq = static_cast<int32_t>(S);
  w.nseg = 1;
  w.batch = P;
  w.flags = kFlagFinal | kFlagCausal;
  w.b_q_rows = S;
  w.b_k_rows = replicate ? 0 : S;
  w.b_o_rows = S;
  w.b_lse_heads = G;
  w.seg[0].mem_row = 0;
  w.seg[0].pos = 0;
  w.seg[0].len = static_cast<int32_t>(S);
  L.items.push_back(w);
  if ((rc = launch_items(L, in_dt, qh, P * S, replicate ? k : kh, replicate ? v : vh,
                         replicate ? S : P * S, s)) != CP_OK)
    return rc;
  if (stage == 1) return ok();
  if ((rc = cp_head_to_seq(oh, out, out_dt, S, H, D, P, stream)) != CP_OK) return rc;
  return ok();
}

int cp_ulysses_forward(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                       int H, int Hkv, int D, int P, void* out, cp_dtype out_dt, float* lse,
                       void* workspace, cp_stream_t stream) {
  return ulysses_impl(q, k, v, in_dt, S, H, Hkv, D, P, out, out_dt, lse, workspace, stream, -1);
}

int cp_ulysses_stage(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S,
                     int H, int Hkv, int D, int P, void* out, cp_dtype out_dt, float* lse,
                     void* workspace, int stage, cp_stream_t stream) {
  if (stage < 0 || stage > 2) return fail(CP_ERR_ARG, "stage=%d outside [0,2]", stage);
  return ulysses_impl(q, k, v, in_dt, S, H, Hkv, D, P, out, out_dt, lse, workspace, stream, stage);
}

// Ulysses degree checks shared by the host-buffer variant: P divides H and
// divides Hkv or is a multiple of it.
static int check_ulysses_degree(int H, int Hkv, int P, bool* replicate) {
  if (P < 1 || P > CP_MAX_RANKS) return fail(CP_ERR_ARG, "P=%d outside [1,%d]", P, CP_MAX_RANKS);
  *replicate = P > Hkv && P % Hkv == 0;
  if (H % P != 0 || (!*replicate && Hkv % P != 0))
    return fail(CP_ERR_SHAPE,
                "Ulysses degree P=%d must divide H=%d and either divide Hkv=%d or be a "
                "multiple of it",
                P, H, Hkv);
  return CP_OK;
}

// Device staging of cp_ulysses_forward_host: every group's compact q, k, v,
// out (k, v: one KV head per group when the heads are replicated) and lse.
// With a ring inside each group (USP), one group's fp32 accumulator follows.
struct UlyssesHostStaging {
  int64_t q, k, v, out, lse, acc, total;
};

static UlyssesHostStaging ulysses_host_staging(int64_t S, int H, int Hkv, int D, int P,
                                               bool replicate, cp_dtype in_dt, cp_dtype out_dt,
                                               bool ring = false) {
  const int64_t ei = elem_bytes(in_dt), eo = elem_bytes(out_dt);
  const int64_t gkv = replicate ? 1 : Hkv / P;
  UlyssesHostStaging h;
  h.q = 0;
  h.k = h.q + pad256(S * H * D * ei);
  h.v = h.k + pad256(P * S * gkv * D * ei);
  h.out = h.v + pad256(P * S * gkv * D * ei);
  h.lse = h.out + pad256(S * H * D * eo);
  h.acc = h.lse + pad256(S * H * 4);
  h.total = h.acc + (ring && out_dt == CP_BF16 ? pad256(S * (H / P) * D * 4) : 0);
  return h;
}

int64_t cp_ulysses_host_workspace_size(int64_t S, int H, int Hkv, int D, int P, cp_dtype in_dt,
                                       cp_dtype out_dt) {
  if (S < 1 || H < 1 || Hkv < 1 || D < 1) return fail(CP_ERR_ARG, "bad sizes");
  if (!valid_dtype(in_dt) || !valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown dtype");
  bool replicate = false;
  const int rc = check_ulysses_degree(H, Hkv, P, &replicate);
  if (rc != CP_OK) return rc;
  ok();
  return ulysses_host_staging(S, H, Hkv, D, P, replicate, in_dt, out_dt).total;
}

// Pr = 0: each group's causal attention is one cp_attn_block; Pr >= 1: a
// ring of Pr virtual ranks in `layout` over the group's sequence (USP).
static int ulysses_host_impl(const void* hq, const void* hk, const void* hv, cp_dtype in_dt,
                             int64_t S, int H, int Hkv, int D, int P, int Pr, cp_layout layout,
                             void* hout, cp_dtype out_dt, float* hlse, void* workspace,
                             cp_stream_t stream, cp_stream_t copy_stream) {
  int rc = check_heads_dims(in_dt, H, Hkv, D);
  if (rc != CP_OK) return rc;
  if (!valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown output dtype %d", int(out_dt));
  if (S < 1 || S >= (int64_t(1) << 31))
    return fail(CP_ERR_ARG, "S=%lld out of range", (long long)S);
  bool replicate = false;
  if ((rc = check_ulysses_degree(H, Hkv, P, &replicate)) != CP_OK) return rc;
  if (Pr > 0 && (rc = check_ring(in_dt, S, H / P, replicate ? 1 : Hkv / P, D, Pr, layout,
                                 out_dt)) != CP_OK)
    return rc;
  if (!hq || !hk || !hv || !hout || !hlse || !workspace)
    return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(workspace)) return fail(CP_ERR_ALIGN, "workspace must be 16-byte aligned");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t xs = reinterpret_cast<cudaStream_t>(copy_stream);
  const int G = H / P, Gkv = replicate ? 1 : Hkv / P;
  const size_t ei = elem_bytes(in_dt), eo = elem_bytes(out_dt), rows = static_cast<size_t>(S);
  const UlyssesHostStaging st =
      ulysses_host_staging(S, H, Hkv, D, P, replicate, in_dt, out_dt, Pr > 0);
  char* ws = static_cast<char*>(workspace);
  const size_t qw = static_cast<size_t>(G) * D * ei, kw = static_cast<size_t>(Gkv) * D * ei;
  const size_t ow = static_cast<size_t>(G) * D * eo, lw = static_cast<size_t>(G) * S * 4;
  HostGroupPipeline pl(cs, xs, P);
  // rank p's heads land in its own compact block: the seq -> head all-to-all
  for (int p = 0; p < P && pl.ok(); ++p) {
    // KV heads of group p: its Gkv heads, or (replicated) the one its query
    // heads read
    const int kv0 = replicate ? (p * G) / (H / Hkv) : p * Gkv;
    pl.in(ws + st.q + p * rows * qw, static_cast<const char*>(hq) + p * qw, qw,
          static_cast<size_t>(H) * D * ei, rows);
    pl.in(ws + st.k + p * rows * kw, static_cast<const char*>(hk) + kv0 * D * ei, kw,
          static_cast<size_t>(Hkv) * D * ei, rows);
    pl.in(ws + st.v + p * rows * kw, static_cast<const char*>(hv) + kv0 * D * ei, kw,
          static_cast<size_t>(Hkv) * D * ei, rows);
    pl.inputs_done(p);
  }
  for (int p = 0; p < P && pl.ok(); ++p) {
    pl.compute_begin(p);
    char* out_p = ws + st.out + p * rows * ow;
    float* lse_p = reinterpret_cast<float*>(ws + st.lse + p * lw);
    char* q_p = ws + st.q + p * rows * qw;
    char* k_p = ws + st.k + p * rows * kw;
    char* v_p = ws + st.v + p * rows * kw;
    if (Pr > 0 && ring_runs_fused(in_dt, layout)) {
      rc = ring_fused_impl(q_p, k_p, v_p, S, G, Gkv, D, Pr, layout, out_p, out_dt, lse_p, cs);
      if (rc != CP_OK) return rc;
    } else if (Pr > 0) {
      for (int t = 0; t < Pr; ++t) {
        rc = ring_step_impl(q_p, k_p, v_p, in_dt, S, G, Gkv, D, Pr, layout, t, out_p, out_dt,
                            lse_p, ws + st.acc, cs, nullptr, nullptr, t > 0);
        if (rc != CP_OK) return rc;
      }
    } else {
      rc = cp_attn_block(q_p, k_p, v_p, in_dt, S, S, G, Gkv, D, 0, 0, 1, 0.f, out_p, out_dt, lse_p,
                         stream);
      if (rc != CP_OK) return rc;
    }
    pl.compute_end(p);
    // ... and back to its heads of hout: the head -> seq all-to-all
    pl.out(static_cast<char*>(hout) + p * ow, out_p, ow, static_cast<size_t>(H) * D * eo, rows);
    pl.out(hlse + static_cast<size_t>(p) * G * S, reinterpret_cast<const char*>(lse_p), lw, lw, 1);
  }
  pl.finish();
  if (!pl.ok()) return cuda_fail(pl.error(), "host Ulysses copies");
  return ok();
}

int cp_ulysses_forward_host(const void* hq, const void* hk, const void* hv, cp_dtype in_dt,
                            int64_t S, int H, int Hkv, int D, int P, void* hout, cp_dtype out_dt,
                            float* hlse, void* workspace, cp_stream_t stream,
                            cp_stream_t copy_stream) {
  return ulysses_host_impl(hq, hk, hv, in_dt, S, H, Hkv, D, P, 0, CP_ZIGZAG, hout, out_dt, hlse,
                           workspace, stream, copy_stream);
}

int64_t cp_usp_host_workspace_size(int64_t S, int H, int Hkv, int D, int Pu, cp_dtype in_dt,
                                   cp_dtype out_dt) {
  if (S < 1 || H < 1 || Hkv < 1 || D < 1) return fail(CP_ERR_ARG, "bad sizes");
  if (!valid_dtype(in_dt) || !valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown dtype");
  bool replicate = false;
  const int rc = check_ulysses_degree(H, Hkv, Pu, &replicate);
  if (rc != CP_OK) return rc;
  ok();
  return ulysses_host_staging(S, H, Hkv, D, Pu, replicate, in_dt, out_dt, true).total;
}

int cp_usp_forward_host(const void* hq, const void* hk, const void* hv, cp_dtype in_dt,
                        int64_t S, int H, int Hkv, int D, int Pu, int Pr, cp_layout layout,
                        void* hout, cp_dtype out_dt, float* hlse, void* workspace,
                        cp_stream_t stream, cp_stream_t copy_stream) {
  if (Pr < 1) return fail(CP_ERR_ARG, "Pr=%d must be >= 1", Pr);
  return ulysses_host_impl(hq, hk, hv, in_dt, S, H, Hkv, D, Pu, Pr, layout, hout, out_dt, hlse,
                           workspace, stream, copy_stream);
}

int64_t cp_usp_workspace_size(int64_t S, int H, int Hkv, int D, cp_dtype in_dt,
                              cp_dtype out_dt) {
  const int64_t u = cp_ulysses_workspace_size(S, H, Hkv, D, in_dt, out_dt);
  if (u < 0) return u;
  // plus the ring's fp32 accumulator for a bf16 output
  return u + (out_dt == CP_BF16 ? pad256(S * H * D * 4) : 0);
}

// stage -1: the whole forward; 0: seq_to_head of q, k, v; 1 .. Pr: ring
// step stage-1; Pr + 1: head_to_seq of the output.
static int usp_impl(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S, int H,
                    int Hkv, int D, int Pu, int Pr, cp_layout layout, void* out, cp_dtype out_dt,
                    float* lse, void* workspace, cp_stream_t stream, int stage) {
  int rc = check_heads_dims(in_dt, H, Hkv, D);
  if (rc != CP_OK) return rc;
  if (!valid_dtype(out_dt)) return fail(CP_ERR_DTYPE, "unknown output dtype %d", int(out_dt));
  if (Pu < 1 || Pu > CP_MAX_RANKS)
    return fail(CP_ERR_ARG, "Pu=%d outside [1,%d]", Pu, CP_MAX_RANKS);
  if (S < 1 || S >= (int64_t(1) << 28))
    return fail(CP_ERR_ARG, "S=%lld out of range", (long long)S);
  if (S % Pu != 0) return fail(CP_ERR_SHAPE, "S=%lld is not a multiple of Pu=%d", (long long)S, Pu);
  const bool replicate = Pu > Hkv && Pu % Hkv == 0;
  if (H % Pu != 0 || (!replicate && Hkv % Pu != 0))
    return fail(CP_ERR_SHAPE,
                "Ulysses degree Pu=%d must divide H=%d and either divide Hkv=%d or be a "
                "multiple of it",
                Pu, H, Hkv);
  const int G = H / Pu, Gkv = replicate ? Hkv : Hkv / Pu;
  if ((rc = check_ring(in_dt, S, G, Gkv, D, Pr, layout, out_dt)) != CP_OK) return rc;
  if (!q || !k || !v || !out || !lse || !workspace)
    return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(workspace))
    return fail(CP_ERR_ALIGN, "q, k, v, out and workspace must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t ei = elem_bytes(in_dt), eo = elem_bytes(out_dt);
  char* ws = static_cast<char*>(workspace);
  void* qh = ws;
  void* kh = ws + pad256(S * H * D * ei);
  void* vh = static_cast<char*>(kh) + pad256(S * Hkv * D * ei);
  void* oh = static_cast<char*>(vh) + pad256(S * Hkv * D * ei);
  void* acc = static_cast<char*>(oh) + pad256(S * H * D * eo);
  if (stage > Pr + 1) return fail(CP_ERR_ARG, "stage=%d outside [0,%d]", stage, Pr + 1);
  if (stage < 0 || stage == 0) {
    if ((rc = cp_seq_to_head(q, qh, in_dt, S, H, D, Pu, stream)) != CP_OK) return rc;
    if (!replicate) {
      if ((rc = cp_seq_to_head(k, kh, in_dt, S, Hkv, D, Pu, stream)) != CP_OK) return rc;
      if ((rc = cp_seq_to_head(v, vh, in_dt, S, Hkv, D, Pu, stream)) != CP_OK) return rc;
    }
    if (stage == 0) return ok();
  }
  if (stage == Pr + 1) return cp_head_to_seq(oh, out, out_dt, S, H, D, Pu, stream);
  // a ring of Pr virtual ranks over each head group's whole sequence, all Pu
  // groups in every launch
  const bool striped = layout == CP_STRIPED;
  RingBatch rb;
  rb.batch = Pu;
  rb.b_q_rows = striped ? S / Pr : S;
  rb.b_k_rows = replicate ? 0 : rb.b_q_rows;
  rb.b_o_rows = S;
  rb.b_lse_heads = G;
  rb.b_q_heads = replicate ? G : 0;
  rb.kv_group = replicate ? H / Hkv : G / Gkv;
  rb.q_rows = Pu * S;
  rb.k_rows = replicate ? S : Pu * S;
  if (ring_runs_fused(in_dt, layout)) {
    // the whole ring in one launch (stage 1; stages 2 .. Pr have nothing left)
    if (stage < 0 || stage == 1) {
      rc = ring_fused_impl(qh, replicate ? k : kh, replicate ? v : vh, S, G, Gkv, D, Pr, layout,
                           oh, out_dt, lse, s, &rb);
      if (rc != CP_OK) return rc;
    }
  } else {
    for (int t = 0; t < Pr; ++t) {
      if (stage > 0 && stage != t + 1) continue;
      // a step overlaps the previous one only when both run in this call
      rc = ring_step_impl(qh, replicate ? k : kh, replicate ? v : vh, in_dt, S, G, Gkv, D, Pr,
                          layout, t, oh, out_dt, lse, acc, s, nullptr, &rb, stage < 0 && t > 0);
      if (rc != CP_OK) return rc;
    }
  }
  if (stage > 0) return ok();
  if ((rc = cp_head_to_seq(oh, out, out_dt, S, H, D, Pu, stream)) != CP_OK) return rc;
  return ok();
}

int cp_usp_forward(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S, int H,
                   int Hkv, int D, int Pu, int Pr, cp_layout layout, void* out, cp_dtype out_dt,
                   float* lse, void* workspace, cp_stream_t stream) {
  return usp_impl(q, k, v, in_dt, S, H, Hkv, D, Pu, Pr, layout, out, out_dt, lse, workspace,
                  stream, -1);
}

int cp_usp_stage(const void* q, const void* k, const void* v, cp_dtype in_dt, int64_t S, int H,
                 int Hkv, int D, int Pu, int Pr, cp_layout layout, void* out, cp_dtype out_dt,
                 float* lse, void* workspace, int stage, cp_stream_t stream) {
  if (stage < 0) return fail(CP_ERR_ARG, "stage=%d is negative", stage);
  return usp_impl(q, k, v, in_dt, S, H, Hkv, D, Pu, Pr, layout, out, out_dt, lse, workspace,
                  stream, stage);
}

int64_t cp_attn_block_backward_workspace_size(int64_t Sq, int H) {
  if (Sq < 0 || H < 1) return fail(CP_ERR_ARG, "bad sizes");
  ok();
  return pad256(Sq * H * 4);
}

int cp_attn_block_backward(const void* q, const void* k, const void* v, const void* out,
                           const void* dout, const float* lse, cp_dtype in_dt, int64_t Sq,
                           int64_t Sk, int H, int Hkv, int D, int64_t q_offset, int64_t k_offset,
                           int causal, float scale, void* dq, void* dk, void* dv,
                           cp_dtype grad_dt, void* workspace, cp_stream_t stream) {
  int rc = check_bwd_common(in_dt, H, Hkv, D, grad_dt);
  if (rc != CP_OK) return rc;
  if (Sq < 0 || Sk < 0 || Sq >= (int64_t(1) << 31) || Sk >= (int64_t(1) << 31))
    return fail(CP_ERR_ARG, "Sq=%lld / Sk=%lld out of range", (long long)Sq, (long long)Sk);
  if (std::llabs(q_offset) >= (int64_t(1) << 40) || std::llabs(k_offset) >= (int64_t(1) << 40))
    return fail(CP_ERR_ARG, "offsets out of range");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t ge = elem_bytes(grad_dt);
  if ((Sq > 0 && (!q || !out || !dout || !lse || !dq || !workspace)) ||
      (Sk > 0 && (!k || !v || !dk || !dv)))
    return fail(CP_ERR_ARG, "null pointer argument");
  for (const void* x : {q, k, v, out, dout, static_cast<const void*>(dq),
                        static_cast<const void*>(dk), static_cast<const void*>(dv),
                        static_cast<const void*>(workspace)})
    if (x && !aligned16(x))
      return fail(CP_ERR_ALIGN, "tensors and workspace must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3) != 0)
    return fail(CP_ERR_ALIGN, "lse must be 4-byte aligned");
  if (Sq == 0 || Sk == 0) {
    // no pairs: every gradient is zero
    cudaError_t e = cudaSuccess;
    if (Sq > 0) e = cudaMemsetAsync(dq, 0, Sq * H * D * ge, s);
    if (e == cudaSuccess && Sk > 0) e = cudaMemsetAsync(dk, 0, Sk * Hkv * D * ge, s);
    if (e == cudaSuccess && Sk > 0) e = cudaMemsetAsync(dv, 0, Sk * Hkv * D * ge, s);
    return e == cudaSuccess ? ok() : cuda_fail(e, "memset");
  }
  float* delta = static_cast<float*>(workspace);
  cudaError_t e = launch_delta(in_dt, out, dout, delta, Sq, H, D, Sq, s);
  if (e != cudaSuccess) return cuda_fail(e, "delta launch");
  const bool f32 = grad_dt == CP_F32;
  BwdArgs a{q, k, v, dout, Sq, Sk, H, Hkv, 1, causal ? 1 : 0, in_dt, D,
            scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(D)),
            lse, delta, Sq, grad_dt, dq, dk, dv,
            f32 ? static_cast<float*>(dq) : nullptr, f32 ? static_cast<float*>(dk) : nullptr,
            f32 ? static_cast<float*>(dv) : nullptr};
  std::vector<BwdTask> tasks(2);
  tasks[0].dkdv = true;
  BwdItem kv{};
  kv.stat = BwdSeg{0, k_offset, static_cast<int32_t>(Sk), 0};
  kv.str[0] = BwdSeg{0, q_offset, static_cast<int32_t>(Sq), 0};
  kv.nstr = 1;
  tasks[0].items.push_back(kv);
  tasks[0].chunk.push_back(0);
  tasks[1].dkdv = false;
  BwdItem qi{};
  qi.stat = BwdSeg{0, q_offset, static_cast<int32_t>(Sq), 0};
  qi.str[0] = BwdSeg{0, k_offset, static_cast<int32_t>(Sk), 0};
  qi.nstr = 1;
  tasks[1].items.push_back(qi);
  tasks[1].chunk.push_back(0);
  rc = run_bwd_tasks(a, tasks, s);
  return rc == CP_OK ? ok() : rc;
}

int64_t cp_ring_backward_workspace_size(int64_t S, int H, int Hkv, int D, cp_dtype grad_dt) {
  if (S < 0 || H < 1 || Hkv < 1 || D < 1) return fail(CP_ERR_ARG, "bad sizes");
  if (!valid_dtype(grad_dt)) return fail(CP_ERR_DTYPE, "unknown gradient dtype %d", int(grad_dt));
  ok();
  int64_t b = pad256(S * H * 4);
  if (grad_dt == CP_BF16) b += pad256(S * H * D * 4) + 2 * pad256(S * Hkv * D * 4);
  return b;
}

// Launch `launch` of the ring backward's per-step schedule (fused = false:
// -1 delta, 2t dK/dV of step t, 2t + 1 dQ of step t) or of its two-launch
// schedule (fused = true: -1 delta, 0 dK/dV, 1 dQ).
static int ring_backward_launch(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse, cp_dtype in_dt, int64_t S,
                                int H, int Hkv, int D, int P, cp_layout layout, int launch,
                                void* dq, void* dk, void* dv, cp_dtype grad_dt, void* workspace,
                                cp_stream_t stream, bool fused) {
  int rc = check_bwd_common(in_dt, H, Hkv, D, grad_dt);
  if (rc != CP_OK) return rc;
  if ((rc = check_ring(in_dt, S, H, Hkv, D, P, layout, grad_dt)) != CP_OK) return rc;
  if (fused && !ring_bwd_runs_fused(in_dt, layout))
    return fail(in_dt != CP_BF16 ? CP_ERR_DTYPE : CP_ERR_ARG,
                "the two-launch ring backward needs bf16 inputs");
  const int nl = fused ? 2 : 2 * P;
  if (launch < -1 || launch >= nl)
    return fail(CP_ERR_ARG, "launch=%d outside [-1,%d)", launch, nl);
  if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv || !workspace)
    return fail(CP_ERR_ARG, "null pointer argument");
  for (const void* x : {q, k, v, out, dout, static_cast<const void*>(dq),
                        static_cast<const void*>(dk), static_cast<const void*>(dv),
                        static_cast<const void*>(workspace)})
    if (!aligned16(x)) return fail(CP_ERR_ALIGN, "tensors and workspace must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3) != 0)
    return fail(CP_ERR_ALIGN, "lse must be 4-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  float* delta = reinterpret_cast<float*>(ws);
  if (launch == -1) {
    cudaError_t e = launch_delta(in_dt, out, dout, delta, S, H, D, S, s);
    return e == cudaSuccess ? ok() : cuda_fail(e, "delta launch");
  }
  const bool f32 = grad_dt == CP_F32;
  // bf16 gradients: fp32 accumulators after delta (dq, then dk, then dv)
  char* acc0 = ws + pad256(S * H * 4);
  char* acc1 = acc0 + pad256(S * H * D * 4);
  char* acc2 = acc1 + pad256(S * Hkv * D * 4);
  float* acc_q = f32 ? static_cast<float*>(dq) : reinterpret_cast<float*>(acc0);
  float* acc_k = f32 ? static_cast<float*>(dk) : reinterpret_cast<float*>(acc1);
  float* acc_v = f32 ? static_cast<float*>(dv) : reinterpret_cast<float*>(acc2);
  const bool striped = layout == CP_STRIPED;
  BwdArgs a{q, k, v, dout, S, S, H, Hkv, striped ? P : 1, 1, in_dt, D,
            1.0f / std::sqrt(static_cast<float>(D)), lse, delta, S, grad_dt, dq, dk, dv,
            acc_q, acc_k, acc_v};
  std::vector<BwdTask> tasks =
      fused ? ring_bwd_fused_tasks(S, P, layout) : ring_bwd_tasks(S, P, layout);
  rc = run_bwd_tasks(a, tasks, s, launch);
  return rc == CP_OK ? ok() : rc;
}

int cp_ring_backward_step(const void* q, const void* k, const void* v, const void* out,
                          const void* dout, const float* lse, cp_dtype in_dt, int64_t S, int H,
                          int Hkv, int D, int P, cp_layout layout, int launch, void* dq,
                          void* dk, void* dv, cp_dtype grad_dt, void* workspace,
                          cp_stream_t stream) {
  return ring_backward_launch(q, k, v, out, dout, lse, in_dt, S, H, Hkv, D, P, layout, launch,
                              dq, dk, dv, grad_dt, workspace, stream, false);
}

int cp_ring_backward_fused_step(const void* q, const void* k, const void* v, const void* out,
                                const void* dout, const float* lse, cp_dtype in_dt, int64_t S,
                                int H, int Hkv, int D, int P, cp_layout layout, int launch,
                                void* dq, void* dk, void* dv, cp_dtype grad_dt, void* workspace,
                                cp_stream_t stream) {
  return ring_backward_launch(q, k, v, out, dout, lse, in_dt, S, H, Hkv, D, P, layout, launch,
                              dq, dk, dv, grad_dt, workspace, stream, true);
}

int cp_ring_backward(const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, cp_dtype in_dt, int64_t S, int H,
                     int Hkv, int D, int P, cp_layout layout, void* dq, void* dk, void* dv,
                     cp_dtype grad_dt, void* workspace, cp_stream_t stream) {
  // the tensor-core path runs the ring in two launches (every step inside
  // each), the rest one dK/dV and one dQ launch per step
  const bool fused = ring_bwd_runs_fused(in_dt, layout);
  const int nl = fused ? 2 : 2 * P;
  for (int l = -1; l < nl; ++l) {
    const int rc = ring_backward_launch(q, k, v, out, dout, lse, in_dt, S, H, Hkv, D, P, layout,
                                        l, dq, dk, dv, grad_dt, workspace, stream, fused);
    if (rc != CP_OK) return rc;
  }
  return ok();
}

// Device staging of cp_ring_backward_host: every group's compact inputs
// (q, k, v, out, dout, lse) and gradients (dq, dk, dv), then one group's
// ring backward workspace.
struct BwdHostStaging {
  int64_t q, k, v, out, dout, lse, dq, dk, dv, ws, total;
};

static BwdHostStaging bwd_host_staging(int64_t S, int H, int Hkv, int D, int groups,
                                       cp_dtype in_dt, cp_dtype grad_dt) {
  const int64_t ei = elem_bytes(in_dt), eg = elem_bytes(grad_dt);
  BwdHostStaging h;
  h.q = 0;
  h.k = h.q + pad256(S * H * D * ei);
  h.v = h.k + pad256(S * Hkv * D * ei);
  h.out = h.v + pad256(S * Hkv * D * ei);
  h.dout = h.out + pad256(S * H * D * ei);
  h.lse = h.dout + pad256(S * H * D * ei);
  h.dq = h.lse + pad256(S * H * 4);
  h.dk = h.dq + pad256(S * H * D * eg);
  h.dv = h.dk + pad256(S * Hkv * D * eg);
  h.ws = h.dv + pad256(S * Hkv * D * eg);
  h.total = h.ws + cp_ring_backward_workspace_size(S, H / groups, Hkv / groups, D, grad_dt);
  return h;
}

int64_t cp_ring_backward_host_workspace_size(int64_t S, int H, int Hkv, int D, int groups,
                                             cp_dtype in_dt, cp_dtype grad_dt) {
  if (S < 1 || H < 1 || Hkv < 1 || D < 1) return fail(CP_ERR_ARG, "bad sizes");
  if (!valid_dtype(in_dt) || !valid_dtype(grad_dt)) return fail(CP_ERR_DTYPE, "unknown dtype");
  if (groups < 1 || Hkv % groups != 0)
    return fail(CP_ERR_SHAPE, "groups=%d must divide Hkv=%d", groups, Hkv);
  ok();
  return bwd_host_staging(S, H, Hkv, D, groups, in_dt, grad_dt).total;
}

int cp_ring_backward_host(const void* hq, const void* hk, const void* hv, const void* hout,
                          const void* hdout, const float* hlse, cp_dtype in_dt, int64_t S,
                          int H, int Hkv, int D, int P, cp_layout layout, void* hdq, void* hdk,
                          void* hdv, cp_dtype grad_dt, int groups, void* workspace,
                          cp_stream_t stream, cp_stream_t copy_stream) {
  int rc = check_bwd_common(in_dt, H, Hkv, D, grad_dt);
  if (rc != CP_OK) return rc;
  if ((rc = check_ring(in_dt, S, H, Hkv, D, P, layout, grad_dt)) != CP_OK) return rc;
  if (groups < 1 || Hkv % groups != 0)
    return fail(CP_ERR_SHAPE, "groups=%d must divide Hkv=%d", groups, Hkv);
  if (!hq || !hk || !hv || !hout || !hdout || !hlse || !hdq || !hdk || !hdv || !workspace)
    return fail(CP_ERR_ARG, "null pointer argument");
  if (!aligned16(workspace)) return fail(CP_ERR_ALIGN, "workspace must be 16-byte aligned");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t xs = reinterpret_cast<cudaStream_t>(copy_stream);
  const int G = groups, Hg = H / G, Hkg = Hkv / G;
  const size_t ei = elem_bytes(in_dt), eg = elem_bytes(grad_dt);
  const BwdHostStaging st = bwd_host_staging(S, H, Hkv, D, G, in_dt, grad_dt);
  char* ws = static_cast<char*>(workspace);
  const size_t rows = static_cast<size_t>(S);
  // one group's slice of a [S, heads, D] tensor: width w bytes out of pitch
  auto slice = [&](int heads_g, size_t e) { return static_cast<size_t>(heads_g) * D * e; };
  HostGroupPipeline pl(cs, xs, G);
  // group g's slice of a host tensor [S, heads_total, D] <-> compact device
  auto h2d = [&](int64_t dev_off, const void* h, int heads_total, int heads_g, int g, size_t e) {
    const size_t w = slice(heads_g, e);
    pl.in(ws + dev_off + g * rows * w, static_cast<const char*>(h) + g * w, w,
          slice(heads_total, e), rows);
  };
  auto d2h = [&](void* h, int64_t dev_off, int heads_total, int heads_g, int g, size_t e) {
    const size_t w = slice(heads_g, e);
    pl.out(static_cast<char*>(h) + g * w, ws + dev_off + g * rows * w, w, slice(heads_total, e),
           rows);
  };
  for (int g = 0; g < G && pl.ok(); ++g) {
    h2d(st.q, hq, H, Hg, g, ei);
    h2d(st.k, hk, Hkv, Hkg, g, ei);
    h2d(st.v, hv, Hkv, Hkg, g, ei);
    h2d(st.out, hout, H, Hg, g, ei);
    h2d(st.dout, hdout, H, Hg, g, ei);
    const size_t lg = rows * Hg * 4;  // group g's lse rows, contiguous in [H, S]
    pl.in(ws + st.lse + g * lg, hlse + static_cast<size_t>(g) * Hg * S, lg, lg, 1);
    pl.inputs_done(g);
  }
  for (int g = 0; g < G && pl.ok(); ++g) {
    pl.compute_begin(g);
    auto at = [&](int64_t off, int heads_g, size_t e) {
      return ws + off + g * rows * slice(heads_g, e);
    };
    rc = cp_ring_backward(at(st.q, Hg, ei), at(st.k, Hkg, ei), at(st.v, Hkg, ei),
                          at(st.out, Hg, ei), at(st.dout, Hg, ei),
                          reinterpret_cast<const float*>(ws + st.lse + g * rows * Hg * 4), in_dt, S,
                          Hg, Hkg, D, P, layout, at(st.dq, Hg, eg), at(st.dk, Hkg, eg),
                          at(st.dv, Hkg, eg), grad_dt, ws + st.ws, stream);
    if (rc != CP_OK) return rc;
    pl.compute_end(g);
    d2h(hdq, st.dq, H, Hg, g, eg);
    d2h(hdk, st.dk, Hkv, Hkg, g, eg);
    d2h(hdv, st.dv, Hkv, Hkg, g, eg);
  }
  pl.finish();
  if (!pl.ok()) return cuda_fail(pl.error(), "host ring backward copies");
  return ok();
}

int cp_check_device_error(cp_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int* st = device_status_ptr();
  if (st == nullptr) return fail(CP_ERR_CUDA, "device status word unavailable");
  int v = 0;
  e = cudaMemcpy(&v, st, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "status reset");
    if ((v & 0xff) == kDevErrBounds) {
      static const char* const sites[] = {
          "?", "forward query tile", "forward K/V tile", "fp32 forward row",
          "backward stationary tile", "backward streamed tile", "fp32 backward row"};
      const int site = v >> 8;
      return fail(CP_ERR_BOUNDS, "a device-side bounds check failed: %s (site %d)",
                  sites[site >= 1 && site <= 6 ? site : 0], site);
    }
    return fail(CP_ERR_TIMEOUT, "a device-side wait expired (status %d)", v);
  }
  return ok();
}

int cp_debug_bounds(void) { return kDebugBounds ? 1 : 0; }

int cp_selftest_wait_timeout(int timeout_us, cp_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 2000000) return fail(CP_ERR_ARG, "timeout_us out of range");
  int* st = device_status_ptr();
  if (st == nullptr) return fail(CP_ERR_CUDA, "device status word unavailable");
  cudaError_t e = launch_wait_timeout_selftest(static_cast<uint64_t>(timeout_us) * 1000ull, st,
                                               reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ok() : cuda_fail(e, "self-test launch");
}

}  // extern "C"
