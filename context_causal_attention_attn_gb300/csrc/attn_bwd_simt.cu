// Backward of block attention for fp32 inputs on the CUDA cores (the toy
// configuration of [CP-handbook] "上下文并行：Ring Attention 与 Ulysses",
// section "哪些运算可以直接切": fp32, D = 16); the same gradients as the
// tensor-core kernels (attn_bwd_tc.cu), in fp32 throughout with accurate
// expf:
//   p_ij = exp(scale q_i.k_j - lse_i),  ds_ij = p_ij (do_i.v_j - delta_i),
//   dq_i = scale sum_j ds_ij k_j,  dk_j = scale sum_i ds_ij q_i,
//   dv_j = sum_i p_ij do_i.
// One warp per (row, head); lane l holds elements l, l + 32, ... of the
// head dimension and dot products reduce across the warp.  Work items,
// flags and output layouts are those of the tensor-core kernels.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"

namespace cpattn {

namespace {

constexpr int kWarpsPerBlock = 4;

template <int E>
__device__ __forceinline__ float warp_dot(const float (&a)[E], const float (&b)[E]) {
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) s = fmaf(a[e], b[e], s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// row r of segment g -> token (the row of the [rows, heads, D] tensors)
__device__ __forceinline__ int64_t seg_token(const BwdSeg& g, int64_t r, int stride) {
  return g.stripe + static_cast<int64_t>(stride) * (g.row + r);
}

template <int D>
__device__ __forceinline__ void load_vec(const float* base, float (&x)[(D + 31) / 32], int lane) {
  constexpr int E = (D + 31) / 32;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = lane + 32 * e;
    x[e] = d < D ? base[d] : 0.f;
  }
}

// Store one gradient row: accumulate into / write the fp32 buffer, or write
// the finished value in out_dt.
template <int D>
__device__ __forceinline__ void store_grad(const BwdParams& p, int flags, float* acc, void* out,
                                           int64_t el, const float (&g)[(D + 31) / 32],
                                           float mul, int lane) {
  constexpr int E = (D + 31) / 32;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int d = lane + 32 * e;
    if (d >= D) continue;
    float v = g[e] * mul;
    if (flags & kBwdAccumulate) v += acc[el + d];
    if (flags & kBwdFinal) {
      if (p.out_dt == 1) {
        // round to nearest even bf16
        const uint32_t u = __float_as_uint(v);
        const uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
        static_cast<uint16_t*>(out)[el + d] = static_cast<uint16_t>(r);
      } else {
        static_cast<float*>(out)[el + d] = v;
      }
    } else {
      acc[el + d] = v;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    bwd_dq_simt_kernel(const float* __restrict__ q, const float* __restrict__ k,
                       const float* __restrict__ v, const float* __restrict__ dout,
                       BwdParams p, int* dev_err) {
  constexpr int E = (D + 31) / 32;
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  int ii = 0;
  while (ii + 1 < p.nitems && w >= p.cta_start[ii + 1]) ++ii;
  if (w >= p.cta_start[p.nitems]) return;
  const BwdItem& it = p.items[ii];
  const int local = w - p.cta_start[ii];
  const int r = local % it.stat.len;
  const int h = local / it.stat.len;
  const int kvh = h / (p.H / p.Hkv);
  const int64_t tok = seg_token(it.stat, r, p.stride);
  const int64_t qpos = it.stat.pos + r;
  // bounds-checked build: the query row (also its lse / delta column and
  // dq row) lies inside its tensors
  if (kDebugBounds && !bounds_ok(tok >= 0 && tok < p.q_rows && tok < p.ld && h < p.H,
                                 dev_err, kSiteBwdSimt))
    return;
  float qi[E], doi[E], dq[E];
  load_vec<D>(q + (tok * p.H + h) * D, qi, lane);
  load_vec<D>(dout + (tok * p.H + h) * D, doi, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) dq[e] = 0.f;
  const float lse = p.lse[static_cast<int64_t>(h) * p.ld + tok];
  const float dl = p.delta[static_cast<int64_t>(h) * p.ld + tok];
  if (lse != -CUDART_INF_F) {
    for (int s = 0; s < it.nstr; ++s) {
      const BwdSeg& g = it.str[s];
      for (int j = 0; j < g.len; ++j) {
        if (p.causal && g.pos + j > qpos) break;
        const int64_t kt = seg_token(g, j, p.stride);
        if (kDebugBounds && !bounds_ok(kt >= 0 && kt < p.k_rows, dev_err, kSiteBwdSimt)) break;
        float kj[E], vj[E];
        load_vec<D>(k + (kt * p.Hkv + kvh) * D, kj, lane);
        load_vec<D>(v + (kt * p.Hkv + kvh) * D, vj, lane);
        const float pij = expf(warp_dot<E>(qi, kj) * p.scale - lse);
        const float ds = pij * (warp_dot<E>(doi, vj) - dl);
#pragma unroll
        for (int e = 0; e < E; ++e) dq[e] = fmaf(ds, kj[e], dq[e]);
      }
    }
  }
  store_grad<D>(p, it.flags, p.acc0, p.out0, (tok * p.H + h) * D, dq, p.scale, lane);
}

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    bwd_dkdv_simt_kernel(const float* __restrict__ q, const float* __restrict__ k,
                         const float* __restrict__ v, const float* __restrict__ dout,
                         BwdParams p, int* dev_err) {
  constexpr int E = (D + 31) / 32;
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  int ii = 0;
  while (ii + 1 < p.nitems && w >= p.cta_start[ii + 1]) ++ii;
  if (w >= p.cta_start[p.nitems]) return;
  const BwdItem& it = p.items[ii];
  const int local = w - p.cta_start[ii];
  const int r = local % it.stat.len;
  const int kvh = local / it.stat.len;
  const int grp = p.H / p.Hkv;
  const int64_t tok = seg_token(it.stat, r, p.stride);
  const int64_t kpos = it.stat.pos + r;
  // bounds-checked build: the key row (also its dk / dv row) lies inside
  // its tensors
  if (kDebugBounds &&
      !bounds_ok(tok >= 0 && tok < p.k_rows && kvh < p.Hkv, dev_err, kSiteBwdSimt))
    return;
  float kj[E], vj[E], dk[E], dv[E];
  load_vec<D>(k + (tok * p.Hkv + kvh) * D, kj, lane);
  load_vec<D>(v + (tok * p.Hkv + kvh) * D, vj, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) dk[e] = dv[e] = 0.f;
  for (int g = 0; g < grp; ++g) {
    const int h = kvh * grp + g;
    for (int s = 0; s < it.nstr; ++s) {
      const BwdSeg& seg = it.str[s];
      for (int i = 0; i < seg.len; ++i) {
        if (p.causal && seg.pos + i < kpos) continue;
        const int64_t qt = seg_token(seg, i, p.stride);
        if (kDebugBounds &&
            !bounds_ok(qt >= 0 && qt < p.q_rows && qt < p.ld, dev_err, kSiteBwdSimt))
          break;
        const float lse = p.lse[static_cast<int64_t>(h) * p.ld + qt];
        if (lse == -CUDART_INF_F) continue;
        const float dl = p.delta[static_cast<int64_t>(h) * p.ld + qt];
        float qi[E], doi[E];
        load_vec<D>(q + (qt * p.H + h) * D, qi, lane);
        load_vec<D>(dout + (qt * p.H + h) * D, doi, lane);
        const float pij = expf(warp_dot<E>(qi, kj) * p.scale - lse);
        const float ds = pij * (warp_dot<E>(doi, vj) - dl);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          dv[e] = fmaf(pij, doi[e], dv[e]);
          dk[e] = fmaf(ds, qi[e], dk[e]);
        }
      }
    }
  }
  const int64_t el = (tok * p.Hkv + kvh) * D;
  store_grad<D>(p, it.flags, p.acc0, p.out0, el, dv, 1.f, lane);
  store_grad<D>(p, it.flags, p.acc1, p.out1, el, dk, p.scale, lane);
}

// delta[h][row] = sum_d dO . O (fp32), one warp per row-head
template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    bwd_delta_f32_kernel(const float* __restrict__ out, const float* __restrict__ dout,
                         float* __restrict__ delta, int64_t rows, int H, int64_t ld) {
  constexpr int E = (D + 31) / 32;
  const int lane = threadIdx.x & 31;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (w >= rows * H) return;
  float a[E], b[E];
  load_vec<D>(out + w * D, a, lane);
  load_vec<D>(dout + w * D, b, lane);
  const float s = warp_dot<E>(a, b);
  if (lane == 0) delta[(w % H) * ld + w / H] = s;
}

template <template <int> class F, typename... A>
cudaError_t dispatch_d(int D, A... a) {
  switch (D) {
    case 16: return F<16>::run(a...);
    case 32: return F<32>::run(a...);
    case 64: return F<64>::run(a...);
    case 128: return F<128>::run(a...);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
struct RunDq {
  static cudaError_t run(const void* q, const void* k, const void* v, const void* dout,
                         const BwdParams* p, int warps, int* dev_err, cudaStream_t s) {
    const int blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    bwd_dq_simt_kernel<D><<<blocks, kWarpsPerBlock * 32, 0, s>>>(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
        static_cast<const float*>(dout), *p, dev_err);
    return cudaGetLastError();
  }
};

template <int D>
struct RunDkdv {
  static cudaError_t run(const void* q, const void* k, const void* v, const void* dout,
                         const BwdParams* p, int warps, int* dev_err, cudaStream_t s) {
    const int blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    bwd_dkdv_simt_kernel<D><<<blocks, kWarpsPerBlock * 32, 0, s>>>(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
        static_cast<const float*>(dout), *p, dev_err);
    return cudaGetLastError();
  }
};

template <int D>
struct RunDelta {
  static cudaError_t run(const void* out, const void* dout, float* delta, int64_t rows, int H,
                         int64_t ld, cudaStream_t s) {
    const int64_t warps = rows * H;
    const int blocks = static_cast<int>((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
    bwd_delta_f32_kernel<D><<<blocks, kWarpsPerBlock * 32, 0, s>>>(
        static_cast<const float*>(out), static_cast<const float*>(dout), delta, rows, H, ld);
    return cudaGetLastError();
  }
};

}  // namespace

// One warp per (stationary row, head) of every item: the warp count.
int attn_bwd_simt_warps(const BwdItem& it, int heads) { return it.stat.len * heads; }

// p.cta_start holds warp offsets here.
cudaError_t launch_attn_bwd_simt(bool dkdv, const void* q, const void* k, const void* v,
                                 const void* dout, const BwdParams& p, int D, int warps,
                                 int* dev_err, cudaStream_t s) {
  return dkdv ? dispatch_d<RunDkdv>(D, q, k, v, dout, &p, warps, dev_err, s)
              : dispatch_d<RunDq>(D, q, k, v, dout, &p, warps, dev_err, s);
}

cudaError_t launch_bwd_delta_f32(const void* out, const void* dout, float* delta, int64_t rows,
                                 int H, int D, int64_t ld, cudaStream_t s) {
  return dispatch_d<RunDelta>(D, out, dout, delta, rows, H, ld, s);
}

}  // namespace cpattn
