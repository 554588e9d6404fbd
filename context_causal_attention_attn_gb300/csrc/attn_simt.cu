// fp32 block attention on the CUDA cores (fp32 FMA), for fp32 inputs with a
// small head dimension, such as the handbook's own toy shapes (D = 16).
//
// Same contract as the tensor-core kernel ([CP-handbook] "上下文并行：Ring
// Attention 与 Ulysses", section "哪些运算可以直接切"; merge from the self-test
// answers): one thread owns one (query row, head); it walks the visible keys
// of the item's segments in order with an fp32 online softmax (natural-log
// domain, accurate expf/logf), then writes or LSE-merges its row.  The
// tensor cores cannot serve this path: tf32 would miss an absolute error of
// 1e-5 against fp64.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"

namespace cpattn {

constexpr int kSimtRows = 128;  // query rows per block (one head)

template <int D>
__global__ void __launch_bounds__(kSimtRows)
    attn_fwd_simt_kernel(const __grid_constant__ AttnParams p, int* dev_err) {
  int ii = 0;
  while (ii + 1 < p.nitems && static_cast<int>(blockIdx.x) >= p.cta_start[ii + 1]) ++ii;
  const WorkItem& it = p.items[ii];
  int local = static_cast<int>(blockIdx.x) - p.cta_start[ii];
  const int head = local % p.H;
  local /= p.H;
  const int b = local % it.batch;
  local /= it.batch;
  const int nblk = (it.sq + kSimtRows - 1) / kSimtRows;
  const int row = (nblk - 1 - local) * kSimtRows + static_cast<int>(threadIdx.x);
  if (row >= it.sq) return;
  const int kvh = (b * p.b_q_heads + head) / p.kv_group;
  const bool causal = (it.flags & kFlagCausal) != 0;
  const int64_t qp = it.q_pos + row;

  const int64_t qrow_i = it.q_mem_row + static_cast<int64_t>(b) * it.b_q_rows + row;
  const int64_t qtok = it.q_stripe + static_cast<int64_t>(p.stripe) * qrow_i;
  if (kDebugBounds) {
    // the row of q, of out / acc (out has the rows of q) and of lse
    const int64_t orow = it.o_row + static_cast<int64_t>(b) * it.b_o_rows +
                         static_cast<int64_t>(row) * it.o_stride;
    const int64_t lcol = it.lse_col + static_cast<int64_t>(row) * it.o_stride;
    const int64_t lh = static_cast<int64_t>(head) + static_cast<int64_t>(b) * it.b_lse_heads;
    if (!bounds_ok(qrow_i >= 0 && qrow_i < p.q_rows / p.stripe && it.q_stripe >= 0 &&
                       it.q_stripe < p.stripe && kvh >= 0 && kvh < p.Hkv && orow >= 0 &&
                       orow < p.q_rows && lcol >= 0 && lcol < p.ld_lse &&
                       lh < static_cast<int64_t>(p.H) * it.batch,
                   dev_err, kSiteFwdSimt))
      return;
  }
  const float* qrow =
      static_cast<const float*>(p.q) + (qtok * p.H + head) * static_cast<int64_t>(D);
  float q[D];
#pragma unroll
  for (int d = 0; d < D; d += 4) {
    const float4 t = *reinterpret_cast<const float4*>(qrow + d);
    q[d] = t.x * p.scale;
    q[d + 1] = t.y * p.scale;
    q[d + 2] = t.z * p.scale;
    q[d + 3] = t.w * p.scale;
  }
  float m = -CUDART_INF_F, l = 0.f;
  float acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;

  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);
  const int64_t kb = static_cast<int64_t>(b) * it.b_k_rows;
  for (int s = 0; s < it.nseg; ++s) {
    const KSeg& sg = it.seg[s];
    int n = sg.len;
    if (causal) {
      const int64_t vis = qp - sg.pos + 1;
      if (vis <= 0) break;
      if (vis < n) n = static_cast<int>(vis);
    }
    for (int j = 0; j < n; ++j) {
      if (kDebugBounds && !bounds_ok(sg.mem_row + kb + j >= 0 &&
                                         sg.mem_row + kb + j < p.k_rows / p.kv_stripe &&
                                         sg.stripe >= 0 && sg.stripe < p.kv_stripe,
                                     dev_err, kSiteFwdSimt))
        break;
      const int64_t ktok = sg.stripe + static_cast<int64_t>(p.kv_stripe) * (sg.mem_row + kb + j);
      const int64_t off = (ktok * p.Hkv + kvh) * static_cast<int64_t>(D);
      const float* kr = K + off;
      float sc = 0.f;
#pragma unroll
      for (int d = 0; d < D; d += 4) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(kr + d));
        sc = fmaf(q[d], t.x, sc);
        sc = fmaf(q[d + 1], t.y, sc);
        sc = fmaf(q[d + 2], t.z, sc);
        sc = fmaf(q[d + 3], t.w, sc);
      }
      const float* vr = V + off;
      float pw, corr;
      if (sc > m) {
        corr = expf(m - sc);  // 0 when m = -inf
        m = sc;
        pw = 1.f;
      } else {
        corr = 1.f;
        pw = expf(sc - m);
      }
      l = fmaf(l, corr, pw);
#pragma unroll
      for (int d = 0; d < D; d += 4) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(vr + d));
        acc[d] = fmaf(acc[d], corr, pw * t.x);
        acc[d + 1] = fmaf(acc[d + 1], corr, pw * t.y);
        acc[d + 2] = fmaf(acc[d + 2], corr, pw * t.z);
        acc[d + 3] = fmaf(acc[d + 3], corr, pw * t.w);
      }
    }
  }

  // ---------------------------------------------------------- epilogue
  // l == 0 exactly when no key was visible (a NaN score leaves l NaN, which
  // then reaches lse and out)
  const float lse_blk = l != 0.f ? m + logf(l) : -CUDART_INF_F;
  const int64_t orow =
      it.o_row + static_cast<int64_t>(b) * it.b_o_rows + static_cast<int64_t>(row) * it.o_stride;
  const int64_t oel = (orow * p.H + head) * static_cast<int64_t>(D);
  const int64_t lse_head = static_cast<int64_t>(head) + static_cast<int64_t>(b) * it.b_lse_heads;
  float* lse_ptr =
      p.lse + lse_head * p.ld_lse + it.lse_col + static_cast<int64_t>(row) * it.o_stride;
  const bool merge = (it.flags & kFlagMerge) != 0;
  const bool final_out = (it.flags & kFlagFinal) != 0;
  float w_acc = 0.f, w_blk = 1.f, lse_new = lse_blk;
  if (merge) {
    const float a = *lse_ptr;
    const float hi = fmaxf(a, lse_blk);
    if (a == -CUDART_INF_F && lse_blk == -CUDART_INF_F) {  // both empty (not NaN)
      w_blk = 0.f;
      lse_new = -CUDART_INF_F;
    } else {
      lse_new = hi + log1pf(expf(-fabsf(a - lse_blk)));
      w_acc = expf(a - lse_new);
      w_blk = expf(lse_blk - lse_new);
    }
  }
  const float c_blk = l != 0.f ? w_blk / l : 0.f;
  float* accp = p.acc + oel;
#pragma unroll
  for (int d = 0; d < D; d += 4) {
    float4 o = make_float4(acc[d] * c_blk, acc[d + 1] * c_blk, acc[d + 2] * c_blk,
                           acc[d + 3] * c_blk);
    if (merge) {
      const float4 a = *reinterpret_cast<const float4*>(accp + d);
      o.x = fmaf(a.x, w_acc, o.x);
      o.y = fmaf(a.y, w_acc, o.y);
      o.z = fmaf(a.z, w_acc, o.z);
      o.w = fmaf(a.w, w_acc, o.w);
    }
    if (final_out && p.out_dt == 1) {
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(
          reinterpret_cast<__nv_bfloat16*>(p.out) + oel + d);
      o2[0] = __floats2bfloat162_rn(o.x, o.y);
      o2[1] = __floats2bfloat162_rn(o.z, o.w);
    } else {
      float* dst = final_out ? reinterpret_cast<float*>(p.out) + oel : accp;
      *reinterpret_cast<float4*>(dst + d) = o;
    }
  }
  *lse_ptr = lse_new;
}

cudaError_t launch_attn_simt(const AttnParams& p, int ctas, int* dev_err, cudaStream_t stream) {
  switch (p.D) {
    case 16: attn_fwd_simt_kernel<16><<<ctas, kSimtRows, 0, stream>>>(p, dev_err); break;
    case 32: attn_fwd_simt_kernel<32><<<ctas, kSimtRows, 0, stream>>>(p, dev_err); break;
    case 64: attn_fwd_simt_kernel<64><<<ctas, kSimtRows, 0, stream>>>(p, dev_err); break;
    case 128: attn_fwd_simt_kernel<128><<<ctas, kSimtRows, 0, stream>>>(p, dev_err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int attn_simt_ctas(const WorkItem& it, int H) {
  return ((it.sq + kSimtRows - 1) / kSimtRows) * it.batch * H;
}

}  // namespace cpattn
