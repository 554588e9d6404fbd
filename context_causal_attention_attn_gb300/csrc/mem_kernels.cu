// HBM-bound kernels of libcpattn: the LSE merge, the Ulysses seq<->head
// permutation, the backward's delta, the empty-block fill, the
// failure-detection self-test, and the device status word.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <type_traits>

#include "internal.h"
#include "sm100.cuh"

namespace cpattn {

__device__ int g_dev_status;

// Resident blocks per SM used to size the grid-stride kernels below.
constexpr int kStreamThreads = 256;

// Device address of g_dev_status on the current device (looked up once per
// device with that device current; the symbol's name is only a host-side
// stand-in in host code).
int* device_status_ptr() {
  static PerDeviceOnce once;
  static int* ptrs[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const cudaError_t e = once_per_device(once, [dev] {
    void* p = nullptr;
    const cudaError_t r = cudaGetSymbolAddress(&p, g_dev_status);
    if (r == cudaSuccess) ptrs[dev] = static_cast<int*>(p);
    return r;
  });
  return e == cudaSuccess ? ptrs[dev] : nullptr;
}

static int stream_grid(int64_t work_items) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t resident = static_cast<int64_t>(sms) * (2048 / kStreamThreads);
  const int64_t need = (work_items + kStreamThreads - 1) / kStreamThreads;
  return static_cast<int>(need < resident ? (need > 0 ? need : 1) : resident);
}

// ------------------------------------------------------------- LSE merge
// [CP-handbook] "上下文并行：Ring Attention 与 Ulysses", self-test answers /
// section "Ring Attention：KV 沿环传一圈": acc <- acc (+) blk.
// Row-heads are visited head-major (h, i) so that the lse accesses of a warp
// are contiguous and every out row-head is one contiguous run of D floats.
// A group of L lanes owns one row-head (L = D/4 up to 32); the lse values of
// the row-head are read by all its lanes before one lane writes the merged
// value back, and the group lives inside one warp (__syncwarp orders it).
template <int L>
__global__ void __launch_bounds__(kStreamThreads)
    lse_merge_kernel(float* __restrict__ out_acc, float* __restrict__ lse_acc,
                     const float* __restrict__ out_blk, const float* __restrict__ lse_blk,
                     int64_t Sq, int H, int D, int vec_per_lane) {
  constexpr int GROUPS_PER_WARP = 32 / L;
  constexpr int U = 4;  // row-head groups per warp per trip, all loads issued first
  const int lane = threadIdx.x & 31;
  const int grp = lane / L;
  const int sub = lane % L;
  const int64_t n_rh = Sq * H;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  constexpr int64_t kStep = static_cast<int64_t>(GROUPS_PER_WARP) * U;
  for (int64_t base = warp_id * kStep; base < n_rh; base += warps_total * kStep) {
    for (int v = 0; v < vec_per_lane; ++v) {
      float lsa[U], lsb[U];
      float4 x[U], y[U];
      int64_t off[U];
      bool act[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t rh = base + u * GROUPS_PER_WARP + grp;  // head-major: h * Sq + i
        act[u] = rh < n_rh;
        lsa[u] = -CUDART_INF_F;
        lsb[u] = -CUDART_INF_F;
        off[u] = 0;
        if (act[u]) {
          const int64_t h = rh / Sq;
          const int64_t i = rh - h * Sq;
          off[u] = (i * H + h) * static_cast<int64_t>(D) / 4 + v * L + sub;
          lsa[u] = lse_acc[rh];
          lsb[u] = lse_blk[rh];
          x[u] = reinterpret_cast<const float4*>(out_acc)[off[u]];
          y[u] = __ldcs(reinterpret_cast<const float4*>(out_blk) + off[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!act[u]) continue;
        // Natural-log domain with the accurate expf / log1pf: the kernel is
        // bound by HBM, so the exact-rounding functions cost nothing and
        // keep fp32 merges within a few ulp of the exact result.  A -inf
        // side gets weight exp(-inf) = 0; both -inf leave (-inf, 0); a NaN
        // side makes the result NaN.
        const float la = lsa[u], lb = lsb[u];
        const float hi = fmaxf(la, lb);
        float wa = 0.f, wb = 0.f, lse = -CUDART_INF_F;
        if (!(la == -CUDART_INF_F && lb == -CUDART_INF_F)) {
          lse = hi + log1pf(expf(-fabsf(la - lb)));
          wa = expf(la - lse);
          wb = expf(lb - lse);
        }
        reinterpret_cast<float4*>(out_acc)[off[u]] =
            make_float4(fmaf(x[u].x, wa, y[u].x * wb), fmaf(x[u].y, wa, y[u].y * wb),
                        fmaf(x[u].z, wa, y[u].z * wb), fmaf(x[u].w, wa, y[u].w * wb));
        lsa[u] = lse;
      }
      // every lane of a group has read the old lse before one writes the new
      __syncwarp();
      if (v == vec_per_lane - 1 && sub == 0) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (act[u]) lse_acc[base + u * GROUPS_PER_WARP + grp] = lsa[u];
      }
      __syncwarp();
    }
  }
}

cudaError_t launch_lse_merge(float* out_acc, float* lse_acc, const float* out_blk,
                             const float* lse_blk, int64_t Sq, int H, int D, cudaStream_t s) {
  const int d4 = D / 4;
  int L = d4 >= 32 ? 32 : d4;
  const int vpl = d4 / L;
  const int64_t n_rh = Sq * H;
  const int grid = stream_grid(n_rh * L / 4);
  // one instantiation per lanes-per-row-head L
  auto go = [&](auto kind) {
    constexpr int kL = decltype(kind)::value;
    lse_merge_kernel<kL><<<grid, kStreamThreads, 0, s>>>(out_acc, lse_acc, out_blk, lse_blk, Sq,
                                                         H, D, vpl);
  };
  switch (L) {
    case 1: go(std::integral_constant<int, 1>{}); break;
    case 2: go(std::integral_constant<int, 2>{}); break;
    case 4: go(std::integral_constant<int, 4>{}); break;
    case 8: go(std::integral_constant<int, 8>{}); break;
    case 16: go(std::integral_constant<int, 16>{}); break;
    case 32: go(std::integral_constant<int, 32>{}); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// --------------------------------------------------------------- permute
// Division by a run-time invariant with a multiply-high (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994,
// round-up variant): for 0 <= n < 2^31 and 1 <= d < 2^31,
//   l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1,
//   n / d = (umulhi(m, n) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
  static FastDiv make(uint32_t d) {
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    f.l = l;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
    return f;
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return (__umulhi(m, n) + n) >> l;
  }
};

// dst[b][a][w] = src[a][b][w] for src [A][B][W] and dst [B][A][W] (W in
// vectors).  seq_to_head is (A, B) = (S, P); head_to_seq is (P, S).
// Each thread moves UNROLL vectors per trip with all loads issued first.
template <typename VT, int UNROLL>
__global__ void __launch_bounds__(kStreamThreads)
    permute_kernel(const VT* __restrict__ src, VT* __restrict__ dst, uint32_t total,
                   FastDiv fw, FastDiv fa, uint32_t B) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t e0 = blockIdx.x * blockDim.x + threadIdx.x; e0 < total; e0 += stride * UNROLL) {
    VT v[UNROLL];
    uint32_t dsti[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const uint32_t e = e0 + u * stride;
      dsti[u] = e;
      if (e < total) {
        const uint32_t t = fw.div(e);
        const uint32_t w = e - t * fw.d;
        const uint32_t b = fa.div(t);
        const uint32_t a = t - b * fa.d;
        v[u] = __ldcs(src + ((static_cast<uint64_t>(a) * B + b) * fw.d + w));
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u)
      if (dsti[u] < total) __stcs(dst + dsti[u], v[u]);
  }
}

// 64-bit-index variant for tensors beyond 2^31 vectors.
template <typename VT>
__global__ void __launch_bounds__(kStreamThreads)
    permute_kernel64(const VT* __restrict__ src, VT* __restrict__ dst, int64_t total, int64_t W,
                     int64_t A, int64_t B) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += stride) {
    const int64_t t = e / W, w = e - t * W;
    const int64_t b = t / A, a = t - b * A;
    dst[e] = src[(a * B + b) * W + w];
  }
}

template <typename VT>
static cudaError_t launch_perm_t(const void* src, void* dst, int64_t A, int64_t B, int64_t W,
                                 cudaStream_t s) {
  const int64_t total = A * B * W;
  const int grid = stream_grid(total);
  if (total < (int64_t(1) << 31)) {
    permute_kernel<VT, 4><<<grid, kStreamThreads, 0, s>>>(
        static_cast<const VT*>(src), static_cast<VT*>(dst), static_cast<uint32_t>(total),
        FastDiv::make(static_cast<uint32_t>(W)), FastDiv::make(static_cast<uint32_t>(A)),
        static_cast<uint32_t>(B));
  } else {
    permute_kernel64<VT><<<grid, kStreamThreads, 0, s>>>(static_cast<const VT*>(src),
                                                          static_cast<VT*>(dst), total, W, A, B);
  }
  return cudaGetLastError();
}

// Swap the two outer dimensions of src [A][B][run_bytes] into dst [B][A][run_bytes].
cudaError_t launch_permute(const void* src, void* dst, int64_t A, int64_t B, int64_t run_bytes,
                           cudaStream_t s) {
  const uintptr_t align = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                          static_cast<uintptr_t>(run_bytes);
  if ((align & 15) == 0) return launch_perm_t<uint4>(src, dst, A, B, run_bytes / 16, s);
  if ((align & 7) == 0) return launch_perm_t<uint2>(src, dst, A, B, run_bytes / 8, s);
  if ((align & 3) == 0) return launch_perm_t<uint32_t>(src, dst, A, B, run_bytes / 4, s);
  if ((align & 1) == 0) return launch_perm_t<uint16_t>(src, dst, A, B, run_bytes / 2, s);
  return launch_perm_t<uint8_t>(src, dst, A, B, run_bytes, s);
}

// ------------------------------------------------------------ empty block
// Rows that see no key: out = 0 (fp32 or bf16), lse = -inf.
__global__ void fill_empty_kernel(void* out, int out_bytes_per_el, int64_t n_out, float* lse,
                                  int64_t n_lse) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_out;
       e += stride) {
    if (out_bytes_per_el == 4)
      static_cast<float*>(out)[e] = 0.f;
    else
      static_cast<uint16_t*>(out)[e] = 0;
  }
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n_lse;
       e += stride)
    lse[e] = -CUDART_INF_F;
}

cudaError_t launch_fill_empty(void* out, int out_bytes_per_el, int64_t n_out, float* lse,
                              int64_t n_lse, cudaStream_t s) {
  const int grid = stream_grid(n_out > n_lse ? n_out : n_lse);
  fill_empty_kernel<<<grid, kStreamThreads, 0, s>>>(out, out_bytes_per_el, n_out, lse, n_lse);
  return cudaGetLastError();
}

// ------------------------------------------------------ backward delta
// delta[h][row] = sum_d dO[row,h,d] * O[row,h,d]: the row term of
// ds = p (dp - delta) in the backward of softmax attention, from the final
// (merged) output.  bf16 inputs [rows, H, 128]; 16 lanes own one row-head
// (8 elements = 16 bytes each), row-heads visited in memory order so that
// a warp reads 512 contiguous bytes of each tensor per trip.
__device__ __forceinline__ float dot_bf16x8(uint4 a, uint4 b) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s = fmaf(__uint_as_float(av[i] << 16), __uint_as_float(bv[i] << 16), s);
    s = fmaf(__uint_as_float(av[i] & 0xffff0000u), __uint_as_float(bv[i] & 0xffff0000u), s);
  }
  return s;
}

__global__ void __launch_bounds__(kStreamThreads)
    bwd_delta_kernel(const uint4* __restrict__ out, const uint4* __restrict__ dout,
                     float* __restrict__ delta, int64_t rows, int H, int64_t ld) {
  constexpr int U = 4;  // row-heads per half-warp per trip, all loads first
  const int64_t n_rh = rows * H;
  const int sub = threadIdx.x & 15;
  const int64_t groups = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 4);
  const int64_t g0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 4;
  // the loop bound is taken per warp (both half-warps run every trip, so
  // the shuffles see all 32 lanes)
  for (int64_t wbase = g0 & ~int64_t(1); wbase < n_rh; wbase += U * groups) {
    const int64_t base = wbase + (g0 & 1);
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t rh = base + u * groups;
      if (rh < n_rh) {
        a[u] = __ldcs(out + rh * 16 + sub);
        b[u] = __ldcs(dout + rh * 16 + sub);
      } else {
        a[u] = b[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float s = dot_bf16x8(a[u], b[u]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      const int64_t rh = base + u * groups;
      if (sub == 0 && rh < n_rh) delta[(rh % H) * ld + rh / H] = s;
    }
  }
}

cudaError_t launch_bwd_delta(const void* out, const void* dout, float* delta, int64_t rows, int H,
                             int64_t ld, cudaStream_t s) {
  const int grid = stream_grid(rows * H * 16);
  bwd_delta_kernel<<<grid, kStreamThreads, 0, s>>>(static_cast<const uint4*>(out),
                                                   static_cast<const uint4*>(dout), delta, rows, H,
                                                   ld);
  return cudaGetLastError();
}

// ------------------------------------------------------ timeout self-test
// One thread waits on an mbarrier that nothing arrives at; the bounded wait
// expires and the kernel records the timeout status, then returns.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int* dev_err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = sm100::smem_u32(&bar);
    sm100::mbar_init(b, 1);
    sm100::fence_mbar_init();
    if (!sm100::mbar_wait(b, 0, limit_ns, nullptr)) atomicCAS(dev_err, 0, kDevErrTimeout);
  }
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int* dev_err, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, dev_err);
  return cudaGetLastError();
}

}  // namespace cpattn
