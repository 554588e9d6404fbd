// cp_ring_forward_noalloc: the ring forward for callers that may not
// allocate device memory.
//
// cp_ring_forward with a bf16 output, when it runs the ring step by step
// (fp32 inputs, or the striped layout), needs an fp32 accumulator of S*H*D
// floats as scratch, which the caller normally allocates and passes as the
// workspace.  Some callers cannot do that: code that runs inside another
// framework's fixed device-memory budget (an inference engine plugin whose
// memory is all handed out up front by the host framework), or code on a
// latency-critical path where a cudaMalloc/cudaFree would synchronise the
// device and stall every other stream.  For them this file keeps the
// accumulator in a file-scope device array instead, so the call needs no
// workspace and allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include <stdio.h>

#include "../../include/cpattn.h"

namespace cpattn {
int set_last_error(int code, const char* msg);
bool ring_runs_fused(cp_dtype in_dt, cp_layout layout);
}

namespace {

// Scratch shared by every call on a device.  64 MiB = 16 Mi fp32 values,
// i.e. S*H*D <= 16,777,216 (S = 4096 at H = 32, D = 128).  Every GPU that
// loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = size_t(64) << 20;
static __device__ __align__(256) float g_ring_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_ring_scratch on the current device.  In host code the
// symbol's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return -1;
  if (dev < 0 || dev >= kMaxDevices) return -2;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_ring_scratch);
    if (e != cudaSuccess || p == nullptr) return -1;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return 0;
}

}  // namespace

extern "C" int cp_ring_forward_noalloc(const void* q, const void* k, const void* v,
                                       cp_dtype in_dt, int64_t S, int H, int Hkv, int D, int P,
                                       cp_layout layout, void* out, cp_dtype out_dt, float* lse,
                                       cp_stream_t stream) {
  // same validation and error reporting as the workspace version
  int64_t need = cp_ring_workspace_size(S, H, D, out_dt);
  if (need < 0) return static_cast<int>(need);
  // a ring cp_ring_forward runs in one launch keeps no accumulator
  if (cpattn::ring_runs_fused(in_dt, layout)) need = 0;
  if (static_cast<uint64_t>(need) > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "cp_ring_forward_noalloc: S*H*D*4 = %lld bytes exceeds the built-in scratch of "
             "%lld bytes (S*H*D <= %lld); use cp_ring_forward with a workspace",
             (long long)need, (long long)kScratchBytes, (long long)(kScratchBytes / 4));
    return cpattn::set_last_error(CP_ERR_SHAPE, msg);
  }
  void* scratch = nullptr;
  if (need > 0 && scratch_address(&scratch) != 0)
    return cpattn::set_last_error(CP_ERR_CUDA,
                                  "cp_ring_forward_noalloc: cudaGetSymbolAddress of the "
                                  "scratch array failed on the current device");
  return cp_ring_forward(q, k, v, in_dt, S, H, Hkv, D, P, layout, out, out_dt, lse, scratch,
                         stream);
}
