// noalloc.cu -- psa_attention_bwd_noalloc: the fused PSA backward without a
// caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: a plugin inside a framework that owns every device allocation and
// forbids allocating while work is being enqueued, or a latency-critical loop in
// which cudaMalloc / cudaFree would synchronise the device.  For them the
// per-head softmax statistic (delta, one float per head and position) lives in a
// fixed array in this library's own device memory instead of a workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the library
// holds it (kMaxDeltaFloats * 4 bytes = 4 MiB) until the process exits.  Host code
// cannot use the variable's name as a device address, so the first call on each
// device (with that device current) looks the address up with
// cudaGetSymbolAddress and caches it per device.
#include <atomic>

#include <cuda_runtime.h>

#include "../../include/psa.h"

namespace {

// Largest B * num_heads * H * W the array holds (one float each).
constexpr size_t kMaxDeltaFloats = size_t(1) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_delta[kMaxDeltaFloats];

std::atomic<void*> g_delta_addr[kMaxDevices];

// Device address of g_noalloc_delta on the current device (looked up once per device).
psa_status_t delta_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PSA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PSA_ERR_UNSUPPORTED;
  void* p = g_delta_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || !p) return PSA_ERR_CUDA;
    g_delta_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return PSA_OK;
}

}  // namespace

extern "C" psa_status_t psa_attention_bwd_noalloc(const void* qkv_nchw, const void* out_nchw,
                                                  const void* dout_nchw, const float* lse,
                                                  const void* dvres_nchw, void* dqkv_nchw,
                                                  psa_shape_t shape, float scale,
                                                  cudaStream_t stream) {
  // the checks psa_attention_bwd makes first (required pointers, the shape), then
  // the capacity of the array, then everything else psa_attention_bwd checks
  if (!qkv_nchw || !out_nchw || !dout_nchw || !lse || !dqkv_nchw) return PSA_ERR_INVALID_ARG;
  const size_t ws = psa_attention_bwd_workspace_size(shape);
  if (ws == 0) return PSA_ERR_INVALID_ARG;
  if ((size_t)shape.B * shape.num_heads * shape.H * shape.W > kMaxDeltaFloats)
    return PSA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  psa_status_t e = delta_scratch(&scratch);
  if (e != PSA_OK) return e;
  // The array is psa_attention_bwd's workspace.  The two-kernel backward's dQ
  // kernel writes every delta value of this call before the dK/dV kernel reads
  // it; the one-kernel backward beyond 512 positions (chosen when its dQ
  // accumulator fits) stores each accumulator row at the first key tile before it
  // reads it at the next; up to 512 positions nothing touches the array.  So
  // nothing an earlier call left needs clearing, and only calls that use the
  // array can race on it.
  return psa_attention_bwd(qkv_nchw, out_nchw, dout_nchw, lse, dvres_nchw, dqkv_nchw, scratch,
                           kMaxDeltaFloats * sizeof(float), shape, scale, stream);
}
