// api.cu -- the C ABI of include/psa.h: host-side validation, TMA tensor maps and
// launches.  No entry point allocates, frees or synchronises (except
// psa_get_last_device_error, which is documented to synchronise).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "../../include/psa.h"
#include "attn.cuh"
#include "ptx.cuh"
#include "layout.cuh"

namespace psa {
__device__ int g_device_error = 0;

namespace {
// One CTA of one warp waits, through the same bounded wait as the attention
// kernels, on an mbarrier that nothing ever arrives at, so the wait gives up
// after limit_ns, records PSA_ERR_TIMEOUT in g_device_error and the kernel
// returns.  Nothing is left waiting and no global memory besides the error word
// is touched.
__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncwarp();
  mbar_wait(&bar, 0, &abort, limit_ns);
}
}  // namespace

int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  int n = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t set_max_dynamic_smem(const void* kern, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;  // (kernel, device)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kern, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({kern, dev});
  return e;
}
}  // namespace psa

namespace {

using psa::BwdArgs;
using psa::FwdArgs;

constexpr float kLog2e = 1.4426950408889634074f;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(psa_dtype_t t) { return t == PSA_DTYPE_F32 ? 4 : 2; }

psa_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? PSA_OK : PSA_ERR_CUDA; }

psa_status_t check_shape(const psa_shape_t& s) {
  if (s.B <= 0 || s.num_heads <= 0 || s.key_dim <= 0 || s.H <= 0 || s.W <= 0)
    return PSA_ERR_INVALID_ARG;
  if (s.dtype != PSA_DTYPE_F32 && s.dtype != PSA_DTYPE_BF16) return PSA_ERR_INVALID_ARG;
  if (s.key_dim > 128) return PSA_ERR_UNSUPPORTED;  // layout tiles stage KD x 64 in shared memory
  // every index of the largest tensor must fit the kernels' int coordinates
  const long long n = (long long)s.H * s.W;
  const long long big = (long long)s.B * s.num_heads * 4 * s.key_dim * n;
  if (n > (1LL << 30) || big > (1LL << 40) || (long long)s.B * s.num_heads * 4 * s.key_dim > (1LL << 30))
    return PSA_ERR_UNSUPPORTED;
  return PSA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time
// dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

CUtensorMapSwizzle swizzle_for(uint32_t inner_bytes) {
  return inner_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
}

// 3-D bf16 map over [BH, N, d] (d contiguous), box {d, box_rows, 1}.
bool map_rows(CUtensorMap* m, const void* base, int BH, int N, int d, int box_rows = 128) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {(cuuint32_t)d, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(d * 2),
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map over an NCHW tensor viewed as [rows, N] (N contiguous), box {64, box_rows}.
bool map_nchw(CUtensorMap* m, const void* base, long long rows, int N, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over the 2-D [rows, N] view of an NCHW output for TMA stores of
// whole tiles: box {128 positions, box_rows channel rows}, no swizzle (the
// staging tile is plain row-major).
bool map_nchw_store(CUtensorMap* m, void* base, long long rows, int N, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of the QKV convolution: w [cout, cin] (box {64, 128}) and x viewed as
// 3-D (N, cin, B) (box {64, 64, 1}); positions and channels past the ends read as 0.
bool map_conv(CUtensorMap* mw, CUtensorMap* mx, CUtensorMap* mo, const void* w, const void* x,
              void* out, int B, int cin, int cout, int N) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t wd[2] = {(cuuint64_t)cin, (cuuint64_t)cout};
  cuuint64_t ws[1] = {(cuuint64_t)cin * 2};
  cuuint32_t wb[2] = {64, 128};
  cuuint32_t e2[2] = {1, 1};
  if (enc(mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), wd, ws, wb, e2,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cuuint64_t xd[3] = {(cuuint64_t)N, (cuuint64_t)cin, (cuuint64_t)B};
  cuuint64_t xs[2] = {(cuuint64_t)N * 2, (cuuint64_t)cin * N * 2};
  cuuint32_t xb[3] = {64, 64, 1};
  cuuint32_t e3[3] = {1, 1, 1};
  if (enc(mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), xd, xs, xb, e3,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  // output tiles for TMA stores: 64 positions x 128 output channels of one batch item
  cuuint64_t od[3] = {(cuuint64_t)N, (cuuint64_t)cout, (cuuint64_t)B};
  cuuint64_t os[2] = {(cuuint64_t)N * 2, (cuuint64_t)cout * N * 2};
  cuuint32_t ob[3] = {64, 128, 1};
  return enc(mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, od, os, ob, e3,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

psa_status_t check_fa2(const void* const* ptrs, int nptr, int BH, int n_ctx, int head_dim,
                       float scale, psa_dtype_t dtype) {
  for (int i = 0; i < nptr; ++i) {
    if (!ptrs[i]) return PSA_ERR_INVALID_ARG;
    if (!aligned16(ptrs[i])) return PSA_ERR_ALIGNMENT;
  }
  if (BH <= 0 || n_ctx <= 0 || head_dim <= 0 || !isfinite(scale) || !(scale > 0.f))
    return PSA_ERR_INVALID_ARG;
  if (dtype != PSA_DTYPE_F32 && dtype != PSA_DTYPE_BF16) return PSA_ERR_INVALID_ARG;
  if (head_dim != 32 && head_dim != 64) return PSA_ERR_UNSUPPORTED;
  if ((long long)BH > 65535 || (long long)n_ctx > (1LL << 28)) return PSA_ERR_UNSUPPORTED;
  return PSA_OK;
}

}  // namespace

extern "C" {

const char* psa_status_string(psa_status_t s) {
  switch (s) {
    case PSA_OK: return "PSA_OK";
    case PSA_ERR_INVALID_ARG: return "PSA_ERR_INVALID_ARG: null pointer, non-positive size or bad enum";
    case PSA_ERR_UNSUPPORTED: return "PSA_ERR_UNSUPPORTED: size or dtype not implemented";
    case PSA_ERR_ALIGNMENT: return "PSA_ERR_ALIGNMENT: pointer or row not 16-byte aligned";
    case PSA_ERR_CUDA: return "PSA_ERR_CUDA: a CUDA call or launch failed";
    case PSA_ERR_TIMEOUT: return "PSA_ERR_TIMEOUT: an on-chip wait gave up";
  }
  return "unknown psa_status_t";
}

psa_status_t psa_debug_wait_timeout(unsigned long long limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > 100000000ull) return PSA_ERR_INVALID_ARG;
  psa::wait_timeout_probe_kernel<<<1, 32, 0, stream>>>((uint64_t)limit_ns);
  return from_cuda(cudaGetLastError());
}

psa_status_t psa_qkv_conv(const void* x, const void* w, const float* bias, void* qkv, int B,
                          int cin, int cout, int H, int W, cudaStream_t st) {
  if (!x || !w || !qkv) return PSA_ERR_INVALID_ARG;
  if (B <= 0 || cin <= 0 || cout <= 0 || H <= 0 || W <= 0) return PSA_ERR_INVALID_ARG;
  const long long N = (long long)H * W;
  if (N > (1LL << 30) || (long long)B * cin * N > (1LL << 40) || (long long)B * cout * N > (1LL << 40) ||
      (long long)B * cout > (1LL << 30) || (long long)B * cin > (1LL << 30))
    return PSA_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(w) || !aligned16(qkv) || (bias && (reinterpret_cast<uintptr_t>(bias) & 3)))
    return PSA_ERR_ALIGNMENT;
  psa::ConvArgs a{};
  a.B = B;
  a.cin = cin;
  a.cout = cout;
  a.N = (int)N;
  a.bias = bias;
  a.out = static_cast<__nv_bfloat16*>(qkv);
  if (cin % 8 == 0 && N % 8 == 0) {
    CUtensorMap mw, mx, mo;
    if (!map_conv(&mw, &mx, &mo, w, x, qkv, B, cin, cout, (int)N)) return PSA_ERR_CUDA;
    return from_cuda(psa::launch_qkv_conv_tc(mw, mx, mo, a, st));
  }
  if (cout > 65535 || B > 65535) return PSA_ERR_UNSUPPORTED;
  return from_cuda(psa::launch_qkv_conv_simt(x, w, a, st));
}

psa_status_t psa_get_last_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, psa::g_device_error, sizeof(int)) != cudaSuccess) return PSA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(psa::g_device_error, &zero, sizeof(int)) != cudaSuccess) return PSA_ERR_CUDA;
  }
  return v == 0 ? PSA_OK : (psa_status_t)v;
}

// ---------------------------------------------------------------- layout entry points
psa_status_t psa_pack_qkv(const void* qkv, void* packed, psa_shape_t s, cudaStream_t st) {
  if (!qkv || !packed) return PSA_ERR_INVALID_ARG;
  psa_status_t e = check_shape(s);
  if (e != PSA_OK) return e;
  if (!aligned16(qkv) || !aligned16(packed)) return PSA_ERR_ALIGNMENT;
  return from_cuda(psa::launch_pack_qkv(qkv, packed, s.B, s.num_heads, s.key_dim, s.H * s.W,
                                        elem_bytes(s.dtype), st));
}

psa_status_t psa_unpack_qkv(const void* packed, void* qkv, psa_shape_t s, cudaStream_t st) {
  if (!qkv || !packed) return PSA_ERR_INVALID_ARG;
  psa_status_t e = check_shape(s);
  if (e != PSA_OK) return e;
  if (!aligned16(qkv) || !aligned16(packed)) return PSA_ERR_ALIGNMENT;
  return from_cuda(psa::launch_unpack_qkv(packed, qkv, s.B, s.num_heads, s.key_dim, s.H * s.W,
                                          elem_bytes(s.dtype), st));
}

psa_status_t psa_extract_v(const void* qkv, void* v, psa_shape_t s, cudaStream_t st) {
  if (!qkv || !v) return PSA_ERR_INVALID_ARG;
  psa_status_t e = check_shape(s);
  if (e != PSA_OK) return e;
  if (!aligned16(qkv) || !aligned16(v)) return PSA_ERR_ALIGNMENT;
  if ((2LL * s.key_dim * s.H * s.W * elem_bytes(s.dtype)) % 16 != 0) return PSA_ERR_ALIGNMENT;
  return from_cuda(psa::launch_extract_v(qkv, v, s.B, s.num_heads, s.key_dim, s.H * s.W,
                                         elem_bytes(s.dtype), st));
}

psa_status_t psa_merge_attn(const void* o_lo, const void* o_hi, void* out, psa_shape_t s,
                            cudaStream_t st) {
  if (!o_lo || !o_hi || !out) return PSA_ERR_INVALID_ARG;
  psa_status_t e = check_shape(s);
  if (e != PSA_OK) return e;
  if (!aligned16(o_lo) || !aligned16(o_hi) || !aligned16(out)) return PSA_ERR_ALIGNMENT;
  return from_cuda(psa::launch_merge_attn(o_lo, o_hi, out, s.B, s.num_heads, s.key_dim,
                                          s.H * s.W, elem_bytes(s.dtype), st));
}

psa_status_t psa_unmerge_attn(const void* dout, void* do_lo, void* do_hi, psa_shape_t s,
                              cudaStream_t st) {
  if (!dout || !do_lo || !do_hi) return PSA_ERR_INVALID_ARG;
  psa_status_t e = check_shape(s);
  if (e != PSA_OK) return e;
  if (!aligned16(dout) || !aligned16(do_lo) || !aligned16(do_hi)) return PSA_ERR_ALIGNMENT;
  return from_cuda(psa::launch_unmerge_attn(dout, do_lo, do_hi, s.B, s.num_heads, s.key_dim,
                                            s.H * s.W, elem_bytes(s.dtype), st));
}

// ---------------------------------------------------------------- Flash Attention 2
psa_status_t flash_attn2_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                             int BH, int n_ctx, int head_dim, float scale, psa_dtype_t dtype,
                             cudaStream_t st) {
  const void* ptrs[4] = {q, k, v, o};
  psa_status_t e = check_fa2(ptrs, 4, BH, n_ctx, head_dim, scale, dtype);
  if (e != PSA_OK) return e;
  if (lse && !aligned16(lse)) return PSA_ERR_ALIGNMENT;
  if (dtype == PSA_DTYPE_F32) {
    psa::SimtArgs a{};
    a.q = q; a.k = k; a.v = v; a.out = o; a.lse = lse;
    a.N = n_ctx; a.BH = BH; a.nh = 1; a.scale = scale;
    return from_cuda(psa::launch_simt_fwd(a, false, false, head_dim, st));
  }
  CUtensorMap mq, mk, mv;
  // the forward walks 128-query tiles against 64-key tiles
  if (!map_rows(&mq, q, BH, n_ctx, head_dim, 128) || !map_rows(&mk, k, BH, n_ctx, head_dim, 64) ||
      !map_rows(&mv, v, BH, n_ctx, head_dim, 64))
    return PSA_ERR_CUDA;
  FwdArgs a{};
  a.N = n_ctx;
  a.BH = BH;
  a.nh = 1;
  a.scale_log2 = scale * kLog2e;
  a.out = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  return from_cuda(psa::launch_fa2_fwd_bf16(mq, mk, mv, a, head_dim, st));
}

psa_status_t flash_attn2_bwd_dq(const void* q, const void* k, const void* v, const void* o,
                                const void* do_, const float* lse, float* delta, void* dq, int BH,
                                int n_ctx, int head_dim, float scale, psa_dtype_t dtype,
                                cudaStream_t st) {
  const void* ptrs[8] = {q, k, v, o, do_, lse, delta, dq};
  psa_status_t e = check_fa2(ptrs, 8, BH, n_ctx, head_dim, scale, dtype);
  if (e != PSA_OK) return e;
  if (dtype == PSA_DTYPE_F32) {
    psa::SimtArgs a{};
    a.q = q; a.k = k; a.v = v; a.o = o; a.dO = do_; a.dq = dq;
    a.lse = const_cast<float*>(lse); a.delta = delta;
    a.N = n_ctx; a.BH = BH; a.nh = 1; a.scale = scale;
    return from_cuda(psa::launch_simt_bwd_dq(a, false, false, head_dim, st));
  }
  CUtensorMap mq, mk, mv, mdo;
  // the dQ kernel walks 128-query tiles against 64-key tiles
  if (!map_rows(&mq, q, BH, n_ctx, head_dim, 128) || !map_rows(&mk, k, BH, n_ctx, head_dim, 64) ||
      !map_rows(&mv, v, BH, n_ctx, head_dim, 64) || !map_rows(&mdo, do_, BH, n_ctx, head_dim, 128))
    return PSA_ERR_CUDA;
  BwdArgs a{};
  a.N = n_ctx;
  a.BH = BH;
  a.nh = 1;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.lse = lse;
  a.delta = delta;
  a.o = static_cast<const __nv_bfloat16*>(o);
  a.dO = static_cast<const __nv_bfloat16*>(do_);
  a.dq = static_cast<__nv_bfloat16*>(dq);
  return from_cuda(psa::launch_fa2_bwd_dq(mq, mk, mv, mdo, a, BH, head_dim, st));
}

psa_status_t flash_attn2_bwd_dkdv(const void* q, const void* k, const void* v, const void* do_,
                                  const float* lse, const float* delta, void* dk, void* dv,
                                  int BH, int n_ctx, int head_dim, float scale,
                                  psa_dtype_t dtype, cudaStream_t st) {
  const void* ptrs[8] = {q, k, v, do_, lse, delta, dk, dv};
  psa_status_t e = check_fa2(ptrs, 8, BH, n_ctx, head_dim, scale, dtype);
  if (e != PSA_OK) return e;
  if (dtype == PSA_DTYPE_F32) {
    psa::SimtArgs a{};
    a.q = q; a.k = k; a.v = v; a.dO = do_; a.dk = dk; a.dv = dv;
    a.lse = const_cast<float*>(lse); a.delta = const_cast<float*>(delta);
    a.N = n_ctx; a.BH = BH; a.nh = 1; a.scale = scale;
    return from_cuda(psa::launch_simt_bwd_dkdv(a, false, false, head_dim, st));
  }
  CUtensorMap mq, mk, mv, mdo;
  // the dK/dV kernel walks 128-key tiles against 64-query tiles
  if (!map_rows(&mq, q, BH, n_ctx, head_dim, 64) || !map_rows(&mk, k, BH, n_ctx, head_dim, 128) ||
      !map_rows(&mv, v, BH, n_ctx, head_dim, 128) || !map_rows(&mdo, do_, BH, n_ctx, head_dim, 64))
    return PSA_ERR_CUDA;
  BwdArgs a{};
  a.N = n_ctx;
  a.BH = BH;
  a.nh = 1;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.lse = lse;
  a.delta = const_cast<float*>(delta);
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  return from_cuda(psa::launch_fa2_bwd_dkdv(mq, mk, mv, mdo, a, BH, head_dim, st));
}

// ---------------------------------------------------------------- fused PSA
namespace {
// NCHW channel rows of N bf16 elements start on 16-byte boundaries, as the TMA
// tensor maps of the tensor-core kernels require.
bool tma_rows(const psa_shape_t& s) { return ((long long)s.H * s.W * 2) % 16 == 0; }

// Arguments of the CUDA-core kernels for an NCHW problem (inputs and outputs set
// by the caller).
psa::SimtArgs simt_nchw(const void* qkv, const psa_shape_t& s, float scale) {
  psa::SimtArgs a{};
  a.q = a.k = a.v = qkv;
  a.N = s.H * s.W;
  a.BH = s.B * s.num_heads;
  a.nh = s.num_heads;
  a.qkv_ch = s.num_heads * 4 * s.key_dim;
  a.out_ch = s.num_heads * 2 * s.key_dim;
  a.scale = scale;
  return a;
}

// The forward kernels write any of out, lse, v_nchw (PsaExtractV) and out_res
// (out + V) that is not null; at least one of out, out_res is required.
psa_status_t fused_fwd(const void* qkv, void* out, float* lse, void* v_nchw, void* out_res,
                       psa_shape_t s, float scale, cudaStream_t st) {
  if (!qkv || (!out && !out_res)) return PSA_ERR_INVALID_ARG;
  psa_status_t e = check_shape(s);
  if (e != PSA_OK) return e;
  if (!isfinite(scale) || !(scale > 0.f)) return PSA_ERR_INVALID_ARG;
  if (s.key_dim != 32 && s.key_dim != 64) return PSA_ERR_UNSUPPORTED;
  if ((long long)s.B * s.num_heads > 65535) return PSA_ERR_UNSUPPORTED;
  if (!aligned16(qkv) || (out && !aligned16(out)) || (lse && !aligned16(lse)) ||
      (v_nchw && !aligned16(v_nchw)) || (out_res && !aligned16(out_res)))
    return PSA_ERR_ALIGNMENT;
  const int N = s.H * s.W;
  const int nh = s.num_heads, KD = s.key_dim;
  if (s.dtype == PSA_DTYPE_F32 || !tma_rows(s)) {
    // fp32, or channel rows a tensor map cannot address: CUDA cores
    psa::SimtArgs a = simt_nchw(qkv, s, scale);
    a.out = out;
    a.out_res = out_res;
    a.lse = lse;
    e = from_cuda(psa::launch_simt_fwd(a, true, s.dtype == PSA_DTYPE_BF16, KD, st));
  } else {
    CUtensorMap mqk, mv, mout, mvres;
    const long long rows = (long long)s.B * nh * 4 * KD, orows = (long long)s.B * nh * 2 * KD;
    if (!map_nchw(&mqk, qkv, rows, N, KD) || !map_nchw(&mv, qkv, rows, N, 2 * KD))
      return PSA_ERR_CUDA;
    // Out and the extracted V are written by TMA stores: Out from the staged tile,
    // V straight from the K/V stage (same box and swizzle as the V load)
    mout = mv;
    mvres = mv;
    if ((out && !map_nchw_store(&mout, out, orows, N, 2 * KD)) ||
        (v_nchw && !map_nchw(&mvres, v_nchw, orows, N, 2 * KD)))
      return PSA_ERR_CUDA;
    FwdArgs a{};
    a.N = N;
    a.BH = s.B * nh;
    a.nh = nh;
    a.qkv_ch = nh * 4 * KD;
    a.out_ch = nh * 2 * KD;
    a.vres_ch = nh * 2 * KD;
    a.scale_log2 = scale * kLog2e;
    a.out = static_cast<__nv_bfloat16*>(out);
    a.lse = lse;
    a.vres = static_cast<__nv_bfloat16*>(v_nchw);  // PsaExtractV fused into the forward
    a.out_res = static_cast<__nv_bfloat16*>(out_res);
    a.qkv = static_cast<const __nv_bfloat16*>(qkv);
    return from_cuda(psa::launch_psa_fwd_bf16(mqk, mv, mout, mvres, a, KD, st));
  }
  if (e != PSA_OK || !v_nchw) return e;
  return from_cuda(psa::launch_extract_v(qkv, v_nchw, s.B, nh, KD, N, elem_bytes(s.dtype), st));
}
}  // namespace

psa_status_t psa_attention_fwd(const void* qkv, void* out, float* lse, void* v_nchw,
                               psa_shape_t s, float scale, cudaStream_t st) {
  if (!out) return PSA_ERR_INVALID_ARG;
  return fused_fwd(qkv, out, lse, v_nchw, nullptr, s, scale, st);
}

psa_status_t psa_attention_fwd_residual(const void* qkv, void* out_res, void* out, float* lse,
                                        psa_shape_t s, float scale, cudaStream_t st) {
  if (!out_res) return PSA_ERR_INVALID_ARG;
  return fused_fwd(qkv, out, lse, nullptr, out_res, s, scale, st);
}

namespace {
size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

// delta [BH, N] fp32: what the two-kernel backward needs
size_t delta_ws_bytes(const psa_shape_t& s) {
  return round256((size_t)s.B * s.num_heads * s.H * s.W * sizeof(float));
}

// the dQ accumulator [BH, N, 32] fp32 of the one-kernel backward beyond
// kFusedBwdMaxN positions (0 where that form does not apply)
size_t long_fused_ws_bytes(const psa_shape_t& s) {
  const long long N = (long long)s.H * s.W;
  if (s.key_dim != 32 || s.dtype != PSA_DTYPE_BF16 || (N * 2) % 16 != 0 ||
      N <= psa::kFusedBwdMaxN || N > psa::kFusedBwdMaxNLong)
    return 0;
  return round256((size_t)s.B * s.num_heads * N * 32 * sizeof(float));
}
}  // namespace

size_t psa_attention_bwd_workspace_size(psa_shape_t s) {
  if (check_shape(s) != PSA_OK) return 0;
  const size_t a = delta_ws_bytes(s), b = long_fused_ws_bytes(s);
  return a > b ? a : b;
}

namespace {
// Host-side checks shared by the fused backward entry points (no CUDA call).
psa_status_t validate_bwd(const void* qkv, const void* dout, const float* lse, const void* dqkv,
                          const float* delta, const void* dvres, const void* out, bool need_out,
                          const psa_shape_t& s, float scale) {
  if (!qkv || !dout || !lse || !dqkv || !delta || (need_out && !out)) return PSA_ERR_INVALID_ARG;
  psa_status_t e = check_shape(s);
  if (e != PSA_OK) return e;
  if (!isfinite(scale) || !(scale > 0.f)) return PSA_ERR_INVALID_ARG;
  if (s.key_dim != 32 && s.key_dim != 64) return PSA_ERR_UNSUPPORTED;
  if ((long long)s.B * s.num_heads > 65535) return PSA_ERR_UNSUPPORTED;
  if (!aligned16(qkv) || !aligned16(dout) || !aligned16(lse) || !aligned16(dqkv) ||
      !aligned16(delta) || (dvres && !aligned16(dvres)) || (out && !aligned16(out)))
    return PSA_ERR_ALIGNMENT;
  return PSA_OK;
}

// The backward on CUDA cores (fp32, or rows a tensor map cannot address).
bool simt_bwd(const psa_shape_t& s) { return s.dtype == PSA_DTYPE_F32 || !tma_rows(s); }

psa::SimtArgs simt_bwd_args(const void* qkv, const void* out, const void* dout, const float* lse,
                            const void* dvres, void* dqkv, float* delta, const psa_shape_t& s,
                            float scale) {
  psa::SimtArgs a = simt_nchw(qkv, s, scale);
  a.o = out;
  a.dO = dout;
  a.dvres = dvres;
  a.dq = a.dk = a.dv = dqkv;
  a.lse = const_cast<float*>(lse);
  a.delta = delta;
  return a;
}

// Tensor maps and kernel arguments of a validated fused backward call.
psa_status_t make_bwd(const void* qkv, const void* dout, const float* lse, const void* dqkv,
                      const float* delta, const void* dvres, const void* out,
                      const psa_shape_t& s, float scale, CUtensorMap* mqk, CUtensorMap* mv,
                      CUtensorMap* mdo, CUtensorMap* mo, BwdArgs* a) {
  const int N = s.H * s.W;
  const int nh = s.num_heads, KD = s.key_dim;
  const long long rows = (long long)s.B * nh * 4 * KD;
  const long long out_rows = (long long)s.B * nh * 2 * KD;
  if (!map_nchw(mqk, qkv, rows, N, KD) || !map_nchw(mv, qkv, rows, N, 2 * KD) ||
      !map_nchw(mdo, dout, out_rows, N, 2 * KD) ||
      (out && !map_nchw(mo, out, out_rows, N, 2 * KD)))
    return PSA_ERR_CUDA;
  *a = BwdArgs{};
  a->N = N;
  a->BH = s.B * nh;
  a->nh = nh;
  a->qkv_ch = nh * 4 * KD;
  a->out_ch = nh * 2 * KD;
  a->scale = scale;
  a->scale_log2 = scale * kLog2e;
  a->lse = lse;
  a->delta = const_cast<float*>(delta);
  a->o = static_cast<const __nv_bfloat16*>(out);
  a->dO = static_cast<const __nv_bfloat16*>(dout);
  a->dvres = static_cast<const __nv_bfloat16*>(dvres);
  a->dq = a->dk = a->dv = static_cast<__nv_bfloat16*>(const_cast<void*>(dqkv));
  return PSA_OK;
}
}  // namespace

psa_status_t psa_attention_bwd_dq(const void* qkv, const void* out, const void* dout,
                                  const float* lse, float* delta, void* dqkv, psa_shape_t s,
                                  float scale, cudaStream_t st) {
  CUtensorMap mqk, mv, mdo, mo;
  BwdArgs a;
  psa_status_t e = validate_bwd(qkv, dout, lse, dqkv, delta, nullptr, out, true, s, scale);
  if (e != PSA_OK) return e;
  if (simt_bwd(s))
    return from_cuda(psa::launch_simt_bwd_dq(
        simt_bwd_args(qkv, out, dout, lse, nullptr, dqkv, delta, s, scale), true,
        s.dtype == PSA_DTYPE_BF16, s.key_dim, st));
  e = make_bwd(qkv, dout, lse, dqkv, delta, nullptr, out, s, scale, &mqk, &mv, &mdo, &mo, &a);
  if (e != PSA_OK) return e;
  return from_cuda(psa::launch_psa_bwd_dq(mqk, mv, mdo, mo, a, s.B * s.num_heads, s.key_dim, st));
}

psa_status_t psa_attention_bwd_dkdv(const void* qkv, const void* dout, const float* lse,
                                    const float* delta, const void* dvres, void* dqkv,
                                    psa_shape_t s, float scale, cudaStream_t st) {
  CUtensorMap mqk, mv, mdo;
  BwdArgs a;
  psa_status_t e = validate_bwd(qkv, dout, lse, dqkv, delta, dvres, nullptr, false, s, scale);
  if (e != PSA_OK) return e;
  if (simt_bwd(s))
    return from_cuda(psa::launch_simt_bwd_dkdv(
        simt_bwd_args(qkv, nullptr, dout, lse, dvres, dqkv, const_cast<float*>(delta), s, scale),
        true, s.dtype == PSA_DTYPE_BF16, s.key_dim, st));
  e = make_bwd(qkv, dout, lse, dqkv, delta, dvres, nullptr, s, scale, &mqk, &mv, &mdo, nullptr, &a);
  if (e != PSA_OK) return e;
  return from_cuda(psa::launch_psa_bwd_dkdv(mqk, mv, mdo, a, s.B * s.num_heads, s.key_dim, st));
}

psa_status_t psa_attention_bwd(const void* qkv, const void* out, const void* dout,
                               const float* lse, const void* dvres, void* dqkv, void* ws,
                               size_t ws_bytes, psa_shape_t s, float scale, cudaStream_t st) {
  if (!ws) return PSA_ERR_INVALID_ARG;
  psa_status_t e = check_shape(s);
  if (e != PSA_OK) return e;
  if (ws_bytes < delta_ws_bytes(s)) return PSA_ERR_INVALID_ARG;
  float* delta = static_cast<float*>(ws);
  // validate both launches completely before issuing either
  CUtensorMap mqk, mv, mdo, mo, mqk2, mv2, mdo2;
  BwdArgs a_dq, a_kv;
  e = validate_bwd(qkv, dout, lse, dqkv, delta, nullptr, out, true, s, scale);
  if (e == PSA_OK) e = validate_bwd(qkv, dout, lse, dqkv, delta, dvres, nullptr, false, s, scale);
  if (e != PSA_OK) return e;
  if (simt_bwd(s)) {
    // delta from the dQ kernel, in the workspace, then dK / dV
    const psa::SimtArgs a = simt_bwd_args(qkv, out, dout, lse, dvres, dqkv, delta, s, scale);
    const bool bf16 = s.dtype == PSA_DTYPE_BF16;
    e = from_cuda(psa::launch_simt_bwd_dq(a, true, bf16, s.key_dim, st));
    if (e != PSA_OK) return e;
    return from_cuda(psa::launch_simt_bwd_dkdv(a, true, bf16, s.key_dim, st));
  }
  if (e == PSA_OK)
    e = make_bwd(qkv, dout, lse, dqkv, delta, nullptr, out, s, scale, &mqk, &mv, &mdo, &mo, &a_dq);
  if (e == PSA_OK)
    e = make_bwd(qkv, dout, lse, dqkv, delta, dvres, nullptr, s, scale, &mqk2, &mv2, &mdo2, nullptr,
                 &a_kv);
  if (e != PSA_OK) return e;
  const int BH = s.B * s.num_heads;
  const size_t long_ws = long_fused_ws_bytes(s);
  if (s.key_dim == 32 &&
      (s.H * s.W <= psa::kFusedBwdMaxN || (long_ws > 0 && ws_bytes >= long_ws))) {
    // one kernel per head produces delta, dQ, dK and dV from a single walk over
    // its tiles (the workspace holds the dQ accumulator beyond kFusedBwdMaxN
    // positions and is not used below)
    a_dq.dvres = static_cast<const __nv_bfloat16*>(dvres);
    return from_cuda(psa::launch_psa_bwd_fused(mqk, mv, mdo, a_dq, s.key_dim, st));
  }
  e = from_cuda(psa::launch_psa_bwd_dq(mqk, mv, mdo, mo, a_dq, BH, s.key_dim, st));
  if (e != PSA_OK) return e;
  return from_cuda(psa::launch_psa_bwd_dkdv(mqk2, mv2, mdo2, a_kv, BH, s.key_dim, st));
}

}  // extern "C"
