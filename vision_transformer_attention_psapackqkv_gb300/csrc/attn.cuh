// attn.cuh -- launch interfaces of the attention kernels (forward and backward).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace psa {

struct FwdArgs {
  int N;             // sequence length (queries = keys)
  int BH;            // heads x batch
  int nh;            // heads per batch (NCHW layout)
  int qkv_ch;        // channels per batch of the QKV tensor (NCHW layout)
  int out_ch;        // channels per batch of the output (NCHW layout)
  int vres_ch;       // channels per batch of the extracted V (NCHW layout)
  float scale_log2;  // scale * log2(e), > 0
  __nv_bfloat16* out;   // may be null when out_res is not
  float* lse;        // [BH, N] natural-log LSE, may be null
  __nv_bfloat16* vres;  // NCHW: PsaExtractV output [B, vres_ch, N], may be null
  // NCHW residual path: out_res = Out + V (V read from qkv at the query
  // positions), written when not null
  __nv_bfloat16* out_res;
  const __nv_bfloat16* qkv;
};

// bf16 tcgen05 forward, persistent grid.  Raw: 3-D maps over [BH, N, d] (box {d, 128, 1}).
cudaError_t launch_fa2_fwd_bf16(const CUtensorMap& mQ, const CUtensorMap& mK,
                                const CUtensorMap& mV, const FwdArgs& a, int d,
                                cudaStream_t st);
// NCHW: 2-D maps over [B*qkv_ch, N] with boxes {64, KD} (Q, K) and {64, 2*KD} (V);
// mOut over [B*out_ch, N] with box {128, 2*KD}, no swizzle (TMA store of a.out);
// mVres over [B*vres_ch, N] like mV (TMA store of a.vres).  A map whose pointer
// is null is never used.
cudaError_t launch_psa_fwd_bf16(const CUtensorMap& mQK, const CUtensorMap& mV,
                                const CUtensorMap& mOut, const CUtensorMap& mVres,
                                const FwdArgs& a, int KD, cudaStream_t st);

// CUDA-core path (attn_simt.cu): fp32 or bf16 storage, any N, fp32 arithmetic.
// Raw layout: q, k, v, o, dO, dq, dk, dv are [BH, N, d] planes.  NCHW layout: q, k,
// v point at the QKV tensor, dq, dk, dv at dQKV, o / dO / dvres / out / out_res
// at [B, nh*2*KD, N] tensors.  Null outputs are skipped (out, out_res, lse).
struct SimtArgs {
  const void *q, *k, *v, *o, *dO, *dvres;
  void *out, *out_res, *dq, *dk, *dv;
  float* lse;    // forward: written (nullable); backward: read
  float* delta;  // [BH, N]: written by the dQ kernel, read by the dK/dV kernel
  int N, BH, nh, qkv_ch, out_ch;
  float scale;
};
cudaError_t launch_simt_fwd(const SimtArgs& a, bool nchw, bool bf16, int dqk, cudaStream_t st);
cudaError_t launch_simt_bwd_dq(const SimtArgs& a, bool nchw, bool bf16, int dqk, cudaStream_t st);
cudaError_t launch_simt_bwd_dkdv(const SimtArgs& a, bool nchw, bool bf16, int dqk,
                                 cudaStream_t st);

// Launches kern with programmatic stream serialization: its CTAs may become
// resident and run their prologue (barrier set-up, tensor memory allocation)
// while the previous kernel of the stream finishes; the kernels call pdl_wait()
// before their first global memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Multiprocessor count of the current device, queried once per device (devices of
// one process may differ, e.g. a partitioned GPU next to a whole one).
int device_sm_count();

// Raises the dynamic shared memory limit of kernel `kern` to `bytes` on the
// current device (a per-device attribute), once per kernel and device.
cudaError_t set_max_dynamic_smem(const void* kern, int bytes);

struct BwdArgs {
  int N;
  int BH;
  int nh;
  int qkv_ch;        // NCHW: channels per batch of QKV / dQKV
  int out_ch;        // NCHW: channels per batch of Out / dOut / dVres
  float scale;       // softmax scale (natural units)
  float scale_log2;  // scale * log2(e)
  const float* lse;  // [BH, N] natural-log LSE from the forward
  float* delta;      // [BH, N] rowsum(dO o O)
  const __nv_bfloat16* o;     // raw: [BH, N, dv]; NCHW: out [B, out_ch, N]
  const __nv_bfloat16* dO;    // raw: [BH, N, dv]; NCHW: dout [B, out_ch, N]
  const __nv_bfloat16* dvres; // NCHW: optional gradient of the extracted V
  __nv_bfloat16* dq;          // raw: [BH, N, dqk]; NCHW: dqkv [B, qkv_ch, N]
  __nv_bfloat16* dk;          // raw: [BH, N, dqk]; NCHW: dqkv
  __nv_bfloat16* dv;          // raw: [BH, N, dv];  NCHW: dqkv
};

// Raw layout maps: mQ/mK box {d, 128, 1}; mV/mDO box {d, 128, 1}.
cudaError_t launch_fa2_bwd_dq(const CUtensorMap& mQ, const CUtensorMap& mK,
                              const CUtensorMap& mV, const CUtensorMap& mDO,
                              const BwdArgs& a, int BH, int d, cudaStream_t st);
cudaError_t launch_fa2_bwd_dkdv(const CUtensorMap& mQ, const CUtensorMap& mK,
                                const CUtensorMap& mV, const CUtensorMap& mDO,
                                const BwdArgs& a, int BH, int d, cudaStream_t st);
// NCHW maps: mQK box {64, KD} and mV box {64, 2KD} over QKV; mDO box {64, 2KD} over dOut,
// mO the same box over Out.
cudaError_t launch_psa_bwd_dq(const CUtensorMap& mQK, const CUtensorMap& mV,
                              const CUtensorMap& mDO, const CUtensorMap& mO, const BwdArgs& a,
                              int BH, int KD, cudaStream_t st);
cudaError_t launch_psa_bwd_dkdv(const CUtensorMap& mQK, const CUtensorMap& mV,
                                const CUtensorMap& mDO, const BwdArgs& a, int BH, int KD,
                                cudaStream_t st);

// Backward of a whole head per CTA (NCHW, KD = 32, N <= kFusedBwdMaxNLong,
// N % 8 == 0): one kernel computes delta (from a.o and a.dO, on chip), dQ, dK and
// dV.  Up to kFusedBwdMaxN positions a.delta is not used; beyond, a.delta points
// at an fp32 workspace of BH * N * 32 floats that accumulates dQ.  Same maps as
// launch_psa_bwd_dkdv.
constexpr int kFusedBwdMaxN = 512;
constexpr int kFusedBwdMaxNLong = 2048;
cudaError_t launch_psa_bwd_fused(const CUtensorMap& mQK, const CUtensorMap& mV,
                                 const CUtensorMap& mDO, const BwdArgs& a, int KD,
                                 cudaStream_t st);

// QKV 1x1 convolution (qkv_conv.cu): out [B, cout, N] = w [cout, cin] . x [B, cin, N]
// + bias [cout] (nullable, fp32), bf16 storage, fp32 accumulation.
struct ConvArgs {
  int B, cin, cout, N;
  const float* bias;
  __nv_bfloat16* out;
};
// Tensor cores: mW 2-D over w (box {64, 128}), mX 3-D over x (box {64, 64, 1}),
// mOut 3-D over out (box {64, 128, 1}), all with the 128-byte swizzle; needs
// cin % 8 == 0 and N % 8 == 0.
cudaError_t launch_qkv_conv_tc(const CUtensorMap& mW, const CUtensorMap& mX,
                               const CUtensorMap& mOut, const ConvArgs& a, cudaStream_t st);
// CUDA cores, any shape.
cudaError_t launch_qkv_conv_simt(const void* x, const void* w, const ConvArgs& a, cudaStream_t st);

}  // namespace psa
