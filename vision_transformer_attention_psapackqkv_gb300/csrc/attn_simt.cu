// attn_simt.cu -- Flash Attention 2 on CUDA cores (vision-rs book, page "Custom
// Kernels", section "Flash Attention 2": online softmax, forward, dQ backward and
// dK/dV backward as separate kernels), for what the tensor-core kernels do not
// take: fp32 storage (whose 1e-4 bound rules out bf16 or tf32 operands) and NCHW
// maps whose channel rows are not 16-byte multiples (N * 2 % 16 != 0, e.g. 7 x 7
// or 13 x 13), which a TMA tensor map cannot address.  Storage is fp32 or bf16,
// arithmetic is fp32 throughout, outputs are rounded once; plain global loads
// reach any alignment.
//
// Layouts as in the tensor-core kernels: kNCHW = false reads [BH, N, d] planes,
// kNCHW = true reads the QKV conv output [B, nh*4*KD, N] directly (per head
// [Q | K | V_lo | V_hi]; both V halves together as DV = 2 KD channels, one
// softmax), writes Out [B, nh*2*KD, N] and dQKV in the QKV layout.
//
//   forward: one thread per query row; 32-key tiles of K and V in shared memory;
//            O = sum_j p_j V_j / sum_j p_j with a running maximum; Out + V for the
//            residual path when requested.
//   dQ:      one thread per query row: delta = dO . O (written for the dK/dV
//            kernel), then over 32-key tiles P = exp(scale q.k - lse),
//            dS = P (dO . v - delta), dQ += dS k; dQ = scale dQ.
//   dK/dV:   one thread per key row, over 32-query tiles of Q, dO, lse, delta:
//            dV += P dO,  dK += dS q;  dK = scale dK, dV (+ dVres).
#include <cuda_bf16.h>
#include <math.h>

#include "attn.cuh"

namespace psa {

namespace {

__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// Element addressing of one head's operands.
template <int DQK, int DV, bool kNCHW>
struct HeadIdx {
  int bh, b, hd, N, qkv_ch, out_ch;
  __device__ HeadIdx(int bh_, const SimtArgs& a)
      : bh(bh_), b(bh_ / a.nh), hd(bh_ % a.nh), N(a.N), qkv_ch(a.qkv_ch), out_ch(a.out_ch) {}
  // plane 0 = Q / dQ (DQK wide), 1 = K / dK (DQK), 2 = V / dV (DV, both halves)
  __device__ long long qkv(int plane, int n, int d) const {
    if (kNCHW) return ((long long)b * qkv_ch + hd * 4 * DQK + plane * DQK + d) * N + n;
    const int width = plane == 2 ? DV : DQK;
    return ((long long)bh * N + n) * width + d;
  }
  // Out / dOut / dVres, DV wide
  __device__ long long out(int n, int c) const {
    if (kNCHW) return ((long long)b * out_ch + hd * DV + c) * N + n;
    return ((long long)bh * N + n) * DV + c;
  }
};

template <typename T, int DQK, int DV, bool kNCHW>
__global__ void __launch_bounds__(128) attn_fwd_simt_kernel(const SimtArgs a) {
  constexpr int TK = 32;
  __shared__ float sk[TK][DQK];
  __shared__ float sv[TK][DV];
  const HeadIdx<DQK, DV, kNCHW> ix(blockIdx.y, a);
  const int N = a.N, i = blockIdx.x * 128 + threadIdx.x;
  const T *Q = static_cast<const T*>(a.q), *K = static_cast<const T*>(a.k),
          *V = static_cast<const T*>(a.v);
  float qr[DQK];
#pragma unroll
  for (int d = 0; d < DQK; ++d) qr[d] = (i < N) ? ldf(Q + ix.qkv(0, i, d)) : 0.f;
  float acc[DV];
#pragma unroll
  for (int c = 0; c < DV; ++c) acc[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int kv0 = 0; kv0 < N; kv0 += TK) {
    __syncthreads();
    for (int e = threadIdx.x; e < TK * DQK; e += 128) {
      const int jj = e / DQK, d = e % DQK;
      sk[jj][d] = (kv0 + jj < N) ? ldf(K + ix.qkv(1, kv0 + jj, d)) : 0.f;
    }
    for (int e = threadIdx.x; e < TK * DV; e += 128) {
      const int jj = e / DV, c = e % DV;
      sv[jj][c] = (kv0 + jj < N) ? ldf(V + ix.qkv(2, kv0 + jj, c)) : 0.f;
    }
    __syncthreads();
    const int nv = min(TK, N - kv0);
    float s[TK];
    float mx = m;
#pragma unroll
    for (int jj = 0; jj < TK; ++jj) {
      float dot = 0.f;
#pragma unroll
      for (int d = 0; d < DQK; ++d) dot = fmaf(qr[d], sk[jj][d], dot);
      s[jj] = (jj < nv) ? dot * a.scale : -INFINITY;
      mx = fmaxf(mx, s[jj]);
    }
    const float corr = expf(m - mx);  // m = -inf on the first tile gives 0
    l *= corr;
#pragma unroll
    for (int c = 0; c < DV; ++c) acc[c] *= corr;
    m = mx;
#pragma unroll
    for (int jj = 0; jj < TK; ++jj) {
      const float p = expf(s[jj] - m);
      l += p;
#pragma unroll
      for (int c = 0; c < DV; ++c) acc[c] = fmaf(p, sv[jj][c], acc[c]);
    }
  }
  if (i >= N) return;
  const float inv_l = 1.f / l;
  T* out = static_cast<T*>(a.out);
  T* out_res = static_cast<T*>(a.out_res);
  for (int c = 0; c < DV; ++c) {
    const long long o = ix.out(i, c);
    if (out) stf(out + o, acc[c] * inv_l);
    if (out_res) stf(out_res + o, acc[c] * inv_l + ldf(V + ix.qkv(2, i, c)));  // Out + V
  }
  if (a.lse) a.lse[(long long)ix.bh * N + i] = m + logf(l);
}

template <typename T, int DQK, int DV, bool kNCHW>
__global__ void __launch_bounds__(128) attn_bwd_dq_simt_kernel(const SimtArgs a) {
  constexpr int TK = 32;
  __shared__ float sk[TK][DQK];
  __shared__ float sv[TK][DV];
  const HeadIdx<DQK, DV, kNCHW> ix(blockIdx.y, a);
  const int N = a.N, i = blockIdx.x * 128 + threadIdx.x;
  const bool live = i < N;
  const T *Q = static_cast<const T*>(a.q), *K = static_cast<const T*>(a.k),
          *V = static_cast<const T*>(a.v), *O = static_cast<const T*>(a.o),
          *G = static_cast<const T*>(a.dO);
  float qr[DQK], g[DV];
  float D = 0.f;
#pragma unroll
  for (int d = 0; d < DQK; ++d) qr[d] = live ? ldf(Q + ix.qkv(0, i, d)) : 0.f;
#pragma unroll
  for (int c = 0; c < DV; ++c) {
    g[c] = live ? ldf(G + ix.out(i, c)) : 0.f;
    if (live) D = fmaf(g[c], ldf(O + ix.out(i, c)), D);
  }
  const long long row = (long long)ix.bh * N + i;
  if (live) a.delta[row] = D;
  const float lse = live ? a.lse[row] : 0.f;
  float dq[DQK];
#pragma unroll
  for (int d = 0; d < DQK; ++d) dq[d] = 0.f;
  for (int kv0 = 0; kv0 < N; kv0 += TK) {
    __syncthreads();
    for (int e = threadIdx.x; e < TK * DQK; e += 128) {
      const int jj = e / DQK, d = e % DQK;
      sk[jj][d] = (kv0 + jj < N) ? ldf(K + ix.qkv(1, kv0 + jj, d)) : 0.f;
    }
    for (int e = threadIdx.x; e < TK * DV; e += 128) {
      const int jj = e / DV, c = e % DV;
      sv[jj][c] = (kv0 + jj < N) ? ldf(V + ix.qkv(2, kv0 + jj, c)) : 0.f;
    }
    __syncthreads();
    const int nv = min(TK, N - kv0);
    for (int jj = 0; jj < nv; ++jj) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int d = 0; d < DQK; ++d) s = fmaf(qr[d], sk[jj][d], s);
#pragma unroll
      for (int c = 0; c < DV; ++c) dp = fmaf(g[c], sv[jj][c], dp);
      const float p = expf(s * a.scale - lse);
      const float ds = p * (dp - D);
#pragma unroll
      for (int d = 0; d < DQK; ++d) dq[d] = fmaf(ds, sk[jj][d], dq[d]);
    }
  }
  if (!live) return;
  T* dQ = static_cast<T*>(a.dq);
#pragma unroll
  for (int d = 0; d < DQK; ++d) stf(dQ + ix.qkv(0, i, d), dq[d] * a.scale);
}

template <typename T, int DQK, int DV, bool kNCHW>
__global__ void __launch_bounds__(128) attn_bwd_dkdv_simt_kernel(const SimtArgs a) {
  constexpr int TQ = 32;
  __shared__ float sq[TQ][DQK];
  __shared__ float sg[TQ][DV];
  __shared__ float sl[TQ], sd[TQ];
  const HeadIdx<DQK, DV, kNCHW> ix(blockIdx.y, a);
  const int N = a.N, j = blockIdx.x * 128 + threadIdx.x;
  const bool live = j < N;
  const T *Q = static_cast<const T*>(a.q), *K = static_cast<const T*>(a.k),
          *V = static_cast<const T*>(a.v), *G = static_cast<const T*>(a.dO);
  float kr[DQK], vr[DV], dk[DQK], dv[DV];
#pragma unroll
  for (int d = 0; d < DQK; ++d) {
    kr[d] = live ? ldf(K + ix.qkv(1, j, d)) : 0.f;
    dk[d] = 0.f;
  }
#pragma unroll
  for (int c = 0; c < DV; ++c) {
    vr[c] = live ? ldf(V + ix.qkv(2, j, c)) : 0.f;
    dv[c] = 0.f;
  }
  for (int q0 = 0; q0 < N; q0 += TQ) {
    __syncthreads();
    for (int e = threadIdx.x; e < TQ * DQK; e += 128) {
      const int ii = e / DQK, d = e % DQK;
      sq[ii][d] = (q0 + ii < N) ? ldf(Q + ix.qkv(0, q0 + ii, d)) : 0.f;
    }
    for (int e = threadIdx.x; e < TQ * DV; e += 128) {
      const int ii = e / DV, c = e % DV;
      sg[ii][c] = (q0 + ii < N) ? ldf(G + ix.out(q0 + ii, c)) : 0.f;
    }
    for (int ii = threadIdx.x; ii < TQ; ii += 128) {
      const long long row = (long long)ix.bh * N + q0 + ii;
      sl[ii] = (q0 + ii < N) ? a.lse[row] : 0.f;
      sd[ii] = (q0 + ii < N) ? a.delta[row] : 0.f;
    }
    __syncthreads();
    const int nq = min(TQ, N - q0);
    for (int ii = 0; ii < nq; ++ii) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int d = 0; d < DQK; ++d) s = fmaf(sq[ii][d], kr[d], s);
#pragma unroll
      for (int c = 0; c < DV; ++c) dp = fmaf(sg[ii][c], vr[c], dp);
      const float p = expf(s * a.scale - sl[ii]);
      const float ds = p * (dp - sd[ii]);
#pragma unroll
      for (int c = 0; c < DV; ++c) dv[c] = fmaf(p, sg[ii][c], dv[c]);
#pragma unroll
      for (int d = 0; d < DQK; ++d) dk[d] = fmaf(ds, sq[ii][d], dk[d]);
    }
  }
  if (!live) return;
  T* dK = static_cast<T*>(a.dk);
  T* dV = static_cast<T*>(a.dv);
  const T* R = static_cast<const T*>(a.dvres);
#pragma unroll
  for (int d = 0; d < DQK; ++d) stf(dK + ix.qkv(1, j, d), dk[d] * a.scale);
#pragma unroll
  for (int c = 0; c < DV; ++c) {
    float x = dv[c];
    if (R) x += ldf(R + ix.out(j, c));
    stf(dV + ix.qkv(2, j, c), x);
  }
}

enum class Kind { kFwd, kDq, kDkdv };

template <typename T, int DQK, int DV, bool kNCHW>
cudaError_t run(Kind kind, const SimtArgs& a, cudaStream_t st) {
  const dim3 grid((a.N + 127) / 128, a.BH);
  if (kind == Kind::kFwd)
    attn_fwd_simt_kernel<T, DQK, DV, kNCHW><<<grid, 128, 0, st>>>(a);
  else if (kind == Kind::kDq)
    attn_bwd_dq_simt_kernel<T, DQK, DV, kNCHW><<<grid, 128, 0, st>>>(a);
  else
    attn_bwd_dkdv_simt_kernel<T, DQK, DV, kNCHW><<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(Kind kind, const SimtArgs& a, bool nchw, int dqk, cudaStream_t st) {
  if (nchw) {
    if (dqk == 32) return run<T, 32, 64, true>(kind, a, st);
    return run<T, 64, 128, true>(kind, a, st);
  }
  if (dqk == 32) return run<T, 32, 32, false>(kind, a, st);
  return run<T, 64, 64, false>(kind, a, st);
}

cudaError_t launch(Kind kind, const SimtArgs& a, bool nchw, bool bf16, int dqk, cudaStream_t st) {
  if ((dqk != 32 && dqk != 64) || a.N <= 0 || a.BH <= 0 || a.BH > 65535)
    return cudaErrorInvalidValue;
  return bf16 ? dispatch<__nv_bfloat16>(kind, a, nchw, dqk, st)
              : dispatch<float>(kind, a, nchw, dqk, st);
}

}  // namespace

cudaError_t launch_simt_fwd(const SimtArgs& a, bool nchw, bool bf16, int dqk, cudaStream_t st) {
  return launch(Kind::kFwd, a, nchw, bf16, dqk, st);
}
cudaError_t launch_simt_bwd_dq(const SimtArgs& a, bool nchw, bool bf16, int dqk, cudaStream_t st) {
  return launch(Kind::kDq, a, nchw, bf16, dqk, st);
}
cudaError_t launch_simt_bwd_dkdv(const SimtArgs& a, bool nchw, bool bf16, int dqk,
                                 cudaStream_t st) {
  return launch(Kind::kDkdv, a, nchw, bf16, dqk, st);
}

}  // namespace psa
