// attn_fwd.cu -- Flash Attention 2 forward (vision-rs book, page "Custom Kernels",
// section "Flash Attention 2"): O = softmax(scale * Q K^T) V with an online
// softmax over key tiles; the N x N score matrix only ever exists one 128 x 128
// tile at a time, in tensor memory.
//
// bf16 path (tcgen05, sm_103a).  One CTA owns 128 query rows of one head and
// walks the key tiles:
//   warp 4   TMA producer: Q once, then K/V tiles into a 2-stage ring.
//   warp 5   MMA issuer (one thread) and TMEM owner:
//              S_j = Q K_j^T          -> TMEM (two 128-column buffers, so S_{j+1}
//                                        is computed while S_j is in the softmax)
//              O  += P_j V_j          -> TMEM (DV columns), P_j from shared memory
//   warps 0-3 softmax, one thread per query row (= TMEM lane): read the S row,
//            running max in the log2 domain, p = 2^(s - m) rounded to bf16 into
//            P_j (K-major, 128-byte swizzle), running sum; O is rescaled in TMEM
//            only when a row max grows by more than 2^8 (the result is exact
//            either way because O and the sum share the stale max); epilogue
//            O / l and LSE.
// Layouts: kNCHW = false reads [BH, N, D] planes through 3-D tensor maps (Q, K
// K-major; V MN-major for the P.V product); kNCHW = true reads the QKV conv
// output [B, nh*4*KD, N] directly (Q, K MN-major; V K-major), which fuses
// PsaPackQkv, the two V-half runs (one softmax, DV = 2*KD) and PsaMergeAttn.
//
// fp32 path (CUDA cores): the same online softmax with one thread per query
// row and fp32 arithmetic throughout (a 1e-4 bound rules out tf32 inputs).
#include <math.h>

#include "attn.cuh"
#include "ptx.cuh"

namespace psa {

namespace {

template <int DQK, int DV, bool kNCHW>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128, STAGES = 2;
  static constexpr int kThreads = 192;
  static constexpr uint32_t Q_BYTES = BM * DQK * 2;
  static constexpr uint32_t K_BYTES = BN * DQK * 2;
  static constexpr uint32_t V_BYTES = BN * DV * 2;
  static constexpr uint32_t P_BYTES = BM * BN * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * K_BYTES;
  static constexpr uint32_t OFF_P = OFF_V + STAGES * V_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t TM_S = 0, TM_O = 2 * BN;
  static constexpr uint32_t QK_R = kNCHW ? 128 : 2 * DQK;
  static constexpr uint32_t Q_ROWS = kNCHW ? DQK : BM;
  static constexpr uint32_t K_ROWS = kNCHW ? DQK : BN;
  static constexpr uint32_t V_R = kNCHW ? 128 : 2 * DV;
  static constexpr uint32_t V_ROWS = kNCHW ? DV : BN;
  static_assert(DQK % 16 == 0 && DV % 32 == 0 && DV <= 128, "tile shape");
  static_assert(TM_O + DV <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Drains (with a time limit only) a barrier phase that a TMA copy will complete.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
}

template <int DQK, int DV, bool kNCHW>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQK,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using C = FwdCfg<DQK, DV, kNCHW>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V,
                 sP = sbase + C::OFF_P;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;    // [2]
  uint64_t* pv_done = bars + 9;   // [2]
  uint64_t* mma_done = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int q0 = blockIdx.x * C::BM;
  const int N = args.N;
  const int nkv = (N + C::BN - 1) / C::BN;
  // NCHW: channel row of this head's Q block in the 2-D [B*qkv_ch, N] view.
  const int ch0 = kNCHW ? (bh / args.nh) * args.qkv_ch + (bh % args.nh) * 4 * DQK : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(kv_full + i, 1);
      mbar_init(kv_empty + i, 1);
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
      mbar_init(pv_done + i, 1);
    }
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      if (kNCHW) {
        for (int b = 0; b < C::BM / 64; ++b)
          tma_load_2d(smem + C::OFF_Q + b * (DQK * 128), &tmQK, q_full, q0 + 64 * b, ch0);
      } else {
        tma_load_3d(smem + C::OFF_Q, &tmQK, q_full, 0, q0, bh);
      }
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % C::STAGES;
        if (j >= C::STAGES && !mbar_wait(&kv_empty[st], ((j / C::STAGES) - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&kv_full[st], C::K_BYTES + C::V_BYTES);
        unsigned char* dK = smem + C::OFF_K + st * C::K_BYTES;
        unsigned char* dV = smem + C::OFF_V + st * C::V_BYTES;
        const int kv0 = j * C::BN;
        if (kNCHW) {
          for (int b = 0; b < C::BN / 64; ++b) {
            tma_load_2d(dK + b * (DQK * 128), &tmK, &kv_full[st], kv0 + 64 * b, ch0 + DQK);
            tma_load_2d(dV + b * (DV * 128), &tmV, &kv_full[st], kv0 + 64 * b, ch0 + 2 * DQK);
          }
        } else {
          tma_load_3d(dK, &tmK, &kv_full[st], 0, kv0, bh);
          tma_load_3d(dV, &tmV, &kv_full[st], 0, kv0, bh);
        }
        issued = j + 1;
      }
      if (*abort) {  // let copies still in flight land before the CTA exits
        drain_wait(q_full, 0);
        for (int j = (issued > C::STAGES ? issued - C::STAGES : 0); j < issued; ++j)
          drain_wait(&kv_full[j % C::STAGES], (j / C::STAGES) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const SmemTile tQ{sQ, C::QK_R, C::Q_ROWS};
      const uint32_t idPV = idesc_bf16_f32(128, DV, false, !kNCHW);
      auto issue_pv = [&](int i) -> bool {
        if (!mbar_wait(&p_full[i & 1], (i >> 1) & 1, abort)) return false;
        tc_fence_after();
        const SmemTile tP{sP + (i & 1) * C::P_BYTES, 128, C::BM};
        const SmemTile tV{sV + (i % C::STAGES) * C::V_BYTES, C::V_R, C::V_ROWS};
        const int valid = min(C::BN, N - i * C::BN);
        const int kend = (valid + 15) & ~15;
        for (int k = 0; k < kend; k += 16) {
          const uint64_t a = desc_kmajor(tP, k);
          const uint64_t b = kNCHW ? desc_kmajor(tV, k) : desc_mnmajor(tV, k);
          mma_bf16(tmem + C::TM_O, a, b, idPV, (i > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(&pv_done[i & 1]);
        mma_commit(&kv_empty[i % C::STAGES]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, abort);
      for (int j = 0; ok && j < nkv; ++j) {
        const int st = j % C::STAGES;
        if (!mbar_wait(&kv_full[st], (j / C::STAGES) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const SmemTile tK{sK + st * C::K_BYTES, C::QK_R, C::K_ROWS};
        const int valid = min(C::BN, N - j * C::BN);
        const int nS = (valid + 15) & ~15;
        const uint32_t idS = idesc_bf16_f32(128, nS, kNCHW, kNCHW);
        const uint32_t dS = tmem + C::TM_S + (j & 1) * C::BN;
#pragma unroll
        for (int k = 0; k < DQK; k += 16) {
          const uint64_t a = kNCHW ? desc_mnmajor(tQ, k) : desc_kmajor(tQ, k);
          const uint64_t b = kNCHW ? desc_mnmajor(tK, k) : desc_kmajor(tK, k);
          mma_bf16(dS, a, b, idS, k > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[j & 1]);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(nkv - 1);
      mma_commit(mma_done);
      drain_wait(mma_done, 0);  // every MMA retired before TMEM is released
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int r = threadIdx.x;  // query row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = args.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[C::BN];
#pragma unroll
      for (int c = 0; c < C::BN; c += 32)
        tmem_load32(tmem + lane_base + C::TM_S + sb * C::BN + c,
                    *reinterpret_cast<float(*)[32]>(s + c));
      const int valid = min(C::BN, N - j * C::BN);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < C::BN; ++c) {
        s[c] = (c < valid) ? s[c] * sl2 : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      bool need = false;
      if (j == 0)
        m_run = mx;
      else
        need = mx > m_run + 8.f;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? fast_exp2(m_run - mx) : 1.f;
        if (need) m_run = mx;
        l_run *= alpha;
        if (!mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DV; c += 32) {
          float o[32];
          tmem_load32(tmem + lane_base + C::TM_O + c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_store32(tmem + lane_base + C::TM_O + c, o);
        }
      }
      if (j >= 2 && !mbar_wait(&pv_done[sb], ((j - 2) >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      const uint32_t prow = sP + sb * C::P_BYTES;
      float ls = 0.f;
#pragma unroll
      for (int ch = 0; ch < C::BN / 8; ++ch) {
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          p[e] = fast_exp2(s[ch * 8 + e] - m_run);
          ls += p[e];
        }
        st_shared_v4(prow + (ch >> 3) * (C::BM * 128) + swizzled_offset(r, ch & 7, 128),
                     pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
                     pack_bf16x2(p[6], p[7]));
      }
      l_run += ls;
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    // epilogue: O / l in the output layout, LSE in natural-log units
    if (ok && mbar_wait(&pv_done[(nkv - 1) & 1], ((nkv - 1) >> 1) & 1, abort)) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const int q = q0 + r;
      const bool live = q < N;
#pragma unroll
      for (int c = 0; c < DV; c += 32) {
        float o[32];
        tmem_load32(tmem + lane_base + C::TM_O + c, o);
        if (live) {
          if (kNCHW) {
            const int b = bh / args.nh, hd = bh % args.nh;
            __nv_bfloat16* dst =
                args.out + ((long long)b * args.out_ch + hd * DV + c) * N + q;
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[(long long)e * N] = __float2bfloat16_rn(o[e] * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(args.out + ((long long)bh * N + q) * DV + c);
#pragma unroll
            for (int e = 0; e < 32; e += 8)
              dst[e / 8] = make_uint4(pack_bf16x2(o[e] * inv_l, o[e + 1] * inv_l),
                                      pack_bf16x2(o[e + 2] * inv_l, o[e + 3] * inv_l),
                                      pack_bf16x2(o[e + 4] * inv_l, o[e + 5] * inv_l),
                                      pack_bf16x2(o[e + 6] * inv_l, o[e + 7] * inv_l));
          }
        }
      }
      if (live && args.lse) args.lse[(long long)bh * N + q] = (m_run + log2f(l_run)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ fp32 path
template <int DQK, int DV, bool kNCHW>
__global__ void __launch_bounds__(128)
    attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, float* __restrict__ out,
                        float* __restrict__ lse, int N, int nh, int qkv_ch, int out_ch,
                        float scale) {
  constexpr int TK = 32;
  __shared__ float sk[TK][DQK];
  __shared__ float sv[TK][DV];
  const int bh = blockIdx.y;
  const int i = blockIdx.x * 128 + threadIdx.x;
  const int b = bh / nh, hd = bh % nh;
  // element (row n, column d) of the Q / K / V operand of this head
  auto at = [&](const float* base, int plane, int n, int d, int width) -> float {
    if (kNCHW)
      return base[((long long)b * qkv_ch + hd * 4 * DQK + plane * DQK + d) * N + n];
    return base[((long long)bh * N + n) * width + d];
  };
  float qr[DQK];
#pragma unroll
  for (int d = 0; d < DQK; ++d) qr[d] = (i < N) ? at(q, 0, i, d, DQK) : 0.f;
  float acc[DV];
#pragma unroll
  for (int c = 0; c < DV; ++c) acc[c] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int kv0 = 0; kv0 < N; kv0 += TK) {
    __syncthreads();
    for (int e = threadIdx.x; e < TK * DQK; e += 128) {
      const int jj = e / DQK, d = e % DQK;
      sk[jj][d] = (kv0 + jj < N) ? at(k, 1, kv0 + jj, d, DQK) : 0.f;
    }
    for (int e = threadIdx.x; e < TK * DV; e += 128) {
      const int jj = e / DV, c = e % DV;
      sv[jj][c] = (kv0 + jj < N) ? at(v, 2, kv0 + jj, c, DV) : 0.f;
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
      s[jj] = (jj < nv) ? dot * scale : -INFINITY;
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
  for (int c = 0; c < DV; ++c) {
    if (kNCHW)
      out[((long long)b * out_ch + hd * DV + c) * N + i] = acc[c] * inv_l;
    else
      out[((long long)bh * N + i) * DV + c] = acc[c] * inv_l;
  }
  if (lse) lse[(long long)bh * N + i] = m + logf(l);
}

template <int DQK, int DV, bool kNCHW>
cudaError_t launch_tc(const CUtensorMap& mQK, const CUtensorMap& mK, const CUtensorMap& mV,
                      const FwdArgs& a, int BH, cudaStream_t st) {
  using C = FwdCfg<DQK, DV, kNCHW>;
  auto kern = attn_fwd_tc_kernel<DQK, DV, kNCHW>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (attr != cudaSuccess) return attr;
  dim3 grid((a.N + C::BM - 1) / C::BM, BH);
  kern<<<grid, C::kThreads, C::SMEM_BYTES, st>>>(mQK, mK, mV, a);
  return cudaGetLastError();
}

template <int DQK, int DV, bool kNCHW>
cudaError_t launch_f32(const float* q, const float* k, const float* v, float* out, float* lse,
                       int BH, int N, int nh, int qkv_ch, int out_ch, float scale,
                       cudaStream_t st) {
  dim3 grid((N + 127) / 128, BH);
  attn_fwd_f32_kernel<DQK, DV, kNCHW><<<grid, 128, 0, st>>>(q, k, v, out, lse, N, nh, qkv_ch,
                                                          out_ch, scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fa2_fwd_bf16(const CUtensorMap& mQ, const CUtensorMap& mK,
                                const CUtensorMap& mV, const FwdArgs& a, int BH, int d,
                                cudaStream_t st) {
  if (d == 32) return launch_tc<32, 32, false>(mQ, mK, mV, a, BH, st);
  return launch_tc<64, 64, false>(mQ, mK, mV, a, BH, st);
}

cudaError_t launch_psa_fwd_bf16(const CUtensorMap& mQK, const CUtensorMap& mV,
                                const FwdArgs& a, int BH, int KD, cudaStream_t st) {
  if (KD == 32) return launch_tc<32, 64, true>(mQK, mQK, mV, a, BH, st);
  return launch_tc<64, 128, true>(mQK, mQK, mV, a, BH, st);
}

cudaError_t launch_fa2_fwd_f32(const float* q, const float* k, const float* v, float* o,
                               float* lse, int BH, int N, int d, float scale, cudaStream_t st) {
  if (d == 32) return launch_f32<32, 32, false>(q, k, v, o, lse, BH, N, 1, 0, 0, scale, st);
  return launch_f32<64, 64, false>(q, k, v, o, lse, BH, N, 1, 0, 0, scale, st);
}

cudaError_t launch_psa_fwd_f32(const float* qkv, float* out, float* lse, int B, int nh, int KD,
                               int N, float scale, cudaStream_t st) {
  const int BH = B * nh;
  if (KD == 32)
    return launch_f32<32, 64, true>(qkv, qkv, qkv, out, lse, BH, N, nh, nh * 4 * KD,
                                    nh * 2 * KD, scale, st);
  return launch_f32<64, 128, true>(qkv, qkv, qkv, out, lse, BH, N, nh, nh * 4 * KD, nh * 2 * KD,
                                   scale, st);
}

}  // namespace psa
