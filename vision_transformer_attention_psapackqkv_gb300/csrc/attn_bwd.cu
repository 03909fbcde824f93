// attn_bwd.cu -- Flash Attention 2 backward (vision-rs book, page "Custom Kernels",
// section "Flash Attention 2": the dQ backward and the dK/dV backward are separate
// kernels with their own grids).  Both recompute the probabilities from the
// forward's log-sum-exp instead of storing P:
//   P = exp(scale q k^T - lse),  dP = dO V^T,  dS = P o (dP - delta),
//   delta_i = sum_c dO_ic O_ic  (= sum_j P_ij dP_ij),
//   dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// No atomics: every output element is produced by exactly one CTA, so results
// are bitwise reproducible.
//
// dQ kernel: one CTA per (128 query rows, head), walking 64-key tiles.
//   prologue (softmax warps): delta of its row from O and dO, written out for the
//     dK/dV kernel, which therefore runs after this one.
//   MMA:  S_j = Q K_j^T and dP_j = dO V_j^T into TMEM (double-buffered, 4 x 64
//         columns), then dQ += dS_j K_j (dS_j bf16 from shared memory).
//   softmax warps: one thread per query row, P and dS of 64 keys per tile.
// dK/dV kernel: one CTA per (128 key rows, head), walking 64-query tiles.
//   MMA:  S^T_i = K Q_i^T and dP^T_i = V dO_i^T into TMEM (double-buffered), then
//         dV += P^T_i dO_i and dK += dS^T_i Q_i (P^T, dS^T bf16 from shared memory).
//   softmax warps: one thread per key row; lse and delta of the 64 query columns
//         come from shared memory, written there by the producer warp.
// Layouts as in the forward: kNCHW = false uses [BH, N, d] planes, kNCHW = true
// reads QKV / Out / dOut in NCHW and writes dQKV in NCHW (the adjoints of
// PsaMergeAttn and PsaPackQkv are folded into the tile addressing; the optional
// PsaExtractV gradient is added into the V channels).
#include <math.h>

#include "attn.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace psa {

namespace {

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

// ====================================================================== dQ
template <int DQK, int DV, bool kNCHW>
struct DqCfg {
  static constexpr int BM = 128, BN = 64, STAGES = 2, kThreads = 192;
  static constexpr uint32_t Q_BYTES = BM * DQK * 2, DO_BYTES = BM * DV * 2;
  static constexpr uint32_t K_BYTES = BN * DQK * 2, V_BYTES = BN * DV * 2;
  static constexpr uint32_t DS_BYTES = BM * BN * 2;
  static constexpr uint32_t OFF_Q = 0, OFF_DO = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_K = OFF_DO + DO_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * K_BYTES;
  static constexpr uint32_t OFF_DS = OFF_V + STAGES * V_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_DS + 2 * DS_BYTES;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM: S[b] at 128 b, dP[b] at 128 b + 64, dQ at 256
  static constexpr uint32_t TM_DQ = 256;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(TM_DQ + DQK <= TMEM_COLS, "tensor memory");
};

template <int DQK, int DV, bool kNCHW>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO, const BwdArgs args) {
  using C = DqCfg<DQK, DV, kNCHW>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* ds_full = bars + 7;   // [2]
  uint64_t* ds_free = bars + 9;   // [2]
  uint64_t* mma_done = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, q0 = blockIdx.x * C::BM, N = args.N;
  const int nkv = (N + C::BN - 1) / C::BN;
  const int b = bh / args.nh, hd = bh % args.nh;
  const int ch0 = kNCHW ? b * args.qkv_ch + hd * 4 * DQK : 0;  // Q rows in the QKV view
  const int och0 = kNCHW ? b * args.out_ch + hd * DV : 0;      // rows in the Out view

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(kv_full + i, 1);
      mbar_init(kv_empty + i, 1);
      mbar_init(s_full + i, 1);
      mbar_init(ds_full + i, 128);
      mbar_init(ds_free + i, 1);
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
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, C::Q_BYTES + C::DO_BYTES);
      load_tile<kNCHW, DQK>(smem + C::OFF_Q, &tmQ, q_full, C::BM, q0, bh, ch0);
      load_tile<kNCHW, DV>(smem + C::OFF_DO, &tmDO, q_full, C::BM, q0, bh, och0);
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % C::STAGES;
        if (j >= C::STAGES && !mbar_wait(&kv_empty[st], ((j / C::STAGES) - 1) & 1, abort)) break;
        mbar_arrive_expect_tx(&kv_full[st], C::K_BYTES + C::V_BYTES);
        load_tile<kNCHW, DQK>(smem + C::OFF_K + st * C::K_BYTES, &tmK, &kv_full[st], C::BN,
                              j * C::BN, bh, ch0 + DQK);
        load_tile<kNCHW, DV>(smem + C::OFF_V + st * C::V_BYTES, &tmV, &kv_full[st], C::BN,
                             j * C::BN, bh, ch0 + 2 * DQK);
        issued = j + 1;
      }
      if (*abort) {
        drain_wait(q_full, 0);
        for (int j = (issued > C::STAGES ? issued - C::STAGES : 0); j < issued; ++j)
          drain_wait(&kv_full[j % C::STAGES], (j / C::STAGES) & 1);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const SmemTile tQ = tile_view<kNCHW, DQK>(sbase + C::OFF_Q, C::BM);
      const SmemTile tDO = tile_view<kNCHW, DV>(sbase + C::OFF_DO, C::BM);
      const uint32_t idSP = idesc_bf16_f32(128, C::BN, kNCHW, kNCHW);
      const uint32_t idDQ = idesc_bf16_f32(128, DQK, false, !kNCHW);
      auto issue_dq = [&](int i) -> bool {
        if (!mbar_wait(&ds_full[i & 1], (i >> 1) & 1, abort)) return false;
        tc_fence_after();
        const SmemTile tDS{sbase + C::OFF_DS + (i & 1) * C::DS_BYTES, 128, C::BM};
        const SmemTile tK = tile_view<kNCHW, DQK>(sbase + C::OFF_K + (i % C::STAGES) * C::K_BYTES, C::BN);
        const int valid = min(C::BN, N - i * C::BN);
        const int kend = (valid + 15) & ~15;
        for (int k = 0; k < kend; k += 16)
          mma_bf16(tmem + C::TM_DQ, desc_kmajor(tDS, k), desc_ch_by_pos<kNCHW>(tK, k), idDQ,
                   (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(&ds_free[i & 1]);
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
        const SmemTile tK = tile_view<kNCHW, DQK>(sbase + C::OFF_K + st * C::K_BYTES, C::BN);
        const SmemTile tV = tile_view<kNCHW, DV>(sbase + C::OFF_V + st * C::V_BYTES, C::BN);
        const uint32_t dS = tmem + (j & 1) * 128, dP = dS + 64;
#pragma unroll
        for (int k = 0; k < DQK; k += 16)
          mma_bf16(dS, desc_pos_by_ch<kNCHW>(tQ, k), desc_pos_by_ch<kNCHW>(tK, k), idSP,
                   k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < DV; k += 16)
          mma_bf16(dP, desc_pos_by_ch<kNCHW>(tDO, k), desc_pos_by_ch<kNCHW>(tV, k), idSP,
                   k > 0 ? 1u : 0u);
        mma_commit(&s_full[j & 1]);
        if (j >= 1 && !issue_dq(j - 1)) ok = false;
      }
      if (ok) issue_dq(nkv - 1);
      mma_commit(mma_done);
      drain_wait(mma_done, 0);
    }
  } else {
    const int r = threadIdx.x;
    const int q = q0 + r;
    const bool live = q < N;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    // delta of this row, and the row's lse in the log2 domain
    float D = 0.f, lse2 = 0.f;
    if (live) {
      if (kNCHW) {
        const __nv_bfloat16* o = args.o + (long long)och0 * N + q;
        const __nv_bfloat16* g = args.dO + (long long)och0 * N + q;
#pragma unroll 8
        for (int c = 0; c < DV; ++c) D = fmaf(bf(o[(long long)c * N]), bf(g[(long long)c * N]), D);
      } else {
        const uint4* o = reinterpret_cast<const uint4*>(args.o + ((long long)bh * N + q) * DV);
        const uint4* g = reinterpret_cast<const uint4*>(args.dO + ((long long)bh * N + q) * DV);
#pragma unroll
        for (int c = 0; c < DV / 8; ++c) {
          const uint4 ov = o[c], gv = g[c];
          const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
          const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 of = __bfloat1622float2(o2[e]), gf = __bfloat1622float2(g2[e]);
            D = fmaf(of.x, gf.x, D);
            D = fmaf(of.y, gf.y, D);
          }
        }
      }
      args.delta[(long long)bh * N + q] = D;
      lse2 = args.lse[(long long)bh * N + q] * 1.4426950408889634f;
    }
    const float sl2 = args.scale_log2;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      if (j >= 2 && !mbar_wait(&ds_free[sb], ((j - 2) >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int valid = min(C::BN, N - j * C::BN);
      const uint32_t drow = sbase + C::OFF_DS + sb * C::DS_BYTES;
#pragma unroll
      for (int c0 = 0; c0 < C::BN; c0 += 32) {
        float s[32], dp[32];
        tmem_load32(tmem + lane_base + sb * 128 + c0, s);
        tmem_load32(tmem + lane_base + sb * 128 + 64 + c0, dp);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          float g[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = ch * 8 + e;
            const float p = (c0 + c < valid) ? fast_exp2(fmaf(s[c], sl2, -lse2)) : 0.f;
            g[e] = p * (dp[c] - D);
          }
          st_shared_v4(drow + swizzled_offset(r, (c0 >> 3) + ch, 128), pack_bf16x2(g[0], g[1]),
                       pack_bf16x2(g[2], g[3]), pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ds_full[sb]);
    }
    if (ok && mbar_wait(mma_done, 0, abort)) {
      tc_fence_after();
      float acc[32];
#pragma unroll
      for (int c = 0; c < DQK; c += 32) {
        tmem_load32(tmem + lane_base + C::TM_DQ + c, acc);
        if (live) {
          if (kNCHW) {
            __nv_bfloat16* dst = args.dq + ((long long)ch0 + c) * N + q;
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[(long long)e * N] = __float2bfloat16_rn(acc[e] * args.scale);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(args.dq + ((long long)bh * N + q) * DQK + c);
            const float sc = args.scale;
#pragma unroll
            for (int e = 0; e < 32; e += 8)
              dst[e / 8] = make_uint4(pack_bf16x2(acc[e] * sc, acc[e + 1] * sc),
                                      pack_bf16x2(acc[e + 2] * sc, acc[e + 3] * sc),
                                      pack_bf16x2(acc[e + 4] * sc, acc[e + 5] * sc),
                                      pack_bf16x2(acc[e + 6] * sc, acc[e + 7] * sc));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ====================================================================== dK / dV
template <int DQK, int DV, bool kNCHW>
struct DkvCfg {
  static constexpr int BM = 128 /* keys */, BQ = 64 /* queries per tile */, STAGES = 2;
  static constexpr int kThreads = 192;
  static constexpr uint32_t K_BYTES = BM * DQK * 2, V_BYTES = BM * DV * 2;
  static constexpr uint32_t Q_BYTES = BQ * DQK * 2, DO_BYTES = BQ * DV * 2;
  static constexpr uint32_t STAT_BYTES = 1024;  // lse2[64] + delta[64], padded
  static constexpr uint32_t PT_BYTES = BM * BQ * 2;
  static constexpr uint32_t OFF_K = 0, OFF_V = OFF_K + K_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + V_BYTES;
  static constexpr uint32_t OFF_DO = OFF_Q + STAGES * Q_BYTES;
  static constexpr uint32_t OFF_STAT = OFF_DO + STAGES * DO_BYTES;
  static constexpr uint32_t OFF_PT = OFF_STAT + STAGES * STAT_BYTES;
  static constexpr uint32_t OFF_DST = OFF_PT + 2 * PT_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_DST + 2 * PT_BYTES;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  // TMEM: S^T[b] at 128 b, dP^T[b] at 128 b + 64, dV at 256, dK at 256 + DV
  static constexpr uint32_t TM_DV = 256, TM_DK = 256 + DV;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(TM_DK + DQK <= TMEM_COLS, "tensor memory");
};

template <int DQK, int DV, bool kNCHW>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmDO, const BwdArgs args) {
  using C = DkvCfg<DQK, DV, kNCHW>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;    // [2]
  uint64_t* q_empty = bars + 3;   // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;    // [2]
  uint64_t* pds_free = bars + 9;  // [2]
  uint64_t* mma_done = bars + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, k0 = blockIdx.x * C::BM, N = args.N;
  const int nq = (N + C::BQ - 1) / C::BQ;
  const int b = bh / args.nh, hd = bh % args.nh;
  const int ch0 = kNCHW ? b * args.qkv_ch + hd * 4 * DQK : 0;
  const int och0 = kNCHW ? b * args.out_ch + hd * DV : 0;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full + i, 1 + 32);
      mbar_init(q_empty + i, 1);
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
      mbar_init(pds_free + i, 1);
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
    // producer: K/V once; per query tile Q, dO by TMA and lse / delta by plain loads
    if (lane == 0) {
      mbar_arrive_expect_tx(kv_full, C::K_BYTES + C::V_BYTES);
      load_tile<kNCHW, DQK>(smem + C::OFF_K, &tmK, kv_full, C::BM, k0, bh, ch0 + DQK);
      load_tile<kNCHW, DV>(smem + C::OFF_V, &tmV, kv_full, C::BM, k0, bh, ch0 + 2 * DQK);
    }
    int issued = 0;
    for (int i = 0; i < nq; ++i) {
      const int st = i % C::STAGES;
      if (i >= C::STAGES && !mbar_wait(&q_empty[st], ((i / C::STAGES) - 1) & 1, abort)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&q_full[st], C::Q_BYTES + C::DO_BYTES);
        load_tile<kNCHW, DQK>(smem + C::OFF_Q + st * C::Q_BYTES, &tmQ, &q_full[st], C::BQ,
                              i * C::BQ, bh, ch0);
        load_tile<kNCHW, DV>(smem + C::OFF_DO + st * C::DO_BYTES, &tmDO, &q_full[st], C::BQ,
                             i * C::BQ, bh, och0);
      }
      float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT + st * C::STAT_BYTES);
#pragma unroll
      for (int e = lane; e < C::BQ; e += 32) {
        const int q = i * C::BQ + e;
        const bool in = q < N;
        stat[e] = in ? args.lse[(long long)bh * N + q] * 1.4426950408889634f : INFINITY;
        stat[C::BQ + e] = in ? args.delta[(long long)bh * N + q] : 0.f;
      }
      mbar_arrive(&q_full[st]);
      issued = i + 1;
    }
    if (lane == 0 && *abort) {
      drain_wait(kv_full, 0);
      for (int i = (issued > C::STAGES ? issued - C::STAGES : 0); i < issued; ++i)
        drain_wait(&q_full[i % C::STAGES], (i / C::STAGES) & 1);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      const SmemTile tK = tile_view<kNCHW, DQK>(sbase + C::OFF_K, C::BM);
      const SmemTile tV = tile_view<kNCHW, DV>(sbase + C::OFF_V, C::BM);
      const uint32_t idSP = idesc_bf16_f32(128, C::BQ, kNCHW, kNCHW);
      const uint32_t idDV = idesc_bf16_f32(128, DV, false, !kNCHW);
      const uint32_t idDK = idesc_bf16_f32(128, DQK, false, !kNCHW);
      auto issue_grad = [&](int i) -> bool {
        if (!mbar_wait(&p_full[i & 1], (i >> 1) & 1, abort)) return false;
        tc_fence_after();
        const int st = i % C::STAGES;
        const SmemTile tQ = tile_view<kNCHW, DQK>(sbase + C::OFF_Q + st * C::Q_BYTES, C::BQ);
        const SmemTile tDO = tile_view<kNCHW, DV>(sbase + C::OFF_DO + st * C::DO_BYTES, C::BQ);
        const SmemTile tPt{sbase + C::OFF_PT + (i & 1) * C::PT_BYTES, 128, C::BM};
        const SmemTile tDSt{sbase + C::OFF_DST + (i & 1) * C::PT_BYTES, 128, C::BM};
        const int valid = min(C::BQ, N - i * C::BQ);
        const int kend = (valid + 15) & ~15;
        for (int k = 0; k < kend; k += 16) {
          const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
          mma_bf16(tmem + C::TM_DV, desc_kmajor(tPt, k), desc_ch_by_pos<kNCHW>(tDO, k), idDV, acc);
          mma_bf16(tmem + C::TM_DK, desc_kmajor(tDSt, k), desc_ch_by_pos<kNCHW>(tQ, k), idDK, acc);
        }
        mma_commit(&pds_free[i & 1]);
        mma_commit(&q_empty[st]);
        return true;
      };
      bool ok = mbar_wait(kv_full, 0, abort);
      for (int i = 0; ok && i < nq; ++i) {
        const int st = i % C::STAGES;
        if (!mbar_wait(&q_full[st], (i / C::STAGES) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const SmemTile tQ = tile_view<kNCHW, DQK>(sbase + C::OFF_Q + st * C::Q_BYTES, C::BQ);
        const SmemTile tDO = tile_view<kNCHW, DV>(sbase + C::OFF_DO + st * C::DO_BYTES, C::BQ);
        const uint32_t dS = tmem + (i & 1) * 128, dP = dS + 64;
#pragma unroll
        for (int k = 0; k < DQK; k += 16)
          mma_bf16(dS, desc_pos_by_ch<kNCHW>(tK, k), desc_pos_by_ch<kNCHW>(tQ, k), idSP,
                   k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < DV; k += 16)
          mma_bf16(dP, desc_pos_by_ch<kNCHW>(tV, k), desc_pos_by_ch<kNCHW>(tDO, k), idSP,
                   k > 0 ? 1u : 0u);
        mma_commit(&s_full[i & 1]);
        if (i >= 1 && !issue_grad(i - 1)) ok = false;
      }
      if (ok) issue_grad(nq - 1);
      mma_commit(mma_done);
      drain_wait(mma_done, 0);
    }
  } else {
    const int r = threadIdx.x;  // key row = TMEM lane
    const int key = k0 + r;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = args.scale_log2;
    bool ok = true;
    for (int i = 0; i < nq; ++i) {
      const int sb = i & 1, st = i % C::STAGES;
      if (!mbar_wait(&s_full[sb], (i >> 1) & 1, abort) ||
          !mbar_wait(&q_full[st], (i / C::STAGES) & 1, abort) ||
          (i >= 2 && !mbar_wait(&pds_free[sb], ((i - 2) >> 1) & 1, abort))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* stat = reinterpret_cast<const float*>(smem + C::OFF_STAT + st * C::STAT_BYTES);
      const uint32_t prow = sbase + C::OFF_PT + sb * C::PT_BYTES;
      const uint32_t drow = sbase + C::OFF_DST + sb * C::PT_BYTES;
#pragma unroll
      for (int c0 = 0; c0 < C::BQ; c0 += 32) {
        float s[32], dp[32];
        tmem_load32(tmem + lane_base + sb * 128 + c0, s);
        tmem_load32(tmem + lane_base + sb * 128 + 64 + c0, dp);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          float p[8], g[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = ch * 8 + e;
            p[e] = fast_exp2(fmaf(s[c], sl2, -stat[c0 + c]));  // lse2 = +inf past N
            g[e] = p[e] * (dp[c] - stat[C::BQ + c0 + c]);
          }
          const uint32_t off = swizzled_offset(r, (c0 >> 3) + ch, 128);
          st_shared_v4(prow + off, pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                       pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7]));
          st_shared_v4(drow + off, pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                       pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7]));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    if (ok && mbar_wait(mma_done, 0, abort)) {
      tc_fence_after();
      const bool live = key < N;
      float acc[32];
#pragma unroll
      for (int c = 0; c < DV; c += 32) {
        tmem_load32(tmem + lane_base + C::TM_DV + c, acc);
        if (live) {
          if (kNCHW) {
            __nv_bfloat16* dst = args.dv + ((long long)ch0 + 2 * DQK + c) * N + key;
            const __nv_bfloat16* res =
                args.dvres ? args.dvres + ((long long)och0 + c) * N + key : nullptr;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float x = acc[e];
              if (res) x += bf(res[(long long)e * N]);
              dst[(long long)e * N] = __float2bfloat16_rn(x);
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(args.dv + ((long long)bh * N + key) * DV + c);
#pragma unroll
            for (int e = 0; e < 32; e += 8)
              dst[e / 8] = make_uint4(pack_bf16x2(acc[e], acc[e + 1]), pack_bf16x2(acc[e + 2], acc[e + 3]),
                                      pack_bf16x2(acc[e + 4], acc[e + 5]), pack_bf16x2(acc[e + 6], acc[e + 7]));
          }
        }
      }
      const float sc = args.scale;
#pragma unroll
      for (int c = 0; c < DQK; c += 32) {
        tmem_load32(tmem + lane_base + C::TM_DK + c, acc);
        if (live) {
          if (kNCHW) {
            __nv_bfloat16* dst = args.dk + ((long long)ch0 + DQK + c) * N + key;
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[(long long)e * N] = __float2bfloat16_rn(acc[e] * sc);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(args.dk + ((long long)bh * N + key) * DQK + c);
#pragma unroll
            for (int e = 0; e < 32; e += 8)
              dst[e / 8] = make_uint4(pack_bf16x2(acc[e] * sc, acc[e + 1] * sc),
                                      pack_bf16x2(acc[e + 2] * sc, acc[e + 3] * sc),
                                      pack_bf16x2(acc[e + 4] * sc, acc[e + 5] * sc),
                                      pack_bf16x2(acc[e + 6] * sc, acc[e + 7] * sc));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <typename Cfg, typename K>
cudaError_t launch(K kern, const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                   const CUtensorMap& mDO, const BwdArgs& a, int BH, int tile,
                   cudaStream_t st) {
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (attr != cudaSuccess) return attr;
  dim3 grid((a.N + tile - 1) / tile, BH);
  kern<<<grid, Cfg::kThreads, Cfg::SMEM_BYTES, st>>>(mQ, mK, mV, mDO, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fa2_bwd_dq(const CUtensorMap& mQ, const CUtensorMap& mK,
                              const CUtensorMap& mV, const CUtensorMap& mDO, const BwdArgs& a,
                              int BH, int d, cudaStream_t st) {
  if (d == 32)
    return launch<DqCfg<32, 32, false>>(attn_bwd_dq_kernel<32, 32, false>, mQ, mK, mV, mDO, a, BH, 128, st);
  return launch<DqCfg<64, 64, false>>(attn_bwd_dq_kernel<64, 64, false>, mQ, mK, mV, mDO, a, BH, 128, st);
}

cudaError_t launch_fa2_bwd_dkdv(const CUtensorMap& mQ, const CUtensorMap& mK,
                                const CUtensorMap& mV, const CUtensorMap& mDO,
                                const BwdArgs& a, int BH, int d, cudaStream_t st) {
  if (d == 32)
    return launch<DkvCfg<32, 32, false>>(attn_bwd_dkdv_kernel<32, 32, false>, mQ, mK, mV, mDO, a, BH, 128, st);
  return launch<DkvCfg<64, 64, false>>(attn_bwd_dkdv_kernel<64, 64, false>, mQ, mK, mV, mDO, a, BH, 128, st);
}

cudaError_t launch_psa_bwd_dq(const CUtensorMap& mQK, const CUtensorMap& mV,
                              const CUtensorMap& mDO, const BwdArgs& a, int BH, int KD,
                              cudaStream_t st) {
  if (KD == 32)
    return launch<DqCfg<32, 64, true>>(attn_bwd_dq_kernel<32, 64, true>, mQK, mQK, mV, mDO, a, BH, 128, st);
  return launch<DqCfg<64, 128, true>>(attn_bwd_dq_kernel<64, 128, true>, mQK, mQK, mV, mDO, a, BH, 128, st);
}

cudaError_t launch_psa_bwd_dkdv(const CUtensorMap& mQK, const CUtensorMap& mV,
                                const CUtensorMap& mDO, const BwdArgs& a, int BH, int KD,
                                cudaStream_t st) {
  if (KD == 32)
    return launch<DkvCfg<32, 64, true>>(attn_bwd_dkdv_kernel<32, 64, true>, mQK, mQK, mV, mDO, a, BH, 128, st);
  return launch<DkvCfg<64, 128, true>>(attn_bwd_dkdv_kernel<64, 128, true>, mQK, mQK, mV, mDO, a, BH, 128, st);
}

}  // namespace psa
