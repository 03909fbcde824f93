// attn_bwd_fused.cu -- the PSA attention backward of one head in one CTA, for the
// short sequences of vision feature maps (N <= 512 positions, key_dim 32).
//
// It computes what the dQ and the dK/dV kernels of the Flash Attention 2
// backward compute (vision-rs book, page "Custom Kernels", section "Flash
// Attention 2"):
//   P = exp(scale q k^T - lse),  dP = dO V^T,  dS = P o (dP - delta),
//   delta_i = sum_c dO_ic O_ic,  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO,
// but from a single pass over the (key tile, query tile) pairs of a head: each
// P / dS tile is produced once and feeds all three gradients.  (Split into two
// kernels, every P and dP is computed twice.)  dQ of every query tile of the
// head stays in tensor memory for the whole walk (4 x 32 columns), which is
// what bounds N.
//
// Two launches: psa_bwd_delta_kernel writes delta = rowsum(dO o O) (a
// bandwidth-bound pass over Out and dOut), then the fused kernel.
//
// Layout: QKV / Out / dOut in NCHW, dQKV written in NCHW (the adjoints of
// PsaMergeAttn and PsaPackQkv are folded into the tile addressing, the optional
// PsaExtractV gradient is added into the V channels), as in the split kernels.
//
// Fused kernel: one CTA per SM (persistent over heads), 352 threads:
//   warps 0-7  row threads: warp w serves TMEM lanes 32(w%4).. (key rows) and
//              query columns 64(w/4)..+63 of the 128 x 128 S^T / dP^T tiles;
//              they build P^T and dS^T (bf16, dS^T double-buffered) in shared
//              memory and write dK, dV per key tile and dQ per head;
//   warp 8     TMA producer (K / V per key tile, double-buffered; Q / dO per
//              step in a ring, with the step's lse and delta loaded by all lanes);
//   warp 9     issues S^T = K Q^T (128 TMEM cols) and dP^T = V dO^T (128) and
//              owns the 512 TMEM columns;
//   warp 10    issues the gradient products into dV (64), dK (32) and dQ of up
//              to 4 query tiles (4 x 32).
// Per step (key tile kt, query tile qt):  S^T, dP^T  ->  row threads  ->
//   dV += P^T dO,  dK += dS^T Q,  dQ_qt += dS K  (dS read as the MN-major
//   view of the dS^T tile).  The next step's S^T / dP^T is issued as soon as
//   the row threads hold the current one in registers.
#include <math.h>

#include <algorithm>

#include "attn.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace psa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------------- delta
// delta[bh, q] = sum_c Out[b, head c, q] * dOut[b, head c, q] over the 2*KD output
// channels of head bh (NCHW, positions contiguous): eight positions per thread.
template <int DV>
__global__ void __launch_bounds__(128) psa_bwd_delta_kernel(const BwdArgs args) {
  const int N = args.N;
  const int groups = N / 8;  // N is a multiple of 8
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (long long)args.BH * groups) return;
  const int bh = (int)(t / groups), q0 = (int)(t % groups) * 8;
  const long long row = (long long)(bh / args.nh) * args.out_ch + (bh % args.nh) * DV;
  const __nv_bfloat16* o = args.o + row * N + q0;
  const __nv_bfloat16* g = args.dO + row * N + q0;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
  for (int c = 0; c < DV; ++c) {
    const uint4 ov = *reinterpret_cast<const uint4*>(o + (long long)c * N);
    const uint4 gv = *reinterpret_cast<const uint4*>(g + (long long)c * N);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 of = __bfloat1622float2(o2[e]), gf = __bfloat1622float2(g2[e]);
      acc[2 * e] = fmaf(of.x, gf.x, acc[2 * e]);
      acc[2 * e + 1] = fmaf(of.y, gf.y, acc[2 * e + 1]);
    }
  }
  float4* d = reinterpret_cast<float4*>(args.delta + (long long)bh * N + q0);
  d[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  d[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// ---------------------------------------------------------------------- fused
// One 32-column chunk of this lane's S^T and dP^T rows, loaded with one wait.
__device__ __forceinline__ void load_sp_chunk(uint32_t tS, uint32_t tP, uint32_t (&sv)[32],
                                              uint32_t (&pv)[32]) {
  tmem_load32_async(tS, sv);
  tmem_load32_async(tP, pv);
  tmem_wait_ld();
  tmem_pin(sv);
  tmem_pin(pv);
}

// P^T = 2^(s*sl2 - lse2[q]) (lse2 = +inf for queries >= N gives 0) and
// dS^T = P^T (dP^T - delta[q]) of 32 columns, packed to bf16 pairs.
__device__ __forceinline__ void p_ds_chunk(const uint32_t (&sv)[32], const uint32_t (&pv)[32],
                                           const float* lse2, const float* delta, float sl2,
                                           uint32_t* pw, uint32_t* dw) {
  const float4* l4p = reinterpret_cast<const float4*>(lse2);
  const float4* d4p = reinterpret_cast<const float4*>(delta);
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const float4 l4 = l4p[c / 4], d4 = d4p[c / 4];
    const float p0 = fast_exp2(fmaf(__uint_as_float(sv[c]), sl2, -l4.x));
    const float p1 = fast_exp2(fmaf(__uint_as_float(sv[c + 1]), sl2, -l4.y));
    const float p2 = fast_exp2(fmaf(__uint_as_float(sv[c + 2]), sl2, -l4.z));
    const float p3 = fast_exp2(fmaf(__uint_as_float(sv[c + 3]), sl2, -l4.w));
    pw[c / 2] = pack_bf16x2(p0, p1);
    pw[c / 2 + 1] = pack_bf16x2(p2, p3);
    dw[c / 2] = pack_bf16x2(p0 * (__uint_as_float(pv[c]) - d4.x),
                            p1 * (__uint_as_float(pv[c + 1]) - d4.y));
    dw[c / 2 + 1] = pack_bf16x2(p2 * (__uint_as_float(pv[c + 2]) - d4.z),
                                p3 * (__uint_as_float(pv[c + 3]) - d4.w));
  }
}

template <int DQK, int DV, int ST>
struct FusedCfg {
  static constexpr int BK = 128, BQ = 128, MAXN = kFusedBwdMaxN, MAXT = MAXN / BQ;
  static constexpr int kThreads = 352;
  static constexpr uint32_t K_BYTES = BK * DQK * 2, V_BYTES = BK * DV * 2;
  static constexpr uint32_t Q_BYTES = BQ * DQK * 2, DO_BYTES = BQ * DV * 2;
  static constexpr uint32_t STAGE_BYTES = Q_BYTES + DO_BYTES;
  static constexpr uint32_t HALF_BYTES = BK * 64 * 2;  // 64 query columns of P^T or dS^T
  static constexpr uint32_t OFF_K = 0, OFF_V = OFF_K + 2 * K_BYTES;
  static constexpr uint32_t OFF_STAGE = OFF_V + 2 * V_BYTES;
  static constexpr uint32_t STAT_BYTES = 2 * BQ * 4;  // lse2[128], delta[128] of a stage
  static constexpr uint32_t OFF_PT = OFF_STAGE + ST * STAGE_BYTES;
  static constexpr uint32_t PAIR_BYTES = 2 * HALF_BYTES;  // one buffer of P^T or dS^T
  static constexpr uint32_t OFF_DST = OFF_PT + PAIR_BYTES;  // dS^T: two buffers (step parity)
  static constexpr uint32_t OFF_STAT = OFF_DST + 2 * PAIR_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_STAT + ST * STAT_BYTES;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;
  static constexpr uint32_t TM_ST = 0, TM_DPT = 128, TM_DV = 256, TM_DK = TM_DV + DV;
  static constexpr uint32_t TM_DQ = TM_DK + DQK;
  static_assert(TM_DQ + MAXT * DQK <= 512, "tensor memory");
  static_assert(SMEM_BYTES <= 227 * 1024 && SMEM_BYTES > 114 * 1024, "one CTA per SM");
  static_assert(ST >= 2 && ST <= 4, "stages");
};

struct FusedBars {
  uint64_t kv_full[2], kv_empty[2], q_full[4], q_empty[4];
  uint64_t s_full, s_free, p_full, pt_free, dst_free[2], acc_full, acc_free, mma_done[2];
};

// Descriptor address steps (16-byte units) of the k-th 16-element K step.
// K-major 128-row tile of two 64-column boxes (P^T, dS^T): 32 bytes per step,
// next box after four steps.
__device__ __forceinline__ uint64_t off_kmajor_pair(int kk) {
  return (uint64_t)((kk >> 2) * ((128 * 128) >> 4) + (kk & 3) * (32 >> 4));
}
// NCHW tile of D channel rows per 64-position box, used as [K = positions,
// N = channels]: 32 bytes per step inside a box, next box after four steps.
template <int D>
__device__ __forceinline__ uint64_t off_ch_by_pos(int kk) {
  return (uint64_t)((kk >> 2) * ((D * 128) >> 4) + (kk & 3) * (32 >> 4));
}

template <int DQK, int DV, int ST>
__global__ void __launch_bounds__(352, 1)
    attn_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmDO, const BwdArgs args) {
  using C = FusedCfg<DQK, DV, ST>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  FusedBars& b = *reinterpret_cast<FusedBars*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&b + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = args.N;
  const int nt = (N + C::BQ - 1) / C::BQ;  // key tiles = query tiles
  const int nunits = (int)blockIdx.x < args.BH
                         ? (args.BH - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                         : 0;
  auto head_of = [&](int u) { return (int)blockIdx.x + u * (int)gridDim.x; };
  auto qkv_row = [&](int bh) { return (bh / args.nh) * args.qkv_ch + (bh % args.nh) * 4 * DQK; };
  auto out_row = [&](int bh) { return (bh / args.nh) * args.out_ch + (bh % args.nh) * DV; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.kv_full[i], 1);
      mbar_init(&b.kv_empty[i], 1);
    }
    for (int i = 0; i < ST; ++i) {
      mbar_init(&b.q_full[i], 1 + 32);
      mbar_init(&b.q_empty[i], 1);
    }
    mbar_init(&b.s_full, 1);
    mbar_init(&b.s_free, 256);
    mbar_init(&b.p_full, 256);
    mbar_init(&b.pt_free, 1);
    mbar_init(&b.dst_free[0], 1);
    mbar_init(&b.dst_free[1], 1);
    mbar_init(&b.acc_full, 1);
    mbar_init(&b.acc_free, 256);
    mbar_init(&b.mma_done[0], 1);
    mbar_init(&b.mma_done[1], 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // K / V and Q / dO by lane 0; lse2 / delta of the step's 128 queries by all
    // lanes (33 arrivals complete a stage).  The lse / delta of a whole head sit
    // in the lanes' registers (query lane + 32 i), loaded one head ahead, so no
    // global-memory latency lands between two stages.
    bool ok = true;
    int kvc = 0, qc = 0;
    constexpr int kPer = C::MAXN / 32;
    float hl[kPer], hd[kPer], nl[kPer], nd[kPer];
    auto load_head = [&](int u) {
      const int bh = head_of(u);
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int q = lane + 32 * i;
        const bool in = q < N;
        nl[i] = in ? args.lse[(long long)bh * N + q] * kLog2e : INFINITY;
        nd[i] = in ? args.delta[(long long)bh * N + q] : 0.f;
      }
    };
    if (nunits > 0) load_head(0);
    for (int u = 0; ok && u < nunits; ++u) {
      const int bh = head_of(u);
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        hl[i] = nl[i];
        hd[i] = nd[i];
      }
      if (u + 1 < nunits) load_head(u + 1);
      for (int kt = 0; ok && kt < nt; ++kt) {
        const int kb = kvc & 1;
        if (kvc >= 2 && !mbar_wait(&b.kv_empty[kb], ((kvc >> 1) - 1) & 1, abort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&b.kv_full[kb], C::K_BYTES + C::V_BYTES);
          load_tile<true, DQK>(smem + C::OFF_K + kb * C::K_BYTES, &tmK, &b.kv_full[kb], C::BK,
                               kt * C::BK, bh, qkv_row(bh) + DQK);
          load_tile<true, DV>(smem + C::OFF_V + kb * C::V_BYTES, &tmV, &b.kv_full[kb], C::BK,
                              kt * C::BK, bh, qkv_row(bh) + 2 * DQK);
        }
        ++kvc;
        for (int qt = 0; ok && qt < nt; ++qt) {
          const int st = qc % ST;
          if (qc >= ST && !mbar_wait(&b.q_empty[st], ((qc / ST) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            unsigned char* stage = smem + C::OFF_STAGE + st * C::STAGE_BYTES;
            mbar_arrive_expect_tx(&b.q_full[st], C::STAGE_BYTES);
            load_tile<true, DQK>(stage, &tmQ, &b.q_full[st], C::BQ, qt * C::BQ, bh, qkv_row(bh));
            load_tile<true, DV>(stage + C::Q_BYTES, &tmDO, &b.q_full[st], C::BQ, qt * C::BQ, bh,
                                out_row(bh));
          }
          float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT + st * C::STAT_BYTES);
#pragma unroll
          for (int i = 0; i < kPer; ++i) {
            if (i / 4 == qt) {
              stat[lane + 32 * (i % 4)] = hl[i];
              stat[C::BQ + lane + 32 * (i % 4)] = hd[i];
            }
          }
          mbar_arrive(&b.q_full[st]);
          ++qc;
        }
      }
    }
    if (lane == 0 && *abort) {
      for (int i = max(0, kvc - 2); i < kvc; ++i) drain_wait(&b.kv_full[i & 1], (i >> 1) & 1);
      for (int i = max(0, qc - ST); i < qc; ++i) drain_wait(&b.q_full[i % ST], (i / ST) & 1);
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing threads share the tensor pipe: warp 9 issues S^T / dP^T, warp
    // 10 the gradient products, so the waits of one stream are covered by the
    // other's MMAs (a thread that waits issues nothing, and the pipe holds
    // little more than the MMA it is executing).
    if (lane == 0) {
      const uint64_t dK0 = desc_mnmajor(tile_view<true, DQK>(sbase + C::OFF_K, C::BK), 0);
      const uint64_t dV0 = desc_mnmajor(tile_view<true, DV>(sbase + C::OFF_V, C::BK), 0);
      const uint64_t dQ0 = desc_mnmajor(tile_view<true, DQK>(sbase + C::OFF_STAGE, C::BQ), 0);
      const uint64_t dDO0 =
          desc_mnmajor(tile_view<true, DV>(sbase + C::OFF_STAGE + C::Q_BYTES, C::BQ), 0);
      // [K = positions, N = channels] views for the gradient products
      const uint64_t dKb0 = desc_kmajor(tile_view<true, DQK>(sbase + C::OFF_K, C::BK), 0);
      const uint64_t dQb0 = desc_kmajor(tile_view<true, DQK>(sbase + C::OFF_STAGE, C::BQ), 0);
      const uint64_t dDOb0 =
          desc_kmajor(tile_view<true, DV>(sbase + C::OFF_STAGE + C::Q_BYTES, C::BQ), 0);
      const uint64_t dPT0 = desc_kmajor(SmemTile{sbase + C::OFF_PT, 128, C::BK}, 0);
      const uint64_t dDST0 = desc_kmajor(SmemTile{sbase + C::OFF_DST, 128, C::BK}, 0);
      const uint64_t dDS0 = desc_mnmajor(SmemTile{sbase + C::OFF_DST, 128, C::BK}, 0);
      constexpr uint64_t kStepCh = (16 * 128) >> 4;  // 16 channel rows (or 16 key rows of dS^T)
      const uint32_t idS_full = idesc_bf16_f32(128, C::BQ, true, true);
      const uint32_t idDV = idesc_bf16_f32(128, DV, false, false);
      const uint32_t idDK = idesc_bf16_f32(128, DQK, false, false);
      const uint32_t idDQ = idesc_bf16_f32(128, DQK, true, false);

      auto issue_sdp = [&](int u, int kt, int qt) -> bool {
        const int kvi = u * nt + kt, s = kvi * nt + qt, st = s % ST, kb = kvi & 1;
        if ((qt == 0 && !mbar_wait(&b.kv_full[kb], (kvi >> 1) & 1, abort)) ||
            !mbar_wait(&b.q_full[st], (s / ST) & 1, abort) ||
            (s >= 1 && !mbar_wait(&b.s_free, (s - 1) & 1, abort)))
          return false;
        tc_fence_after();
        const uint64_t dK = dK0 + (uint64_t)(kb * C::K_BYTES >> 4);
        const uint64_t dV = dV0 + (uint64_t)(kb * C::V_BYTES >> 4);
        const uint64_t dQ = dQ0 + (uint64_t)(st * C::STAGE_BYTES >> 4);
        const uint64_t dDO = dDO0 + (uint64_t)(st * C::STAGE_BYTES >> 4);
        const int vq = min(C::BQ, N - qt * C::BQ);
        const uint32_t id = vq == C::BQ ? idS_full : idesc_bf16_f32(128, (vq + 15) & ~15, true, true);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
          mma_bf16(tmem + C::TM_ST, dK + kk * kStepCh, dQ + kk * kStepCh, id, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_bf16(tmem + C::TM_DPT, dV + kk * kStepCh, dDO + kk * kStepCh, id, kk > 0 ? 1u : 0u);
        mma_commit(&b.s_full);
        return true;
      };
      auto issue_grad = [&](int u, int kt, int qt) -> bool {
        const int kvi = u * nt + kt, s = kvi * nt + qt, st = s % ST, kb = kvi & 1;
        if (!mbar_wait(&b.p_full, s & 1, abort) ||
            (qt == 0 && kvi >= 1 && !mbar_wait(&b.acc_free, (kvi - 1) & 1, abort)))
          return false;
        tc_fence_after();
        const uint64_t dQb = dQb0 + (uint64_t)(st * C::STAGE_BYTES >> 4);
        const uint64_t dDOb = dDOb0 + (uint64_t)(st * C::STAGE_BYTES >> 4);
        const uint64_t dKb = dKb0 + (uint64_t)(kb * C::K_BYTES >> 4);
        const int vq = min(C::BQ, N - qt * C::BQ), vk = min(C::BK, N - kt * C::BK);
        // dV first, so P^T is released early; dS^T is double-buffered by step parity
        const uint64_t dDST = dDST0 + (uint64_t)((s & 1) * C::PAIR_BYTES >> 4);
        const uint64_t dDS = dDS0 + (uint64_t)((s & 1) * C::PAIR_BYTES >> 4);
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          if (kk * 16 < vq)
            mma_bf16(tmem + C::TM_DV, dPT0 + off_kmajor_pair(kk), dDOb + off_ch_by_pos<DV>(kk),
                     idDV, (qt > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&b.pt_free);
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          if (kk * 16 < vq)
            mma_bf16(tmem + C::TM_DK, dDST + off_kmajor_pair(kk), dQb + off_ch_by_pos<DQK>(kk),
                     idDK, (qt > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk) {
          if (kk * 16 < vk)
            mma_bf16(tmem + C::TM_DQ + qt * DQK, dDS + kk * kStepCh, dKb + off_ch_by_pos<DQK>(kk),
                     idDQ, (kt > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&b.dst_free[s & 1]);
        mma_commit(&b.q_empty[st]);
        if (qt == nt - 1) {
          mma_commit(&b.kv_empty[kb]);
          mma_commit(&b.acc_full);
        }
        return true;
      };

      // steps in order: qt fastest, then kt, then head
      bool ok = true;
      for (int u = 0; ok && u < nunits; ++u)
        for (int kt = 0; ok && kt < nt; ++kt)
          for (int qt = 0; ok && qt < nt; ++qt)
            ok = warp == 9 ? issue_sdp(u, kt, qt) : issue_grad(u, kt, qt);
      mma_commit(&b.mma_done[warp - 9]);
      drain_wait(&b.mma_done[warp - 9], 0);
    }
  } else {
    // ------------------------------------------------------------ row threads
    const int wl = warp & 3, half = warp >> 2;
    const int r = wl * 32 + lane;  // TMEM lane: key row of S^T, query row of dQ
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const int c0 = half * 64;      // first query column of this thread
    const float sl2 = args.scale_log2, sc = args.scale;
    bool ok = true;
    for (int u = 0; ok && u < nunits; ++u) {
      const int bh = head_of(u);
      for (int kt = 0; ok && kt < nt; ++kt) {
        const int kvi = u * nt + kt;
        const int vk = min(C::BK, N - kt * C::BK);
        const bool krows = wl * 32 < vk;
        for (int qt = 0; qt < nt; ++qt) {
          const int s = kvi * nt + qt, st = s % ST;
          const int vq = min(C::BQ, N - qt * C::BQ);
          const int mine = vq - c0;
          const int kend = mine > 0 ? (min(mine, 64) + 15) & ~15 : 0;
          const bool active = krows && mine > 0;
          if (!mbar_wait(&b.s_full, s & 1, abort) ||
              !mbar_wait(&b.q_full[st], (s / ST) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Two 32-column chunks; the first is packed before the second is loaded,
          // which keeps at most 96 row values live.  S^T / dP^T go back to the MMA
          // warp once both chunks are in registers.
          uint32_t pw[32], dw[32];  // packed P^T and dS^T of the 64 columns
          const float* lrow =
              reinterpret_cast<const float*>(smem + C::OFF_STAT + st * C::STAT_BYTES) + c0;
          const float* drow = lrow + C::BQ;
          const uint32_t tS = tmem + lane_base + C::TM_ST + c0;
          const uint32_t tP = tmem + lane_base + C::TM_DPT + c0;
          if (active) {
            uint32_t sv[32], pv[32];
            load_sp_chunk(tS, tP, sv, pv);
            if (kend <= 32) {
              tc_fence_before();
              mbar_arrive(&b.s_free);
            }
            p_ds_chunk(sv, pv, lrow, drow, sl2, pw, dw);
            if (kend > 32) {
              load_sp_chunk(tS + 32, tP + 32, sv, pv);
              tc_fence_before();
              mbar_arrive(&b.s_free);
              p_ds_chunk(sv, pv, lrow + 32, drow + 32, sl2, pw + 16, dw + 16);
            }
          } else {
            tc_fence_before();
            mbar_arrive(&b.s_free);
          }
          // P^T once the dV products of the previous step are done, dS^T once the
          // dK / dQ products of two steps back are done
          if (s >= 1 && !mbar_wait(&b.pt_free, (s - 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (active) store_row64(sbase + C::OFF_PT + half * C::HALF_BYTES, r, kend, pw);
          if (s >= 2 && !mbar_wait(&b.dst_free[s & 1], ((s >> 1) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (active)
            store_row64(sbase + C::OFF_DST + (s & 1) * C::PAIR_BYTES + half * C::HALF_BYTES, r,
                        kend, dw);
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&b.p_full);
        }
        if (!ok) break;
        // ---- key tile done: dV (warps 0-3) and dK (warps 4-7) of its keys
        if (!mbar_wait(&b.acc_full, kvi & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (krows) {
          const int key = kt * C::BK + r;
          const bool live = key < N;
          float acc[32];
          if (half == 0) {
#pragma unroll
            for (int c = 0; c < DV; c += 32) {
              tmem_load32(tmem + lane_base + C::TM_DV + c, acc);
              if (live) {
                __nv_bfloat16* dst = args.dv + ((long long)qkv_row(bh) + 2 * DQK + c) * N + key;
                const __nv_bfloat16* res =
                    args.dvres ? args.dvres + ((long long)out_row(bh) + c) * N + key : nullptr;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  float x = acc[e];
                  if (res) x += bf(res[(long long)e * N]);
                  dst[(long long)e * N] = __float2bfloat16_rn(x);
                }
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < DQK; c += 32) {
              tmem_load32(tmem + lane_base + C::TM_DK + c, acc);
              if (live) {
                __nv_bfloat16* dst = args.dk + ((long long)qkv_row(bh) + DQK + c) * N + key;
#pragma unroll
                for (int e = 0; e < 32; ++e) dst[(long long)e * N] = __float2bfloat16_rn(acc[e] * sc);
              }
            }
          }
        }
        // ---- last key tile of the head: dQ of every query tile
        if (kt == nt - 1) {
          for (int qt = half; qt < nt; qt += 2) {
            if (wl * 32 >= N - qt * C::BQ) continue;
            const int q = qt * C::BQ + r;
            float acc[32];
#pragma unroll
            for (int c = 0; c < DQK; c += 32) {
              tmem_load32(tmem + lane_base + C::TM_DQ + qt * DQK + c, acc);
              if (q < N) {
                __nv_bfloat16* dst = args.dq + ((long long)qkv_row(bh) + c) * N + q;
#pragma unroll
                for (int e = 0; e < 32; ++e) dst[(long long)e * N] = __float2bfloat16_rn(acc[e] * sc);
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&b.acc_free);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_psa_bwd_fused(const CUtensorMap& mQK, const CUtensorMap& mV,
                                 const CUtensorMap& mDO, const BwdArgs& a, int KD,
                                 cudaStream_t st) {
  if (KD != 32 || a.N > kFusedBwdMaxN || a.N <= 0 || a.N % 8 != 0 || a.BH <= 0 || !a.delta)
    return cudaErrorInvalidValue;
  const long long threads = (long long)a.BH * (a.N / 8);
  psa_bwd_delta_kernel<64><<<(unsigned)((threads + 127) / 128), 128, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  using Cfg = FusedCfg<32, 64, 3>;
  auto kern = attn_bwd_fused_kernel<32, 64, 3>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (attr != cudaSuccess) return attr;
  const int ctas = std::min(device_sm_count(), a.BH);
  kern<<<ctas, Cfg::kThreads, Cfg::SMEM_BYTES, st>>>(mQK, mQK, mV, mDO, a);
  return cudaGetLastError();
}

}  // namespace psa
