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
// One launch: at the start of each head the row threads compute the head's
// delta = rowsum(dO o O) from Out and dOut (while the head's first tiles load),
// so no separate pass over Out and dOut runs and delta never leaves the SM.
//
// Layout: QKV / Out / dOut in NCHW, dQKV written in NCHW (the adjoints of
// PsaMergeAttn and PsaPackQkv are folded into the tile addressing, the optional
// PsaExtractV gradient is added into the V channels), as in the split kernels.
//
// Fused kernel: one CTA per SM (persistent over heads), 896 threads.  A step is
// (key tile kt of 128 keys, query sub-tile j of 64 queries); dQ is accumulated
// per 128-query tile, i.e. once every two steps.
//   warps 0-15 row threads: warp w serves TMEM lanes 32(w%4).. (key rows) and
//              query columns 16(w/4)..+15 of the step (four warps per SM
//              sub-partition, so one warp's waits overlap the others'
//              exponentials); they turn S^T / dP^T into bf16 P^T and dS^T, which
//              they write into their own TMEM lanes (for dV and dK) and dS^T also
//              into shared memory (for dQ, which needs it transposed), and
//              compute each head's delta at its start;
//   warp 16    TMA producer (K / V per key tile, double-buffered; Q / dO per step
//              in a ring; lse2 of a head into shared memory, from registers
//              loaded one head ahead);
//   warps 17-21 issue the products, one thread each: S^T = K Q^T and dP^T =
//              V dO^T into TMEM (64 + 64 columns) as soon as the row threads
//              hold the previous step's in registers (warp 17 also owns the 512
//              columns); dV += P^T dO and dK += dS^T Q (P^T, dS^T read as the A
//              operand from tensor memory); dQ of up to 4 query tiles (4 x 32);
//   warps 22-23 idle;
//   warps 24-27 epilogue: read dV / dK of a finished key tile out of tensor
//              memory, hand the accumulators back, and write them to dQKV (with
//              dVres); read and write dQ once a head is done.
// The products of step s+1 run while the row threads work on step s; P^T and
// dS^T are double-buffered in tensor memory and dS^T pair-buffered in shared
// memory, so neither side waits for the other's previous step.  Five issuing
// threads keep the tensor pipe fed (one thread alone issues one MMA per ~130
// cycles).  Keeping P^T and
// dS^T out of shared memory for dV and dK halves the shared-memory traffic of a
// step, which the MMAs' operand reads, the row threads' stores and the TMA
// fills otherwise share.  The row
// threads never wait for a key tile's products to drain: the epilogue warps do,
// while the rows already work on the next key tile's first steps.
//   dV += P^T dO,  dK += dS^T Q  (per step);  dQ_t += dS K  (dS read as the
//   MN-major view of the two dS^T halves of tile t).
#include <math.h>

#include <algorithm>

#include "attn.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace psa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf(const __nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------------- fused
// P^T = 2^(s*sl2 - lse2[q]) and dS^T = P^T (dP^T - delta[q]) of NC columns,
// packed to bf16 pairs.  The stats come negated (nlse2 = -lse2, -inf for
// queries >= N, which gives P = 0; ndelta = -delta), so that every step is one
// paired FP32 instruction for two columns.
template <int NC>
__device__ __forceinline__ void p_ds_chunk(const uint32_t (&sv)[NC], const uint32_t (&pv)[NC],
                                           const float* nlse2, const float* ndelta, float sl2,
                                           uint32_t* pw, uint32_t* dw) {
  const float2* l2p = reinterpret_cast<const float2*>(nlse2);
  const float2* d2p = reinterpret_cast<const float2*>(ndelta);
  const float2 sl2x2 = make_float2(sl2, sl2);
#pragma unroll
  for (int c = 0; c < NC; c += 2) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])),
                                sl2x2, l2p[c / 2]);
    const float2 p = make_float2(fast_exp2(x.x), fast_exp2(x.y));
    const float2 g =
        __fadd2_rn(make_float2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])), d2p[c / 2]);
    const float2 ds = __fmul2_rn(p, g);
    pw[c / 2] = pack_bf16x2(p.x, p.y);
    dw[c / 2] = pack_bf16x2(ds.x, ds.y);
  }
}

// kLong: up to kFusedBwdMaxNLong positions; dQ of each 128-query tile and key
// tile is a partial sum that the epilogue warps add into an fp32 accumulator in
// the workspace, in key-tile order.  Otherwise (up to kFusedBwdMaxN positions)
// dQ of every query tile stays in tensor memory for the whole head.
template <int DQK, int DV, int ST, bool kLong>
struct FusedCfg {
  static constexpr int BK = 128, BQ = 64, QT = 128;
  static constexpr int MAXN = kLong ? kFusedBwdMaxNLong : kFusedBwdMaxN, MAXQT = MAXN / QT;
  static constexpr int CHUNK = 512;  // positions per pass of the delta computation
  static constexpr int kRowWarps = 16, kThreads = 32 * kRowWarps + 384;
  // producer, then the issuers of S^T (TMEM owner), dP^T, dV, dK and dQ, two idle
  // warps, then four epilogue warps (warp % 4 = TMEM lane quadrant)
  static constexpr int kProducer = kRowWarps, kIssS = kRowWarps + 1, kIssLast = kIssS + 4;
  static constexpr int kEpiWarp0 = kRowWarps + 8, kEpiThreads = 128;
  static constexpr uint32_t K_BYTES = BK * DQK * 2, V_BYTES = BK * DV * 2;
  static constexpr uint32_t Q_BYTES = BQ * DQK * 2, DO_BYTES = BQ * DV * 2;
  static constexpr uint32_t STAGE_BYTES = Q_BYTES + DO_BYTES;
  static constexpr uint32_t HALF_BYTES = BK * 64 * 2;  // 128 keys x 64 queries, bf16
  static constexpr uint32_t PAIR_BYTES = 2 * HALF_BYTES;  // dS^T of a 128-query tile
  static constexpr uint32_t HSTAT_BYTES = 2 * MAXN * 4;  // -lse2[MAXN], -delta[MAXN] of a head
  static constexpr uint32_t OFF_K = 0, OFF_V = OFF_K + 2 * K_BYTES;
  static constexpr uint32_t OFF_STAGE = OFF_V + 2 * V_BYTES;
  static constexpr uint32_t OFF_DST = OFF_STAGE + ST * STAGE_BYTES;  // dS^T: two pair buffers
  static constexpr uint32_t OFF_HSTAT = OFF_DST + 2 * PAIR_BYTES;  // two heads
  static constexpr uint32_t OFF_DSCR = OFF_HSTAT + 2 * HSTAT_BYTES;  // delta partial sums
  static constexpr uint32_t OFF_BAR = OFF_DSCR + 8 * CHUNK * 4;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + 512 + 1024;
  // TMEM columns: S^T, dP^T (fp32), then P^T_b and dS^T_b (bf16 pairs, 32 columns
  // per 64 queries, b = step parity), dV, dK, then dQ: of up to 4 query tiles, or
  // (kLong) two buffers of one query tile's partial sum
  static constexpr uint32_t TM_S = 0, TM_DP = 64, TM_PT = 128, TM_DST = 192;
  static constexpr uint32_t TM_DV = 256, TM_DK = TM_DV + DV;
  static constexpr uint32_t TM_DQ = TM_DK + DQK;
  static_assert(TM_DQ + (kLong ? 2 : MAXQT) * DQK <= 512, "tensor memory");
  static_assert(MAXN % CHUNK == 0 && 8 * 64 == CHUNK, "delta passes of 512 positions");
  static_assert(SMEM_BYTES <= 227 * 1024 && SMEM_BYTES > 114 * 1024, "one CTA per SM");
  static_assert(kEpiWarp0 % 4 == 0, "epilogue warps cover the four lane quadrants in order");
  static_assert(ST >= 2 && ST <= 8, "stages");
};

struct FusedBars {
  uint64_t kv_full[2], kv_empty[2], q_full[8], q_empty[8];
  uint64_t s_full, s_free, p_full[2], g_done[2], hs_full[2], hs_free[2];
  uint64_t acc_full, acc_free, dq_full[2], dq_free[2], mma_done[5];
  uint64_t dl_part, dl_full;  // a head's delta: partial sums written, delta written
};
static_assert(sizeof(FusedBars) + 8 <= 512, "barrier area");

// NCHW tile of D channel rows per 64-position box, used as [K = positions,
// N = channels]: 32 bytes per 16-position step inside a box, next box after four.
template <int D>
__device__ __forceinline__ uint64_t off_ch_by_pos(int kk) {
  return (uint64_t)((kk >> 2) * ((D * 128) >> 4) + (kk & 3) * (32 >> 4));
}

template <int DQK, int DV, int ST, bool kLong>
__global__ void __launch_bounds__(896, 1)
    attn_bwd_fused_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __grid_constant__ CUtensorMap tmDO, const BwdArgs args) {
  using C = FusedCfg<DQK, DV, ST, kLong>;
  static_assert(DQK == 32 && DV == 64, "tile split of the epilogue");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  FusedBars& b = *reinterpret_cast<FusedBars*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&b + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = args.N;
  const int nkt = (N + C::BK - 1) / C::BK;  // key tiles
  const int nqs = (N + C::BQ - 1) / C::BQ;  // 64-query steps per key tile
  const int nqt = (N + C::QT - 1) / C::QT;  // 128-query dQ tiles
  const int nunits = (int)blockIdx.x < args.BH
                         ? (args.BH - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                         : 0;
  auto head_of = [&](int u) { return (int)blockIdx.x + u * (int)gridDim.x; };
  auto qkv_row = [&](int bh) { return (bh / args.nh) * args.qkv_ch + (bh % args.nh) * 4 * DQK; };
  auto out_row = [&](int bh) { return (bh / args.nh) * args.out_ch + (bh % args.nh) * DV; };

  if (threadIdx.x == 0) {
    // arrival counts: K / V are read by the S^T, dP^T and dQ issuers, a Q / dO
    // stage by the S^T, dP^T, dV and dK issuers; S^T / dP^T come from two
    // issuers, P^T / dS^T are read by the dV, dK and dQ issuers, and the dV / dK
    // accumulators are filled by two
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.kv_full[i], 1);
      mbar_init(&b.kv_empty[i], 3);
      mbar_init(&b.p_full[i], 32 * C::kRowWarps);
      mbar_init(&b.g_done[i], 3);
      mbar_init(&b.hs_full[i], 32);
      mbar_init(&b.hs_free[i], 32 * C::kRowWarps);
    }
    for (int i = 0; i < 5; ++i) mbar_init(&b.mma_done[i], 1);
    mbar_init(&b.s_full, 2);
    mbar_init(&b.s_free, 32 * C::kRowWarps);
    for (int i = 0; i < ST; ++i) {
      mbar_init(&b.q_full[i], 1);
      mbar_init(&b.q_empty[i], 4);
    }
    mbar_init(&b.acc_full, 2);
    mbar_init(&b.acc_free, C::kEpiThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b.dq_full[i], 1);
      mbar_init(&b.dq_free[i], C::kEpiThreads);
    }
    mbar_init(&b.dl_part, 32 * C::kRowWarps);
    mbar_init(&b.dl_full, 32 * C::kRowWarps);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kIssS) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // set-up done: the next kernel may start its own; the previous one must have
  // finished before this grid reads or writes global memory
  pdl_launch_dependents();
  pdl_wait();

  if (warp == C::kProducer) {
    // ------------------------------------------------------------ TMA producer
    // K / V and Q / dO by lane 0.  The negated lse2 of a whole head is written to
    // shared memory by all lanes (double-buffered by head parity); its first 512
    // positions come from registers (query lane + 32 i) loaded one head ahead, so
    // no global-memory latency lands between two stages.  (The row threads add
    // the head's delta.)
    bool ok = true;
    int kvc = 0, qc = 0;
    constexpr int kPer = C::CHUNK / 32;
    // raw lse values: nothing consumes them until they are written to shared
    // memory, so the loads stay in flight while the producer goes on issuing
    // copies (scaling them at load time would stall it on the loads)
    float nl[kPer];
    auto load_chunk = [&](int bh, int c0) {
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int q = c0 + lane + 32 * i;
        nl[i] = q < N ? args.lse[(long long)bh * N + q] : 0.f;
      }
    };
    if (nunits > 0) load_chunk(head_of(0), 0);
    for (int u = 0; ok && u < nunits; ++u) {
      const int bh = head_of(u);
      if (u >= 2 && !mbar_wait(&b.hs_free[u & 1], ((u >> 1) - 1) & 1, abort)) {
        ok = false;
        break;
      }
      float* hst = reinterpret_cast<float*>(smem + C::OFF_HSTAT + (u & 1) * C::HSTAT_BYTES);
      for (int c0 = 0; c0 < C::MAXN; c0 += C::CHUNK) {
        if (c0 > 0) load_chunk(bh, c0);
#pragma unroll
        for (int i = 0; i < kPer; ++i)
          hst[c0 + lane + 32 * i] = c0 + lane + 32 * i < N ? -nl[i] * kLog2e : -INFINITY;
      }
      mbar_arrive(&b.hs_full[u & 1]);
      if (u + 1 < nunits) load_chunk(head_of(u + 1), 0);
      for (int kt = 0; ok && kt < nkt; ++kt) {
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
        for (int j = 0; ok && j < nqs; ++j) {
          const int st = qc % ST;
          if (qc >= ST && !mbar_wait(&b.q_empty[st], ((qc / ST) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            unsigned char* stage = smem + C::OFF_STAGE + st * C::STAGE_BYTES;
            mbar_arrive_expect_tx(&b.q_full[st], C::STAGE_BYTES);
            load_tile<true, DQK>(stage, &tmQ, &b.q_full[st], C::BQ, j * C::BQ, bh, qkv_row(bh));
            load_tile<true, DV>(stage + C::Q_BYTES, &tmDO, &b.q_full[st], C::BQ, j * C::BQ, bh,
                                out_row(bh));
          }
          ++qc;
        }
      }
    }
    if (lane == 0 && *abort) {
      for (int i = max(0, kvc - 2); i < kvc; ++i) drain_wait(&b.kv_full[i & 1], (i >> 1) & 1);
      for (int i = max(0, qc - ST); i < qc; ++i) drain_wait(&b.q_full[i % ST], (i / ST) & 1);
    }
  } else if (warp >= C::kIssS && warp <= C::kIssLast) {
    // ------------------------------------------------------------ MMA issuers
    // Five issuing threads, one per product and accumulator: a single thread
    // issues at most one tcgen05.mma per ~130 cycles whatever the shape (measured
    // on GB300), while the pipe itself takes one every ~46-55 cycles at N = 32 /
    // 64 when several threads feed it.  Each accumulator has one issuer, so every
    // sum runs in a fixed order and results stay bitwise reproducible.
    if (lane == 0) {
      const int role = warp - C::kIssS;
      // S^T = K Q^T, dP^T = V dO^T: positions x channels tiles, MN-major, K = channels
      const uint64_t dK0 = desc_mnmajor(tile_view<true, DQK>(sbase + C::OFF_K, C::BK), 0);
      const uint64_t dV0 = desc_mnmajor(tile_view<true, DV>(sbase + C::OFF_V, C::BK), 0);
      const uint64_t dQ0 = desc_mnmajor(tile_view<true, DQK>(sbase + C::OFF_STAGE, C::BQ), 0);
      const uint64_t dDO0 =
          desc_mnmajor(tile_view<true, DV>(sbase + C::OFF_STAGE + C::Q_BYTES, C::BQ), 0);
      // [K = positions, N = channels] views: dO and Q (one 64-position box) for
      // dV / dK, K (two boxes) for dQ
      const uint64_t dDOb0 =
          desc_kmajor(tile_view<true, DV>(sbase + C::OFF_STAGE + C::Q_BYTES, C::BQ), 0);
      const uint64_t dQb0 = desc_kmajor(tile_view<true, DQK>(sbase + C::OFF_STAGE, C::BQ), 0);
      const uint64_t dKb0 = desc_kmajor(tile_view<true, DQK>(sbase + C::OFF_K, C::BK), 0);
      // dS of a 128-query tile: the MN-major view of its two dS^T halves (128 key
      // rows x 64 queries each, K-major)
      const uint64_t dDS0 = desc_mnmajor(SmemTile{sbase + C::OFF_DST, 128, C::BK}, 0);
      constexpr uint64_t kStep16Rows = (16 * 128) >> 4;
      const uint32_t idS_full = idesc_bf16_f32(128, C::BQ, true, true);
      const uint32_t idDV = idesc_bf16_f32(128, DV, false, false);
      const uint32_t idDK = idesc_bf16_f32(128, DQK, false, false);
      const uint32_t idDQ = idesc_bf16_f32(128, DQK, true, false);

      // S^T (role 0) or dP^T (role 1) of step s, as soon as the row threads hold
      // step s - 1's in registers
      auto issue_sdp = [&](int u, int kt, int j) -> bool {
        const int kvi = u * nkt + kt, s = kvi * nqs + j, st = s % ST, kb = kvi & 1;
        if ((j == 0 && !mbar_wait(&b.kv_full[kb], (kvi >> 1) & 1, abort)) ||
            !mbar_wait(&b.q_full[st], (s / ST) & 1, abort) ||
            (s >= 1 && !mbar_wait(&b.s_free, (s - 1) & 1, abort)))
          return false;
        tc_fence_after();
        const int vq = min(C::BQ, N - j * C::BQ);
        const uint32_t id = vq == C::BQ ? idS_full : idesc_bf16_f32(128, (vq + 15) & ~15, true, true);
        if (role == 0) {
          const uint64_t dK = dK0 + (uint64_t)(kb * C::K_BYTES >> 4);
          const uint64_t dQ = dQ0 + (uint64_t)(st * C::STAGE_BYTES >> 4);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            mma_bf16(tmem + C::TM_S, dK + kk * kStep16Rows, dQ + kk * kStep16Rows, id, kk > 0 ? 1u : 0u);
        } else {
          const uint64_t dV = dV0 + (uint64_t)(kb * C::V_BYTES >> 4);
          const uint64_t dDO = dDO0 + (uint64_t)(st * C::STAGE_BYTES >> 4);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            mma_bf16(tmem + C::TM_DP, dV + kk * kStep16Rows, dDO + kk * kStep16Rows, id, kk > 0 ? 1u : 0u);
        }
        mma_commit(&b.s_full);
        mma_commit(&b.q_empty[st]);
        if (j == nqs - 1) mma_commit(&b.kv_empty[kb]);
        return true;
      };
      // dV += P^T dO (role 2) or dK += dS^T Q (role 3) of step s, A from TMEM
      auto issue_dvdk = [&](int u, int kt, int j) -> bool {
        const int kvi = u * nkt + kt, s = kvi * nqs + j, st = s % ST, bb = s & 1;
        if (!mbar_wait(&b.p_full[bb], (s >> 1) & 1, abort) ||
            !mbar_wait(&b.q_full[st], (s / ST) & 1, abort) ||
            (j == 0 && kvi >= 1 && !mbar_wait(&b.acc_free, (kvi - 1) & 1, abort)))
          return false;
        tc_fence_after();
        const int vq = min(C::BQ, N - j * C::BQ);
        if (role == 2) {
          const uint64_t dDOb = dDOb0 + (uint64_t)(st * C::STAGE_BYTES >> 4);
          const uint32_t tPT = tmem + C::TM_PT + 32 * bb;  // 8 columns per 16 queries
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            if (kk * 16 < vq)
              mma_bf16_ts(tmem + C::TM_DV, tPT + 8 * kk, dDOb + 2 * kk, idDV, (j > 0 || kk > 0) ? 1u : 0u);
        } else {
          const uint64_t dQb = dQb0 + (uint64_t)(st * C::STAGE_BYTES >> 4);
          const uint32_t tDST = tmem + C::TM_DST + 32 * bb;
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            if (kk * 16 < vq)
              mma_bf16_ts(tmem + C::TM_DK, tDST + 8 * kk, dQb + 2 * kk, idDK, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&b.q_empty[st]);
        mma_commit(&b.g_done[bb]);
        if (j == nqs - 1) mma_commit(&b.acc_full);
        return true;
      };
      // dQ_t += dS K (role 4) once both halves of query tile t (or its only one)
      // are stored; every step, so that g_done counts this thread's reads of the
      // dS^T pair buffers.  kLong: the product of this key tile alone, into one of
      // two TMEM buffers the epilogue warps add into the workspace
      auto issue_dq = [&](int u, int kt, int j) -> bool {
        const int kvi = u * nkt + kt, s = kvi * nqs + j, kb = kvi & 1, bb = s & 1;
        const bool dq_step = (j & 1) || j == nqs - 1;
        const int qt = j >> 1, pi = kvi * nqt + qt, pb = pi & 1;
        // the first dQ product of a head (or, kLong, of a buffer) overwrites the
        // accumulators the epilogue warps read out before
        const bool first_dq = kt == 0 && dq_step && j <= 1;
        const bool wait_free = kLong ? (dq_step && pi >= 2) : (first_dq && u >= 1);
        const int free_bar = kLong ? pb : 0;
        const uint32_t free_parity = kLong ? (((pi >> 1) - 1) & 1) : ((u - 1) & 1);
        if (!mbar_wait(&b.p_full[bb], (s >> 1) & 1, abort) ||
            (j == 0 && !mbar_wait(&b.kv_full[kb], (kvi >> 1) & 1, abort)) ||
            (wait_free && !mbar_wait(&b.dq_free[free_bar], free_parity, abort)))
          return false;
        tc_fence_after();
        if (dq_step) {
          const int vk = min(C::BK, N - kt * C::BK);
          const uint64_t dDS = dDS0 + (uint64_t)(pb * C::PAIR_BYTES >> 4);
          const uint64_t dKb = dKb0 + (uint64_t)(kb * C::K_BYTES >> 4);
          const uint32_t dst = tmem + C::TM_DQ + (kLong ? pb : qt) * DQK;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            if (kk * 16 < vk)
              mma_bf16(dst, dDS + kk * kStep16Rows, dKb + off_ch_by_pos<DQK>(kk), idDQ,
                       ((!kLong && kt > 0) || kk > 0) ? 1u : 0u);
          }
          if (kLong) mma_commit(&b.dq_full[pb]);
        }
        mma_commit(&b.g_done[bb]);
        if (j == nqs - 1) {
          mma_commit(&b.kv_empty[kb]);
          if (!kLong && kt == nkt - 1) mma_commit(&b.dq_full[0]);
        }
        return true;
      };

      // steps in order: j fastest, then kt, then head
      bool ok = true;
      for (int u = 0; ok && u < nunits; ++u)
        for (int kt = 0; ok && kt < nkt; ++kt)
          for (int j = 0; ok && j < nqs; ++j)
            ok = role <= 1 ? issue_sdp(u, kt, j) : role <= 3 ? issue_dvdk(u, kt, j) : issue_dq(u, kt, j);
      mma_commit(&b.mma_done[role]);
      drain_wait(&b.mma_done[role], 0);
    }
  } else if (warp >= C::kEpiWarp0) {
    // ------------------------------------------------------------ epilogue warps
    // One thread per TMEM lane (key row of dV / dK, query row of a dQ tile).
    const int wl = warp & 3;
    const int r = wl * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const float sc = args.scale;
    bool ok = true;
    // dQ rows of query tile qt: the 32 values of this lane, scaled and rounded
    auto store_dq = [&](int bh, int qt, const float (&acc)[32]) {
      const int q = qt * C::QT + r;
      if (q >= N) return;
      __nv_bfloat16* dst = args.dq + (long long)qkv_row(bh) * N + q;
#pragma unroll
      for (int e = 0; e < 32; ++e) dst[(long long)e * N] = __float2bfloat16_rn(acc[e] * sc);
    };
    for (int u = 0; ok && u < nunits; ++u) {
      const int bh = head_of(u);
      for (int kt = 0; kt < nkt; ++kt) {
        const int kvi = u * nkt + kt;
        if (kLong) {
          // this key tile's dQ of every query tile, added in key-tile order into the
          // fp32 accumulator of the head in the workspace ([BH, N, 32]); the last
          // key tile writes the result
          for (int qt = 0; ok && qt < nqt; ++qt) {
            const int pi = kvi * nqt + qt, pb = pi & 1;
            if (!mbar_wait(&b.dq_full[pb], (pi >> 1) & 1, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            float acc[32];
            tmem_load32(tmem + lane_base + C::TM_DQ + pb * DQK, acc);
            tc_fence_before();
            mbar_arrive(&b.dq_free[pb]);
            const int q = qt * C::QT + r;
            if (q >= N) continue;
            float4* part = reinterpret_cast<float4*>(args.delta + ((long long)bh * N + q) * DQK);
            if (kt > 0) {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float4 p4 = part[e];
                acc[4 * e] += p4.x;
                acc[4 * e + 1] += p4.y;
                acc[4 * e + 2] += p4.z;
                acc[4 * e + 3] += p4.w;
              }
            }
            if (kt < nkt - 1) {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                part[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
            } else {
              store_dq(bh, qt, acc);
            }
          }
          if (!ok) break;
        }
        if (!mbar_wait(&b.acc_full, kvi & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dV (column groups 0, 1: 32 channels each) and dK (group 2) of this key
        // tile's rows, one group at a time; the accumulators go back to the
        // gradient issuers as soon as the last group is in registers
        const int key = kt * C::BK + r;
        const bool live = key < N;
#pragma unroll 1
        for (int g = 0; g < 3; ++g) {
          float acc[32];
          tmem_load32(tmem + lane_base + C::TM_DV + 32 * g, acc);  // dK follows dV's 64 columns
          if (g == 2) {
            tc_fence_before();
            mbar_arrive(&b.acc_free);
          }
          if (!live) continue;
          if (g < 2) {
            __nv_bfloat16* dst = args.dv + ((long long)qkv_row(bh) + 2 * DQK + 32 * g) * N + key;
            const __nv_bfloat16* res =
                args.dvres ? args.dvres + ((long long)out_row(bh) + 32 * g) * N + key : nullptr;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float x = acc[e];
              if (res) x += bf(res[(long long)e * N]);
              dst[(long long)e * N] = __float2bfloat16_rn(x);
            }
          } else {
            __nv_bfloat16* dst = args.dk + ((long long)qkv_row(bh) + DQK) * N + key;
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[(long long)e * N] = __float2bfloat16_rn(acc[e] * sc);
          }
        }
      }
      if (!ok || kLong) continue;
      // the head's last products are done: dQ of every 128-query tile
      if (!mbar_wait(&b.dq_full[0], u & 1, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int qt = 0; qt < nqt; ++qt) {
        float acc[32];
        tmem_load32(tmem + lane_base + C::TM_DQ + qt * DQK, acc);
        store_dq(bh, qt, acc);
      }
      tc_fence_before();
      mbar_arrive(&b.dq_free[0]);
    }
  } else if (warp < C::kRowWarps) {
    // ------------------------------------------------------------ row threads
    const int wl = warp & 3, cq = warp >> 2;
    const int r = wl * 32 + lane;  // TMEM lane: key row of S^T, query row of dQ
    const uint32_t lane_base = (uint32_t)(wl * 32) << 16;
    const int c0 = cq * 16;        // first query column of this thread in a step
    const float sl2 = args.scale_log2;
    bool ok = true;
    int dlc = 0;  // delta passes done (phase of dl_part / dl_full)
    for (int u = 0; ok && u < nunits; ++u) {
      const int bh = head_of(u);
      float* hst = reinterpret_cast<float*>(smem + C::OFF_HSTAT + (u & 1) * C::HSTAT_BYTES);
      // delta[q] = sum_c Out[c, q] dOut[c, q] over the head's DV channels, while
      // its first tiles load, 512 positions per pass.  Thread t = 64 s + g sums
      // channels 8s .. 8s+7 at positions 8g .. 8g+7 of the pass; the eight channel
      // slices meet in a scratch area of shared memory.
      static_assert(C::kRowWarps * 32 == C::CHUNK && DV == 64, "one thread per 8 x 8 block");
      for (int p0 = 0; ok && p0 < N; p0 += C::CHUNK) {
        const int t = threadIdx.x, g = t & 63, sl8 = t >> 6;
        float part[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) part[e] = 0.f;
        if (p0 + 8 * g < N) {
          const long long base = ((long long)out_row(bh) + 8 * sl8) * N + p0 + 8 * g;
          uint4 ov[8], dv[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            ov[c] = __ldg(reinterpret_cast<const uint4*>(args.o + base + (long long)c * N));
            dv[c] = __ldg(reinterpret_cast<const uint4*>(args.dO + base + (long long)c * N));
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t ow[4] = {ov[c].x, ov[c].y, ov[c].z, ov[c].w};
            const uint32_t dw4[4] = {dv[c].x, dv[c].y, dv[c].z, dv[c].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 o2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[e]));
              const float2 d2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw4[e]));
              part[2 * e] = fmaf(o2.x, d2.x, part[2 * e]);
              part[2 * e + 1] = fmaf(o2.y, d2.y, part[2 * e + 1]);
            }
          }
        }
        float* scratch = reinterpret_cast<float*>(smem + C::OFF_DSCR);
        float4* sp = reinterpret_cast<float4*>(scratch + sl8 * C::CHUNK + 8 * g);
        sp[0] = make_float4(part[0], part[1], part[2], part[3]);
        sp[1] = make_float4(part[4], part[5], part[6], part[7]);
        mbar_arrive(&b.dl_part);
        if (!mbar_wait(&b.dl_part, dlc & 1, abort)) {
          ok = false;
          break;
        }
        float dsum = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) dsum += scratch[k * C::CHUNK + t];
        hst[C::MAXN + p0 + t] = p0 + t < N ? -dsum : 0.f;
        mbar_arrive(&b.dl_full);
        if (!mbar_wait(&b.dl_full, dlc & 1, abort)) {
          ok = false;
          break;
        }
        ++dlc;
      }
      if (!ok) break;
      if (!mbar_wait(&b.hs_full[u & 1], (u >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      for (int kt = 0; ok && kt < nkt; ++kt) {
        const int kvi = u * nkt + kt;
        const int vk = min(C::BK, N - kt * C::BK);
        const bool krows = wl * 32 < vk;
        for (int j = 0; j < nqs; ++j) {
          const int s = kvi * nqs + j, bb = s & 1;
          const int qt = j >> 1, pi = kvi * nqt + qt, pb = pi & 1;
          const int vq = min(C::BQ, N - j * C::BQ);
          const int mine = vq - c0;
          const bool active = krows && mine > 0;
          if (!mbar_wait(&b.s_full, s & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t pw[8], dw[8];  // packed P^T and dS^T of this thread's 16 queries
          if (active) {
            uint32_t sv[16], pv[16];
            tmem_load16_async(tmem + lane_base + C::TM_S + c0, sv);
            tmem_load16_async(tmem + lane_base + C::TM_DP + c0, pv);
            tmem_wait_ld();
            tmem_pin(sv);
            tmem_pin(pv);
            tc_fence_before();
            mbar_arrive(&b.s_free);
            const float* lrow = hst + j * C::BQ + c0;
            p_ds_chunk<16>(sv, pv, lrow, lrow + C::MAXN, sl2, pw, dw);
          } else {
            tc_fence_before();
            mbar_arrive(&b.s_free);
          }
          // the P^T / dS^T TMEM buffers s & 1 were last read by the products of
          // step s - 2, and the dS^T pair buffer by those of step s - 3 or s - 4:
          // all done once the products of step s - 2 are (one issuing thread,
          // commits cover all earlier MMAs)
          if (s >= 2 && !mbar_wait(&b.g_done[bb], ((s >> 1) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          if (active) {
            tmem_store8_async(tmem + lane_base + C::TM_PT + 32 * bb + c0 / 2, pw);
            tmem_store8_async(tmem + lane_base + C::TM_DST + 32 * bb + c0 / 2, dw);
          }
          if (active) {
            const uint32_t half = sbase + C::OFF_DST + pb * C::PAIR_BYTES + (j & 1) * C::HALF_BYTES;
#pragma unroll
            for (int i = 0; i < 2; ++i)
              st_shared_v4(half + swizzled_offset(r, c0 / 8 + i, 128), dw[4 * i], dw[4 * i + 1],
                           dw[4 * i + 2], dw[4 * i + 3]);
          }
          if (active) {
            tmem_wait_st();
            fence_proxy_async_smem();  // (only active threads stored dS^T)
          }
          tc_fence_before();
          mbar_arrive(&b.p_full[bb]);
        }
        if (!ok) break;
      }
      mbar_arrive(&b.hs_free[u & 1]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kIssS) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_psa_bwd_fused(const CUtensorMap& mQK, const CUtensorMap& mV,
                                 const CUtensorMap& mDO, const BwdArgs& a, int KD,
                                 cudaStream_t st) {
  if (KD != 32 || a.N > kFusedBwdMaxNLong || a.N <= 0 || a.N % 8 != 0 || a.BH <= 0 || !a.o ||
      !a.dO || (a.N > kFusedBwdMaxN && !a.delta))
    return cudaErrorInvalidValue;
  const int ctas = std::min(device_sm_count(), a.BH);
  if (a.N <= kFusedBwdMaxN) {
    using Cfg = FusedCfg<32, 64, 4, false>;
    auto kern = attn_bwd_fused_kernel<32, 64, 4, false>;
    const cudaError_t attr = set_max_dynamic_smem((const void*)kern, Cfg::SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    return launch_pdl(kern, dim3(ctas), dim3(Cfg::kThreads), Cfg::SMEM_BYTES, st, mQK, mQK, mV,
                      mDO, a);
  }
  using Cfg = FusedCfg<32, 64, 4, true>;
  auto kern = attn_bwd_fused_kernel<32, 64, 4, true>;
  const cudaError_t attr = set_max_dynamic_smem((const void*)kern, Cfg::SMEM_BYTES);
  if (attr != cudaSuccess) return attr;
  return launch_pdl(kern, dim3(ctas), dim3(Cfg::kThreads), Cfg::SMEM_BYTES, st, mQK, mQK, mV, mDO,
                    a);
}

}  // namespace psa
