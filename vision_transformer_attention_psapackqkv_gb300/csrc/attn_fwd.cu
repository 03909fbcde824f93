// attn_fwd.cu -- Flash Attention 2 forward (vision-rs book, page "Custom Kernels",
// section "Flash Attention 2"): O = softmax(scale * Q K^T) V with an online
// softmax over key tiles; the N x N score matrix only ever exists one 128 x 64
// tile at a time, in tensor memory.
//
// bf16 path (tcgen05, sm_103a): a persistent kernel.  Each CTA runs NWG
// independent 128-query-row pipelines ("slots"); tiles are dealt to the S slots
// of the grid round by round, in slot order in even rounds and in reverse slot
// order in odd ones.  Tiles are numbered full query tiles first (t -> head
// t / nfull, query tile t % nfull), then the partial last tile of every head
// (t -> head t - BH*nfull), so that the cheap partial tiles fill the last rounds
// and go to the slots that took the fewest full tiles.  Warp roles:
//   warps 4w .. 4w+3   softmax of slot w: one thread per query row (= TMEM lane)
//                      (split rows: warps 0-7 of the single slot, see below)
//   next warp (P)      TMA producer: per slot, Q (double- or single-buffered)
//                      and a 2- to 4-stage ring of 64-key K/V tiles
//   warp P + 1         S issuer (one thread) and TMEM owner; per slot
//                        S_k = Q K_k^T -> TMEM (64 columns), issued as soon as
//                        the softmax holds S_{k-1} in registers, so it overlaps
//                        the exponentials of tile k-1
//   warp P + 2         P.V issuer (one thread): O += P_k V_k -> TMEM (DV
//                      columns), P_k read from tensor memory (A operand;
//                      double-buffered)
//   warp P + 3         store warp (NCHW): TMA stores of each finished O tile and
//                      bulk copies of its LSE, from a shared-memory staging tile
// The bf16 kernels run persistent grids; with one slot per CTA two CTAs share
// an SM (and its tensor core), which interleaves their softmax and MMA phases.
// Split rows (kSplit, short sequences): warps 0-3 and 4-7 both cover the 128 rows,
// each thread owning one 32-key half of every tile with its own running max and
// sum and its own O accumulator in TMEM (P.V k-steps of half h go to accumulator
// h); the epilogue merges the halves, O = (O_0 2^(m_0-m) + O_1 2^(m_1-m)) / l.
// Every CTA sets up its barriers and TMEM, lets the next kernel of the stream
// start (programmatic dependent launch) and waits for the previous one before
// touching global memory.
// Softmax: running max in the log2 domain; p = 2^(scale*log2e*s - m) rounded to
// bf16 and written by each thread into its own TMEM lane (two per 32-bit column),
// where the P.V product reads it as its A operand, so P never passes through
// shared memory; O is rescaled in TMEM only when a row
// max grows by more than 2^8 (exact either way, since O and the running sum
// share the stale max).  Epilogue: O / l in the output layout and the LSE.
// The row threads issue no global store in the NCHW layout: an mbarrier arrive
// has release semantics, so every hand-off after a global store would wait for
// that store to be acknowledged (measured ~0.7-1k cycles per step); they stage O
// and the LSE in shared memory for the store warp instead.
// Layouts: kNCHW = false reads [BH, N, D] planes (Q, K K-major; V MN-major);
// kNCHW = true reads the QKV conv output [B, nh*4*KD, N] directly (Q, K
// MN-major; V K-major), which fuses PsaPackQkv, both V-half runs (one softmax,
// DV = 2*KD), PsaMergeAttn, and optionally PsaExtractV (for the slot whose query
// tile covers a key tile, the S issuer TMA-stores that V tile from its K/V stage).
//
// fp32 storage and maps whose rows TMA cannot address run on CUDA cores
// (attn_simt.cu).
#include <math.h>

#include <algorithm>

#include "attn.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace psa {

namespace {

constexpr float kLn2 = 0.69314718055994530942f;

template <int DQK, int DV, bool kNCHW, int NWG, int QBUF, int ST, bool kSplit>
struct FwdCfg {
  // 64-key tiles keep a whole S row in ~64 registers of its thread; with kSplit
  // two threads share a query row, each owning one 32-key half of every tile
  // with its own running max / sum and its own O accumulator
  static constexpr int BM = 128, BN = 64, STAGES = ST;
  static_assert(ST >= 2 && ST <= 4 && QBUF >= 1 && QBUF <= 2, "buffering");
  static_assert(!kSplit || NWG == 1, "split rows run one slot per CTA");
  static constexpr int H = kSplit ? 2 : 1;  // softmax threads per query row
  static constexpr int HC = BN / H;         // S columns per softmax thread
  static constexpr int kRowThreads = 128 * H;  // softmax threads of a slot
  static constexpr int kSoftmaxWarps = 4 * NWG * H;
  // control warps: TMA producer, S issuer (TMEM owner), P.V issuer, and the store
  // warp that writes the staged output tiles (NCHW) with TMA
  static constexpr int kProducerWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
  static constexpr int kPvWarp = kSoftmaxWarps + 2, kStoreWarp = kSoftmaxWarps + 3;
  static constexpr int kThreads = 32 * kSoftmaxWarps + 128;
  static constexpr uint32_t Q_BYTES = BM * DQK * 2;
  static constexpr uint32_t K_BYTES = BN * DQK * 2;
  static constexpr uint32_t V_BYTES = BN * DV * 2;
  // per-slot shared memory region
  static constexpr uint32_t SL_Q = 0;
  static constexpr uint32_t SL_K = SL_Q + QBUF * Q_BYTES;
  static constexpr uint32_t SL_V = SL_K + STAGES * K_BYTES;
  // split rows: per tile parity, (max, sum) of both halves of every row
  static constexpr uint32_t SL_ML = SL_V + STAGES * V_BYTES;
  // NCHW: the finished O tile (DV channel rows of BM positions, bf16, unswizzled)
  // and its BM LSE values, staged for the store warp's TMA stores
  static constexpr uint32_t SL_OUT = SL_ML + (kSplit ? 2 * 2 * BM * 8 : 0);
  static constexpr uint32_t OUT_BYTES = kNCHW ? DV * BM * 2 : 0;
  static constexpr uint32_t SL_LSE = SL_OUT + OUT_BYTES;
  static constexpr uint32_t SL_BYTES = SL_LSE + (kNCHW ? 1024 : 0);
  static constexpr uint32_t OFF_BAR = NWG * SL_BYTES;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + 512 + 1024;
  // tensor memory per slot w: S (BN columns) at TM_SLOT * w, then H O accumulators
  // (DV columns each; accumulator h sums the P.V products of key half h), then P
  // in two buffers of BN / 2 columns (bf16 pairs)
  static constexpr uint32_t TM_O = BN;
  static constexpr uint32_t TM_P = BN + H * DV;
  static constexpr uint32_t TM_SLOT = (TM_P + BN <= 128) ? 128 : 256;
  static_assert(TM_P + BN <= 256, "tensor memory per slot");
  static_assert(SL_ML % 1024 == 0 && SL_OUT % 1024 == 0 && SL_LSE % 1024 == 0,
                "1024-byte aligned (max, sum) and staging areas");
  static_assert(BM * 4 <= 1024, "LSE staging");
  static constexpr uint32_t TMEM_COLS = NWG * TM_SLOT < 32 ? 32 : NWG * TM_SLOT;
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation");
  static_assert(DQK % 16 == 0 && DV % 32 == 0 && DV <= 128, "tile shape");
  static_assert(SL_BYTES % 1024 == 0, "1024-byte aligned slot regions");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct SlotBars {
  uint64_t q_full[2], q_empty[2], kv_full[4], kv_empty[4];
  uint64_t s_full, s_free, p_full[2], pv_done[2], o_free;  // P / P.V per P buffer
  uint64_t ml_ready;  // split rows: both halves' (max, sum) of the tile are in shared memory
  uint64_t out_full, out_free;  // NCHW: the staged O / LSE tile is written / stored
};

// Loads this thread's NC-column S row from TMEM into registers with a single
// wait (columns >= kend were not written by this tile's MMA and are not loaded).
template <int NC>
__device__ __forceinline__ void load_s_row(uint32_t srow, int kend, uint32_t (&s)[NC]) {
  using Chunk = uint32_t[32];
#pragma unroll
  for (int c = 0; c < NC; c += 32)
    if (c < kend) tmem_load32_async(srow + c, *reinterpret_cast<Chunk*>(s + c));
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < NC; c += 32) tmem_pin(*reinterpret_cast<Chunk*>(s + c));
}

// Online-softmax step of one row held in registers.  Raw scores s (scale sl2 =
// scale*log2(e) > 0; columns past the last valid key hold -inf, so their p is 0)
// become p = 2^(s*sl2 - m) packed as bf16 pairs into the front half of s; m / l
// are the running max (log2 domain) and sum.  Returns the factor the O
// accumulator must be scaled by (1 if the max moved by no more than 2^8, in which
// case the stale max is kept).  Full and partial key tiles run this one code
// path: a separate partial-tile form, taken once per query tile, measured ~5 %
// slower for the whole forward at N = 400.
template <int NC>
__device__ __forceinline__ float softmax_row(uint32_t (&s)[NC], float sl2, bool first,
                                             float& m_run, float& l_run) {
  // two new columns per three-input max, four independent chains
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int c = 0; c < NC; c += 8) {
    m0 = fmax3(m0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    m1 = fmax3(m1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
    m2 = fmax3(m2, __uint_as_float(s[c + 4]), __uint_as_float(s[c + 5]));
    m3 = fmax3(m3, __uint_as_float(s[c + 6]), __uint_as_float(s[c + 7]));
  }
  const float mx = fmax3(m0, m1, fmaxf(m2, m3)) * sl2;
  float alpha = 1.f;
  if (first) {
    m_run = mx;
  } else if (mx > m_run + 8.f) {
    alpha = fast_exp2(m_run - mx);
    m_run = mx;
  }
  // exponent arguments and the running sum two columns at a time (paired FP32
  // instructions: half the issue slots of scalar FMA / add)
  const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(-m_run, -m_run);
  float2 l01 = make_float2(0.f, 0.f), l23 = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < NC; c += 4) {
    const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])),
                                  sl2x2, nm2);
    const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])),
                                  sl2x2, nm2);
    const float2 p01 = make_float2(fast_exp2(x01.x), fast_exp2(x01.y));
    const float2 p23 = make_float2(fast_exp2(x23.x), fast_exp2(x23.y));
    l01 = __fadd2_rn(l01, p01);
    l23 = __fadd2_rn(l23, p23);
    s[c / 2] = pack_bf16x2(p01.x, p01.y);
    s[c / 2 + 1] = pack_bf16x2(p23.x, p23.y);
  }
  l_run = l_run * alpha + ((l01.x + l01.y) + (l23.x + l23.y));
  return alpha;
}

// Head and query tile of tile t: the BH * nfull full 128-row tiles come first,
// then one partial tile per head (when N is not a multiple of 128).
__device__ __forceinline__ void tile_coords(int t, int BH, int nfull, int& bh, int& qt) {
  if (t < BH * nfull) {
    bh = t / nfull;
    qt = t - bh * nfull;
  } else {
    bh = t - BH * nfull;
    qt = nfull;
  }
}

// Tile of slot `slot` in its round i: slot order in even rounds, reverse slot
// order in odd ones.  At N = 400 (1024 tiles on 304 slots, 256 of them 16-row
// partial tiles) no slot then takes three full tiles and a partial one: the
// longest slot holds three full tiles or two full and two partial ones.
__device__ __forceinline__ int slot_tile(int slot, int i, int nslots) {
  return (i & 1) ? (i + 1) * nslots - 1 - slot : i * nslots + slot;
}
// Number of tiles slot `slot` of `nslots` owns out of T.
__device__ __forceinline__ int slot_tiles(int slot, int nslots, int T) {
  const int rounds = T / nslots, rem = T - rounds * nslots;
  const int pos = (rounds & 1) ? nslots - 1 - slot : slot;
  return rounds + (pos < rem ? 1 : 0);
}

// Writes channels [ch, ch + n) of O's row r (query q; live: q < N) of head bh.
// NCHW: into the staging tile (channel rows of 128 positions, bf16) when Out is
// wanted, and Out + V (V read at the query position) straight to out_res when the
// residual output is wanted; raw layout: 16-byte stores of the row.
template <int DQK, int DV, bool kNCHW, int n>
__device__ __forceinline__ void emit_row(const FwdArgs& args, int N, uint32_t stg, int bh, int r,
                                         int q, bool live, int ch, const float (&o)[n]) {
  if (kNCHW) {
    if (args.out) {
#pragma unroll
      for (int e = 0; e < n; ++e) st_shared_bf16(stg + ((ch + e) * 128 + r) * 2, o[e]);
    }
    if (args.out_res && live) {
      const long long orow =
          ((long long)(bh / args.nh) * args.out_ch + (bh % args.nh) * DV + ch) * N + q;
      const __nv_bfloat16* vsrc =
          args.qkv + ((long long)(bh / args.nh) * args.qkv_ch + (bh % args.nh) * 4 * DQK + 2 * DQK + ch) *
                         N + q;
#pragma unroll
      for (int e = 0; e < n; ++e)
        args.out_res[orow + (long long)e * N] =
            __float2bfloat16_rn(o[e] + __bfloat162float(vsrc[(long long)e * N]));
    }
  } else if (live) {
    uint4* dst = reinterpret_cast<uint4*>(args.out + ((long long)bh * N + q) * DV + ch);
#pragma unroll
    for (int e = 0; e < n; e += 8)
      dst[e / 8] = make_uint4(pack_bf16x2(o[e], o[e + 1]), pack_bf16x2(o[e + 2], o[e + 3]),
                              pack_bf16x2(o[e + 4], o[e + 5]), pack_bf16x2(o[e + 6], o[e + 7]));
  }
}

template <int DQK, int DV, bool kNCHW, int NWG, int QBUF, int ST, bool kSplit>
__global__ void __launch_bounds__(128 * NWG * (kSplit ? 2 : 1) + 128, NWG == 1 ? 2 : 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQK,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmOut,
                       const __grid_constant__ CUtensorMap tmVres, const FwdArgs args) {
  using C = FwdCfg<DQK, DV, kNCHW, NWG, QBUF, ST, kSplit>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  SlotBars* bars = reinterpret_cast<SlotBars*>(smem + C::OFF_BAR);
  uint64_t* mma_done = reinterpret_cast<uint64_t*>(bars + NWG);  // one per issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 2);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = args.N;
  const int nkv = (N + C::BN - 1) / C::BN;
  const int nqt = (N + C::BM - 1) / C::BM;
  const int nfull = N / C::BM;  // full query tiles per head
  const int T = args.BH * nqt;
  const int nslots = gridDim.x * NWG;

  if (threadIdx.x == 0) {
    for (int w = 0; w < NWG; ++w) {
      SlotBars& b = bars[w];
      for (int i = 0; i < 2; ++i) {
        mbar_init(&b.q_full[i], 1);
        mbar_init(&b.q_empty[i], 1);
      }
      for (int i = 0; i < C::STAGES; ++i) {
        mbar_init(&b.kv_full[i], 1);
        // K read by S, V by P.V: one commit each; NCHW: and the S issuer's arrival
        // once its PsaExtractV store has read the stage
        mbar_init(&b.kv_empty[i], kNCHW ? 3 : 2);
      }
      mbar_init(&b.s_full, 1);
      mbar_init(&b.s_free, C::kRowThreads);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&b.p_full[i], C::kRowThreads);
        mbar_init(&b.pv_done[i], 1);
      }
      mbar_init(&b.o_free, C::kRowThreads);
      mbar_init(&b.ml_ready, C::kRowThreads);
      mbar_init(&b.out_full, C::kRowThreads);
      mbar_init(&b.out_free, 1);
    }
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
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

  int ntiles[NWG];
  int max_tiles = 0;
#pragma unroll
  for (int w = 0; w < NWG; ++w) {
    ntiles[w] = slot_tiles(blockIdx.x * NWG + w, nslots, T);
    max_tiles = max(max_tiles, ntiles[w]);
  }
  // first channel row of head bh in the 2-D [B * qkv_ch, N] view of the QKV tensor
  auto head_row = [&](int bh) { return (bh / args.nh) * args.qkv_ch + (bh % args.nh) * 4 * DQK; };

  // the control warpgroup (producer, MMA issuer, two idle warps) hands registers
  // to the softmax warpgroups
  if (warp >= C::kSoftmaxWarps) {
  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQK);
      tma_prefetch_desc(&tmV);
      bool ok = true;
      int q_issued[NWG], kv_issued[NWG];
#pragma unroll
      for (int w = 0; w < NWG; ++w) q_issued[w] = kv_issued[w] = 0;
      // Q of tile i goes to buffer i % QBUF; with two buffers, Q of tile i + 1 is
      // fetched right after the first K/V tile of tile i so that it has landed
      // when tile i ends
      auto issue_q = [&](int w, int i) -> bool {
        SlotBars& b = bars[w];
        const int t = slot_tile(blockIdx.x * NWG + w, i, nslots);
        int bh, qt;
        tile_coords(t, args.BH, nfull, bh, qt);
        const int q0 = qt * C::BM;
        const int qb = i % QBUF;
        if (i >= QBUF && !mbar_wait(&b.q_empty[qb], ((i / QBUF) - 1) & 1, abort)) return false;
        mbar_arrive_expect_tx(&b.q_full[qb], C::Q_BYTES);
        load_tile<kNCHW, DQK>(smem + w * C::SL_BYTES + C::SL_Q + qb * C::Q_BYTES, &tmQK,
                              &b.q_full[qb], C::BM, q0, bh, kNCHW ? head_row(bh) : 0);
        q_issued[w] = i + 1;
        return true;
      };
#pragma unroll
      for (int w = 0; w < NWG; ++w)
        if (ok && ntiles[w] > 0) ok = issue_q(w, 0);
      for (int i = 0; ok && i < max_tiles; ++i) {
        if (QBUF == 1 && i > 0) {
#pragma unroll
          for (int w = 0; w < NWG; ++w)
            if (ok && i < ntiles[w]) ok = issue_q(w, i);
        }
        for (int j = 0; ok && j < nkv; ++j) {
#pragma unroll
          for (int w = 0; w < NWG; ++w) {
            if (i >= ntiles[w]) continue;
            SlotBars& b = bars[w];
            const int t = slot_tile(blockIdx.x * NWG + w, i, nslots);
            int bh, qt_unused;
            tile_coords(t, args.BH, nfull, bh, qt_unused);
            const int g = i * nkv + j, st = g % C::STAGES;
            if (g >= C::STAGES && !mbar_wait(&b.kv_empty[st], ((g / C::STAGES) - 1) & 1, abort)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&b.kv_full[st], C::K_BYTES + C::V_BYTES);
            unsigned char* sl = smem + w * C::SL_BYTES;
            const int row = kNCHW ? head_row(bh) : 0;
            load_tile<kNCHW, DQK>(sl + C::SL_K + st * C::K_BYTES, &tmK, &b.kv_full[st], C::BN,
                                  j * C::BN, bh, row + DQK);
            load_tile<kNCHW, DV>(sl + C::SL_V + st * C::V_BYTES, &tmV, &b.kv_full[st], C::BN,
                                 j * C::BN, bh, row + 2 * DQK);
            kv_issued[w] = g + 1;
          }
          if (QBUF == 2 && j == 0) {
#pragma unroll
            for (int w = 0; w < NWG; ++w)
              if (ok && i + 1 < ntiles[w]) ok = issue_q(w, i + 1);
          }
        }
      }
      if (*abort) {
        // let the copies issued last on every buffer land before the CTA exits
#pragma unroll
        for (int w = 0; w < NWG; ++w) {
          for (int i = max(0, q_issued[w] - QBUF); i < q_issued[w]; ++i)
            drain_wait(&bars[w].q_full[i % QBUF], (i / QBUF) & 1);
          for (int g = max(0, kv_issued[w] - C::STAGES); g < kv_issued[w]; ++g)
            drain_wait(&bars[w].kv_full[g % C::STAGES], (g / C::STAGES) & 1);
        }
      }
    }
  } else if (warp == C::kMmaWarp || warp == C::kPvWarp) {
    // ------------------------------------------------------------ MMA issuers
    // S and P.V are issued by two threads: one thread issues at most one
    // tcgen05.mma per ~130 cycles whatever its shape (measured), so S of the next
    // tile does not queue behind the four P.V products of this one.
    if (lane == 0) {
      const bool s_role = warp == C::kMmaWarp;
      // descriptors of buffer 0 / stage 0 of slot 0; the others are fixed offsets
      const uint64_t dQ0 = desc_pos_by_ch<kNCHW>(tile_view<kNCHW, DQK>(sbase + C::SL_Q, C::BM), 0);
      const uint64_t dK0 = desc_pos_by_ch<kNCHW>(tile_view<kNCHW, DQK>(sbase + C::SL_K, C::BN), 0);
      const uint64_t dV0 = desc_ch_by_pos<kNCHW>(tile_view<kNCHW, DV>(sbase + C::SL_V, C::BN), 0);
      constexpr uint64_t kStepQK = kstep_pos_by_ch<kNCHW, DQK>();
      constexpr uint64_t kStepV = kstep_ch_by_pos<kNCHW, DV>();
      const uint32_t idS_full = idesc_bf16_f32(128, C::BN, kNCHW, kNCHW);
      const uint32_t idPV = idesc_bf16_f32(128, DV, false, !kNCHW);
      // query tile and V-slab row of each slot's current tile for the PsaExtractV
      // stores, worked out once per tile (integer divisions off the per-step path)
      int vqt[NWG], vrow0[NWG];
      auto issue_s = [&](int w, int i, int j) -> bool {
        SlotBars& b = bars[w];
        const int k = i * nkv + j;
        if ((j == 0 && !mbar_wait(&b.q_full[i % QBUF], (i / QBUF) & 1, abort)) ||
            !mbar_wait(&b.kv_full[k % C::STAGES], (k / C::STAGES) & 1, abort) ||
            (k >= 1 && !mbar_wait(&b.s_free, (k - 1) & 1, abort)))
          return false;
        tc_fence_after();
        const uint64_t slot_off = (uint64_t)(w * C::SL_BYTES) >> 4;
        const uint64_t dQ = dQ0 + slot_off + (uint64_t)((i % QBUF) * C::Q_BYTES >> 4);
        const uint64_t dK = dK0 + slot_off + (uint64_t)((k % C::STAGES) * C::K_BYTES >> 4);
        const int valid = min(C::BN, N - j * C::BN);
        const uint32_t idS =
            valid == C::BN ? idS_full : idesc_bf16_f32(128, (valid + 15) & ~15, kNCHW, kNCHW);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
          mma_bf16(tmem + w * C::TM_SLOT, dQ + kk * kStepQK, dK + kk * kStepQK, idS,
                   kk > 0 ? 1u : 0u);
        mma_commit(&b.s_full);
        mma_commit(&b.kv_empty[k % C::STAGES]);
        if (j == nkv - 1) mma_commit(&b.q_empty[i % QBUF]);
        if (kNCHW) {
          // PsaExtractV: the slot whose query tile covers key tile j stores V tile j
          // (already in shared memory for P.V) to the NCHW output with TMA; the
          // stage is released once the store has read it
          if (args.vres != nullptr) {
            if (j == 0) {
              int bh, qt;
              tile_coords(slot_tile(blockIdx.x * NWG + w, i, nslots), args.BH, nfull, bh, qt);
              vqt[w] = qt;
              vrow0[w] = (bh / args.nh) * args.vres_ch + (bh % args.nh) * DV;
            }
            if ((j * C::BN) / C::BM == vqt[w]) {
              const unsigned char* vt =
                  smem + w * C::SL_BYTES + C::SL_V + (k % C::STAGES) * C::V_BYTES;
              const int vrow = vrow0[w];
#pragma unroll
              for (int bx = 0; bx < C::BN / 64; ++bx)
                tma_store_2d(&tmVres, vt + bx * (DV * 128), j * C::BN + 64 * bx, vrow);
              bulk_commit();
              bulk_wait_read_all();
            }
          }
          mbar_arrive(&b.kv_empty[k % C::STAGES]);
        }
        return true;
      };
      auto issue_pv = [&](int w, int i, int j) -> bool {
        SlotBars& b = bars[w];
        const int k = i * nkv + j;
        if (!mbar_wait(&b.p_full[k & 1], (k >> 1) & 1, abort) ||
            (j == 0 && i >= 1 && !mbar_wait(&b.o_free, (i - 1) & 1, abort)))
          return false;
        tc_fence_after();
        const uint64_t slot_off = (uint64_t)(w * C::SL_BYTES) >> 4;
        // P of this tile: 8 TMEM columns (16 keys) per k-step
        const uint32_t tP = tmem + w * C::TM_SLOT + C::TM_P + (k & 1) * (C::BN / 2);
        const uint64_t dV = dV0 + slot_off + (uint64_t)((k % C::STAGES) * C::V_BYTES >> 4);
        const uint32_t tO = tmem + w * C::TM_SLOT + C::TM_O;
        const int valid = min(C::BN, N - j * C::BN);
        // k-steps of key half h accumulate into O accumulator h
        constexpr int KH = C::HC / 16;
        if (valid == C::BN) {
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            mma_bf16_ts(tO + (kk / KH) * DV, tP + kk * 8, dV + kk * kStepV, idPV,
                        (j > 0 || kk % KH > 0) ? 1u : 0u);
        } else {
          for (int kk = 0; kk * 16 < valid; ++kk)
            mma_bf16_ts(tO + (kk / KH) * DV, tP + kk * 8, dV + kk * kStepV, idPV,
                        (j > 0 || kk % KH > 0) ? 1u : 0u);
        }
        mma_commit(&b.pv_done[k & 1]);
        mma_commit(&b.kv_empty[k % C::STAGES]);
        return true;
      };
      bool ok = true;
      for (int i = 0; ok && i < max_tiles; ++i)
        for (int j = 0; ok && j < nkv; ++j)
          for (int w = 0; ok && w < NWG; ++w)
            if (i < ntiles[w]) ok = s_role ? issue_s(w, i, j) : issue_pv(w, i, j);
      uint64_t* done = &mma_done[s_role ? 0 : 1];
      mma_commit(done);
      drain_wait(done, 0);  // every MMA retired before TMEM is released
      if (kNCHW && s_role) bulk_wait_all();
    }
  } else if (warp == C::kStoreWarp) {
    // ------------------------------------------------------------ store warp
    // NCHW: once the row threads have staged a finished tile (O rows of BM
    // positions, LSE), one TMA store writes O (positions >= N are clipped) and a
    // bulk copy the LSE of the live rows; the staging area is handed back once the
    // copies have read it.  Row threads thus issue no global stores.
    if (kNCHW && lane == 0) {
      tma_prefetch_desc(&tmOut);
      bool ok = true;
      for (int i = 0; ok && i < max_tiles; ++i)
        for (int w = 0; ok && w < NWG; ++w) {
          if (i >= ntiles[w]) continue;
          SlotBars& b = bars[w];
          if (!mbar_wait(&b.out_full, i & 1, abort)) {
            ok = false;
            break;
          }
          int bh, qt;
          tile_coords(slot_tile(blockIdx.x * NWG + w, i, nslots), args.BH, nfull, bh, qt);
          const int q0 = qt * C::BM;
          const unsigned char* sl = smem + w * C::SL_BYTES;
          if (args.out)
            tma_store_2d(&tmOut, sl + C::SL_OUT, q0,
                         (bh / args.nh) * args.out_ch + (bh % args.nh) * DV);
          if (args.lse)  // N % 8 == 0: a multiple of 32 bytes
            bulk_store(args.lse + (long long)bh * N + q0, sl + C::SL_LSE,
                       (uint32_t)min(C::BM, N - q0) * 4u);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(&b.out_free);
        }
      bulk_wait_all();
    }
  }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int w = kSplit ? 0 : warp >> 2;  // slot
    const int h = kSplit ? warp >> 2 : 0;  // key half of every tile this thread owns
    const int wq = warp & 3;               // TMEM lane quadrant
    const int r = wq * 32 + lane;          // query row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    // S, and the O accumulator of this thread's key half
    const uint32_t tS = tmem + w * C::TM_SLOT, tO = tS + C::TM_O + h * DV;
    const uint32_t sl = sbase + w * C::SL_BYTES;
    SlotBars& b = bars[w];
    const float sl2 = args.scale_log2;
    const int my_tiles = slot_tiles(blockIdx.x * NWG + w, nslots, T);
    bool ok = true;
    // Epilogue of this slot's tile i (m_run / l_run: the running max and sum of
    // this thread's row): O / l and the LSE in natural-log units.  NCHW: the row
    // threads stage both in shared memory for the store warp (no global store on
    // their path); raw layout: 16-byte stores of the thread's own row.  The next
    // tile's first P.V waits for o_free, arrived once O has been read.  (Running
    // it after the next tile's first P hand-off instead measured slower: the
    // next tile's state stays live across it and spills.)
    auto finish_tile = [&](int i, float m_run, float l_run) -> bool {
      int bh, qt;
      tile_coords(slot_tile(blockIdx.x * NWG + w, i, nslots), args.BH, nfull, bh, qt);
      const int q0 = qt * C::BM, q = q0 + r;
      const bool active = wq * 32 < N - q0, live = q < N;
      const int klast = i * nkv + nkv - 1;
      // split rows: the row's (max, sum) go to the other half while the last P.V
      // runs (the exchange area alternates with the tile parity)
      float* ml = reinterpret_cast<float*>(smem + w * C::SL_BYTES + C::SL_ML) + (i & 1) * 512;
      if (kSplit) {
        ml[h * 256 + 2 * r] = m_run;
        ml[h * 256 + 2 * r + 1] = l_run;
        mbar_arrive(&b.ml_ready);
      }
      if (!mbar_wait(&b.pv_done[klast & 1], (klast >> 1) & 1, abort)) return false;
      tc_fence_after();
      // NCHW: the staging area is free once the previous tile's stores have read it
      if (kNCHW && i > 0 && !mbar_wait(&b.out_free, (i - 1) & 1, abort)) return false;
      float lse = 0.f;
      if (kSplit) {
        // both halves' (max, sum) of the row, then this thread writes channels
        // [h * DV/2, (h + 1) * DV/2) of O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / l
        if (!mbar_wait(&b.ml_ready, i & 1, abort)) return false;
        const float m0 = ml[2 * r], l0 = ml[2 * r + 1];
        const float m1 = ml[256 + 2 * r], l1 = ml[256 + 2 * r + 1];
        // a half without any valid key (N <= 32) has l = 0 and an unwritten accumulator
        const float mx = l1 > 0.f ? fmaxf(m0, m1) : m0;
        const float f0 = fast_exp2(m0 - mx), f1 = l1 > 0.f ? fast_exp2(m1 - mx) : 0.f;
        const float l = l0 * f0 + l1 * f1;
        const float c0s = f0 / l, c1s = f1 / l;
        if (active) {
#pragma unroll 1
          for (int c = 0; c < DV / 2; c += 16) {
            const int ch = h * (DV / 2) + c;
            uint32_t a0[16], a1[16];
            tmem_load16_async(tS + C::TM_O + lane_base + ch, a0);
            tmem_load16_async(tS + C::TM_O + DV + lane_base + ch, a1);
            tmem_wait_ld();
            tmem_pin(a0);
            tmem_pin(a1);
            float o[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              o[e] = l1 > 0.f ? __uint_as_float(a0[e]) * c0s + __uint_as_float(a1[e]) * c1s
                              : __uint_as_float(a0[e]) * c0s;
            emit_row<DQK, DV, kNCHW>(args, N, sl + C::SL_OUT, bh, r, q, live, ch, o);
          }
        }
        lse = (mx + log2f(l)) * kLn2;
      } else if (active) {
        const float inv_l = 1.f / l_run;
#pragma unroll 1
        for (int c = 0; c < DV; c += 32) {
          float o[32];
          tmem_load32(tO + lane_base + c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= inv_l;
          emit_row<DQK, DV, kNCHW>(args, N, sl + C::SL_OUT, bh, r, q, live, c, o);
        }
        lse = (m_run + log2f(l_run)) * kLn2;
      }
      tc_fence_before();
      mbar_arrive(&b.o_free);
      if (h == 0 && active && args.lse) {
        if (kNCHW)
          st_shared_f32(sl + C::SL_LSE + r * 4, lse);
        else if (live)
          args.lse[(long long)bh * N + q] = lse;
      }
      if (kNCHW) {
        if (active) fence_proxy_async_smem();  // (only active warps wrote the staging tile)
        mbar_arrive(&b.out_full);
      }
      return true;
    };
    for (int i = 0; ok && i < my_tiles; ++i) {
      const int t = slot_tile(blockIdx.x * NWG + w, i, nslots);
      int bh, qt;
      tile_coords(t, args.BH, nfull, bh, qt);
      const int q0 = qt * C::BM;
      const bool active = wq * 32 < N - q0;  // the warp has live rows
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkv; ++j) {
        const int k = i * nkv + j;
        const int valid = min(C::BN, N - j * C::BN);
        // valid columns of this thread's half, and the columns the products wrote
        const int vh = min(max(valid - h * C::HC, 0), C::HC);
        const int kend = (vh + 15) & ~15;
        if (!mbar_wait(&b.s_full, k & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // this thread's part of the S row goes to registers at once, so the S buffer
        // is handed back to the MMA warp (which starts S_{k+1}) before the
        // exponentials
        uint32_t s[C::HC];
        if (active && kend > 0) load_s_row(tS + lane_base + h * C::HC, kend, s);
        tc_fence_before();
        mbar_arrive(&b.s_free);
        float alpha = 1.f;
        if (active && vh > 0) {
          // a partial tile: the columns past the last valid key (and those the
          // products did not write) become -inf; a half without a valid key has
          // nothing to add
          if (vh < C::HC) {
#pragma unroll
            for (int c = 0; c < C::HC; ++c)
              if (c >= vh) s[c] = 0xff800000u;
          }
          alpha = softmax_row<C::HC>(s, sl2, j == 0, m_run, l_run);
        }
        // P buffer k & 1 was last read by P.V of k - 2
        if (k >= 2 && !mbar_wait(&b.pv_done[k & 1], ((k >> 1) - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (active) {
          // this thread's P (keys >= N already zeroed) into its TMEM lane, beside
          // the other half's
          const uint32_t tP = tS + C::TM_P + (k & 1) * (C::BN / 2) + h * (C::HC / 2) + lane_base;
#pragma unroll
          for (int c = 0; c < C::HC / 2; c += 16) tmem_store16_async(tP + c, s + c);
          tmem_wait_st();
          // O may only be rescaled once every earlier P.V has landed in it
          const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
          if (rescale && !mbar_wait(&b.pv_done[(k - 1) & 1], ((k - 1) >> 1) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (rescale) {
#pragma unroll 1
            for (int c = 0; c < DV; c += 32) {
              float o[32];
              tmem_load32(tO + lane_base + c, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_store32(tO + lane_base + c, o);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&b.p_full[k & 1]);
      }
      if (!ok) break;
      if (!finish_tile(i, m_run, l_run)) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int DQK, int DV, bool kNCHW, int NWG, int QBUF, int ST, bool kSplit>
cudaError_t launch_tc(const CUtensorMap& mQK, const CUtensorMap& mK, const CUtensorMap& mV,
                      const CUtensorMap& mOut, const CUtensorMap& mVres, const FwdArgs& a,
                      cudaStream_t st) {
  using C = FwdCfg<DQK, DV, kNCHW, NWG, QBUF, ST, kSplit>;
  auto kern = attn_fwd_tc_kernel<DQK, DV, kNCHW, NWG, QBUF, ST, kSplit>;
  const cudaError_t attr = set_max_dynamic_smem((const void*)kern, C::SMEM_BYTES);
  if (attr != cudaSuccess) return attr;
  // persistent grid: one CTA per SM with two slots, or two single-slot CTAs per SM
  const long long T = (long long)a.BH * ((a.N + C::BM - 1) / C::BM);
  const long long per_sm = NWG == 1 ? 2 : 1;
  const long long ctas = std::min<long long>(per_sm * device_sm_count(), (T + NWG - 1) / NWG);
  return launch_pdl(kern, dim3((unsigned)ctas), dim3(C::kThreads), C::SMEM_BYTES, st, mQK, mK,
                    mV, mOut, mVres, a);
}

}  // namespace

cudaError_t launch_fa2_fwd_bf16(const CUtensorMap& mQ, const CUtensorMap& mK,
                                const CUtensorMap& mV, const FwdArgs& a, int d,
                                cudaStream_t st) {
  // <DQK, DV, layout, slots per CTA, Q buffers, K/V stages, split rows>: two CTAs
  // per SM, each within half of the SM's shared memory and tensor memory
  // (split rows measured slower on long sequences: the hand-off chain between the
  // row threads and the MMA warp, not the per-row exponentials, sets their pace)
  // (the raw layout stores O from the row threads: the output maps are unused)
  if (d == 32) return launch_tc<32, 32, false, 1, 2, 4, false>(mQ, mK, mV, mV, mV, a, st);
  return launch_tc<64, 64, false, 1, 1, 3, false>(mQ, mK, mV, mV, mV, a, st);
}

cudaError_t launch_psa_fwd_bf16(const CUtensorMap& mQK, const CUtensorMap& mV,
                                const CUtensorMap& mOut, const CUtensorMap& mVres,
                                const FwdArgs& a, int KD, cudaStream_t st) {
  // split rows for the short sequences of vision feature maps (N = 400: 41.7 against
  // 42.7 us), one thread per row beyond (N = 1600: 267 against 291 us)
  if (KD == 32 && a.N <= 512)
    return launch_tc<32, 64, true, 1, 2, 4, true>(mQK, mQK, mV, mOut, mVres, a, st);
  if (KD == 32) return launch_tc<32, 64, true, 1, 2, 4, false>(mQK, mQK, mV, mOut, mVres, a, st);
  // DV = 128: two accumulators would not leave room for a second CTA's tensor memory
  return launch_tc<64, 128, true, 1, 1, 2, false>(mQK, mQK, mV, mOut, mVres, a, st);
}

}  // namespace psa
