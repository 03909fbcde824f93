// qkv_conv.cu -- the QKV 1x1 convolution that produces the NCHW tensor PsaPackQkv
// (and the fused PSA forward) reads (vision-rs book, page "Custom Kernels", section
// "Position-Sensitive Attention (PSA)": PsaPackQkv takes a QKV conv's NCHW
// output):  qkv[b, o, n] = bias[o] + sum_c w[o, c] x[b, c, n].
//
// Per batch item this is the dense product W [cout x cin] . X_b [cin x N], so it
// runs on the tensor cores: a persistent kernel, one CTA per SM, walks output
// tiles of 128 output channels x 128 positions of one batch item.  Up to 512
// input channels (and two or more tiles per CTA) a weight-resident form below
// keeps each CTA's 128 W rows in shared memory; the general form streams W
// with X:
//   warp 4     TMA producer: per 64-channel K block, the W block (128 rows of 64
//              input channels, K-major, 128-byte swizzle) and the X block (two
//              boxes of 64 positions x 64 channel rows straight from NCHW: the
//              MN-major B operand) into a 4-stage ring;
//   warp 5     MMA issuer (one thread) and TMEM owner: 128 x 128 x 16 products
//              into one of two fp32 accumulators (128 columns each), so the next
//              tile's products run while the previous tile is written out;
//   warps 0-3  epilogue: thread = output channel (TMEM lane); adds the bias,
//              rounds to bf16 once and writes 8 positions per 16-byte store.
// Positions beyond N and input channels beyond cin read as zeros (TMA fill); the
// epilogue writes only real rows and positions.  Every wait is bounded, as in the
// attention kernels.
//
// Shapes the tensor maps cannot address (cin or N not a multiple of 8, i.e.
// rows that are not 16-byte multiples) run a CUDA-core kernel with fp32
// accumulation instead.
#include <cuda_bf16.h>

#include <algorithm>

#include "attn.cuh"
#include "ptx.cuh"

namespace psa {

namespace {

constexpr int kBM = 128, kBN = 128, kBK = 64, kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;       // 16 KB
constexpr uint32_t kBBytes = kBK * kBN * 2;       // 16 KB (two 64-position boxes)
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kOffBar = kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
constexpr int kThreads = 192;

struct ConvBars {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_free[2], mma_done;
};

struct TileCoord {
  int b, nt, mt;
};

// Tiles numbered with the output-channel tile fastest, so the CTAs working at the
// same time share the X block of one batch item and position tile in L2.
__device__ __forceinline__ TileCoord tile_coord(int t, int nmt, int nnt) {
  TileCoord c;
  c.mt = t % nmt;
  const int r = t / nmt;
  c.nt = r % nnt;
  c.b = r / nnt;
  return c;
}

__global__ void __launch_bounds__(kThreads, 1)
    qkv_conv_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const ConvArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  ConvBars& bar = *reinterpret_cast<ConvBars*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(&bar + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nmt = (a.cout + kBM - 1) / kBM, nnt = (a.N + kBN - 1) / kBN;
  const int nkb = (a.cin + kBK - 1) / kBK;
  const int T = a.B * nmt * nnt;
  const int ntiles = (int)blockIdx.x < T ? (T - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar.full[i], 1);
      mbar_init(&bar.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.acc_full[i], 1);
      mbar_init(&bar.acc_free[i], 128);
    }
    mbar_init(&bar.mma_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      int g = 0;
      bool ok = true;
      for (int i = 0; ok && i < ntiles; ++i) {
        const TileCoord c = tile_coord((int)blockIdx.x + i * (int)gridDim.x, nmt, nnt);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int st = g % kStages;
          if (g >= kStages && !mbar_wait(&bar.empty[st], ((g / kStages) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          unsigned char* stage = smem + st * kStageBytes;
          mbar_arrive_expect_tx(&bar.full[st], kStageBytes);
          tma_load_2d(stage, &tmW, &bar.full[st], kb * kBK, c.mt * kBM);
          tma_load_3d(stage + kABytes, &tmX, &bar.full[st], c.nt * kBN, kb * kBK, c.b);
          tma_load_3d(stage + kABytes + kBBytes / 2, &tmX, &bar.full[st], c.nt * kBN + 64, kb * kBK,
                      c.b);
        }
      }
      if (*abort)
        for (int j = std::max(0, g - kStages); j < g; ++j)
          drain_wait(&bar.full[j % kStages], (j / kStages) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // A = W block (128 rows of 64 channels, K-major); B = X block (64 channel
      // rows of 64-position boxes: positions x channels, MN-major)
      const uint64_t dA0 = desc_kmajor(SmemTile{sbase, 128, kBM}, 0);
      const uint64_t dB0 = desc_mnmajor(SmemTile{sbase + kABytes, 128, kBK}, 0);
      constexpr uint64_t kStepA = 32 >> 4, kStepB = (16 * 128) >> 4;
      const uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, true);
      int g = 0;
      bool ok = true;
      for (int i = 0; ok && i < ntiles; ++i) {
        const int ab = i & 1;
        if (i >= 2 && !mbar_wait(&bar.acc_free[ab], ((i >> 1) - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int st = g % kStages;
          if (!mbar_wait(&bar.full[st], (g / kStages) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t so = (uint64_t)(st * kStageBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16(tmem + ab * kBN, dA0 + so + kk * kStepA, dB0 + so + kk * kStepB, idesc,
                     (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&bar.empty[st]);
        }
        if (ok) mma_commit(&bar.acc_full[ab]);
      }
      mma_commit(&bar.mma_done);
      drain_wait(&bar.mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int r = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int i = 0; i < ntiles; ++i) {
      const int ab = i & 1;
      const TileCoord c = tile_coord((int)blockIdx.x + i * (int)gridDim.x, nmt, nnt);
      if (!mbar_wait(&bar.acc_full[ab], (i >> 1) & 1, abort)) break;
      tc_fence_after();
      const int o = c.mt * kBM + r;
      const bool live = o < a.cout;
      const float bias = (live && a.bias) ? a.bias[o] : 0.f;
      __nv_bfloat16* dst = a.out + ((long long)c.b * a.cout + o) * a.N + c.nt * kBN;
#pragma unroll 1
      for (int col = 0; col < kBN; col += 32) {
        float acc[32];
        tmem_load32(tmem + ab * kBN + lane_base + col, acc);
        if (!live) continue;
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          if (c.nt * kBN + col + e < a.N)  // N % 8 == 0: whole groups of 8
            *reinterpret_cast<uint4*>(dst + col + e) = make_uint4(
                pack_bf16x2(acc[e] + bias, acc[e + 1] + bias),
                pack_bf16x2(acc[e + 2] + bias, acc[e + 3] + bias),
                pack_bf16x2(acc[e + 4] + bias, acc[e + 5] + bias),
                pack_bf16x2(acc[e + 6] + bias, acc[e + 7] + bias));
        }
      }
      tc_fence_before();
      mbar_arrive(&bar.acc_free[ab]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// Weight-resident form (cin <= kWresMaxCin): the CTAs form nmt groups, group m
// computes every (batch item, position tile) of output-channel tile m, and each
// of its CTAs loads that tile's W rows once (128 x cin, K-major, one 16 KB
// block per 64 input channels) and keeps them in shared memory, so per output
// tile only the X blocks stream through the ring: half the L2-to-SM traffic of
// the form above, which reloads W for every tile.
constexpr int kWresMaxCin = 512;
constexpr uint32_t kXStageBytes = kBBytes;  // one 64-channel X block per stage
constexpr int kXStages = 4;
constexpr uint32_t kStgBytes = kBM * kBN * 2;  // 32 KB: two boxes of 128 rows x 128 bytes

template <bool kTmaStore>
__global__ void __launch_bounds__(kThreads, 1)
    qkv_conv_wres_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmOut, const ConvArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = align1024(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  const int nmt = (a.cout + kBM - 1) / kBM, nnt = (a.N + kBN - 1) / kBN;
  const int nkb = (a.cin + kBK - 1) / kBK;
  const uint32_t w_bytes = (uint32_t)nkb * kABytes;
  // the finished tile is staged (two 64-position boxes of 128 channel rows, 128-byte
  // swizzle) and written by TMA stores: a thread's own stores would each hit 32
  // channel rows with 16 bytes of a 32-byte sector
  const uint32_t off_x = w_bytes, off_stg = off_x + kXStages * kXStageBytes;
  const uint32_t off_bar = off_stg + (kTmaStore ? kStgBytes : 0);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + off_bar);
  uint64_t* empty = full + kXStages;
  uint64_t* acc_full = empty + kXStages;
  uint64_t* acc_free = acc_full + 2;
  uint64_t* w_full = acc_free + 2;  // W block kb landed (kWresMaxCin / kBK of them)
  uint64_t* stg_full = w_full + kWresMaxCin / kBK;  // the epilogue threads staged a tile
  uint64_t* stg_free = stg_full + 1;  // its stores have read the staging area
  uint64_t* mma_done = stg_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // group mt = blockIdx % nmt; its G CTAs take the (batch, position tile) pairs
  // p = gi, gi + G, ...
  const int G = (int)gridDim.x / nmt;
  const int mt = (int)blockIdx.x % nmt, gi = (int)blockIdx.x / nmt;
  const int P = a.B * nnt;
  const int ntiles = gi < P ? (P - gi + G - 1) / G : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kXStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], 128);
    }
    for (int kb = 0; kb < kWresMaxCin / kBK; ++kb) mbar_init(&w_full[kb], 1);
    mbar_init(stg_full, 128);
    mbar_init(stg_free, 1);
    mbar_init(mma_done, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmW);
      tma_prefetch_desc(&tmX);
      if (ntiles > 0) {
        for (int kb = 0; kb < nkb; ++kb) {
          mbar_arrive_expect_tx(&w_full[kb], kABytes);
          tma_load_2d(smem + kb * kABytes, &tmW, &w_full[kb], kb * kBK, mt * kBM);
        }
      }
      int g = 0;
      bool ok = true;
      for (int i = 0; ok && i < ntiles; ++i) {
        const int p = gi + i * G, b = p / nnt, nt = p - b * nnt;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int st = g % kXStages;
          if (g >= kXStages && !mbar_wait(&empty[st], ((g / kXStages) - 1) & 1, abort)) {
            ok = false;
            break;
          }
          unsigned char* stage = smem + off_x + st * kXStageBytes;
          mbar_arrive_expect_tx(&full[st], kXStageBytes);
          tma_load_3d(stage, &tmX, &full[st], nt * kBN, kb * kBK, b);
          tma_load_3d(stage + kXStageBytes / 2, &tmX, &full[st], nt * kBN + 64, kb * kBK, b);
        }
      }
      if (*abort) {
        if (ntiles > 0)
          for (int kb = 0; kb < nkb; ++kb) drain_wait(&w_full[kb], 0);
        for (int j = std::max(0, g - kXStages); j < g; ++j)
          drain_wait(&full[j % kXStages], (j / kXStages) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t dA0 = desc_kmajor(SmemTile{sbase, 128, kBM}, 0);
      const uint64_t dB0 = desc_mnmajor(SmemTile{sbase + off_x, 128, kBK}, 0);
      constexpr uint64_t kStepA = 32 >> 4, kStepB = (16 * 128) >> 4;
      const uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, true);
      int g = 0;
      bool ok = true;
      for (int i = 0; ok && i < ntiles; ++i) {
        const int ab = i & 1;
        if (i >= 2 && !mbar_wait(&acc_free[ab], ((i >> 1) - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int st = g % kXStages;
          if ((i == 0 && !mbar_wait(&w_full[kb], 0, abort)) ||
              !mbar_wait(&full[st], (g / kXStages) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ao = (uint64_t)(kb * kABytes) >> 4;
          const uint64_t bo = (uint64_t)(st * kXStageBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16(tmem + ab * kBN, dA0 + ao + kk * kStepA, dB0 + bo + kk * kStepB, idesc,
                     (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[st]);
        }
        if (ok) mma_commit(&acc_full[ab]);
      }
      mma_commit(mma_done);
      drain_wait(mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue warps
    const int r = warp * 32 + lane;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int o = mt * kBM + r;
    const bool live = o < a.cout;
    const float bias = (live && a.bias) ? a.bias[o] : 0.f;
    if constexpr (!kTmaStore) {
      for (int i = 0; i < ntiles; ++i) {
        const int ab = i & 1;
        const int p = gi + i * G, b = p / nnt, nt = p - b * nnt;
        if (!mbar_wait(&acc_full[ab], (i >> 1) & 1, abort)) break;
        tc_fence_after();
        __nv_bfloat16* dst = a.out + ((long long)b * a.cout + o) * a.N + nt * kBN;
#pragma unroll 1
        for (int col = 0; col < kBN; col += 32) {
          float acc[32];
          tmem_load32(tmem + ab * kBN + lane_base + col, acc);
          if (!live) continue;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            if (nt * kBN + col + e < a.N)  // N % 8 == 0: whole groups of 8
              *reinterpret_cast<uint4*>(dst + col + e) = make_uint4(
                  pack_bf16x2(acc[e] + bias, acc[e + 1] + bias),
                  pack_bf16x2(acc[e + 2] + bias, acc[e + 3] + bias),
                  pack_bf16x2(acc[e + 4] + bias, acc[e + 5] + bias),
                  pack_bf16x2(acc[e + 6] + bias, acc[e + 7] + bias));
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_free[ab]);
      }
    } else {
      const uint32_t stg = sbase + off_stg;
      bool ok = true;
      for (int i = 0; ok && i < ntiles; ++i) {
        const int ab = i & 1;
        const int p = gi + i * G, b = p / nnt, nt = p - b * nnt;
        if (!mbar_wait(&acc_full[ab], (i >> 1) & 1, abort)) break;
        if (i >= 1 && !mbar_wait(stg_free, (i - 1) & 1, abort)) break;
        tc_fence_after();
#pragma unroll 1
        for (int col = 0; col < kBN; col += 32) {
          float acc[32];
          tmem_load32(tmem + ab * kBN + lane_base + col, acc);
          // row r of box col / 64, 16-byte chunks (col % 64) / 8 .. + 3, swizzled
          const uint32_t row = stg + (col >> 6) * (kStgBytes / 2) + r * 128;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            const uint32_t chunk = ((col & 63) + e) >> 3;
            st_shared_v4(row + ((chunk ^ (r & 7)) << 4), pack_bf16x2(acc[e] + bias, acc[e + 1] + bias),
                         pack_bf16x2(acc[e + 2] + bias, acc[e + 3] + bias),
                         pack_bf16x2(acc[e + 4] + bias, acc[e + 5] + bias),
                         pack_bf16x2(acc[e + 6] + bias, acc[e + 7] + bias));
          }
        }
        tc_fence_before();
        mbar_arrive(&acc_free[ab]);
        fence_proxy_async_smem();
        mbar_arrive(stg_full);
        if (threadIdx.x == 0) {
          // rows >= cout and positions >= N fall outside the tensor and are dropped
          ok = mbar_wait(stg_full, i & 1, abort);
          if (ok) {
            const int x0 = nt * kBN;
            tma_store_3d(&tmOut, smem + off_stg, x0, mt * kBM, b);
            if (x0 + 64 < a.N) tma_store_3d(&tmOut, smem + off_stg + kStgBytes / 2, x0 + 64, mt * kBM, b);
            bulk_commit();
            bulk_wait_read_all();
            mbar_arrive(stg_free);
          }
        }
      }
      if (threadIdx.x == 0) bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// CUDA cores, any shape: one thread per output position of one output channel.
__global__ void __launch_bounds__(128) qkv_conv_simt_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const __nv_bfloat16* __restrict__ w,
                                                           const ConvArgs a) {
  const int n = blockIdx.x * 128 + threadIdx.x, o = blockIdx.y, b = blockIdx.z;
  if (n >= a.N) return;
  float acc = a.bias ? a.bias[o] : 0.f;
  const __nv_bfloat16* xb = x + (long long)b * a.cin * a.N + n;
  const __nv_bfloat16* wo = w + (long long)o * a.cin;
  for (int c = 0; c < a.cin; ++c)
    acc = fmaf(__bfloat162float(wo[c]), __bfloat162float(xb[(long long)c * a.N]), acc);
  a.out[((long long)b * a.cout + o) * a.N + n] = __float2bfloat16_rn(acc);
}

}  // namespace

cudaError_t launch_qkv_conv_tc(const CUtensorMap& mW, const CUtensorMap& mX,
                               const CUtensorMap& mOut, const ConvArgs& a, cudaStream_t st) {
  const cudaError_t attr = set_max_dynamic_smem((const void*)qkv_conv_tc_kernel, kSmemBytes);
  if (attr != cudaSuccess) return attr;
  const long long T = (long long)a.B * ((a.cout + kBM - 1) / kBM) * ((a.N + kBN - 1) / kBN);
  if (T <= 0 || T > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int sms = device_sm_count();
  const int nmt = (a.cout + kBM - 1) / kBM;
  const long long P = (long long)a.B * ((a.N + kBN - 1) / kBN);  // tiles per channel tile
  if (a.cin <= kWresMaxCin && nmt <= sms && P >= 2LL * (sms / nmt)) {
    // nmt groups of G CTAs, two or more tiles per CTA (a CTA with a single tile
    // gains nothing from keeping W); up to 256 input channels the tile leaves
    // through TMA stores (with 512 that measured slower than the threads' own
    // stores)
    const int G = sms / nmt;
    const int nkb = (a.cin + kBK - 1) / kBK;
    const bool tma_store = a.cin <= 256;
    const uint32_t smem = (uint32_t)nkb * kABytes + kXStages * kXStageBytes +
                          (tma_store ? kStgBytes : 0) + 256 + 1024;
    // (the attribute is set once per device: the largest W this form takes)
    constexpr uint32_t kMaxSmem =
        (kWresMaxCin / kBK) * kABytes + kXStages * kXStageBytes + kStgBytes + 256 + 1024;
    static_assert(kMaxSmem <= 227 * 1024, "shared memory");
    auto kern = tma_store ? qkv_conv_wres_kernel<true> : qkv_conv_wres_kernel<false>;
    const cudaError_t wattr = set_max_dynamic_smem((const void*)kern, kMaxSmem);
    if (wattr != cudaSuccess) return wattr;
    return launch_pdl(kern, dim3(G * nmt), dim3(kThreads), smem, st, mW, mX, mOut, a);
  }
  const int ctas = (int)std::min<long long>(sms, T);
  return launch_pdl(qkv_conv_tc_kernel, dim3(ctas), dim3(kThreads), kSmemBytes, st, mW, mX, a);
}

cudaError_t launch_qkv_conv_simt(const void* x, const void* w, const ConvArgs& a, cudaStream_t st) {
  if (a.cout > 65535 || a.B > 65535) return cudaErrorInvalidValue;
  const dim3 grid((a.N + 127) / 128, a.cout, a.B);
  qkv_conv_simt_kernel<<<grid, 128, 0, st>>>(static_cast<const __nv_bfloat16*>(x),
                                             static_cast<const __nv_bfloat16*>(w), a);
  return cudaGetLastError();
}

}  // namespace psa
