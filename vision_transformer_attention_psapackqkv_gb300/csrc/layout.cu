// layout.cu -- PsaPackQkv, PsaExtractV, PsaMergeAttn and their adjoints
// (vision-rs book, page "Custom Kernels", section "Position-Sensitive Attention (PSA)").
//
// All five are pure element permutations, so they move raw bits (T = uint16_t for
// bf16, uint32_t for fp32) and are bit-exact by construction.  Two transposes
// cover four of them:
//   channels_to_rows: a block of KD channels x N positions (NCHW, positions
//     contiguous) -> N rows x KD (row-major, KD contiguous).   pack, unmerge
//   rows_to_channels: the inverse direction.                   unpack, merge
// Each CTA moves a tile of channels x positions through shared memory so that
// both the global loads and the global stores are coalesced: for bf16 with
// 16-byte aligned rows (N % 8 == 0, KD % 8 == 0, every shape the fused kernels
// take) in 16-byte vectors on both sides; otherwise (fp32, or rows that are not
// 16-byte multiples) one element per thread.  ExtractV is a strided copy of
// contiguous per-head slabs in 16-byte vectors.
#include <stdint.h>

#include "attn.cuh"
#include "layout.cuh"
#include "ptx.cuh"

namespace psa {

namespace {

constexpr int kTileN = 64;
constexpr int kThreads = 256;

// One unit = one (b, head, plane s).  Source channel of element d:
//   b * ch_per_batch + head * ch_per_head + s * KD + d   (NCHW side)
// Row-major side: plane pointer rows[s], row (b * nh + head) * N + n.
struct TransposeArgs {
  const void* nchw_src;
  void* nchw_dst;
  const void* rows_src[4];
  void* rows_dst[4];
  int nh, KD, N, planes;
  long long ch_per_batch, ch_per_head;
};

template <typename T>
__global__ void __launch_bounds__(kThreads) channels_to_rows_kernel(TransposeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* tile = reinterpret_cast<T*>(smem_raw);  // [KD][kTileN + 1]
  const int ntiles = (a.N + kTileN - 1) / kTileN;
  const int unit = blockIdx.x / ntiles;
  const int s = unit % a.planes;
  const int bhd = unit / a.planes;  // b * nh + head
  const int head = bhd % a.nh, b = bhd / a.nh;
  const int n0 = (blockIdx.x % ntiles) * kTileN;
  const int nvalid = min(kTileN, a.N - n0);
  const T* src = static_cast<const T*>(a.nchw_src) +
                 ((long long)b * a.ch_per_batch + (long long)head * a.ch_per_head +
                  (long long)s * a.KD) * a.N;
  for (int idx = threadIdx.x; idx < a.KD * kTileN; idx += kThreads) {
    const int d = idx / kTileN, n = idx % kTileN;
    if (n < nvalid) tile[d * (kTileN + 1) + n] = src[(long long)d * a.N + n0 + n];
  }
  __syncthreads();
  T* dst = static_cast<T*>(a.rows_dst[s]) + ((long long)bhd * a.N + n0) * a.KD;
  for (int idx = threadIdx.x; idx < nvalid * a.KD; idx += kThreads) {
    const int n = idx / a.KD, d = idx % a.KD;
    dst[idx] = tile[d * (kTileN + 1) + n];
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) rows_to_channels_kernel(TransposeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* tile = reinterpret_cast<T*>(smem_raw);  // [KD][kTileN + 1]
  const int ntiles = (a.N + kTileN - 1) / kTileN;
  const int unit = blockIdx.x / ntiles;
  const int s = unit % a.planes;
  const int bhd = unit / a.planes;
  const int head = bhd % a.nh, b = bhd / a.nh;
  const int n0 = (blockIdx.x % ntiles) * kTileN;
  const int nvalid = min(kTileN, a.N - n0);
  const T* src = static_cast<const T*>(a.rows_src[s]) + ((long long)bhd * a.N + n0) * a.KD;
  for (int idx = threadIdx.x; idx < nvalid * a.KD; idx += kThreads) {
    const int n = idx / a.KD, d = idx % a.KD;
    tile[d * (kTileN + 1) + n] = src[idx];
  }
  __syncthreads();
  T* dst = static_cast<T*>(a.nchw_dst) +
           ((long long)b * a.ch_per_batch + (long long)head * a.ch_per_head +
            (long long)s * a.KD) * a.N;
  for (int idx = threadIdx.x; idx < a.KD * kTileN; idx += kThreads) {
    const int d = idx / kTileN, n = idx % kTileN;
    if (n < nvalid) dst[(long long)d * a.N + n0 + n] = tile[d * (kTileN + 1) + n];
  }
}

// ---------------------------------------------------------------- 16-byte vectors
// The same two transposes for bf16 when every channel row and every position row
// starts on a 16-byte boundary (N % 8 == 0 and KD % 8 == 0): each CTA moves a tile
// of KD channels x up to 512 positions of one (batch, head, plane); global and
// shared memory are only read and written in 16-byte vectors (8 elements), and
// shared memory holds the tile as 16-byte chunks (chunk (d, c) = channel d,
// positions 8c .. 8c+7), row-major with the chunk index XOR-ed with (d / 8) % 8.
// The position-row side works on 8 x 8 blocks (8 channels x 8 positions per
// thread, transposed in registers with byte permutes): its warp reads or writes
// the chunks (8g + i, c) of 8 c and 4 g per instruction without bank conflicts,
// and in global memory the threads of one c cover whole position rows side by
// side.  The channel-row side moves chunks along the NCHW rows, a warp per row
// and a lane per chunk (up to eight per thread in flight when loading them).
constexpr int kVecTileN = 512;
constexpr int kVecChunks = kVecTileN / 8;  // 16-byte chunks per channel row of the tile

__device__ __forceinline__ int vec_chunk(int d, int c) { return d * kVecChunks + (c ^ ((d >> 3) & 7)); }
constexpr int kWarps = kThreads / 32;
static_assert(kVecChunks == 64, "two 16-byte chunks per lane cover a channel row of the tile");

// Row j of the 8 x 8 transpose of 16-bit elements held as eight 16-byte vectors:
// in[i] holds elements (i, 0..7) (two per 32-bit word, the lower index in the low
// half); the result holds elements (0..7, j).  One byte permute per word: 0x5410
// takes the low halves of its two words, 0x7632 the high halves.
__device__ __forceinline__ uint4 transpose8x8_row(const uint4 (&in)[8], int j) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(in);  // w[4 i + k]
  const int k = j >> 1;
  const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
  return make_uint4(__byte_perm(w[0 * 4 + k], w[1 * 4 + k], sel),
                    __byte_perm(w[2 * 4 + k], w[3 * 4 + k], sel),
                    __byte_perm(w[4 * 4 + k], w[5 * 4 + k], sel),
                    __byte_perm(w[6 * 4 + k], w[7 * 4 + k], sel));
}

// Plane pointer s of four without a local-memory copy of the array.
template <typename P>
__device__ __forceinline__ P plane_ptr(const P (&p)[4], int s) {
  return s == 0 ? p[0] : s == 1 ? p[1] : s == 2 ? p[2] : p[3];
}

__global__ void __launch_bounds__(kThreads, 4) channels_to_rows_vec_kernel(const TransposeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* tile = reinterpret_cast<uint4*>(smem_raw);  // KD x kVecChunks chunks
  // launched with programmatic dependent launch: the next kernel may start its
  // CTAs once every CTA here has begun; this one waits for the previous kernel
  pdl_launch_dependents();
  pdl_wait();
  const int ntiles = (a.N + kVecTileN - 1) / kVecTileN;
  const int unit = blockIdx.x / ntiles;
  const int s = unit % a.planes;
  const int bhd = unit / a.planes;  // b * nh + head
  const int head = bhd % a.nh, b = bhd / a.nh;
  const int n0 = (blockIdx.x % ntiles) * kVecTileN;
  const int nvalid = min(kVecTileN, a.N - n0);
  const int cvalid = nvalid / 8;  // N % 8 == 0, so the tile holds whole chunks
  const uint16_t* src = static_cast<const uint16_t*>(a.nchw_src) +
                        ((long long)b * a.ch_per_batch + (long long)head * a.ch_per_head +
                         (long long)s * a.KD) * a.N + n0;
  // channel rows d = warp + kWarps i, 16-byte chunks c = lane + 32 h of each row
  // (cvalid <= 64): a warp reads 512 contiguous bytes per instruction, eight loads
  // in flight per thread, and no index needs a division
  const int wid = threadIdx.x >> 5, ln = threadIdx.x & 31;
  for (int d0 = wid; d0 < a.KD; d0 += 4 * kWarps) {
    uint4 v[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int d = d0 + i * kWarps, c = ln + 32 * h;
        if (d < a.KD && c < cvalid)
          v[i][h] = __ldg(reinterpret_cast<const uint4*>(src + (long long)d * a.N + 8 * c));
      }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int d = d0 + i * kWarps, c = ln + 32 * h;
        if (d < a.KD && c < cvalid) tile[vec_chunk(d, c)] = v[i][h];
      }
  }
  __syncthreads();
  // one item = channels 8g .. 8g+7 x positions 8c .. 8c+7: eight chunk reads, a
  // register transpose, eight position-row writes (the dvec threads of one c
  // write whole position rows side by side)
  const int dvec = a.KD / 8;
  uint4* dst = reinterpret_cast<uint4*>(plane_ptr(a.rows_dst, s)) +
               ((long long)bhd * a.N + n0) * dvec;
  const int nitems = dvec * cvalid;
  // item idx -> (c, g) = (idx / dvec, idx % dvec); dvec = KD / 8 is a power of two
  // for every power-of-two key_dim, where a shift replaces the division
  const bool pow2 = (dvec & (dvec - 1)) == 0;
  const int lg = 31 - __clz(dvec);
  for (int idx = threadIdx.x; idx < nitems; idx += kThreads) {
    const int c = pow2 ? idx >> lg : idx / dvec, g = idx - c * dvec;
    uint4 in[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) in[i] = tile[vec_chunk(8 * g + i, c)];
#pragma unroll
    for (int j = 0; j < 8; ++j) dst[(long long)(8 * c + j) * dvec + g] = transpose8x8_row(in, j);
  }
}

__global__ void __launch_bounds__(kThreads, 4) rows_to_channels_vec_kernel(const TransposeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint4* tile = reinterpret_cast<uint4*>(smem_raw);
  pdl_launch_dependents();  // (programmatic dependent launch, as above)
  pdl_wait();
  const int ntiles = (a.N + kVecTileN - 1) / kVecTileN;
  const int unit = blockIdx.x / ntiles;
  const int s = unit % a.planes;
  const int bhd = unit / a.planes;
  const int head = bhd % a.nh, b = bhd / a.nh;
  const int n0 = (blockIdx.x % ntiles) * kVecTileN;
  const int nvalid = min(kVecTileN, a.N - n0);
  const int cvalid = nvalid / 8;
  const int dvec = a.KD / 8;
  const uint4* src = reinterpret_cast<const uint4*>(plane_ptr(a.rows_src, s)) +
                     ((long long)bhd * a.N + n0) * dvec;
  // one item = positions 8c .. 8c+7 x channels 8g .. 8g+7: eight position-row
  // reads (eight in flight), a register transpose, eight chunk writes
  const int nitems = dvec * cvalid;
  const bool pow2 = (dvec & (dvec - 1)) == 0;  // (as in the other direction)
  const int lg = 31 - __clz(dvec);
  for (int idx = threadIdx.x; idx < nitems; idx += kThreads) {
    const int c = pow2 ? idx >> lg : idx / dvec, g = idx - c * dvec;
    uint4 in[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) in[j] = __ldg(src + (long long)(8 * c + j) * dvec + g);
#pragma unroll
    for (int i = 0; i < 8; ++i) tile[vec_chunk(8 * g + i, c)] = transpose8x8_row(in, i);
  }
  __syncthreads();
  uint16_t* dst = static_cast<uint16_t*>(a.nchw_dst) +
                  ((long long)b * a.ch_per_batch + (long long)head * a.ch_per_head +
                   (long long)s * a.KD) * a.N + n0;
  // channel rows d = warp + kWarps i, chunks c = lane + 32 h (as the loads of the
  // other direction)
  const int wid = threadIdx.x >> 5, ln = threadIdx.x & 31;
  for (int d = wid; d < a.KD; d += kWarps)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = ln + 32 * h;
      if (c < cvalid) *reinterpret_cast<uint4*>(dst + (long long)d * a.N + 8 * c) = tile[vec_chunk(d, c)];
    }
}

// Copies `slabs` contiguous slabs of slab_vec 16-byte vectors from src (slab
// stride src_stride_vec) to dst (slab stride dst_stride_vec).
__global__ void __launch_bounds__(kThreads)
    strided_slab_copy_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                             long long slabs, long long slab_vec, long long src_stride_vec,
                             long long dst_stride_vec) {
  pdl_launch_dependents();  // (programmatic dependent launch)
  pdl_wait();
  const long long total = slabs * slab_vec;
  for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < total;
       i += (long long)gridDim.x * kThreads) {
    const long long sl = i / slab_vec, e = i % slab_vec;
    dst[sl * dst_stride_vec + e] = src[sl * src_stride_vec + e];
  }
}

template <typename T>
cudaError_t launch_transpose(bool to_rows, const TransposeArgs& a, int B, cudaStream_t st) {
  // one CTA per (64-position tile, unit); the flat index stays below 2^31 for
  // every shape the entry points accept
  const long long tiles = (long long)((a.N + kTileN - 1) / kTileN) * B * a.nh * a.planes;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  dim3 grid((unsigned)tiles);
  const size_t smem = (size_t)a.KD * (kTileN + 1) * sizeof(T);
  if (to_rows)
    channels_to_rows_kernel<T><<<grid, kThreads, smem, st>>>(a);
  else
    rows_to_channels_kernel<T><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t transpose(bool to_rows, const TransposeArgs& a, int B, int elem_bytes,
                      cudaStream_t st) {
  if (elem_bytes == 2 && a.N % 8 == 0 && a.KD % 8 == 0) {
    // bf16 with 16-byte aligned channel and position rows: 16-byte vectors
    const long long tiles =
        (long long)((a.N + kVecTileN - 1) / kVecTileN) * B * a.nh * a.planes;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)a.KD * kVecTileN * 2;  // up to 128 KB (KD = 128)
    const cudaError_t attr = set_max_dynamic_smem(
        to_rows ? (const void*)channels_to_rows_vec_kernel : (const void*)rows_to_channels_vec_kernel,
        128 * kVecTileN * 2);  // the largest tile (key_dim 128), set once per device
    if (attr != cudaSuccess) return attr;
    return to_rows ? launch_pdl(channels_to_rows_vec_kernel, dim3((unsigned)tiles), dim3(kThreads),
                                smem, st, a)
                   : launch_pdl(rows_to_channels_vec_kernel, dim3((unsigned)tiles), dim3(kThreads),
                                smem, st, a);
  }
  return elem_bytes == 2 ? launch_transpose<uint16_t>(to_rows, a, B, st)
                         : launch_transpose<uint32_t>(to_rows, a, B, st);
}

}  // namespace

cudaError_t launch_pack_qkv(const void* qkv, void* packed, int B, int nh, int KD, int N,
                            int elem_bytes, cudaStream_t st) {
  TransposeArgs a{};
  a.nchw_src = qkv;
  const long long plane = (long long)B * nh * N * KD * elem_bytes;
  for (int s = 0; s < 4; ++s) a.rows_dst[s] = static_cast<char*>(packed) + s * plane;
  a.nh = nh; a.KD = KD; a.N = N; a.planes = 4;
  a.ch_per_batch = (long long)nh * 4 * KD;
  a.ch_per_head = 4 * KD;
  return transpose(true, a, B, elem_bytes, st);
}

cudaError_t launch_unpack_qkv(const void* packed, void* qkv, int B, int nh, int KD, int N,
                              int elem_bytes, cudaStream_t st) {
  TransposeArgs a{};
  a.nchw_dst = qkv;
  const long long plane = (long long)B * nh * N * KD * elem_bytes;
  for (int s = 0; s < 4; ++s) a.rows_src[s] = static_cast<const char*>(packed) + s * plane;
  a.nh = nh; a.KD = KD; a.N = N; a.planes = 4;
  a.ch_per_batch = (long long)nh * 4 * KD;
  a.ch_per_head = 4 * KD;
  return transpose(false, a, B, elem_bytes, st);
}

cudaError_t launch_merge_attn(const void* o_lo, const void* o_hi, void* out, int B, int nh,
                              int KD, int N, int elem_bytes, cudaStream_t st) {
  TransposeArgs a{};
  a.nchw_dst = out;
  a.rows_src[0] = o_lo;
  a.rows_src[1] = o_hi;
  a.nh = nh; a.KD = KD; a.N = N; a.planes = 2;
  a.ch_per_batch = (long long)nh * 2 * KD;
  a.ch_per_head = 2 * KD;
  return transpose(false, a, B, elem_bytes, st);
}

cudaError_t launch_unmerge_attn(const void* dout, void* do_lo, void* do_hi, int B, int nh,
                                int KD, int N, int elem_bytes, cudaStream_t st) {
  TransposeArgs a{};
  a.nchw_src = dout;
  a.rows_dst[0] = do_lo;
  a.rows_dst[1] = do_hi;
  a.nh = nh; a.KD = KD; a.N = N; a.planes = 2;
  a.ch_per_batch = (long long)nh * 2 * KD;
  a.ch_per_head = 2 * KD;
  return transpose(true, a, B, elem_bytes, st);
}

cudaError_t launch_extract_v(const void* qkv, void* v, int B, int nh, int KD, int N,
                             int elem_bytes, cudaStream_t st) {
  // Per head the V section is 2*KD consecutive channels, i.e. one contiguous slab
  // of 2*KD*N elements; slabs repeat every 4*KD*N elements in qkv and every
  // 2*KD*N elements in v.  Callers guarantee 2*KD*N*elem_bytes % 16 == 0.
  const long long slab_bytes = 2LL * KD * N * elem_bytes;
  const long long slab_vec = slab_bytes / 16;
  const long long slabs = (long long)B * nh;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(qkv) + slab_bytes);
  const long long total = slabs * slab_vec;
  long long blocks = (total + kThreads - 1) / kThreads;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (blocks < 1) blocks = 1;
  return launch_pdl(strided_slab_copy_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, st, src,
                    static_cast<uint4*>(v), slabs, slab_vec, 2 * slab_vec, slab_vec);
}

}  // namespace psa
