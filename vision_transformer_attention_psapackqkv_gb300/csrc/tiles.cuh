// tiles.cuh -- how the attention kernels move operand tiles: TMA loads of
// sequence tiles in either layout, the shared-memory view of a loaded tile, and the
// tcgen05 descriptor of that view for either operand orientation.
//
// Raw layout [BH, N, D]: one 3-D box {D, rows, 1}: `rows` rows of D bf16 (D*2
//   bytes, swizzle of the same width).
// NCHW layout [B, channels, N]: rows/64 boxes {64 positions, D channels}: D rows
//   of 128 bytes per box, 128-byte swizzle, boxes D*128 bytes apart.
#pragma once

#include "ptx.cuh"

namespace psa {

template <bool kNCHW, int D>
__device__ __forceinline__ void load_tile(unsigned char* dst, const CUtensorMap* map,
                                          uint64_t* bar, int rows_tile, int pos0, int bh,
                                          int ch) {
  if (kNCHW) {
    for (int b = 0; b < rows_tile / 64; ++b)
      tma_load_2d(dst + b * (D * 128), map, bar, pos0 + 64 * b, ch);
  } else {
    tma_load_3d(dst, map, bar, 0, pos0, bh);
  }
}

template <bool kNCHW, int D>
__device__ __forceinline__ SmemTile tile_view(uint32_t base, int rows_tile) {
  return kNCHW ? SmemTile{base, 128u, (uint32_t)D}
               : SmemTile{base, (uint32_t)(2 * D), (uint32_t)rows_tile};
}

// Operand whose M/N runs over sequence positions and whose K runs over the D channels.
template <bool kNCHW>
__device__ __forceinline__ uint64_t desc_pos_by_ch(const SmemTile& t, int k) {
  return kNCHW ? desc_mnmajor(t, k) : desc_kmajor(t, k);
}
// Operand whose N runs over the D channels and whose K runs over sequence positions.
template <bool kNCHW>
__device__ __forceinline__ uint64_t desc_ch_by_pos(const SmemTile& t, int k) {
  return kNCHW ? desc_kmajor(t, k) : desc_mnmajor(t, k);
}

// Amount to add to a descriptor (in its 16-byte address units) per 16-element K
// step, for the two orientations above.  Valid while the steps stay inside one
// 64-position box (tiles of at most 64 positions along K):
//   positions x channels, K = channels: NCHW steps 16 channel rows of 128 bytes;
//     raw steps 32 bytes along a row;
//   channels x positions, K = positions: NCHW steps 32 bytes along a row; raw
//     steps 16 position rows of 2*D bytes.
template <bool kNCHW, int D>
constexpr uint64_t kstep_pos_by_ch() {
  return kNCHW ? (16 * 128) >> 4 : 32 >> 4;
}
template <bool kNCHW, int D>
constexpr uint64_t kstep_ch_by_pos() {
  return kNCHW ? 32 >> 4 : (16 * 2 * D) >> 4;
}

// Loads a 64-column S row and the matching dP row (TMEM columns tS, tP) with
// one wait; columns >= kend were not written and are not loaded.
__device__ __forceinline__ void load_sp_rows(uint32_t tS, uint32_t tP, int kend,
                                             uint32_t (&s)[64], uint32_t (&p)[64]) {
  using Chunk = uint32_t[32];
  tmem_load32_async(tS, *reinterpret_cast<Chunk*>(s));
  tmem_load32_async(tP, *reinterpret_cast<Chunk*>(p));
  if (kend > 32) {
    tmem_load32_async(tS + 32, *reinterpret_cast<Chunk*>(s + 32));
    tmem_load32_async(tP + 32, *reinterpret_cast<Chunk*>(p + 32));
  }
  tmem_wait_ld();
  tmem_pin(*reinterpret_cast<Chunk*>(s));
  tmem_pin(*reinterpret_cast<Chunk*>(p));
  tmem_pin(*reinterpret_cast<Chunk*>(s + 32));
  tmem_pin(*reinterpret_cast<Chunk*>(p + 32));
}

// Stores 8 packed bf16x2 words per 16-byte chunk of a 128-row, 64-column K-major
// tile with the 128-byte swizzle (row r, chunks below kend / 8).
__device__ __forceinline__ void store_row64(uint32_t tile, int r, int kend, const uint32_t* w) {
#pragma unroll
  for (int ch = 0; ch < 8; ++ch)
    if (ch * 8 < kend)
      st_shared_v4(tile + swizzled_offset(r, ch, 128), w[ch * 4], w[ch * 4 + 1], w[ch * 4 + 2],
                   w[ch * 4 + 3]);
}

}  // namespace psa
