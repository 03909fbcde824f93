// layout.cuh -- launchers of the PSA layout kernels (element permutations).
#pragma once
#include <cuda_runtime.h>

namespace psa {

cudaError_t launch_pack_qkv(const void* qkv, void* packed, int B, int nh, int KD, int N,
                            int elem_bytes, cudaStream_t st);
cudaError_t launch_unpack_qkv(const void* packed, void* qkv, int B, int nh, int KD, int N,
                              int elem_bytes, cudaStream_t st);
cudaError_t launch_merge_attn(const void* o_lo, const void* o_hi, void* out, int B, int nh,
                              int KD, int N, int elem_bytes, cudaStream_t st);
cudaError_t launch_unmerge_attn(const void* dout, void* do_lo, void* do_hi, int B, int nh,
                                int KD, int N, int elem_bytes, cudaStream_t st);
cudaError_t launch_extract_v(const void* qkv, void* v, int B, int nh, int KD, int N,
                             int elem_bytes, cudaStream_t st);

}  // namespace psa
