/*
 * psa.h -- C ABI of the GB300 (sm_103a) Position-Sensitive Attention library
 * (libpsa_gb300.so).
 *
 * The operations are those of the vision-rs book, page "Custom Kernels":
 *   section "Flash Attention 2"  -- softmax attention over [BATCH*N_HEADS, N_CTX,
 *     HEAD_DIM] tensors with an online softmax (the N x N matrix is never stored);
 *     the forward, the dQ backward and the dK/dV backward are separate kernels.
 *   section "Position-Sensitive Attention (PSA)" -- PsaPackQkv, PsaExtractV and
 *     PsaMergeAttn around Flash Attention 2, which PSA runs once per V half
 *     (V_lo, V_hi) with HEAD_DIM = KEY_DIM.
 *
 * Notation: KD = key_dim, nh = num_heads, N = H*W, BH = B*nh, qkv_h = nh*4*KD,
 * c = nh*2*KD.  Spatial index n = h*W + w; head-batch index bh = b*nh + head.
 * Per head, QKV channels are [Q | K | V_lo | V_hi], each KD wide: channel
 * head*4*KD + s*KD + d holds element d of plane s (0=Q, 1=K, 2=V_lo, 3=V_hi).
 * The merged output channel head*2*KD + t*KD + d holds element d of half t.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers to dense, contiguous buffers owned
 *     by the caller; the library never allocates, frees or synchronises, and
 *     every call is ordered on the given stream.  Pointers must be 16-byte
 *     aligned (PSA_ERR_ALIGNMENT otherwise).
 *   - Arguments come in the order inputs, outputs, workspace, sizes, stream.
 *   - Validation is host-side and happens before any launch: a NULL required
 *     pointer or a non-positive size gives PSA_ERR_INVALID_ARG; a size the
 *     kernels do not implement gives PSA_ERR_UNSUPPORTED; a failed launch gives
 *     PSA_ERR_CUDA.  Nothing is printed and nothing exits.
 *   - Element types: bf16 (PSA_DTYPE_BF16; fp32 accumulation, softmax
 *     probabilities rounded to bf16 before the P.V product, outputs rounded to
 *     nearest-even) or fp32 (PSA_DTYPE_F32; forward only, fp32 arithmetic).
 *     Log-sum-exp and delta arrays are always fp32.
 *   - Kernels that wait on on-chip barriers give up after a bounded time and
 *     record PSA_ERR_TIMEOUT in a device-side error word that
 *     psa_get_last_device_error() reads and clears.
 *   - The attention kernels are launched with programmatic stream
 *     serialization: their CTAs may start their set-up while the previous
 *     kernel of the stream is finishing, but they read and write no global
 *     memory before that kernel has completed, so results are exactly those of
 *     plain stream order.
 */
#ifndef PSA_GB300_H
#define PSA_GB300_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PSA_OK = 0,
    PSA_ERR_INVALID_ARG = 1,
    PSA_ERR_UNSUPPORTED = 2,
    PSA_ERR_ALIGNMENT = 3,
    PSA_ERR_CUDA = 4,
    PSA_ERR_TIMEOUT = 5
} psa_status_t;

typedef enum { PSA_DTYPE_F32 = 0, PSA_DTYPE_BF16 = 1 } psa_dtype_t;

/* One PSA problem: QKV conv output [B, nh*4*KD, H, W] of the given element type. */
typedef struct {
    int B, num_heads, key_dim, H, W;
    psa_dtype_t dtype;
} psa_shape_t;

/* ---- QKV convolution ---------------------------------------------------------- */

/* The QKV 1x1 convolution whose NCHW output PsaPackQkv and the fused PSA forward
 * read ("Custom Kernels", section "Position-Sensitive Attention (PSA)": PsaPackQkv
 * takes a QKV conv's NCHW output): qkv[b, o, n] = bias[o] + sum_c w[o, c] x[b, c, n]
 * for x_nchw [B, cin, H, W], weight [cout, cin] (row-major), bias [cout] fp32
 * (NULL: none) and qkv_nchw [B, cout, H, W]; bf16 storage, fp32 accumulation,
 * outputs rounded once.  On the tensor cores when cin and H*W are multiples of 8,
 * on CUDA cores otherwise.  Pointers 16-byte aligned (bias 4-byte);
 * PSA_ERR_INVALID_ARG for a NULL required pointer or a non-positive size. */
psa_status_t psa_qkv_conv(const void *x_nchw, const void *weight, const float *bias,
                          void *qkv_nchw, int B, int cin, int cout, int H, int W,
                          cudaStream_t stream);

/* ---- layout kernels (bit-exact element copies) ------------------------------ */

/* PsaPackQkv ("Custom Kernels", section "Position-Sensitive Attention (PSA)"):
 * qkv_nchw [B, qkv_h, H, W] -> packed [4, BH, N, KD] (planes Q, K, V_lo, V_hi).
 * Both dtypes; key_dim up to 128 for all layout kernels. */
psa_status_t psa_pack_qkv(const void *qkv_nchw, void *packed, psa_shape_t shape,
                          cudaStream_t stream);

/* Inverse permutation of psa_pack_qkv (the adjoint the backward needs):
 * packed [4, BH, N, KD] -> qkv_nchw [B, qkv_h, H, W]. */
psa_status_t psa_unpack_qkv(const void *packed, void *qkv_nchw, psa_shape_t shape,
                            cudaStream_t stream);

/* PsaExtractV (same section): the V section [V_lo | V_hi] of every head, as NCHW
 * v_nchw [B, c, H, W] (v_nchw[b, head*2KD + j, n] = qkv[b, head*4KD + 2KD + j, n]). */
psa_status_t psa_extract_v(const void *qkv_nchw, void *v_nchw, psa_shape_t shape,
                           cudaStream_t stream);

/* PsaMergeAttn (same section): o_lo, o_hi [BH, N, KD] -> out_nchw [B, c, H, W]. */
psa_status_t psa_merge_attn(const void *o_lo, const void *o_hi, void *out_nchw,
                            psa_shape_t shape, cudaStream_t stream);

/* Inverse of psa_merge_attn (the adjoint the backward needs):
 * dout_nchw [B, c, H, W] -> do_lo, do_hi [BH, N, KD]. */
psa_status_t psa_unmerge_attn(const void *dout_nchw, void *do_lo, void *do_hi,
                              psa_shape_t shape, cudaStream_t stream);

/* ---- Flash Attention 2 on [BH, N, HEAD_DIM] ("Flash Attention 2" section) ---- */

/* Forward: o = softmax(scale * q k^T) v, lse = log-sum-exp of each score row
 * (natural log, fp32 [BH, n_ctx]; lse may be NULL).  q, k, v, o are
 * [BH, n_ctx, head_dim] of dtype; head_dim in {32, 64} (PSA_ERR_UNSUPPORTED
 * otherwise).  Non-causal, no mask. */
psa_status_t flash_attn2_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                             int BH, int n_ctx, int head_dim, float scale, psa_dtype_t dtype,
                             cudaStream_t stream);

/* dQ backward: writes delta[bh, i] = sum_c do[bh, i, c] * o[bh, i, c] (fp32
 * [BH, n_ctx], caller-owned) and dq = scale * dS k with dS = P o (dP - delta),
 * P = exp(scale q k^T - lse), dP = do v^T.  lse is the forward's.  bf16 only.
 * Must run before flash_attn2_bwd_dkdv, which reads delta. */
psa_status_t flash_attn2_bwd_dq(const void *q, const void *k, const void *v, const void *o,
                                const void *do_, const float *lse, float *delta, void *dq,
                                int BH, int n_ctx, int head_dim, float scale, psa_dtype_t dtype,
                                cudaStream_t stream);

/* dK/dV backward: dv = P^T do, dk = scale * dS^T q, with delta from
 * flash_attn2_bwd_dq.  bf16 only.  dk, dv are overwritten. */
psa_status_t flash_attn2_bwd_dkdv(const void *q, const void *k, const void *v, const void *do_,
                                  const float *lse, const float *delta, void *dk, void *dv,
                                  int BH, int n_ctx, int head_dim, float scale,
                                  psa_dtype_t dtype, cudaStream_t stream);

/* ---- fused PSA reading and writing NCHW directly ----------------------------- */

/* Forward of the whole PSA attention step: pack, attention over both V halves
 * with one shared softmax (identical to two HEAD_DIM = KD runs), merge; writes
 * out_nchw [B, c, H, W], lse [BH, N] fp32 (nullable) and, when v_nchw is not
 * NULL, the PsaExtractV output [B, c, H, W].  key_dim in {32, 64};
 * N*sizeof(dtype) must be a multiple of 16 (PSA_ERR_ALIGNMENT otherwise);
 * bf16, or fp32 (computed in fp32). */
psa_status_t psa_attention_fwd(const void *qkv_nchw, void *out_nchw, float *lse, void *v_nchw,
                               psa_shape_t shape, float scale, cudaStream_t stream);

/* The same forward with the residual path fused into its epilogue
 * ("Custom Kernels", section "Position-Sensitive Attention (PSA)": PsaExtractV
 * pulls the V section out in NCHW for the residual path, which adds it to the
 * merged attention output): writes out_res [B, c, H, W] = Out + V, each element
 * rounded once, where V is the PsaExtractV output; also writes the plain attention
 * output out and lse [BH, N] when they are not NULL.  The backward of out_res is
 * psa_attention_bwd with dvres_nchw = dout_nchw (the residual adds the upstream
 * gradient into the V channels); it needs out, so callers that train pass out here.
 * Same sizes, dtypes and errors as psa_attention_fwd (out_res is required). */
psa_status_t psa_attention_fwd_residual(const void *qkv_nchw, void *out_res_nchw, void *out_nchw,
                                        float *lse, psa_shape_t shape, float scale,
                                        cudaStream_t stream);

/* Backward of psa_attention_fwd: given qkv, the forward's out and lse, the
 * upstream gradient dout [B, c, H, W] and optionally the gradient dvres of the
 * extracted V (nullable), writes dqkv_nchw [B, qkv_h, H, W] (overwritten, V
 * channels include dvres).  workspace is device memory, 16-byte aligned, of
 * ws_bytes >= psa_attention_bwd_workspace_size(shape) bytes.  Which kernels run:
 *   - key_dim 32, bf16, N <= 512: one kernel per head computes delta on chip and
 *     forms every P and dS once; the workspace is not touched;
 *   - key_dim 32, bf16, 512 < N <= 2048, with the full workspace: the same kernel,
 *     with the dQ accumulator in the workspace;
 *   - otherwise (key_dim 64, longer N, or a workspace of only B*num_heads*N*4
 *     bytes rounded up to 256, the least accepted): the dQ and dK/dV kernels of
 *     the two-kernel form, with delta in the workspace;
 *   - fp32, or rows that are not 16-byte multiples: CUDA-core dQ and dK/dV.
 * key_dim 32 or 64; bf16 or fp32. */
psa_status_t psa_attention_bwd(const void *qkv_nchw, const void *out_nchw, const void *dout_nchw,
                               const float *lse, const void *dvres_nchw, void *dqkv_nchw,
                               void *workspace, size_t ws_bytes, psa_shape_t shape, float scale,
                               cudaStream_t stream);

/* The two kernels psa_attention_bwd runs, for callers that schedule them
 * separately ("Flash Attention 2" section: the dQ and dK/dV backward are separate
 * kernels with their own grids).  psa_attention_bwd_dq writes the Q channels of
 * dqkv_nchw and delta [BH, N] fp32 (rowsum of dOut o Out per head and position);
 * psa_attention_bwd_dkdv then reads delta and writes the K and V channels (V
 * channels include dvres when it is not NULL).  It must run after
 * psa_attention_bwd_dq on the same stream.  Same sizes and errors as
 * psa_attention_bwd. */
psa_status_t psa_attention_bwd_dq(const void *qkv_nchw, const void *out_nchw,
                                  const void *dout_nchw, const float *lse, float *delta,
                                  void *dqkv_nchw, psa_shape_t shape, float scale,
                                  cudaStream_t stream);
psa_status_t psa_attention_bwd_dkdv(const void *qkv_nchw, const void *dout_nchw,
                                    const float *lse, const float *delta,
                                    const void *dvres_nchw, void *dqkv_nchw, psa_shape_t shape,
                                    float scale, cudaStream_t stream);

/* psa_attention_bwd for callers that cannot allocate device memory when they run
 * the backward (for example a plugin whose host framework owns all device
 * allocations, or a latency-critical loop where cudaMalloc / cudaFree would
 * synchronise the device).  The pages have no counterpart: this is a
 * convenience of this library.  Same arguments and results as
 * psa_attention_bwd, minus the workspace.  The delta scratch lives in a fixed
 * 4 MiB array inside the library's device memory, which every GPU that loads the
 * library keeps until the process exits; B * num_heads * H * W may not exceed
 * 1048576.  Errors are checked in this order: a NULL required pointer or an
 * invalid shape (PSA_ERR_INVALID_ARG), then that limit (PSA_ERR_UNSUPPORTED),
 * then every other check of psa_attention_bwd.  The first call on each device,
 * made with that device current, looks up the array's address; make that first
 * call before any stream capture.  The array serves as the workspace of
 * psa_attention_bwd: it holds delta for the two-kernel form (key_dim 64, fp32,
 * rows that are not 16-byte multiples, or N > 2048), or the dQ accumulator of the
 * one-kernel form for key_dim 32 and 512 < N <= 2048 when B * num_heads * N * 32
 * floats fit in it (the two-kernel form otherwise); the one-kernel form for
 * N <= 512 keeps everything on chip and leaves it untouched.  All calls that use
 * the array share it: such calls whose kernels overlap on the GPU (other
 * streams, other threads) race on it, so serialise them.  Nothing in the array
 * needs clearing between calls (each call writes every value it reads before it
 * reads it).  No allocation of any kind is made. */
psa_status_t psa_attention_bwd_noalloc(const void *qkv_nchw, const void *out_nchw,
                                       const void *dout_nchw, const float *lse,
                                       const void *dvres_nchw, void *dqkv_nchw, psa_shape_t shape,
                                       float scale, cudaStream_t stream);

/* Bytes of device workspace for psa_attention_bwd to take its fastest form (0 for
 * an invalid shape): B*num_heads*N*4 rounded up to 256 (delta), or, for key_dim 32
 * and 512 < N <= 2048, B*num_heads*N*32*4 rounded up to 256 (a dQ accumulator). */
size_t psa_attention_bwd_workspace_size(psa_shape_t shape);

/* ---- status ------------------------------------------------------------------- */

/* Static description of a status code. */
const char *psa_status_string(psa_status_t status);

/* Synchronises the stream, then reads and clears the device-side error word
 * (PSA_ERR_TIMEOUT after a bounded on-chip wait gave up; PSA_OK otherwise). */
psa_status_t psa_get_last_device_error(cudaStream_t stream);

/* Diagnostic of the failure path (no counterpart on the pages): launches one warp
 * that waits, through the same bounded on-chip wait as the attention kernels but
 * with a limit of limit_ns nanoseconds (1 .. 100,000,000), on a barrier that
 * nothing arrives at.  The wait gives up, records PSA_ERR_TIMEOUT in the device
 * error word (read it with psa_get_last_device_error) and the kernel returns; the
 * context stays usable.  PSA_ERR_INVALID_ARG for a limit outside that range. */
psa_status_t psa_debug_wait_timeout(unsigned long long limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PSA_GB300_H */
