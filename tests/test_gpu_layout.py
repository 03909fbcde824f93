"""PsaPackQkv / PsaExtractV / PsaMergeAttn and their adjoints on the GPU, bit-exact
against the oracle's element copies (vision-rs book, page "Custom Kernels",
section "Position-Sensitive Attention (PSA)")."""
import numpy as np
import pytest

from helpers import to_device, to_host_bits
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import psa_inputs

pytestmark = pytest.mark.gpu

SHAPES = [
    # (B, nh, KD, H, W, dtype)
    (1, 2, 32, 8, 8, "f32"),       # psa_fwd_f32_n64
    (16, 4, 32, 20, 20, "bf16"),   # psa_fwd_n400
    (32, 8, 32, 40, 40, "bf16"),   # psa_fwdbwd_n1600
    (2, 3, 8, 5, 7, "bf16"),       # ragged: N = 35, tiles of 64 leave a tail
    (3, 1, 64, 1, 1, "f32"),       # a single position
    (1, 2, 16, 9, 15, "f32"),      # N = 135
    # 16-byte vector path (bf16, N % 8 == 0, KD % 8 == 0): tiles of 512 positions
    (1, 2, 64, 12, 12, "bf16"),    # key_dim 64, one partial tile
    (1, 1, 128, 16, 40, "bf16"),   # key_dim 128, N = 640: a full tile and a partial one
    (2, 3, 8, 4, 6, "bf16"),       # key_dim 8, N = 24
    (1, 1, 16, 8, 129, "bf16"),    # N = 1032: two full tiles and one chunk of 8
]


@pytest.mark.parametrize("Bn,nh,KD,H,W,dtype", SHAPES)
def test_layout_kernels_bit_exact(oracle, Bn, nh, KD, H, W, dtype):
    import torch

    qkv_h = psa_inputs(Bn, nh, KD, H, W, dtype, seed=11, with_grad=False)["qkv"]
    qkv = to_device(qkv_h, dtype)
    shape = B.shape_of(qkv, nh, KD)
    N, BH = H * W, Bn * nh

    packed = torch.empty((4, BH, N, KD), dtype=qkv.dtype, device="cuda")
    B.psa_pack_qkv(qkv, packed, shape)
    ref_packed = oracle.pack_qkv(qkv_h, nh, KD)
    np.testing.assert_array_equal(to_host_bits(packed), ref_packed.view(to_host_bits(packed).dtype))

    back = torch.empty_like(qkv)
    B.psa_unpack_qkv(packed, back, shape)
    np.testing.assert_array_equal(to_host_bits(back), to_host_bits(qkv))

    if (2 * KD * N * qkv.element_size()) % 16 == 0:
        v = torch.empty((Bn, nh * 2 * KD, H, W), dtype=qkv.dtype, device="cuda")
        B.psa_extract_v(qkv, v, shape)
        ref_v = oracle.extract_v(qkv_h, nh, KD)
        np.testing.assert_array_equal(to_host_bits(v), ref_v.view(to_host_bits(v).dtype))

    out = torch.empty((Bn, nh * 2 * KD, H, W), dtype=qkv.dtype, device="cuda")
    B.psa_merge_attn(packed[2], packed[3], out, shape)
    ref_out = oracle.merge_attn(ref_packed[2], ref_packed[3], Bn, nh, KD, H, W)
    np.testing.assert_array_equal(to_host_bits(out), ref_out.view(to_host_bits(out).dtype))

    lo = torch.empty((BH, N, KD), dtype=qkv.dtype, device="cuda")
    hi = torch.empty_like(lo)
    B.psa_unmerge_attn(out, lo, hi, shape)
    ref_lo, ref_hi = oracle.unmerge_attn(ref_out, nh, KD)
    np.testing.assert_array_equal(to_host_bits(lo), ref_lo.view(to_host_bits(lo).dtype))
    np.testing.assert_array_equal(to_host_bits(hi), ref_hi.view(to_host_bits(hi).dtype))
    torch.cuda.synchronize()
