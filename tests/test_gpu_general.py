"""General shapes through the fused entry points (vision-rs book, page "Custom
Kernels", sections "Flash Attention 2" and "Position-Sensitive Attention (PSA)"):
feature maps whose channel rows are not 16-byte multiples (N * 2 % 16 != 0: 7 x 7,
5 x 7, 13 x 13, 25 x 25, which no TMA tensor map can address) and fp32 storage in
the backward, both of which run on CUDA cores; each against the fp64 oracle at the
usual bars (bf16: max-abs 1.5e-2, mean-relative 3e-3; fp32: max-abs 1e-4)."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import fa2_inputs, psa_inputs, storage_to_f64

pytestmark = pytest.mark.gpu


def run_fused(ins, nh, KD, dtype, scale, dvres):
    import torch

    qkv = to_device(ins["qkv"], dtype)
    Bn, C, H, W = qkv.shape
    shape = B.shape_of(qkv, nh, KD)
    out = torch.empty((Bn, nh * 2 * KD, H, W), dtype=qkv.dtype, device="cuda")
    lse = torch.empty((Bn * nh, H * W), dtype=torch.float32, device="cuda")
    v = torch.empty_like(out)
    B.psa_attention_fwd(qkv, out, lse, v, shape, scale)
    dout = to_device(ins["dout"], dtype)
    dv = to_device(ins["dvres"], dtype) if dvres else None
    ws = torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    dqkv = torch.full_like(qkv, float("nan"))
    B.psa_attention_bwd(qkv, out, dout, lse, dv, dqkv, ws, shape, scale)
    torch.cuda.synchronize()
    assert B.psa_get_last_device_error() == 0
    return out, lse, v, dqkv


@pytest.mark.parametrize("Bn,nh,KD,H,W,dtype", [
    (2, 2, 32, 7, 7, "bf16"),      # 224-pixel input at stride 32
    (1, 3, 64, 5, 7, "bf16"),
    (1, 2, 32, 13, 13, "bf16"),    # 416-pixel input
    (1, 1, 32, 25, 25, "bf16"),    # N = 625
    (1, 2, 32, 8, 8, "f32"),       # the fp32 configuration, now with its backward
    (2, 1, 64, 5, 7, "f32"),
    (1, 2, 32, 7, 7, "f32"),
])
def test_fused_general_shapes(oracle, Bn, nh, KD, H, W, dtype):
    scale = 1 / math.sqrt(KD)
    ins = psa_inputs(Bn, nh, KD, H, W, dtype, seed=700 + H * W, with_dvres=True)
    out, lse, v, dqkv = run_fused(ins, nh, KD, dtype, scale, dvres=True)
    q64 = storage_to_f64(ins["qkv"], dtype)
    ref_out, ref_lse, ref_v = oracle.psa_fwd(q64, nh, KD, scale)
    assert_close(to_host_f64(out), ref_out, dtype, "out")
    np.testing.assert_allclose(to_host_f64(lse), ref_lse, atol=1e-4 if dtype == "f32" else 2e-3, rtol=0)
    np.testing.assert_array_equal(to_host_f64(v), ref_v)
    ref = oracle.psa_bwd(q64, storage_to_f64(ins["dout"], dtype), nh, KD, scale,
                         dvres=storage_to_f64(ins["dvres"], dtype)).reshape(Bn, nh, 4, KD, -1)
    got = to_host_f64(dqkv).reshape(Bn, nh, 4, KD, -1)
    for s, name in enumerate(("dQ", "dK", "dV_lo", "dV_hi")):
        assert_close(got[:, :, s], ref[:, :, s], dtype, name, output_rounding=dtype == "bf16" and s >= 2)


def test_residual_on_unaligned_map(oracle):
    import torch

    Bn, nh, KD, H, W = 2, 2, 32, 7, 7
    scale = 1 / math.sqrt(KD)
    ins = psa_inputs(Bn, nh, KD, H, W, "bf16", seed=777, with_grad=False)
    qkv = to_device(ins["qkv"], "bf16")
    out_res = torch.empty((Bn, nh * 2 * KD, H, W), dtype=torch.bfloat16, device="cuda")
    B.psa_attention_fwd_residual(qkv, out_res, None, None, B.shape_of(qkv, nh, KD), scale)
    torch.cuda.synchronize()
    ref, _ = oracle.psa_fwd_residual(storage_to_f64(ins["qkv"], "bf16"), nh, KD, scale)
    assert_close(to_host_f64(out_res), ref, "bf16", "out + V", output_rounding=True)


@pytest.mark.parametrize("BH,N,d", [(2, 100, 32), (3, 257, 64), (1, 1, 32)])
def test_fa2_fp32_backward(oracle, BH, N, d):
    import torch

    ins = fa2_inputs(BH, N, d, "f32", seed=800 + N)
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (to_device(ins[n], "f32") for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((BH, N), dtype=torch.float32, device="cuda")
    B.flash_attn2_fwd(q, k, v, o, lse, scale)
    delta = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B.flash_attn2_bwd_dq(q, k, v, o, do, lse, delta, dq, scale)
    B.flash_attn2_bwd_dkdv(q, k, v, do, lse, delta, dk, dv, scale)
    torch.cuda.synchronize()
    ref_dq, ref_dk, ref_dv = oracle.attn_bwd(ins["q"], ins["k"], ins["v"], ins["do"], scale)
    assert_close(to_host_f64(dq), ref_dq, "f32", "dQ")
    assert_close(to_host_f64(dk), ref_dk, "f32", "dK")
    assert_close(to_host_f64(dv), ref_dv, "f32", "dV")
