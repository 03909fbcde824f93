"""psa_attention_fwd_residual: the PSA forward with its residual path fused into
the epilogue, Out + V (vision-rs book, page "Custom Kernels", section
"Position-Sensitive Attention (PSA)": PsaExtractV pulls the V section out in NCHW
for the residual path), against the oracle's out + V; and its backward, which is
psa_attention_bwd with dvres = dOut.  Out + V reaches magnitudes above 4, where
rounding to bf16 alone moves a value by more than 1.5e-2, so the bf16 per-element
bar there is 1.5e-2 + 2^-8 |ref| (mean-relative 3e-3 as everywhere)."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import psa_inputs, storage_to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("with_out", [False, True])
@pytest.mark.parametrize("Bn,nh,KD,H,W,dtype", [
    (2, 2, 32, 20, 20, "bf16"),   # two threads per query row
    (1, 2, 32, 24, 24, "bf16"),   # one thread per query row
    (2, 1, 64, 12, 12, "bf16"),   # key_dim 64
    (1, 2, 32, 8, 8, "f32"),      # fp32
])
def test_residual_forward_and_backward(oracle, with_out, Bn, nh, KD, H, W, dtype):
    import torch

    scale = 1 / math.sqrt(KD)
    ins = psa_inputs(Bn, nh, KD, H, W, dtype, seed=90 + H * W, with_grad=True)
    qkv = to_device(ins["qkv"], dtype)
    shape = B.shape_of(qkv, nh, KD)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out_res = torch.full((Bn, nh * 2 * KD, H, W), float("nan"), dtype=tdt, device="cuda")
    out = torch.empty_like(out_res) if with_out else None
    lse = torch.empty((Bn * nh, H * W), dtype=torch.float32, device="cuda") if with_out else None
    B.psa_attention_fwd_residual(qkv, out_res, out, lse, shape, scale)
    torch.cuda.synchronize()
    q64 = storage_to_f64(ins["qkv"], dtype)
    ref_res, ref_lse = oracle.psa_fwd_residual(q64, nh, KD, scale)
    assert_close(to_host_f64(out_res), ref_res, dtype, "out + V", output_rounding=dtype == "bf16")
    if not with_out:
        return
    ref_out, _, _ = oracle.psa_fwd(q64, nh, KD, scale)
    assert_close(to_host_f64(out), ref_out, dtype, "out")
    np.testing.assert_allclose(to_host_f64(lse), ref_lse, atol=1e-4 if dtype == "f32" else 2e-3, rtol=0)
    if dtype != "bf16":
        return
    # backward of out + V: psa_attention_bwd with dvres = dOut
    dout = to_device(ins["dout"], dtype)
    ws = torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    dqkv = torch.empty_like(qkv)
    B.psa_attention_bwd(qkv, out, dout, lse, dout, dqkv, ws, shape, scale)
    torch.cuda.synchronize()
    d64 = storage_to_f64(ins["dout"], dtype)
    ref = oracle.psa_bwd(q64, d64, nh, KD, scale, dvres=d64).reshape(Bn, nh, 4, KD, -1)
    got = to_host_f64(dqkv).reshape(Bn, nh, 4, KD, -1)
    for s, name in enumerate(("dQ", "dK", "dV_lo", "dV_hi")):
        assert_close(got[:, :, s], ref[:, :, s], "bf16", "residual " + name, output_rounding=s >= 2)
