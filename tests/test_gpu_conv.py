"""psa_qkv_conv, the QKV 1x1 convolution whose NCHW output PsaPackQkv and the fused
PSA forward read (vision-rs book, page "Custom Kernels", section
"Position-Sensitive Attention (PSA)": PsaPackQkv takes a QKV conv's NCHW output),
against the oracle's fp64 convolution; then the conv output fed straight into the
fused PSA forward, against the oracle's attention of the same input.  Outputs
reach magnitudes above 4, where rounding to bf16 alone moves a value by more than
1.5e-2, so the per-element bar is 1.5e-2 + 2^-8 |ref| (mean-relative 3e-3)."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import bf16_to_f64, conv_inputs, f32_to_bf16

pytestmark = pytest.mark.gpu


def run_conv(ins):
    import torch

    x, w = to_device(ins["x"], "bf16"), to_device(ins["w"], "bf16")
    bias = None if ins["bias"] is None else torch.from_numpy(ins["bias"]).cuda()
    Bn, cin, H, W = x.shape
    out = torch.full((Bn, w.shape[0], H, W), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.psa_qkv_conv(x, w, bias, out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("Bn,cin,cout,H,W,bias", [
    (2, 256, 512, 20, 20, True),   # the psa_fwdbwd_n400 block's QKV conv, two batch items
    (1, 512, 1024, 8, 8, True),    # the N = 1600 block's channel counts, a small map
    (3, 72, 200, 9, 8, True),      # partial K block, partial output-channel and position tiles
    (1, 64, 64, 16, 16, False),    # no bias
    (2, 20, 48, 6, 6, True),       # cin % 8 != 0: CUDA cores
    (1, 64, 128, 7, 7, True),      # N = 49: CUDA cores
    # enough tiles for two or more per CTA on 152 SMs: the weight-resident form
    (20, 256, 512, 20, 20, True),  # tiles written by TMA stores (cin <= 256)
    (76, 72, 200, 9, 16, True),    # the same with partial K, channel and position tiles
    (10, 512, 1024, 20, 20, True), # 512 input channels: the threads' own stores
    (152, 328, 136, 8, 10, False), # the same with partial tiles, no bias
])
def test_qkv_conv(oracle, Bn, cin, cout, H, W, bias):
    ins = conv_inputs(Bn, cin, cout, H, W, seed=cin + cout + H, with_bias=bias)
    out = run_conv(ins)
    ref = oracle.qkv_conv(bf16_to_f64(ins["x"]), bf16_to_f64(ins["w"]),
                          None if ins["bias"] is None else ins["bias"].astype(np.float64))
    assert_close(to_host_f64(out), ref, "bf16", "qkv", output_rounding=True)


def test_conv_feeds_the_fused_forward(oracle):
    """x -> QKV conv -> fused PSA forward, all on the GPU, against the oracle's
    attention of the oracle's conv output (rounded to bf16, the storage the
    attention reads)."""
    import torch

    Bn, nh, KD, H, W = 2, 4, 32, 20, 20
    c = nh * 2 * KD
    ins = conv_inputs(Bn, c, nh * 4 * KD, H, W, seed=5)
    qkv = run_conv(ins)
    out = torch.empty((Bn, c, H, W), dtype=torch.bfloat16, device="cuda")
    scale = 1 / math.sqrt(KD)
    B.psa_attention_fwd(qkv, out, None, None, B.shape_of(qkv, nh, KD), scale)
    torch.cuda.synchronize()
    ref_qkv = oracle.qkv_conv(bf16_to_f64(ins["x"]), bf16_to_f64(ins["w"]), ins["bias"].astype(np.float64))
    ref_qkv_bf16 = bf16_to_f64(f32_to_bf16(ref_qkv.astype(np.float32)))
    ref_out, _, _ = oracle.psa_fwd(ref_qkv_bf16, nh, KD, scale)
    assert_close(to_host_f64(out), ref_out, "bf16", "attention of the conv output")
