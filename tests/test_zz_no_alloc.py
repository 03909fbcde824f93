"""psa_attention_bwd_noalloc: the fused PSA backward for callers that cannot
allocate device memory when they run it (a plugin whose host framework owns every
device allocation, or a latency-critical loop where cudaMalloc / cudaFree would
synchronise the device).  Its delta scratch is a fixed array inside the library,
so the caller passes only inputs and outputs.

The test calls it through the C ABI twice in a row and compares each result with
psa_attention_bwd (caller workspace) under the bf16 bars the other tests use.
This file is collected last on purpose."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import psa_inputs

pytestmark = pytest.mark.gpu


def test_noalloc_backward_matches_workspace_backward_twice():
    import torch

    Bn, nh, KD, H, W = 8, 4, 32, 20, 20
    scale = 1.0 / math.sqrt(KD)
    ins = psa_inputs(Bn, nh, KD, H, W, "bf16", seed=77, with_dvres=True)
    qkv, dout, dvres = (to_device(ins[k], "bf16") for k in ("qkv", "dout", "dvres"))
    shape = B.shape_of(qkv, nh, KD)
    out = torch.empty((Bn, nh * 2 * KD, H, W), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((Bn * nh, H * W), dtype=torch.float32, device="cuda")
    B.psa_attention_fwd(qkv, out, lse, None, shape, scale)
    ws = torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(qkv)
    B.psa_attention_bwd(qkv, out, dout, lse, dvres, ref, ws, shape, scale)
    ref_h = to_host_f64(ref)
    for call in range(2):
        got = torch.full_like(qkv, float("nan"))
        B.psa_attention_bwd_noalloc(qkv, out, dout, lse, dvres, got, shape, scale)
        torch.cuda.synchronize()
        assert B.psa_get_last_device_error() == 0
        g = to_host_f64(got).reshape(Bn, nh, 4, KD, -1)
        r = ref_h.reshape(Bn, nh, 4, KD, -1)
        for s, name in enumerate(("dQ", "dK", "dV_lo", "dV_hi")):
            assert_close(g[:, :, s], r[:, :, s], "bf16", f"call {call} {name}", output_rounding=s >= 2)
        assert np.array_equal(g, r), f"call {call}: differs from the workspace backward"


def test_noalloc_backward_rejects_sizes_beyond_its_scratch():
    import torch

    # 1048576 head-positions is the scratch capacity; one batch more is refused
    # before anything is launched
    shape = B.PsaShape(2049, 4, 32, 16, 8, B.PSA_DTYPE_BF16)  # 2049*4*128 > 2^20
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.PsaError) as e:
        B.psa_attention_bwd_noalloc(dummy, dummy, dummy, dummy, None, dummy, shape, 0.1)
    assert e.value.status == 2
