"""psa_attention_bwd_noalloc: the fused PSA backward for callers that cannot
allocate device memory when they run it (a plugin whose host framework owns every
device allocation, or a latency-critical loop where cudaMalloc / cudaFree would
synchronise the device).  Its workspace is a fixed array inside the library, so
the caller passes only inputs and outputs.

The backward uses that array as its workspace: for delta in its two-kernel form
(key_dim 64 below), and as the dQ accumulator of its one-kernel form between 512
and 2048 positions (N = 1600 below); up to 512 positions it leaves the array
alone.  The cases run those forms on different shapes one after the other, plus
one short case.  Each call is made
twice in a row through the C ABI, and each result is compared with the fp64
oracle at the bf16 bars the other tests use, and bit for bit with
psa_attention_bwd given a workspace of its own.  This file is collected last on
purpose."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import psa_inputs, storage_to_f64

pytestmark = pytest.mark.gpu

CASES = [
    # (B, nh, KD, H, W, seed)
    (2, 2, 64, 20, 20, 77),   # key_dim 64: dQ kernel writes delta, dK/dV kernel reads it
    (1, 2, 32, 40, 40, 78),   # N = 1600: one kernel, dQ accumulated in the array
    (2, 2, 64, 8, 12, 79),    # a smaller two-kernel case right after a larger one
    (2, 4, 32, 20, 20, 80),   # key_dim 32, N = 400: one kernel, delta on chip
]


def test_noalloc_backward_matches_oracle_and_workspace_backward(oracle):
    import torch

    for Bn, nh, KD, H, W, seed in CASES:
        scale = 1.0 / math.sqrt(KD)
        ins = psa_inputs(Bn, nh, KD, H, W, "bf16", seed=seed, with_dvres=True)
        qkv, dout, dvres = (to_device(ins[k], "bf16") for k in ("qkv", "dout", "dvres"))
        shape = B.shape_of(qkv, nh, KD)
        out = torch.empty((Bn, nh * 2 * KD, H, W), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((Bn * nh, H * W), dtype=torch.float32, device="cuda")
        B.psa_attention_fwd(qkv, out, lse, None, shape, scale)
        ws = torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
        with_ws = torch.empty_like(qkv)
        B.psa_attention_bwd(qkv, out, dout, lse, dvres, with_ws, ws, shape, scale)
        q64 = storage_to_f64(ins["qkv"], "bf16")
        ref = oracle.psa_bwd(q64, storage_to_f64(ins["dout"], "bf16"), nh, KD, scale,
                             dvres=storage_to_f64(ins["dvres"], "bf16")).reshape(Bn, nh, 4, KD, -1)
        ws_h = to_host_f64(with_ws)
        for call in range(2):
            got = torch.full_like(qkv, float("nan"))
            B.psa_attention_bwd_noalloc(qkv, out, dout, lse, dvres, got, shape, scale)
            torch.cuda.synchronize()
            assert B.psa_get_last_device_error() == 0
            g = to_host_f64(got)
            what = f"KD={KD} {H}x{W} call {call}"
            gr = g.reshape(Bn, nh, 4, KD, -1)
            for s, name in enumerate(("dQ", "dK", "dV_lo", "dV_hi")):
                assert_close(gr[:, :, s], ref[:, :, s], "bf16", f"{what} {name}", output_rounding=s >= 2)
            assert np.array_equal(g, ws_h), f"{what}: differs from psa_attention_bwd with a workspace"


def test_noalloc_backward_rejects_sizes_beyond_its_scratch():
    import torch

    # 1048576 head-positions is the scratch capacity; one batch more is refused
    # before anything is launched
    shape = B.PsaShape(2049, 4, 32, 16, 8, B.PSA_DTYPE_BF16)  # 2049*4*128 > 2^20
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.PsaError) as e:
        B.psa_attention_bwd_noalloc(dummy, dummy, dummy, dummy, None, dummy, shape, 0.1)
    assert e.value.status == 2
    # a missing required pointer is reported first, whatever the size
    with pytest.raises(B.PsaError) as e:
        B.psa_attention_bwd_noalloc(dummy, None, dummy, dummy, None, dummy, shape, 0.1)
    assert e.value.status == 1
