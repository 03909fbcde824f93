"""The fused PSA step captured into a CUDA graph (vision-rs book, page "Custom
Kernels": the attention kernels are launched once per step; capturing the step
removes the host from its critical path).  psa_attention_fwd and
psa_attention_bwd allocate nothing and never synchronise, so the step can be
captured once and replayed; the replayed results must equal an eager run bit for
bit, and a replay on new inputs written into the same buffers must match the
oracle."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import psa_inputs, storage_to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Bn,nh,KD,H,W", [(4, 4, 32, 20, 20), (1, 2, 32, 40, 40), (2, 2, 64, 12, 12)])
def test_step_replays_from_a_cuda_graph(oracle, Bn, nh, KD, H, W):
    import torch

    scale = 1 / math.sqrt(KD)
    ins = psa_inputs(Bn, nh, KD, H, W, "bf16", seed=900 + H * W)
    qkv, dout = to_device(ins["qkv"], "bf16"), to_device(ins["dout"], "bf16")
    shape = B.shape_of(qkv, nh, KD)
    out = torch.empty((Bn, nh * 2 * KD, H, W), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(out)
    lse = torch.empty((Bn * nh, H * W), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    dqkv = torch.empty_like(qkv)

    def step(stream):
        B.psa_attention_fwd(qkv, out, lse, v, shape, scale, stream)
        B.psa_attention_bwd(qkv, out, dout, lse, None, dqkv, ws, shape, scale, stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)  # eager, outside capture: per-device set-up happens here
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, v, lse, dqkv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    for t in (out, v, lse, dqkv):
        t.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, (out, v, lse, dqkv)):
        assert torch.equal(a, b)
    # new inputs in the captured buffers, replayed
    ins2 = psa_inputs(Bn, nh, KD, H, W, "bf16", seed=901 + H * W)
    qkv.copy_(to_device(ins2["qkv"], "bf16"))
    dout.copy_(to_device(ins2["dout"], "bf16"))
    g.replay()
    torch.cuda.synchronize()
    assert B.psa_get_last_device_error() == 0
    q64 = storage_to_f64(ins2["qkv"], "bf16")
    ref_out, _, _ = oracle.psa_fwd(q64, nh, KD, scale)
    assert_close(to_host_f64(out), ref_out, "bf16", "replayed out")
    ref = oracle.psa_bwd(q64, storage_to_f64(ins2["dout"], "bf16"), nh, KD, scale)
    assert_close(to_host_f64(dqkv), ref, "bf16", "replayed dQKV")
