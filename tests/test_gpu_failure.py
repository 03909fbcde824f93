"""The failure path of the bounded on-chip waits: a wait that runs out records
PSA_ERR_TIMEOUT in the device error word, the kernel returns, and the context
stays usable (vision-rs book, page "Custom Kernels", section "Flash Attention 2":
the kernels hand tiles between warps through on-chip barriers; every such wait in
this library gives up after a bounded time instead of hanging).

psa_debug_wait_timeout launches one warp that waits, with a 1 ms limit, on a
barrier nothing arrives at: the same wait routine the attention kernels use.
Nothing faults and nothing is left waiting."""
import math

import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import psa_inputs, storage_to_f64

pytestmark = pytest.mark.gpu

PSA_ERR_TIMEOUT = 5


def test_wait_that_runs_out_reports_timeout_and_context_survives(oracle):
    import torch

    assert B.psa_get_last_device_error() == 0
    B.psa_debug_wait_timeout(1_000_000)
    assert B.psa_get_last_device_error() == PSA_ERR_TIMEOUT
    assert B.psa_get_last_device_error() == 0  # read and cleared
    # the next real call runs normally and matches the oracle
    nh, KD, H, W = 2, 32, 10, 20
    scale = 1 / math.sqrt(KD)
    ins = psa_inputs(2, nh, KD, H, W, "bf16", seed=61)
    qkv = to_device(ins["qkv"], "bf16")
    out = torch.empty((2, nh * 2 * KD, H, W), dtype=torch.bfloat16, device="cuda")
    B.psa_attention_fwd(qkv, out, None, None, B.shape_of(qkv, nh, KD), scale)
    assert B.psa_get_last_device_error() == 0
    ref, _, _ = oracle.psa_fwd(storage_to_f64(ins["qkv"], "bf16"), nh, KD, scale)
    assert_close(to_host_f64(out), ref, "bf16", "out after a timed-out wait")
