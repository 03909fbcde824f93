"""Flash Attention 2 on [BH, N, HEAD_DIM] (vision-rs book, page "Custom Kernels",
section "Flash Attention 2"): forward, dQ and dK/dV kernels against the fp64 oracle
on the same seeded inputs."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import (FA2_SWEEP_BH, FA2_SWEEP_D, FA2_SWEEP_N,
                                                                  FA2_SWEEP_SEED, fa2_inputs,
                                                                  storage_to_f64)

pytestmark = pytest.mark.gpu


def _run_fwd(ins, dtype, scale):
    import torch

    q, k, v = (to_device(ins[n], dtype) for n in ("q", "k", "v"))
    BH, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((BH, N), dtype=torch.float32, device="cuda")
    B.flash_attn2_fwd(q, k, v, o, lse, scale)
    return q, k, v, o, lse


def _run_bwd(q, k, v, o, lse, do, scale):
    import torch

    BH, N, d = q.shape
    delta = torch.empty((BH, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B.flash_attn2_bwd_dq(q, k, v, o, do, lse, delta, dq, scale)
    B.flash_attn2_bwd_dkdv(q, k, v, do, lse, delta, dk, dv, scale)
    return delta, dq, dk, dv


SMALL = [(2, 1, 32), (3, 17, 32), (2, 128, 32), (2, 200, 64), (4, 400, 32), (2, 400, 64),
         (1, 1024, 32), (2, 257, 64), (1, 63, 64)]


@pytest.mark.parametrize("BH,N,d", SMALL)
def test_fwd_bwd_bf16_small(oracle, BH, N, d):
    import torch

    ins = fa2_inputs(BH, N, d, "bf16", seed=100 + N + d)
    scale = 1.0 / math.sqrt(d)
    q, k, v, o, lse = _run_fwd(ins, "bf16", scale)
    f64 = {n: storage_to_f64(a, "bf16") for n, a in ins.items()}
    ref_o, ref_lse = oracle.attn_fwd(f64["q"], f64["k"], f64["v"], scale)
    assert_close(to_host_f64(o), ref_o, "bf16", "O")
    np.testing.assert_allclose(to_host_f64(lse), ref_lse, atol=2e-3, rtol=0)

    do = to_device(ins["do"], "bf16")
    delta, dq, dk, dv = _run_bwd(q, k, v, o, lse, do, scale)
    ref_dq, ref_dk, ref_dv = oracle.attn_bwd(f64["q"], f64["k"], f64["v"], f64["do"], scale)
    assert_close(to_host_f64(dv), ref_dv, "bf16", "dV")
    assert_close(to_host_f64(dk), ref_dk, "bf16", "dK")
    assert_close(to_host_f64(dq), ref_dq, "bf16", "dQ")
    ref_delta = np.sum(f64["do"] * ref_o, axis=-1)
    np.testing.assert_allclose(to_host_f64(delta), ref_delta, atol=3e-2, rtol=0)
    torch.cuda.synchronize()


@pytest.mark.parametrize("BH,N,d", [(2, 64, 32), (3, 100, 64), (1, 1, 32), (2, 300, 32)])
def test_fwd_f32(oracle, BH, N, d):
    ins = fa2_inputs(BH, N, d, "f32", seed=200 + N)
    scale = 1.0 / math.sqrt(d)
    _, _, _, o, lse = _run_fwd(ins, "f32", scale)
    ref_o, ref_lse = oracle.attn_fwd(ins["q"], ins["k"], ins["v"], scale)
    assert_close(to_host_f64(o), ref_o, "f32", "O")
    np.testing.assert_allclose(to_host_f64(lse), ref_lse, atol=1e-4, rtol=0)


def test_reruns_are_bitwise_identical():
    import torch

    ins = fa2_inputs(4, 333, 64, "bf16", seed=9)
    q, k, v, o1, lse1 = _run_fwd(ins, "bf16", 0.125)
    do = to_device(ins["do"], "bf16")
    r1 = _run_bwd(q, k, v, o1, lse1, do, 0.125)
    _, _, _, o2, lse2 = _run_fwd(ins, "bf16", 0.125)
    r2 = _run_bwd(q, k, v, o2, lse2, do, 0.125)
    assert torch.equal(o1, o2) and torch.equal(lse1, lse2)
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


@pytest.mark.parametrize("N", FA2_SWEEP_N)
@pytest.mark.parametrize("d", FA2_SWEEP_D)
def test_sweep_full_size_sampled(oracle, N, d):
    """The raw sweep at its full size (BH=64), in the launch configuration the
    benchmark times: sampled rows of two heads against the oracle, plus the
    gradient-sum identities on every head."""
    import torch

    ins = fa2_inputs(FA2_SWEEP_BH, N, d, "bf16", seed=FA2_SWEEP_SEED)
    scale = 1.0 / math.sqrt(d)
    q, k, v, o, lse = _run_fwd(ins, "bf16", scale)
    do = to_device(ins["do"], "bf16")
    _, dq, dk, dv = _run_bwd(q, k, v, o, lse, do, scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(N + d)
    heads = [0, FA2_SWEEP_BH - 1]
    nrows = 48 if N <= 4096 else 16
    for bh in heads:
        f64 = {n: storage_to_f64(a[bh], "bf16") for n, a in ins.items()}
        rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, nrows)]))
        ref_o, ref_lse = oracle.attn_fwd_rows(f64["q"], f64["k"], f64["v"], scale, rows)
        assert_close(to_host_f64(o[bh, rows]), ref_o, "bf16", f"O rows bh={bh}")
        np.testing.assert_allclose(to_host_f64(lse[bh, rows]), ref_lse, atol=2e-3, rtol=0)
        ref_dq = oracle.attn_bwd_dq_rows(f64["q"], f64["k"], f64["v"], f64["do"], scale, rows)
        assert_close(to_host_f64(dq[bh, rows]), ref_dq, "bf16", f"dQ rows bh={bh}")
        keys = rows[: max(4, len(rows) // 4)]
        ref_dk, ref_dv = oracle.attn_bwd_dkdv_rows(f64["q"], f64["k"], f64["v"], f64["do"], scale, keys)
        assert_close(to_host_f64(dk[bh, keys]), ref_dk, "bf16", f"dK rows bh={bh}")
        assert_close(to_host_f64(dv[bh, keys]), ref_dv, "bf16", f"dV rows bh={bh}")
    # identities that hold at any size: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i
    dk_sum = dk.double().sum(dim=1)
    dv_sum = dv.double().sum(dim=1)
    do_sum = do.double().sum(dim=1)
    scale_dk = dk.double().abs().sum(dim=1)
    assert torch.all(dk_sum.abs() <= 1e-2 * scale_dk + 1e-3)
    assert torch.allclose(dv_sum, do_sum, rtol=0, atol=2e-3 * math.sqrt(N) + 1e-2)
