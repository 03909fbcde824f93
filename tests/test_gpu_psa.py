"""The fused PSA attention step reading and writing NCHW (psa_attention_fwd /
psa_attention_bwd) and the unfused chain PsaPackQkv -> Flash Attention 2 per V half
-> PsaMergeAttn, against the oracle's PSA chain (vision-rs book, page "Custom
Kernels", section "Position-Sensitive Attention (PSA)")."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_bits, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import (PSA_WORKLOADS, psa_inputs,
                                                                  storage_to_f64, workload_inputs)

pytestmark = pytest.mark.gpu


def fused_fwd(qkv, nh, KD, scale, with_lse=True, with_v=True):
    import torch

    Bn, C, H, W = qkv.shape
    shape = B.shape_of(qkv, nh, KD)
    out = torch.empty((Bn, nh * 2 * KD, H, W), dtype=qkv.dtype, device="cuda")
    lse = torch.empty((Bn * nh, H * W), dtype=torch.float32, device="cuda") if with_lse else None
    v = torch.empty_like(out) if with_v else None
    B.psa_attention_fwd(qkv, out, lse, v, shape, scale)
    return out, lse, v


def fused_bwd(qkv, out, dout, lse, dvres, nh, KD, scale):
    import torch

    shape = B.shape_of(qkv, nh, KD)
    ws = torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    dqkv = torch.empty_like(qkv)
    B.psa_attention_bwd(qkv, out, dout, lse, dvres, dqkv, ws, shape, scale)
    return dqkv


def check_psa(oracle, ins, nh, KD, dtype, scale, backward, dvres=False, batches=None):
    """Runs the fused forward (+ backward) on all of `ins`, checks the batches
    `batches` (all when None) against the oracle."""
    import torch

    qkv = to_device(ins["qkv"], dtype)
    out, lse, v = fused_fwd(qkv, nh, KD, scale)
    Bn = qkv.shape[0]
    sel = list(range(Bn)) if batches is None else batches
    q64 = storage_to_f64(ins["qkv"][sel], dtype)
    ref_out, ref_lse, ref_v = oracle.psa_fwd(q64, nh, KD, scale)
    assert_close(to_host_f64(out[sel]), ref_out, dtype, "out")
    lse_sel = to_host_f64(lse.view(Bn, nh, -1)[sel]).reshape(len(sel) * nh, -1)
    np.testing.assert_allclose(lse_sel, ref_lse, atol=1e-4 if dtype == "f32" else 2e-3, rtol=0)
    np.testing.assert_array_equal(to_host_f64(v[sel]), ref_v)  # PsaExtractV is an exact copy
    if not backward:
        return
    dout = to_device(ins["dout"], dtype)
    dv_t = to_device(ins["dvres"], dtype) if dvres else None
    dqkv = fused_bwd(qkv, out, dout, lse, dv_t, nh, KD, scale)
    torch.cuda.synchronize()
    ref_dqkv = oracle.psa_bwd(q64, storage_to_f64(ins["dout"][sel], dtype), nh, KD, scale,
                              dvres=storage_to_f64(ins["dvres"][sel], dtype) if dvres else None)
    got = to_host_f64(dqkv[sel]).reshape(len(sel), nh, 4, KD, -1)
    ref = ref_dqkv.reshape(len(sel), nh, 4, KD, -1)
    for s, name in enumerate(("dQ", "dK", "dV_lo", "dV_hi")):
        assert_close(got[:, :, s], ref[:, :, s], dtype, name, output_rounding=dvres and s >= 2)


def test_psa_fwd_f32_n64(oracle):
    w = PSA_WORKLOADS["psa_fwd_f32_n64"]
    check_psa(oracle, workload_inputs(w), w.num_heads, w.key_dim, "f32", 1 / math.sqrt(w.key_dim), False)


def test_psa_fwd_n400(oracle):
    w = PSA_WORKLOADS["psa_fwd_n400"]
    check_psa(oracle, workload_inputs(w), w.num_heads, w.key_dim, "bf16", 1 / math.sqrt(w.key_dim), False)


def test_psa_fwdbwd_n400_full(oracle):
    w = PSA_WORKLOADS["psa_fwdbwd_n400"]
    check_psa(oracle, workload_inputs(w), w.num_heads, w.key_dim, "bf16", 1 / math.sqrt(w.key_dim), True)


def test_psa_fwdbwd_n400_with_residual_grad(oracle):
    w = PSA_WORKLOADS["psa_fwdbwd_n400"]
    ins = workload_inputs(w, with_dvres=True)
    check_psa(oracle, ins, w.num_heads, w.key_dim, "bf16", 1 / math.sqrt(w.key_dim), True, dvres=True,
              batches=[0, 17, 63])


def test_psa_fwdbwd_n1600_sampled_batches(oracle):
    w = PSA_WORKLOADS["psa_fwdbwd_n1600"]
    check_psa(oracle, workload_inputs(w), w.num_heads, w.key_dim, "bf16", 1 / math.sqrt(w.key_dim), True,
              batches=[0, 31])


RAGGED = [
    # (B, nh, KD, H, W): N = 8, 40, 136, 144 (KD = 64), 264, 72
    (1, 1, 32, 2, 4), (2, 3, 32, 5, 8), (1, 2, 32, 8, 17), (2, 1, 64, 12, 12), (1, 2, 32, 12, 22),
    (3, 2, 64, 8, 9),
    # KD = 32 around the one-kernel backward's tiles and its limit: N = 128, 512, 520;
    # around the single-pass forward's limit: N = 448, 456
    (2, 1, 32, 8, 16), (1, 2, 32, 16, 32), (1, 1, 32, 4, 130), (1, 2, 32, 16, 28), (1, 1, 32, 8, 57),
    # the one-kernel backward beyond 512 positions (dQ accumulated in the workspace):
    # N = 1032 (a 16-position last query step), 2048 (its limit); N = 2056 is past it
    (1, 1, 32, 8, 129), (1, 2, 32, 32, 64), (1, 1, 32, 8, 257),
]


@pytest.mark.parametrize("Bn,nh,KD,H,W", RAGGED)
def test_psa_ragged_bf16(oracle, Bn, nh, KD, H, W):
    ins = psa_inputs(Bn, nh, KD, H, W, "bf16", seed=300 + H * W, with_dvres=True)
    check_psa(oracle, ins, nh, KD, "bf16", 1 / math.sqrt(KD), True, dvres=True)


@pytest.mark.parametrize("Bn,nh,KD,H,W", [(1, 2, 32, 2, 4), (2, 1, 64, 5, 8), (1, 3, 32, 10, 20)])
def test_psa_ragged_f32(oracle, Bn, nh, KD, H, W):
    ins = psa_inputs(Bn, nh, KD, H, W, "f32", seed=400 + H * W, with_grad=False)
    check_psa(oracle, ins, nh, KD, "f32", 1 / math.sqrt(KD), False)


@pytest.mark.parametrize("Bn,nh,KD,H,W", [(2, 3, 32, 5, 8), (1, 2, 32, 20, 20), (2, 1, 64, 12, 12)])
def test_split_backward_entry_points(oracle, Bn, nh, KD, H, W):
    """psa_attention_bwd_dq then psa_attention_bwd_dkdv (the two-kernel backward that
    psa_attention_bwd replaces by one kernel for short KD = 32 sequences)."""
    import torch

    scale = 1 / math.sqrt(KD)
    ins = psa_inputs(Bn, nh, KD, H, W, "bf16", seed=500 + H * W, with_dvres=True)
    qkv = to_device(ins["qkv"], "bf16")
    out, lse, _ = fused_fwd(qkv, nh, KD, scale, with_v=False)
    dout = to_device(ins["dout"], "bf16")
    dvres = to_device(ins["dvres"], "bf16")
    shape = B.shape_of(qkv, nh, KD)
    delta = torch.empty((Bn * nh, H * W), dtype=torch.float32, device="cuda")
    dqkv = torch.empty_like(qkv)
    B.psa_attention_bwd_dq(qkv, out, dout, lse, delta, dqkv, shape, scale)
    B.psa_attention_bwd_dkdv(qkv, dout, lse, delta, dvres, dqkv, shape, scale)
    torch.cuda.synchronize()
    q64 = storage_to_f64(ins["qkv"], "bf16")
    ref = oracle.psa_bwd(q64, storage_to_f64(ins["dout"], "bf16"), nh, KD, scale,
                         dvres=storage_to_f64(ins["dvres"], "bf16")).reshape(Bn, nh, 4, KD, -1)
    got = to_host_f64(dqkv).reshape(Bn, nh, 4, KD, -1)
    for s, name in enumerate(("dQ", "dK", "dV_lo", "dV_hi")):
        assert_close(got[:, :, s], ref[:, :, s], "bf16", "split " + name, output_rounding=s >= 2)
    fused = fused_bwd(qkv, out, dout, lse, dvres, nh, KD, scale)
    torch.cuda.synchronize()
    for s, name in enumerate(("dQ", "dK", "dV_lo", "dV_hi")):
        assert_close(to_host_f64(fused).reshape(Bn, nh, 4, KD, -1)[:, :, s], ref[:, :, s], "bf16",
                     "fused " + name, output_rounding=s >= 2)


@pytest.mark.parametrize("Bn,nh,KD,H,W", [(4, 4, 32, 20, 20), (2, 2, 32, 7, 7), (1, 3, 64, 5, 7)])
def test_unfused_chain_matches_oracle_and_fused(oracle, Bn, nh, KD, H, W):
    """PsaPackQkv -> flash_attn2_fwd (V_lo) -> flash_attn2_fwd (V_hi) -> PsaMergeAttn, and its
    backward through the FA2 dQ / dK-dV kernels and the layout adjoints, also on maps whose
    N * 2 bytes is not a multiple of 16 (7 x 7, 5 x 7)."""
    import torch

    scale = 1 / math.sqrt(KD)
    ins = psa_inputs(Bn, nh, KD, H, W, "bf16", seed=21)
    qkv = to_device(ins["qkv"], "bf16")
    shape = B.shape_of(qkv, nh, KD)
    BH, N = Bn * nh, H * W
    packed = torch.empty((4, BH, N, KD), dtype=torch.bfloat16, device="cuda")
    B.psa_pack_qkv(qkv, packed, shape)
    q, k, vlo, vhi = packed
    o_lo, o_hi = torch.empty_like(q), torch.empty_like(q)
    lse = torch.empty((BH, N), dtype=torch.float32, device="cuda")
    lse2 = torch.empty_like(lse)
    B.flash_attn2_fwd(q, k, vlo, o_lo, lse, scale)
    B.flash_attn2_fwd(q, k, vhi, o_hi, lse2, scale)
    out = torch.empty((Bn, nh * 2 * KD, H, W), dtype=torch.bfloat16, device="cuda")
    B.psa_merge_attn(o_lo, o_hi, out, shape)
    q64 = storage_to_f64(ins["qkv"], "bf16")
    ref_out, ref_lse, _ = oracle.psa_fwd(q64, nh, KD, scale)
    assert_close(to_host_f64(out), ref_out, "bf16", "chain out")
    assert torch.equal(lse, lse2)
    # the fused entry point takes every map (rows that are not 16-byte multiples
    # run on CUDA cores)
    fout, flse, _ = fused_fwd(qkv, nh, KD, scale, with_v=False)
    assert_close(to_host_f64(fout), ref_out, "bf16", "fused out")
    # backward of the chain: unmerge dOut, FA2 backward per half, sum dQ / dK, unpack
    dout = to_device(ins["dout"], "bf16")
    do_lo, do_hi = torch.empty_like(q), torch.empty_like(q)
    B.psa_unmerge_attn(dout, do_lo, do_hi, shape)
    delta = torch.empty_like(lse)
    grads = []
    for o_h, do_h, v_h in ((o_lo, do_lo, vlo), (o_hi, do_hi, vhi)):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        B.flash_attn2_bwd_dq(q, k, v_h, o_h, do_h, lse, delta, dq, scale)
        B.flash_attn2_bwd_dkdv(q, k, v_h, do_h, lse, delta, dk, dv, scale)
        grads.append((dq, dk, dv))
    torch.cuda.synchronize()
    # each FA2 backward call on its own, at the single-rounding bars: the oracle's
    # attention backward of that V half
    p64 = storage_to_f64(oracle.pack_qkv(ins["qkv"], nh, KD), "bf16")
    do64 = [storage_to_f64(x, "bf16") for x in oracle.unmerge_attn(ins["dout"], nh, KD)]
    for half, (dq, dk, dv) in enumerate(grads):
        rq, rk, rv = oracle.attn_bwd(p64[0], p64[1], p64[2 + half], do64[half], scale)
        assert_close(to_host_f64(dq), rq, "bf16", f"half {half} dQ")
        assert_close(to_host_f64(dk), rk, "bf16", f"half {half} dK")
        assert_close(to_host_f64(dv), rv, "bf16", f"half {half} dV")
    dpacked = torch.stack([(grads[0][0].float() + grads[1][0].float()).to(torch.bfloat16),
                           (grads[0][1].float() + grads[1][1].float()).to(torch.bfloat16),
                           grads[0][2], grads[1][2]]).contiguous()
    dqkv = torch.empty_like(qkv)
    B.psa_unpack_qkv(dpacked, dqkv, shape)
    ref_dqkv = oracle.psa_bwd(q64, storage_to_f64(ins["dout"], "bf16"), nh, KD, scale)
    got = to_host_f64(dqkv).reshape(Bn, nh, 4, KD, -1)
    ref = ref_dqkv.reshape(Bn, nh, 4, KD, -1)
    # end to end through the chain: dQ and dK are sums of the two halves' bf16
    # outputs (two roundings, checked per half above at the single-rounding bars);
    # the dV halves carry one
    for s, name in enumerate(("dQ", "dK", "dV_lo", "dV_hi")):
        assert_close(got[:, :, s], ref[:, :, s], "bf16", "chain " + name, roundings=2 if s < 2 else 1)


def test_fused_reruns_are_bitwise_identical():
    import torch

    ins = psa_inputs(8, 4, 32, 20, 20, "bf16", seed=5)
    qkv = to_device(ins["qkv"], "bf16")
    dout = to_device(ins["dout"], "bf16")
    res = []
    for _ in range(2):
        out, lse, v = fused_fwd(qkv, 4, 32, 0.17)
        dqkv = fused_bwd(qkv, out, dout, lse, None, 4, 32, 0.17)
        res.append((out, lse, v, dqkv))
    for a, b in zip(*res):
        assert torch.equal(a, b)
    assert B.psa_get_last_device_error() == 0
