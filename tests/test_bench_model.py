"""The bench's work model against the algorithmic counts written out by hand (no
GPU needed): per head, the forward does S = Q K^T (2 N^2 KD FLOPs) and
O = P [V_lo | V_hi] (2 N^2 2KD), i.e. 192 N^2 at KD = 32; the backward recomputes
S once and does dP, dV, dQ, dK: 2 N^2 (KD + 2KD + 2KD + KD + KD) = 448 N^2.
Bytes are bf16 tensors touched once: QKV [B, 512, N] read, Out and the extracted
V [B, 256, N] written, LSE [BH, N] fp32 written (forward); QKV, Out, dOut read,
dQKV written, LSE read (backward)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_step_model_at_the_headline_workload():
    import bench
    from vision_transformer_attention_psapackqkv_gb300.inputs import PSA_WORKLOADS

    w = PSA_WORKLOADS["psa_fwdbwd_n400"]
    B, N, BH = 64, 400, 256
    kernels, step = bench.work_model(w)
    assert kernels["fwd"]["flops"] == 192 * N * N * BH
    assert kernels["bwd"]["flops"] == 448 * N * N * BH
    assert step["flops"] == (192 + 448) * N * N * BH == 26_214_400_000
    fwd_bytes = B * N * (512 + 256 + 256) * 2 + BH * N * 4
    bwd_bytes = B * N * (512 + 256 + 256 + 512) * 2 + BH * N * 4
    assert kernels["fwd"]["bytes"] == fwd_bytes
    assert kernels["bwd"]["bytes"] == bwd_bytes
    assert step["bytes"] == fwd_bytes + bwd_bytes == 131_891_200


def test_split_backward_model_counts_the_recompute():
    import bench
    from vision_transformer_attention_psapackqkv_gb300.inputs import PSA_WORKLOADS

    w = PSA_WORKLOADS["psa_fwdbwd_n400"]
    kernels, _ = bench.work_model(w)
    n2 = 400 * 400 * 256
    # dQ kernel: S, dP, dQ; dK/dV kernel: S, dP, dV, dK (S and dP formed twice)
    assert kernels["bwd_dq"]["flops"] == n2 * 2 * (32 + 64 + 32)
    assert kernels["bwd_dkdv"]["flops"] == n2 * 2 * (32 + 64 + 64 + 32)


def test_roofline_time_at_the_fallback_peaks():
    import bench

    peaks = bench.FALLBACK_PEAKS
    t_hbm = 131_891_200 / (peaks["hbm_gbs"] * 1e9)
    t_tensor = 26_214_400_000 / (peaks["bf16_tflops_sustained"] * 1e12)
    # HBM-bound: the bytes take longer than the FLOPs at the fallback peaks
    assert t_hbm > t_tensor
    assert t_hbm * 1e6 == pytest.approx(19.3958, rel=1e-4)
