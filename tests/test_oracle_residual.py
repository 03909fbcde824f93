"""Pins of the oracle's residual-path output, out + V (vision-rs book, page
"Custom Kernels", section "Position-Sensitive Attention (PSA)": PsaExtractV pulls
the V section out in NCHW for the residual path, which adds it to the merged
attention output).  Runs without a GPU."""
import math

import numpy as np
import pytest
import torch


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _library_out_plus_v(qkv, nh, KD, scale):
    """The same quantity from library calls: a channel reshape, PyTorch SDPA once per
    V half, and the V channels sliced out of the input."""
    B, C, H, W = qkv.shape
    t = torch.from_numpy(qkv).reshape(B, nh, 4, KD, H * W)
    u = t.permute(2, 0, 1, 4, 3)  # [4, B, nh, N, KD]
    o_lo = torch.nn.functional.scaled_dot_product_attention(u[0], u[1], u[2], scale=scale)
    o_hi = torch.nn.functional.scaled_dot_product_attention(u[0], u[1], u[3], scale=scale)
    out = torch.stack([o_lo, o_hi], dim=2).permute(0, 1, 2, 4, 3).reshape(B, nh * 2 * KD, H, W)
    v = t[:, :, 2:].reshape(B, nh * 2 * KD, H, W)
    return (out + v).numpy()


@pytest.mark.parametrize("B,nh,KD,H,W", [(1, 2, 8, 3, 4), (2, 1, 4, 5, 5), (1, 2, 32, 8, 8)])
def test_residual_matches_library(oracle, B, nh, KD, H, W):
    qkv = _rand((B, nh * 4 * KD, H, W), 80)
    scale = 1 / math.sqrt(KD)
    out_res, lse = oracle.psa_fwd_residual(qkv, nh, KD, scale)
    np.testing.assert_allclose(out_res, _library_out_plus_v(qkv, nh, KD, scale), rtol=1e-12, atol=1e-12)
    _, lse_plain, _ = oracle.psa_fwd(qkv, nh, KD, scale)
    np.testing.assert_array_equal(lse, lse_plain)


def test_residual_with_zero_queries_is_mean_plus_v(oracle):
    """With Q = 0 every score is 0, the softmax is uniform and the attention output of
    a channel is the mean of its V row over all positions: out + V = mean + V."""
    B, nh, KD, H, W = 2, 2, 4, 3, 5
    qkv = _rand((B, nh * 4 * KD, H, W), 81)
    heads = qkv.reshape(B, nh, 4, KD, H, W)
    heads[:, :, 0] = 0.0
    out_res, _ = oracle.psa_fwd_residual(qkv, nh, KD, 0.7)
    v = heads[:, :, 2:].reshape(B, nh * 2 * KD, H * W)
    expect = v.mean(axis=2, keepdims=True) + v
    np.testing.assert_allclose(out_res.reshape(B, nh * 2 * KD, H * W), expect, rtol=0, atol=1e-13)


def test_residual_gradient_is_the_backward_with_dvres_equal_to_dout(oracle):
    """The gradient of sum(dY o (out + V)) is psa_bwd with dvres = dY (the residual adds
    dY into the V channels): central differences of the residual output itself."""
    B, nh, KD, H, W = 1, 2, 2, 2, 3
    qkv = _rand((B, nh * 4 * KD, H, W), 82)
    dy = _rand((B, nh * 2 * KD, H, W), 83)
    scale = 1 / math.sqrt(KD)
    grad = oracle.psa_bwd(qkv, dy, nh, KD, scale, dvres=dy)

    def loss(x):
        return float(np.sum(oracle.psa_fwd_residual(x, nh, KD, scale)[0] * dy))

    h = 1e-6
    for idx in np.ndindex(*qkv.shape):
        xp, xm = qkv.copy(), qkv.copy()
        xp[idx] += h
        xm[idx] -= h
        num = (loss(xp) - loss(xm)) / (2 * h)
        assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (idx, num, grad[idx])
