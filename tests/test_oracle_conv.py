"""Pins of the oracle's QKV 1x1 convolution (vision-rs book, page "Custom Kernels",
section "Position-Sensitive Attention (PSA)": PsaPackQkv takes a QKV conv's NCHW
output).  Runs without a GPU."""
import numpy as np
import pytest
import torch


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("B,cin,cout,H,W", [(2, 8, 12, 3, 5), (1, 16, 64, 4, 4), (3, 5, 7, 1, 9)])
def test_conv_matches_library(oracle, B, cin, cout, H, W):
    x, w, b = _rand((B, cin, H, W), 1), _rand((cout, cin), 2), _rand((cout,), 3)
    got = oracle.qkv_conv(x, w, b)
    ref = torch.nn.functional.conv2d(torch.from_numpy(x), torch.from_numpy(w)[:, :, None, None],
                                     torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.qkv_conv(x, w), ref - b[None, :, None, None], rtol=1e-12, atol=1e-12)


def test_conv_identity_and_channel_selection(oracle):
    """Identity weights return x (+ bias); a one-hot row copies one input channel."""
    x = _rand((2, 6, 3, 4), 4)
    np.testing.assert_array_equal(oracle.qkv_conv(x, np.eye(6)), x)
    bias = np.arange(6.0)
    np.testing.assert_array_equal(oracle.qkv_conv(x, np.eye(6), bias), x + bias[None, :, None, None])
    sel = np.zeros((3, 6))
    sel[0, 5] = sel[1, 0] = sel[2, 2] = 1.0
    np.testing.assert_array_equal(oracle.qkv_conv(x, sel), x[:, [5, 0, 2]])
