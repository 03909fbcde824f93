"""Pins for the oracle's layout routines (PsaPackQkv, PsaExtractV, PsaMergeAttn and
their adjoints), checked against hand-written examples and permutation properties.

Source: vision-rs book, page "Custom Kernels", section "Position-Sensitive Attention (PSA)".
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_hand_examples.json")


def _tagged(B, C, H, W):
    b = np.arange(B).reshape(B, 1, 1, 1)
    c = np.arange(C).reshape(1, C, 1, 1)
    n = np.arange(H * W).reshape(1, 1, H, W)
    return (100 * b + 10 * c + n).astype(np.int64)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_layouts_match_hand_examples(oracle, case):
    B, nh, KD, H, W = case["B"], case["num_heads"], case["key_dim"], case["H"], case["W"]
    qkv = _tagged(B, nh * 4 * KD, H, W)
    packed = oracle.pack_qkv(qkv, nh, KD)
    np.testing.assert_array_equal(packed, np.array(case["packed"]))
    np.testing.assert_array_equal(oracle.extract_v(qkv, nh, KD), np.array(case["extract_v"]))
    merged = oracle.merge_attn(packed[2], packed[3], B, nh, KD, H, W)
    np.testing.assert_array_equal(merged, np.array(case["merge_of_v_planes"]))


SHAPES = [(1, 2, 32, 8, 8), (2, 4, 32, 5, 7), (3, 1, 8, 2, 3), (2, 3, 4, 1, 9)]


@pytest.mark.parametrize("B,nh,KD,H,W", SHAPES)
def test_pack_is_a_permutation_and_matches_a_view(oracle, B, nh, KD, H, W):
    C = nh * 4 * KD
    qkv = np.arange(B * C * H * W, dtype=np.int64).reshape(B, C, H, W)
    packed = oracle.pack_qkv(qkv, nh, KD)
    assert packed.shape == (4, B * nh, H * W, KD)
    # every input element lands exactly once
    np.testing.assert_array_equal(np.sort(packed.ravel()), np.arange(qkv.size))
    # the same layout stated as a reshape/transpose of the channel axis [nh, 4, KD]
    view = qkv.reshape(B, nh, 4, KD, H * W).transpose(2, 0, 1, 4, 3).reshape(4, B * nh, H * W, KD)
    np.testing.assert_array_equal(packed, view)
    # the adjoint undoes it
    np.testing.assert_array_equal(oracle.unpack_qkv(packed, B, nh, KD, H, W), qkv)


@pytest.mark.parametrize("B,nh,KD,H,W", SHAPES)
def test_merge_extract_and_their_inverses(oracle, B, nh, KD, H, W):
    rng = np.random.default_rng(7)
    lo = rng.integers(0, 1 << 16, size=(B * nh, H * W, KD)).astype(np.uint16)
    hi = rng.integers(0, 1 << 16, size=(B * nh, H * W, KD)).astype(np.uint16)
    out = oracle.merge_attn(lo, hi, B, nh, KD, H, W)
    assert out.shape == (B, nh * 2 * KD, H, W)
    np.testing.assert_array_equal(np.sort(out.ravel()), np.sort(np.concatenate([lo.ravel(), hi.ravel()])))
    view = np.stack([lo, hi]).reshape(2, B, nh, H * W, KD).transpose(1, 2, 0, 4, 3).reshape(out.shape)
    np.testing.assert_array_equal(out, view)
    lo2, hi2 = oracle.unmerge_attn(out, nh, KD)
    np.testing.assert_array_equal(lo2, lo)
    np.testing.assert_array_equal(hi2, hi)
    # ExtractV is the V planes of the pack, merged back to NCHW
    qkv = rng.integers(0, 1 << 16, size=(B, nh * 4 * KD, H, W)).astype(np.uint16)
    packed = oracle.pack_qkv(qkv, nh, KD)
    np.testing.assert_array_equal(oracle.extract_v(qkv, nh, KD),
                                  oracle.merge_attn(packed[2], packed[3], B, nh, KD, H, W))


def test_layout_copies_are_bitwise(oracle):
    # float payloads including NaN patterns and -0.0 travel unchanged
    bits = np.array([0x7FC1, 0xFF80, 0x8000, 0x0001, 0x7F80, 0x3F80, 0xBF81, 0x1234], dtype=np.uint16)
    qkv = np.tile(bits, 2 * 4 * 8 * 4 // bits.size).reshape(1, 2 * 4 * 8, 2, 2)
    packed = oracle.pack_qkv(qkv, 2, 8)
    assert packed.dtype == np.uint16
    np.testing.assert_array_equal(oracle.unpack_qkv(packed, 1, 2, 8, 2, 2), qkv)
    f32 = np.frombuffer(np.arange(2 * 4 * 4 * 3, dtype=np.uint32).tobytes(), dtype=np.float32)
    q32 = f32.reshape(1, 2 * 4 * 4, 3, 1).copy()
    np.testing.assert_array_equal(oracle.unpack_qkv(oracle.pack_qkv(q32, 2, 4), 1, 2, 4, 3, 1).view(np.uint32),
                                  q32.view(np.uint32))
