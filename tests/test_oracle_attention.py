"""Pins for the oracle's attention forward and backward.

The oracle is the plain definition of softmax attention (vision-rs book, page
"Custom Kernels", section "Flash Attention 2") and the PSA chain of section
"Position-Sensitive Attention (PSA)".  It is checked here against things other
than itself: hand-derived closed forms (tests/golden), a library routine
(PyTorch's scaled_dot_product_attention and autograd in float64), invariants of
softmax attention, and central finite differences.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "attention_closed_form.json")
_G = json.load(open(GOLDEN))


def _ev(x):
    if isinstance(x, list):
        return [_ev(e) for e in x]
    return float(eval(x, {"__builtins__": {}}, {"log": math.log}))


def _arr(x):
    return np.array(_ev(x), dtype=np.float64)


@pytest.mark.parametrize("case", _G["cases"], ids=lambda c: c["name"])
def test_forward_closed_forms(oracle, case):
    q, k, v = _arr(case["q"])[None], _arr(case["k"])[None], _arr(case["v"])[None]
    o, lse = oracle.attn_fwd(q, k, v, _ev(case["scale"]))
    np.testing.assert_allclose(o[0], _arr(case["o"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0], _arr(case["lse"]), rtol=0, atol=1e-13)
    o_r, lse_r = oracle.attn_fwd_rows(q[0], k[0], v[0], _ev(case["scale"]), np.arange(q.shape[1]))
    np.testing.assert_allclose(o_r, _arr(case["o"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse_r, _arr(case["lse"]), rtol=0, atol=1e-13)


@pytest.mark.parametrize("case", _G["backward_cases"], ids=lambda c: c["name"])
def test_backward_closed_forms(oracle, case):
    q, k, v, do = (_arr(case[n])[None] for n in ("q", "k", "v", "do"))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, _ev(case["scale"]))
    np.testing.assert_allclose(dq[0], _arr(case["dq"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk[0], _arr(case["dk"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv[0], _arr(case["dv"]), rtol=0, atol=1e-13)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("BH,N,dqk,dv", [(2, 17, 8, 8), (3, 33, 4, 16), (1, 64, 32, 64)])
def test_forward_matches_library_sdpa(oracle, BH, N, dqk, dv):
    q, k, v = _rand((BH, N, dqk), 1), _rand((BH, N, dqk), 2), _rand((BH, N, dv), 3)
    scale = 1.0 / math.sqrt(dqk)
    o, lse = oracle.attn_fwd(q, k, v, scale)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=scale).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)
    scores = torch.from_numpy(q) @ torch.from_numpy(k).transpose(1, 2) * scale
    np.testing.assert_allclose(lse, torch.logsumexp(scores, dim=-1).numpy(), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("BH,N,dqk,dv", [(2, 9, 4, 4), (1, 40, 8, 16)])
def test_backward_matches_library_autograd(oracle, BH, N, dqk, dv):
    q, k, v, do = (_rand(s, i) for i, s in enumerate([(BH, N, dqk), (BH, N, dqk), (BH, N, dv), (BH, N, dv)]))
    scale = 0.37
    dq, dk, dvv = oracle.attn_bwd(q, k, v, do, scale)
    tq, tk, tv = (torch.from_numpy(a).requires_grad_() for a in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
    out.backward(torch.from_numpy(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dvv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_softmax_rows_sum_to_one_and_identical_keys_average(oracle):
    BH, N, d = 2, 23, 8
    q, k = _rand((BH, N, d), 4), _rand((BH, N, d), 5)
    ones = np.ones((BH, N, 3))
    o, _ = oracle.attn_fwd(q, k, ones, 0.3)
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-12)
    # identical keys: every row is the mean of V
    v = _rand((BH, N, 5), 6)
    k_same = np.repeat(k[:, :1], N, axis=1)
    o, lse = oracle.attn_fwd(q, k_same, v, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-12)
    # and LSE = s + ln N with s the (common) score
    s = 0.3 * np.einsum("bnd,bd->bn", q, k[:, 0])
    np.testing.assert_allclose(lse, s + math.log(N), atol=1e-12)
    # Q = 0 gives the mean of V as well
    o, _ = oracle.attn_fwd(np.zeros_like(q), k, v, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-12)


def test_single_key_and_dominant_logit(oracle):
    q, k, v = _rand((3, 1, 4), 7), _rand((3, 1, 4), 8), _rand((3, 1, 6), 9)
    o, lse = oracle.attn_fwd(q, k, v, 0.5)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse[:, 0], 0.5 * np.sum(q[:, 0] * k[:, 0], axis=-1), atol=1e-14)
    # one key aligned with the query and scaled up takes all the weight
    N, d = 12, 4
    q = _rand((1, N, d), 10)
    k = _rand((1, N, d), 11) * 0.1
    v = _rand((1, N, 3), 12)
    j = 5
    k[0, j] = 60.0 * q[0, 0]
    o, _ = oracle.attn_fwd(q, k, v, 1.0)
    np.testing.assert_allclose(o[0, 0], v[0, j], atol=1e-9)


def test_permutation_equivariance(oracle):
    BH, N = 2, 19
    q, k, v = _rand((BH, N, 8), 13), _rand((BH, N, 8), 14), _rand((BH, N, 5), 15)
    o, lse = oracle.attn_fwd(q, k, v, 0.4)
    perm = np.random.default_rng(3).permutation(N)
    o2, lse2 = oracle.attn_fwd(q, k[:, perm], v[:, perm], 0.4)
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)
    o3, lse3 = oracle.attn_fwd(q[:, perm], k, v, 0.4)
    np.testing.assert_allclose(o3, o[:, perm], atol=1e-13)
    np.testing.assert_allclose(lse3, lse[:, perm], atol=1e-13)


def test_two_half_runs_equal_one_wide_run(oracle):
    BH, N, KD = 3, 21, 8
    q, k = _rand((BH, N, KD), 16), _rand((BH, N, KD), 17)
    vlo, vhi = _rand((BH, N, KD), 18), _rand((BH, N, KD), 19)
    o_lo, lse_lo = oracle.attn_fwd(q, k, vlo, 1 / math.sqrt(KD))
    o_hi, lse_hi = oracle.attn_fwd(q, k, vhi, 1 / math.sqrt(KD))
    o, lse = oracle.attn_fwd(q, k, np.concatenate([vlo, vhi], -1), 1 / math.sqrt(KD))
    np.testing.assert_allclose(o, np.concatenate([o_lo, o_hi], -1), atol=1e-14)
    np.testing.assert_array_equal(lse_lo, lse_hi)
    np.testing.assert_allclose(lse, lse_lo, atol=1e-14)


def test_backward_invariants(oracle):
    BH, N, dqk, dv = 2, 31, 8, 12
    q, k, v, do = (_rand(s, 20 + i) for i, s in enumerate([(BH, N, dqk), (BH, N, dqk), (BH, N, dv), (BH, N, dv)]))
    dq, dk, dvv = oracle.attn_bwd(q, k, v, do, 0.35)
    # rows of dS sum to zero, so the key gradients sum to zero
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    # rows of P sum to one, so the value gradients sum to the output gradients
    np.testing.assert_allclose(dvv.sum(axis=1), do.sum(axis=1), atol=1e-12)
    # dV is linear in dO
    _, _, dv2 = oracle.attn_bwd(q, k, v, 2.5 * do, 0.35)
    np.testing.assert_allclose(dv2, 2.5 * dvv, atol=1e-12)


def _fd(f, x, idx, h=1e-6):
    xp, xm = x.copy(), x.copy()
    xp[idx] += h
    xm[idx] -= h
    return (f(xp) - f(xm)) / (2 * h)


def test_backward_central_differences(oracle):
    BH, N, dqk, dv = 2, 11, 4, 6
    q, k, v, do = (_rand(s, 30 + i) for i, s in enumerate([(BH, N, dqk), (BH, N, dqk), (BH, N, dv), (BH, N, dv)]))
    scale = 0.6
    dq, dk, dvv = oracle.attn_bwd(q, k, v, do, scale)

    def loss(qq, kk, vv):
        return float(np.sum(oracle.attn_fwd(qq, kk, vv, scale)[0] * do))

    rng = np.random.default_rng(0)
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dvv, 2)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in arr.shape)
            if which == 0:
                num = _fd(lambda x: loss(x, k, v), q, idx)
            elif which == 1:
                num = _fd(lambda x: loss(q, x, v), k, idx)
            else:
                num = _fd(lambda x: loss(q, k, x), v, idx)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (which, idx, num, grad[idx])


def test_sampled_rows_agree_with_whole_heads(oracle):
    BH, N, dqk, dv = 2, 37, 8, 16
    q, k, v, do = (_rand(s, 40 + i) for i, s in enumerate([(BH, N, dqk), (BH, N, dqk), (BH, N, dv), (BH, N, dv)]))
    o, lse = oracle.attn_fwd(q, k, v, 0.3)
    dq, dk, dvv = oracle.attn_bwd(q, k, v, do, 0.3)
    rows = np.array([0, 5, 36, 17])
    for bh in range(BH):
        o_r, lse_r = oracle.attn_fwd_rows(q[bh], k[bh], v[bh], 0.3, rows)
        np.testing.assert_allclose(o_r, o[bh, rows], atol=1e-14)
        np.testing.assert_allclose(lse_r, lse[bh, rows], atol=1e-14)
        np.testing.assert_allclose(oracle.attn_bwd_dq_rows(q[bh], k[bh], v[bh], do[bh], 0.3, rows),
                                   dq[bh, rows], atol=1e-13)
        dk_r, dv_r = oracle.attn_bwd_dkdv_rows(q[bh], k[bh], v[bh], do[bh], 0.3, rows, nthreads=3)
        np.testing.assert_allclose(dk_r, dk[bh, rows], atol=1e-13)
        np.testing.assert_allclose(dv_r, dvv[bh, rows], atol=1e-13)


# ----------------------------------------------------------------------------- PSA chain

def _psa_reference(qkv, nh, KD, scale):
    """The PSA forward stated with library calls: a channel reshape for the pack and
    PyTorch SDPA run once per V half."""
    B, C, H, W = qkv.shape
    t = torch.from_numpy(qkv).reshape(B, nh, 4, KD, H * W).permute(2, 0, 1, 4, 3)  # [4,B,nh,N,KD]
    q, k, vlo, vhi = t[0], t[1], t[2], t[3]
    o_lo = torch.nn.functional.scaled_dot_product_attention(q, k, vlo, scale=scale)
    o_hi = torch.nn.functional.scaled_dot_product_attention(q, k, vhi, scale=scale)
    out = torch.stack([o_lo, o_hi], dim=2)  # [B, nh, 2, N, KD]
    return out.permute(0, 1, 2, 4, 3).reshape(B, nh * 2 * KD, H, W)


@pytest.mark.parametrize("B,nh,KD,H,W", [(1, 2, 8, 3, 4), (2, 1, 4, 5, 5), (1, 2, 32, 8, 8)])
def test_psa_forward_matches_library_chain(oracle, B, nh, KD, H, W):
    qkv = _rand((B, nh * 4 * KD, H, W), 50)
    scale = 1 / math.sqrt(KD)
    out, lse, vres = oracle.psa_fwd(qkv, nh, KD, scale)
    np.testing.assert_allclose(out, _psa_reference(qkv, nh, KD, scale).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(vres, oracle.extract_v(qkv, nh, KD))
    assert lse.shape == (B * nh, H * W)


@pytest.mark.parametrize("with_dvres", [False, True])
def test_psa_backward_matches_library_autograd(oracle, with_dvres):
    B, nh, KD, H, W = 2, 2, 4, 3, 3
    qkv = _rand((B, nh * 4 * KD, H, W), 60)
    dout = _rand((B, nh * 2 * KD, H, W), 61)
    dvres = _rand((B, nh * 2 * KD, H, W), 62) if with_dvres else None
    scale = 1 / math.sqrt(KD)
    dqkv = oracle.psa_bwd(qkv, dout, nh, KD, scale, dvres=dvres)
    t = torch.from_numpy(qkv).requires_grad_()
    out = _psa_reference_t(t, nh, KD, scale)
    loss = (out * torch.from_numpy(dout)).sum()
    if with_dvres:
        vres = t.reshape(B, nh, 4, KD, H, W)[:, :, 2:].reshape(B, nh * 2 * KD, H, W)
        loss = loss + (vres * torch.from_numpy(dvres)).sum()
    loss.backward()
    np.testing.assert_allclose(dqkv, t.grad.numpy(), rtol=1e-11, atol=1e-12)


def _psa_reference_t(t, nh, KD, scale):
    B, C, H, W = t.shape
    u = t.reshape(B, nh, 4, KD, H * W).permute(2, 0, 1, 4, 3)
    o_lo = torch.nn.functional.scaled_dot_product_attention(u[0], u[1], u[2], scale=scale)
    o_hi = torch.nn.functional.scaled_dot_product_attention(u[0], u[1], u[3], scale=scale)
    return torch.stack([o_lo, o_hi], dim=2).permute(0, 1, 2, 4, 3).reshape(B, nh * 2 * KD, H, W)


def test_psa_backward_central_differences(oracle):
    B, nh, KD, H, W = 1, 2, 2, 2, 3
    qkv = _rand((B, nh * 4 * KD, H, W), 70)
    dout = _rand((B, nh * 2 * KD, H, W), 71)
    dvres = _rand((B, nh * 2 * KD, H, W), 72)
    scale = 1 / math.sqrt(KD)
    dqkv = oracle.psa_bwd(qkv, dout, nh, KD, scale, dvres=dvres)

    def loss(x):
        out, _, vres = oracle.psa_fwd(x, nh, KD, scale)
        return float(np.sum(out * dout) + np.sum(vres * dvres))

    for idx in np.ndindex(*qkv.shape):
        num = _fd(loss, qkv, idx)
        assert abs(num - dqkv[idx]) <= 1e-6 * max(1.0, abs(dqkv[idx])), (idx, num, dqkv[idx])


def test_planted_mistakes_are_caught(tmp_path):
    """A plausible mistake planted in a copy of the oracle's C source (built on the
    CPU) must fail the library-routine pin."""
    import ctypes
    import subprocess

    src = open(os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "psa_oracle.c")).read()
    mutations = {
        "dropped_max": ("if (p[j] > m)\n            m = p[j];", ""),
        "wrong_lse": ("return m + log(l);", "return log(l);"),
        "wrong_sign_ds": ("double ds = p[j] * (dp[j] - D);", "double ds = p[j] * (dp[j] + D);"),
        "transposed_dk": ("dk[j * dqk + c] += scale * ds * q[i * dqk + c];",
                          "dk[j * dqk + c] += scale * ds * k[i * dqk + c];"),
    }
    BH, N, d = 1, 5, 3
    q, k, v, do = (_rand((BH, N, d), 80 + i) for i in range(4))
    tq, tk, tv = (torch.from_numpy(a).requires_grad_() for a in (q, k, v))
    ref_o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.7)
    ref_o.backward(torch.from_numpy(do))
    ref_lse = torch.logsumexp(torch.from_numpy(q) @ torch.from_numpy(k).transpose(1, 2) * 0.7, -1).numpy()
    for name, (old, new) in mutations.items():
        assert old in src, name
        path = tmp_path / f"{name}.c"
        path.write_text(src.replace(old, new))
        so = tmp_path / f"{name}.so"
        subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-pthread", str(path), "-o", str(so), "-lm"],
                       check=True)
        lib = ctypes.CDLL(str(so))
        o = np.empty((BH, N, d)); lse = np.empty((BH, N))
        dq = np.empty_like(q); dk = np.empty_like(k); dv = np.empty_like(v)
        P = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        lib.oracle_attn_fwd.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 + [ctypes.c_double, ctypes.c_int]
        lib.oracle_attn_bwd.argtypes = [ctypes.c_void_p] * 7 + [ctypes.c_int] * 4 + [ctypes.c_double, ctypes.c_int]
        lib.oracle_attn_fwd(P(q), P(k), P(v), P(o), P(lse), BH, N, d, d, 0.7, 1)
        lib.oracle_attn_bwd(P(q), P(k), P(v), P(do), P(dq), P(dk), P(dv), BH, N, d, d, 0.7, 1)
        ok = (np.allclose(o, ref_o.detach().numpy(), atol=1e-10) and np.allclose(lse, ref_lse, atol=1e-10)
              and np.allclose(dq, tq.grad.numpy(), atol=1e-10) and np.allclose(dk, tk.grad.numpy(), atol=1e-10)
              and np.allclose(dv, tv.grad.numpy(), atol=1e-10))
        assert not ok, f"planted mistake {name} was not caught"
