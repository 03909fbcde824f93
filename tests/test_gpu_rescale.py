"""The online softmax when a row maximum jumps (vision-rs book, page "Custom
Kernels", section "Flash Attention 2": the forward keeps a running maximum and
sum per query row while it walks the key tiles).

The forward kernels rescale their output accumulator lazily: only when a row's
maximum grows by more than 2^8 after its first key tile.  With i.i.d. N(0, 1)
inputs that never happens, so these inputs plant a direction shared by every
query and by keys whose weight grows along the sequence (or one dominant last
key), which makes the maximum jump by about 2^10 per key tile.  Each case first
checks on the host that the planted inputs do make the maxima jump by more than
2^8 (in base-2 units of the scaled scores, per key group the kernel walks), then
compares the forward with the oracle at the usual bars.

The backward has no such branch (it takes P from the forward's log-sum-exp), but
the dominant-key inputs also exercise it with large logits.  There dV = P^T dO
reaches magnitudes above 4 (one key receives most of the attention), where
rounding to bf16 alone moves a value by more than 1.5e-2, so its per-element bar
is 1.5e-2 + 2^-8 |ref|, with the usual mean-relative bar of 3e-3.  dQ and dK are
not compared on planted inputs, because no kernel that rounds dS to bf16 before
its products and takes delta from the stored bf16 output (as these do, the way
the pages' backward is built) can meet the bars there: dQ_i = scale sum_j dS_ij K_j
and dK_j = scale sum_i dS_ij Q_i weight large shared components of K or Q with
values of dS that cancel exactly in the fp64 oracle (the rows of dS sum to zero,
and dS vanishes for a key that takes all the attention).  Computed in exact
arithmetic from bf16-rounded dS and a delta of the bf16-rounded output, dQ on
these shapes misses the bars by up to 10x (max-abs up to 0.15, mean-relative up
to 2.4e-2) and dK by up to 1.5x.  Every other input in the suite compares all
three gradients."""
import math

import numpy as np
import pytest

from helpers import assert_close, to_device, to_host_f64
from vision_transformer_attention_psapackqkv_gb300 import binding as B
from vision_transformer_attention_psapackqkv_gb300.inputs import (rescale_fa2_inputs,
                                                                  rescale_psa_inputs, storage_to_f64)

pytestmark = pytest.mark.gpu

LOG2E = 1.4426950408889634


def rows_with_jumps(q, k, scale, group, stride):
    """Number of query rows whose running maximum over key groups rises by more than 8
    (base-2 units of scale * q.k): groups are keys [g*stride, g*stride + group)."""
    s = (q @ k.T) * scale * LOG2E
    N = k.shape[0]
    starts = range(0, N, stride)
    m = None
    jumped = np.zeros(q.shape[0], dtype=bool)
    for g0 in starts:
        cols = s[:, g0:min(g0 + group, N)]
        if cols.shape[1] == 0:
            continue
        mx = cols.max(axis=1)
        if m is None:
            m = mx
            continue
        up = mx > m + 8.0
        jumped |= up
        m = np.where(up, mx, m)
    return int(jumped.sum())


@pytest.mark.parametrize("mode", ["growing", "late_key"])
@pytest.mark.parametrize("Bn,nh,KD,H,W", [
    (2, 2, 32, 20, 20),   # N = 400: two threads per query row, one per 32-key half
    (1, 2, 32, 24, 24),   # N = 576: one thread per query row
    (2, 1, 64, 12, 12),   # key_dim 64
])
def test_psa_fused_rescale(oracle, mode, Bn, nh, KD, H, W):
    import torch

    N = H * W
    scale = 1.0 / math.sqrt(KD)
    ins = rescale_psa_inputs(Bn, nh, KD, H, W, seed=31, mode=mode)
    q64 = storage_to_f64(ins["qkv"], "bf16")
    heads = q64.reshape(Bn, nh, 4, KD, N)
    q0, k0 = heads[0, 0, 0].T, heads[0, 0, 1].T
    if KD == 32 and N <= 512:
        # two threads per row, each walking one 32-key half of every 64-key tile
        jumps = [rows_with_jumps(q0, k0, scale, 32, 64), rows_with_jumps(q0, k0[32:], scale, 32, 64)]
    else:
        jumps = [rows_with_jumps(q0, k0, scale, 64, 64)]
    # every half jumps on growing scores; one dominant key sits in one half only
    assert (min(jumps) if mode == "growing" else max(jumps)) >= N // 8, \
        f"planted inputs make too few maxima jump: {jumps}"

    qkv = to_device(ins["qkv"], "bf16")
    shape = B.shape_of(qkv, nh, KD)
    out = torch.empty((Bn, nh * 2 * KD, H, W), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((Bn * nh, N), dtype=torch.float32, device="cuda")
    v = torch.empty_like(out)
    B.psa_attention_fwd(qkv, out, lse, v, shape, scale)
    ref_out, ref_lse, ref_v = oracle.psa_fwd(q64, nh, KD, scale)
    assert_close(to_host_f64(out), ref_out, "bf16", "out")
    np.testing.assert_allclose(to_host_f64(lse), ref_lse, atol=2e-3, rtol=0)
    np.testing.assert_array_equal(to_host_f64(v), ref_v)

    if mode != "late_key":
        return
    dout = to_device(ins["dout"], "bf16")
    ws = torch.empty(B.psa_attention_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    dqkv = torch.empty_like(qkv)
    B.psa_attention_bwd(qkv, out, dout, lse, None, dqkv, ws, shape, scale)
    torch.cuda.synchronize()
    assert B.psa_get_last_device_error() == 0
    assert torch.all(torch.isfinite(dqkv.float()))
    ref = oracle.psa_bwd(q64, storage_to_f64(ins["dout"], "bf16"), nh, KD, scale).reshape(Bn, nh, 4, KD, N)
    got = to_host_f64(dqkv).reshape(Bn, nh, 4, KD, N)
    for s, name in ((2, "dV_lo"), (3, "dV_hi")):
        assert_close(got[:, :, s], ref[:, :, s], "bf16", name, output_rounding=True)


@pytest.mark.parametrize("mode", ["growing", "late_key"])
@pytest.mark.parametrize("BH,N,d", [(3, 400, 32), (2, 333, 64)])
def test_fa2_rescale(oracle, mode, BH, N, d):
    import torch

    scale = 1.0 / math.sqrt(d)
    ins = rescale_fa2_inputs(BH, N, d, seed=41, mode=mode)
    f64 = {n: storage_to_f64(a, "bf16") for n, a in ins.items()}
    assert rows_with_jumps(f64["q"][0], f64["k"][0], scale, 64, 64) >= N // 8

    q, k, v, do = (to_device(ins[n], "bf16") for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty((BH, N), dtype=torch.float32, device="cuda")
    B.flash_attn2_fwd(q, k, v, o, lse, scale)
    ref_o, ref_lse = oracle.attn_fwd(f64["q"], f64["k"], f64["v"], scale)
    assert_close(to_host_f64(o), ref_o, "bf16", "O")
    np.testing.assert_allclose(to_host_f64(lse), ref_lse, atol=2e-3, rtol=0)

    if mode != "late_key":
        return
    delta = torch.empty((BH, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B.flash_attn2_bwd_dq(q, k, v, o, do, lse, delta, dq, scale)
    B.flash_attn2_bwd_dkdv(q, k, v, do, lse, delta, dk, dv, scale)
    torch.cuda.synchronize()
    assert B.psa_get_last_device_error() == 0
    _, _, ref_dv = oracle.attn_bwd(f64["q"], f64["k"], f64["v"], f64["do"], scale)
    assert torch.all(torch.isfinite(dq.float())) and torch.all(torch.isfinite(dk.float()))
    assert_close(to_host_f64(dv), ref_dv, "bf16", "dV", output_rounding=True)
