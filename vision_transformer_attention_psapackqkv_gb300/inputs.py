"""Seeded synthetic inputs for the PSA attention path.

This module is shared by the tests, the smoke check and the benchmark.  It holds
no attention arithmetic: it only draws i.i.d. normal values from a seeded numpy
generator and rounds them to the storage dtype (round-to-nearest-even for bf16),
so that the CUDA path and the CPU oracle receive bit-identical inputs.

bf16 tensors are carried on the host as ``uint16`` bit patterns (numpy has no
bf16); ``bf16_to_f64`` widens them exactly.

Workloads (the five PSA-shaped configurations; N = H*W, KD = key_dim):
  psa_fwd_f32_n64    B=1,  nh=2, KD=32, 8x8   fp32, forward only            seed 1
  psa_fwd_n400       B=16, nh=4, KD=32, 20x20 bf16, forward only            seed 2
  psa_fwdbwd_n400    B=64, nh=4, KD=32, 20x20 bf16, forward+backward        seed 3
  psa_fwdbwd_n1600   B=32, nh=8, KD=32, 40x40 bf16, forward+backward, x0.5  seed 4
  fa2_sweep          BH=64, N in {1024, 4096, 16384}, d in {32, 64}, bf16   seed 5
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class PsaWorkload:
    name: str
    B: int
    num_heads: int
    key_dim: int
    H: int
    W: int
    dtype: str  # "f32" or "bf16"
    backward: bool
    value_scale: float
    seed: int

    @property
    def N(self) -> int:
        return self.H * self.W

    @property
    def qkv_channels(self) -> int:
        return self.num_heads * 4 * self.key_dim

    @property
    def out_channels(self) -> int:
        return self.num_heads * 2 * self.key_dim

    @property
    def BH(self) -> int:
        return self.B * self.num_heads


PSA_WORKLOADS = {
    w.name: w
    for w in (
        PsaWorkload("psa_fwd_f32_n64", 1, 2, 32, 8, 8, "f32", False, 1.0, 1),
        PsaWorkload("psa_fwd_n400", 16, 4, 32, 20, 20, "bf16", False, 1.0, 2),
        PsaWorkload("psa_fwdbwd_n400", 64, 4, 32, 20, 20, "bf16", True, 1.0, 3),
        PsaWorkload("psa_fwdbwd_n1600", 32, 8, 32, 40, 40, "bf16", True, 0.5, 4),
    )
}

FA2_SWEEP_BH = 64
FA2_SWEEP_N = (1024, 4096, 16384)
FA2_SWEEP_D = (32, 64)
FA2_SWEEP_SEED = 5


def normal_f32(shape, seed: int, scale: float = 1.0, stream: int = 0) -> np.ndarray:
    """i.i.d. N(0, 1) * scale in float32 from numpy's default_rng((seed, stream))."""
    rng = np.random.default_rng((seed, stream))
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x = (x * np.float32(scale)).astype(np.float32)
    return x


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


def to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    """float32 values -> storage array (float32 itself, or bf16 bit patterns)."""
    if dtype == "f32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16(x32)
    raise ValueError(dtype)


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_to_f64(a)
    raise ValueError(dtype)


def psa_inputs(B: int, num_heads: int, key_dim: int, H: int, W: int, dtype: str, seed: int,
               value_scale: float = 1.0, with_grad: bool = True, with_dvres: bool = False):
    """QKV [B, nh*4*KD, H, W] and upstream gradient dOut [B, nh*2*KD, H, W] in storage form."""
    C = num_heads * 4 * key_dim
    c = num_heads * 2 * key_dim
    out = {"qkv": to_storage(normal_f32((B, C, H, W), seed, value_scale, 0), dtype)}
    if with_grad:
        out["dout"] = to_storage(normal_f32((B, c, H, W), seed, value_scale, 1), dtype)
    if with_dvres:
        out["dvres"] = to_storage(normal_f32((B, c, H, W), seed, value_scale, 2), dtype)
    return out


def workload_inputs(w: PsaWorkload, with_dvres: bool = False):
    return psa_inputs(w.B, w.num_heads, w.key_dim, w.H, w.W, w.dtype, w.seed, w.value_scale,
                      with_grad=True, with_dvres=with_dvres)


def fa2_inputs(BH: int, N: int, d: int, dtype: str, seed: int, value_scale: float = 1.0):
    """Q, K, V, dO of shape [BH, N, d] in storage form."""
    return {name: to_storage(normal_f32((BH, N, d), seed, value_scale, i), dtype)
            for i, name in enumerate(("q", "k", "v", "do"))}


# --------------------------------------------------------------------------- planted score growth
def planted_direction(d: int, seed: int) -> np.ndarray:
    """A seeded unit vector of length d (float32)."""
    u = normal_f32((d,), seed, 1.0, 7).astype(np.float64)
    return (u / np.linalg.norm(u)).astype(np.float32)


def planted_shifts(N: int, d: int, scale: float, seed: int, mode: str, tile: int = 64,
                   growth_log2: float = 10.0, q_shift: float = 3.0):
    """Additive offsets (float32) for query and key rows of one head that make the
    scores of a query row grow along the key sequence, so that an online softmax
    over key tiles meets a row maximum that rises by more than 2^8 after its first
    tile (the case in which a lazily rescaled accumulator must be rescaled).

    Every query row gets q_shift * u and key row n gets c_n * u, with u a fixed unit
    vector, so a score gains about q_shift * c_n * scale, i.e.
    q_shift * c_n * scale * log2(e) in base-2 units.  mode "growing": c_n rises by
    growth_log2 base-2 units per key tile of `tile` keys (c_n proportional to
    n // tile); mode "late_key": only the last key row is shifted, by
    (N // tile + 1) * growth_log2 base-2 units.  Returns (dq [d], dk [N, d])."""
    u = planted_direction(d, seed)
    per_tile = growth_log2 / (q_shift * scale * 1.4426950408889634)
    c = np.zeros(N, dtype=np.float64)
    if mode == "growing":
        c = (np.arange(N) // tile) * per_tile
    elif mode == "late_key":
        c[N - 1] = (N // tile + 1) * per_tile
    else:
        raise ValueError(mode)
    dq = (q_shift * u).astype(np.float32)
    dk = (c[:, None] * u[None, :]).astype(np.float32)
    return dq, dk


def rescale_fa2_inputs(BH: int, N: int, d: int, seed: int, mode: str = "growing"):
    """fa2_inputs (bf16) with planted_shifts added to Q and K before rounding."""
    scale = 1.0 / np.sqrt(d)
    dq, dk = planted_shifts(N, d, scale, seed, mode)
    out = {}
    for i, name in enumerate(("q", "k", "v", "do")):
        x = normal_f32((BH, N, d), seed, 1.0, i)
        if name == "q":
            x = x + dq[None, None, :]
        elif name == "k":
            x = x + dk[None, :, :]
        out[name] = f32_to_bf16(x.astype(np.float32))
    return out


def rescale_psa_inputs(B: int, num_heads: int, key_dim: int, H: int, W: int, seed: int,
                       mode: str = "growing"):
    """psa_inputs (bf16, with dOut) with planted_shifts added to the Q and K channels
    of every head (positions n = h*W + w) before rounding."""
    N, KD = H * W, key_dim
    scale = 1.0 / np.sqrt(KD)
    dq, dk = planted_shifts(N, KD, scale, seed, mode)
    C = num_heads * 4 * KD
    qkv = normal_f32((B, C, H, W), seed, 1.0, 0).reshape(B, num_heads, 4, KD, N)
    qkv[:, :, 0] += dq[None, None, :, None]
    qkv[:, :, 1] += dk.T[None, None, :, :]
    out = {"qkv": f32_to_bf16(qkv.reshape(B, C, H, W).astype(np.float32))}
    out["dout"] = f32_to_bf16(normal_f32((B, num_heads * 2 * KD, H, W), seed, 1.0, 1))
    return out


def conv_inputs(B: int, cin: int, cout: int, H: int, W: int, seed: int, with_bias: bool = True):
    """Input feature map x [B, cin, H, W] (N(0, 1)), QKV weights w [cout, cin]
    (N(0, 1) / sqrt(cin), so outputs have unit scale) as bf16 bits, and bias [cout]
    (N(0, 0.25), float32) or None.  Synthetic weights: no trained model is involved."""
    x = f32_to_bf16(normal_f32((B, cin, H, W), seed, 1.0, 10))
    w = f32_to_bf16(normal_f32((cout, cin), seed, 1.0 / float(np.sqrt(cin)), 11))
    bias = normal_f32((cout,), seed, 0.5, 12) if with_bias else None
    return {"x": x, "w": w, "bias": bias}
