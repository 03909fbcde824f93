"""fp64 CPU oracle for the Position-Sensitive Attention (PSA) path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; the library's product path never
imports it, and it imports nothing from the library.

The arithmetic lives in ``psa_oracle.c`` (plain loops in double precision); this
module compiles it with gcc and marshals numpy arrays through ctypes.  See the
header of ``psa_oracle.c`` for the passages each routine follows (vision-rs book,
page "Custom Kernels", sections "Flash Attention 2" and "Position-Sensitive
Attention (PSA)") and for the readings taken where the page is silent.

Layout routines (pack / unpack / extract / merge / unmerge) accept arrays of any
dtype and move raw elements, so they are bit-exact references.  Attention
routines take and return float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "psa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpsa_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile psa_oracle.c into a shared library (portable flags, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        for name in ("oracle_pack_qkv", "oracle_unpack_qkv", "oracle_extract_v"):
            getattr(lib, name).argtypes = [P, P, I, I, I, I, I]
        lib.oracle_merge_attn.argtypes = [P, P, P, I, I, I, I, I]
        lib.oracle_unmerge_attn.argtypes = [P, P, P, I, I, I, I, I]
        lib.oracle_attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, D, I]
        lib.oracle_attn_bwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, D, I]
        lib.oracle_attn_fwd_rows.argtypes = [P, P, P, I, I, I, D, P, I, P, P]
        lib.oracle_attn_bwd_dq_rows.argtypes = [P, P, P, P, I, I, I, D, P, I, P]
        lib.oracle_attn_bwd_dkdv_rows.argtypes = [P, P, P, P, I, I, I, D, P, I, P, P, I]
        lib.oracle_psa_fwd.argtypes = [P, P, P, P, I, I, I, I, D, I]
        lib.oracle_psa_bwd.argtypes = [P, P, P, P, I, I, I, I, D, I]
        lib.oracle_psa_fwd_residual.argtypes = [P, P, P, I, I, I, I, D, I]
        lib.oracle_qkv_conv.argtypes = [P, P, P, P, I, I, I, I]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    a = np.asarray(a)
    if dtype is not None:
        a = a.astype(dtype, copy=False)
    return np.ascontiguousarray(a)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------- layouts
def pack_qkv(qkv, num_heads: int, key_dim: int):
    """PsaPackQkv: NCHW [B, nh*4*KD, H, W] -> [4, B*nh, H*W, KD] (raw element copy)."""
    qkv = _c(qkv)
    B, C, H, W = qkv.shape
    assert C == num_heads * 4 * key_dim
    out = np.empty((4, B * num_heads, H * W, key_dim), dtype=qkv.dtype)
    _load().oracle_pack_qkv(_ptr(qkv), _ptr(out), B, num_heads, key_dim, H * W, qkv.itemsize)
    return out


def unpack_qkv(packed, B: int, num_heads: int, key_dim: int, H: int, W: int):
    """Inverse of pack_qkv: [4, B*nh, N, KD] -> [B, nh*4*KD, H, W]."""
    packed = _c(packed)
    out = np.empty((B, num_heads * 4 * key_dim, H, W), dtype=packed.dtype)
    _load().oracle_unpack_qkv(_ptr(packed), _ptr(out), B, num_heads, key_dim, H * W, packed.itemsize)
    return out


def extract_v(qkv, num_heads: int, key_dim: int):
    """PsaExtractV: NCHW [B, nh*4*KD, H, W] -> [B, nh*2*KD, H, W] (raw element copy)."""
    qkv = _c(qkv)
    B, C, H, W = qkv.shape
    out = np.empty((B, num_heads * 2 * key_dim, H, W), dtype=qkv.dtype)
    _load().oracle_extract_v(_ptr(qkv), _ptr(out), B, num_heads, key_dim, H * W, qkv.itemsize)
    return out


def merge_attn(o_lo, o_hi, B: int, num_heads: int, key_dim: int, H: int, W: int):
    """PsaMergeAttn: two [B*nh, N, KD] halves -> NCHW [B, nh*2*KD, H, W]."""
    o_lo, o_hi = _c(o_lo), _c(o_hi)
    assert o_lo.dtype == o_hi.dtype
    out = np.empty((B, num_heads * 2 * key_dim, H, W), dtype=o_lo.dtype)
    _load().oracle_merge_attn(_ptr(o_lo), _ptr(o_hi), _ptr(out), B, num_heads, key_dim, H * W,
                              o_lo.itemsize)
    return out


def unmerge_attn(out, num_heads: int, key_dim: int):
    """Inverse of merge_attn: NCHW [B, nh*2*KD, H, W] -> two [B*nh, N, KD] halves."""
    out = _c(out)
    B, c, H, W = out.shape
    lo = np.empty((B * num_heads, H * W, key_dim), dtype=out.dtype)
    hi = np.empty_like(lo)
    _load().oracle_unmerge_attn(_ptr(out), _ptr(lo), _ptr(hi), B, num_heads, key_dim, H * W,
                                out.itemsize)
    return lo, hi


# --------------------------------------------------------------------------- attention
def attn_fwd(q, k, v, scale: float, nthreads: int | None = None):
    """Softmax attention over [BH, N, d] (float64): returns O [BH, N, dv], LSE [BH, N]."""
    q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
    BH, N, dqk = q.shape
    dv = v.shape[2]
    o = np.empty((BH, N, dv))
    lse = np.empty((BH, N))
    _load().oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), BH, N, dqk, dv,
                            float(scale), nthreads or default_threads())
    return o, lse


def attn_bwd(q, k, v, dout, scale: float, nthreads: int | None = None):
    """Analytic backward of attn_fwd: returns dQ, dK, dV (float64)."""
    q, k, v, dout = (_c(a, np.float64) for a in (q, k, v, dout))
    BH, N, dqk = q.shape
    dv = v.shape[2]
    dq, dk, dvv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dvv),
                            BH, N, dqk, dv, float(scale), nthreads or default_threads())
    return dq, dk, dvv


def attn_fwd_rows(q, k, v, scale: float, rows):
    """Output rows of one head ([N, d] arrays): returns O[rows] and LSE[rows]."""
    q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
    rows = _c(rows, np.int64)
    N, dqk = q.shape
    dv = v.shape[1]
    o = np.empty((len(rows), dv))
    lse = np.empty(len(rows))
    _load().oracle_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), N, dqk, dv, float(scale), _ptr(rows),
                                 len(rows), _ptr(o), _ptr(lse))
    return o, lse


def attn_bwd_dq_rows(q, k, v, dout, scale: float, rows):
    """dQ rows of one head ([N, d] arrays)."""
    q, k, v, dout = (_c(a, np.float64) for a in (q, k, v, dout))
    rows = _c(rows, np.int64)
    N, dqk = q.shape
    dv = v.shape[1]
    dq = np.empty((len(rows), dqk))
    _load().oracle_attn_bwd_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), N, dqk, dv, float(scale),
                                    _ptr(rows), len(rows), _ptr(dq))
    return dq


def attn_bwd_dkdv_rows(q, k, v, dout, scale: float, keys, nthreads: int | None = None):
    """dK and dV rows for the given keys of one head ([N, d] arrays)."""
    q, k, v, dout = (_c(a, np.float64) for a in (q, k, v, dout))
    keys = _c(keys, np.int64)
    N, dqk = q.shape
    dv = v.shape[1]
    dk = np.empty((len(keys), dqk))
    dvv = np.empty((len(keys), dv))
    _load().oracle_attn_bwd_dkdv_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), N, dqk, dv,
                                      float(scale), _ptr(keys), len(keys), _ptr(dk), _ptr(dvv),
                                      nthreads or default_threads())
    return dk, dvv


# --------------------------------------------------------------------------- the PSA chain
def psa_fwd(qkv, num_heads: int, key_dim: int, scale: float, nthreads: int | None = None):
    """PSA forward on NCHW [B, nh*4KD, H, W] (float64): returns out [B, nh*2KD, H, W],
    LSE [B*nh, H*W] and the extracted V [B, nh*2KD, H, W]."""
    qkv = _c(qkv, np.float64)
    B, C, H, W = qkv.shape
    assert C == num_heads * 4 * key_dim
    out = np.empty((B, num_heads * 2 * key_dim, H, W))
    vres = np.empty_like(out)
    lse = np.empty((B * num_heads, H * W))
    _load().oracle_psa_fwd(_ptr(qkv), _ptr(out), _ptr(lse), _ptr(vres), B, num_heads, key_dim,
                           H * W, float(scale), nthreads or default_threads())
    return out, lse, vres


def qkv_conv(x, w, bias=None):
    """QKV 1x1 convolution (float64): x [B, cin, H, W], w [cout, cin], bias [cout] or
    None -> [B, cout, H, W]."""
    x = _c(x, np.float64)
    w = _c(w, np.float64)
    bias = None if bias is None else _c(bias, np.float64)
    B, cin, H, W = x.shape
    cout = w.shape[0]
    assert w.shape == (cout, cin)
    out = np.empty((B, cout, H, W))
    _load().oracle_qkv_conv(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), B, cin, cout, H * W)
    return out


def psa_fwd_residual(qkv, num_heads: int, key_dim: int, scale: float, nthreads: int | None = None):
    """PSA forward with its residual path added (float64): returns out + vres
    [B, nh*2KD, H, W] and LSE [B*nh, H*W]."""
    qkv = _c(qkv, np.float64)
    B, C, H, W = qkv.shape
    assert C == num_heads * 4 * key_dim
    out = np.empty((B, num_heads * 2 * key_dim, H, W))
    lse = np.empty((B * num_heads, H * W))
    _load().oracle_psa_fwd_residual(_ptr(qkv), _ptr(out), _ptr(lse), B, num_heads, key_dim, H * W,
                                    float(scale), nthreads or default_threads())
    return out, lse


def psa_bwd(qkv, dout, num_heads: int, key_dim: int, scale: float, dvres=None,
            nthreads: int | None = None):
    """Gradient of sum(dout o out) (+ sum(dvres o vres)) w.r.t. the NCHW QKV tensor."""
    qkv = _c(qkv, np.float64)
    dout = _c(dout, np.float64)
    dvres = None if dvres is None else _c(dvres, np.float64)
    B, C, H, W = qkv.shape
    dqkv = np.empty_like(qkv)
    _load().oracle_psa_bwd(_ptr(qkv), _ptr(dout), _ptr(dvres), _ptr(dqkv), B, num_heads, key_dim,
                           H * W, float(scale), nthreads or default_threads())
    return dqkv
