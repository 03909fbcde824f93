"""Thin Python binding of libpsa_gb300.so (the C ABI declared in include/psa.h).

Every function carries the C entry point's name and only marshals arguments:
torch tensors become device pointers, the current torch CUDA stream becomes the
cudaStream_t, and a non-OK status raises PsaError.  All computation happens in
the library's kernels; there is no fallback of any kind.  If the shared library
has not been built, the first call raises RuntimeError.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

PSA_OK = 0
PSA_DTYPE_F32 = 0
PSA_DTYPE_BF16 = 1

_lib = None


class PsaError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed with status {status}: {message}")
        self.status = status


class PsaShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("num_heads", ctypes.c_int), ("key_dim", ctypes.c_int),
                ("H", ctypes.c_int), ("W", ctypes.c_int), ("dtype", ctypes.c_int)]


EXPORTED = (
    "psa_qkv_conv", "psa_pack_qkv", "psa_unpack_qkv", "psa_extract_v", "psa_merge_attn", "psa_unmerge_attn",
    "flash_attn2_fwd", "flash_attn2_bwd_dq", "flash_attn2_bwd_dkdv", "psa_attention_fwd",
    "psa_attention_fwd_residual", "psa_attention_bwd", "psa_attention_bwd_dq", "psa_attention_bwd_dkdv", "psa_attention_bwd_noalloc",
    "psa_attention_bwd_workspace_size", "psa_status_string",
    "psa_get_last_device_error", "psa_debug_wait_timeout",
)


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Loads the shared library (built by ``_build.build()`` / ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libpsa_gb300.so is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, F, S, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, PsaShape, ctypes.c_size_t
    sigs = {
        "psa_qkv_conv": [P, P, P, P, I, I, I, I, I, P],
        "psa_pack_qkv": [P, P, S, P],
        "psa_unpack_qkv": [P, P, S, P],
        "psa_extract_v": [P, P, S, P],
        "psa_merge_attn": [P, P, P, S, P],
        "psa_unmerge_attn": [P, P, P, S, P],
        "flash_attn2_fwd": [P, P, P, P, P, I, I, I, F, I, P],
        "flash_attn2_bwd_dq": [P, P, P, P, P, P, P, P, I, I, I, F, I, P],
        "flash_attn2_bwd_dkdv": [P, P, P, P, P, P, P, P, I, I, I, F, I, P],
        "psa_attention_fwd": [P, P, P, P, S, F, P],
        "psa_attention_fwd_residual": [P, P, P, P, S, F, P],
        "psa_attention_bwd": [P, P, P, P, P, P, P, Z, S, F, P],
        "psa_attention_bwd_dq": [P, P, P, P, P, P, S, F, P],
        "psa_attention_bwd_dkdv": [P, P, P, P, P, P, S, F, P],
        "psa_attention_bwd_noalloc": [P, P, P, P, P, P, S, F, P],
        "psa_attention_bwd_workspace_size": [S],
        "psa_status_string": [I],
        "psa_get_last_device_error": [P],
        "psa_debug_wait_timeout": [ctypes.c_ulonglong, P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.psa_attention_bwd_workspace_size.restype = ctypes.c_size_t
    lib.psa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, status: int):
    if status != PSA_OK:
        raise PsaError(fn, status, load().psa_status_string(status).decode())


def dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return PSA_DTYPE_BF16
    if t.dtype == torch.float32:
        return PSA_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def shape_of(qkv, num_heads: int, key_dim: int) -> PsaShape:
    B, C, H, W = qkv.shape
    if C != num_heads * 4 * key_dim:
        raise ValueError(f"QKV has {C} channels, expected num_heads*4*key_dim = {num_heads * 4 * key_dim}")
    return PsaShape(B, num_heads, key_dim, H, W, dtype_code(qkv))


# ------------------------------------------------------------------ QKV convolution
def psa_qkv_conv(x, weight, bias, qkv, stream=None):
    """x [B, cin, H, W] bf16, weight [cout, cin] bf16, bias [cout] fp32 or None -> qkv."""
    Bn, cin, H, W = x.shape
    cout = weight.shape[0]
    _check("psa_qkv_conv", load().psa_qkv_conv(_ptr(x), _ptr(weight), _ptr(bias), _ptr(qkv), Bn, cin,
                                                cout, H, W, _stream(stream)))


# ------------------------------------------------------------------ layout
def psa_pack_qkv(qkv, packed, shape: PsaShape, stream=None):
    _check("psa_pack_qkv", load().psa_pack_qkv(_ptr(qkv), _ptr(packed), shape, _stream(stream)))


def psa_unpack_qkv(packed, qkv, shape: PsaShape, stream=None):
    _check("psa_unpack_qkv", load().psa_unpack_qkv(_ptr(packed), _ptr(qkv), shape, _stream(stream)))


def psa_extract_v(qkv, v_nchw, shape: PsaShape, stream=None):
    _check("psa_extract_v", load().psa_extract_v(_ptr(qkv), _ptr(v_nchw), shape, _stream(stream)))


def psa_merge_attn(o_lo, o_hi, out, shape: PsaShape, stream=None):
    _check("psa_merge_attn", load().psa_merge_attn(_ptr(o_lo), _ptr(o_hi), _ptr(out), shape, _stream(stream)))


def psa_unmerge_attn(dout, do_lo, do_hi, shape: PsaShape, stream=None):
    _check("psa_unmerge_attn",
           load().psa_unmerge_attn(_ptr(dout), _ptr(do_lo), _ptr(do_hi), shape, _stream(stream)))


# ------------------------------------------------------------------ Flash Attention 2
def flash_attn2_fwd(q, k, v, o, lse, scale: float, stream=None):
    BH, N, d = q.shape
    _check("flash_attn2_fwd", load().flash_attn2_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), BH, N, d, float(scale), dtype_code(q),
        _stream(stream)))


def flash_attn2_bwd_dq(q, k, v, o, do, lse, delta, dq, scale: float, stream=None):
    BH, N, d = q.shape
    _check("flash_attn2_bwd_dq", load().flash_attn2_bwd_dq(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(delta), _ptr(dq), BH, N, d,
        float(scale), dtype_code(q), _stream(stream)))


def flash_attn2_bwd_dkdv(q, k, v, do, lse, delta, dk, dv, scale: float, stream=None):
    BH, N, d = q.shape
    _check("flash_attn2_bwd_dkdv", load().flash_attn2_bwd_dkdv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(delta), _ptr(dk), _ptr(dv), BH, N, d,
        float(scale), dtype_code(q), _stream(stream)))


# ------------------------------------------------------------------ fused PSA
def psa_attention_fwd(qkv, out, lse, v_nchw, shape: PsaShape, scale: float, stream=None):
    _check("psa_attention_fwd", load().psa_attention_fwd(
        _ptr(qkv), _ptr(out), _ptr(lse), _ptr(v_nchw), shape, float(scale), _stream(stream)))


def psa_attention_fwd_residual(qkv, out_res, out, lse, shape: PsaShape, scale: float, stream=None):
    _check("psa_attention_fwd_residual", load().psa_attention_fwd_residual(
        _ptr(qkv), _ptr(out_res), _ptr(out), _ptr(lse), shape, float(scale), _stream(stream)))


def psa_attention_bwd_workspace_size(shape: PsaShape) -> int:
    return int(load().psa_attention_bwd_workspace_size(shape))


def psa_attention_bwd(qkv, out, dout, lse, dvres, dqkv, workspace, shape: PsaShape, scale: float,
                      stream=None):
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("psa_attention_bwd", load().psa_attention_bwd(
        _ptr(qkv), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dvres), _ptr(dqkv), _ptr(workspace),
        ws_bytes, shape, float(scale), _stream(stream)))


def psa_attention_bwd_dq(qkv, out, dout, lse, delta, dqkv, shape: PsaShape, scale: float, stream=None):
    _check("psa_attention_bwd_dq", load().psa_attention_bwd_dq(
        _ptr(qkv), _ptr(out), _ptr(dout), _ptr(lse), _ptr(delta), _ptr(dqkv), shape, float(scale),
        _stream(stream)))


def psa_attention_bwd_dkdv(qkv, dout, lse, delta, dvres, dqkv, shape: PsaShape, scale: float, stream=None):
    _check("psa_attention_bwd_dkdv", load().psa_attention_bwd_dkdv(
        _ptr(qkv), _ptr(dout), _ptr(lse), _ptr(delta), _ptr(dvres), _ptr(dqkv), shape, float(scale),
        _stream(stream)))


def psa_attention_bwd_noalloc(qkv, out, dout, lse, dvres, dqkv, shape: PsaShape, scale: float, stream=None):
    _check("psa_attention_bwd_noalloc", load().psa_attention_bwd_noalloc(
        _ptr(qkv), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dvres), _ptr(dqkv), shape, float(scale),
        _stream(stream)))


def psa_get_last_device_error(stream=None) -> int:
    return int(load().psa_get_last_device_error(_stream(stream)))


def psa_debug_wait_timeout(limit_ns: int, stream=None):
    _check("psa_debug_wait_timeout", load().psa_debug_wait_timeout(int(limit_ns), _stream(stream)))


def psa_status_string(status: int) -> str:
    return load().psa_status_string(int(status)).decode()
