"""Shared helpers of the GPU tests: host <-> device conversion of the seeded inputs
and the tolerance checks (the same bars everywhere).

Tolerances against the fp64 oracle:
  layout kernels (pack / unpack / extract / merge / unmerge): bit-exact;
  fp32 attention: max |x - ref| <= 1e-4;
  bf16 attention: max |x - ref| <= 1.5e-2 and sum|x - ref| / sum|ref| <= 3e-3.
"""
import numpy as np

F32_MAX_ABS = 1e-4
BF16_MAX_ABS = 1.5e-2
BF16_MEAN_REL = 3e-3


def to_device(a: np.ndarray, dtype: str):
    import torch

    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def to_host_bits(t) -> np.ndarray:
    """Raw element bits of a device tensor (uint16 for bf16, uint32 for fp32)."""
    import torch

    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy().view(np.uint32)
    raise TypeError(t.dtype)


def to_host_f64(t) -> np.ndarray:
    import torch

    return t.detach().to(torch.float64).cpu().numpy()


def errors(x: np.ndarray, ref: np.ndarray):
    d = np.abs(x - ref)
    denom = float(np.sum(np.abs(ref)))
    return float(d.max()) if d.size else 0.0, (float(d.sum()) / denom if denom > 0 else float(d.sum()))


def assert_close(x: np.ndarray, ref: np.ndarray, dtype: str, what: str = "",
                 output_rounding: bool = False, roundings: int = 1):
    """The bars above.  With output_rounding, each bf16 element may in addition be
    off by half a bf16 ulp of its reference (2^-8 |ref|): used where the outputs
    reach magnitudes >= 4 (a residual gradient added into dV), at which rounding
    to bf16 alone can move a value by more than 1.5e-2.  roundings = 2 is for a sum
    of two results that were each rounded to bf16 before the sum (the two-call
    chain's dQ and dK): its mean-relative bar is twice the single-rounding one."""
    assert x.shape == ref.shape, (what, x.shape, ref.shape)
    assert np.all(np.isfinite(x)), f"{what}: non-finite values"
    max_abs, mean_rel = errors(x, ref)
    if dtype == "f32":
        assert max_abs <= F32_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {F32_MAX_ABS}"
    else:
        if output_rounding:
            excess = float(np.max(np.abs(x - ref) - (BF16_MAX_ABS + np.abs(ref) * 2.0 ** -8)))
            assert excess <= 0, f"{what}: error exceeds 1.5e-2 + 2^-8|ref| by {excess:.3e}"
        else:
            assert max_abs <= BF16_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {BF16_MAX_ABS}"
        bar = BF16_MEAN_REL * roundings
        assert mean_rel <= bar, f"{what}: mean-rel {mean_rel:.3e} > {bar}"
    return max_abs, mean_rel
