"""GB300 (sm_103a) Position-Sensitive Attention: PsaPackQkv -> Flash Attention 2 (per V
half) -> PsaMergeAttn, PsaExtractV, and the dQ / dK-dV backward, as hand-written
CUDA kernels behind the C ABI of include/psa.h.  ``binding`` is the Python view of
that ABI; ``inputs`` draws the seeded synthetic workloads."""

from . import binding  # noqa: F401

__all__ = ["binding", "inputs"]
