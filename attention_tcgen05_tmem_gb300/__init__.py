"""Fused training attention (forward + deterministic backward) for GB300.

The compute runs in hand-written sm_103a CUDA kernels (tcgen05 MMA with
accumulators in tensor memory, TMA-fed shared-memory tiles) behind the C ABI
declared in ``include/attn_train.h``.  This package is the thin Python
binding over that library (``binding``), plus seeded synthetic inputs
(``synth``) and mask-aware FLOP counts (``flops``).
"""
from . import flops, synth  # noqa: F401

__all__ = ["flops", "synth"]
