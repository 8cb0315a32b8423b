"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws random numbers and
names shapes, so both the CUDA path and the fp64 oracle take their inputs
from here.

Recipe (the same for every workload): each tensor is drawn as fp32 N(0, 1)
from its own ``torch.Generator`` seeded with ``seed * 16 + index`` (Q=0, K=1,
V=2, dO=3), then rounded once to bf16 (round-to-nearest-even).  Both sides
consume the rounded values; the oracle widens them to fp64.

The shapes follow the pages' workloads: the CS336 README's benchmark grid
(B=8, one head, d in {16, 32, 64}, S in {256, 1024, 4096}), the SpecForge
post's long-context EAGLE3 training (16K tokens, GQA, TTT steps that append
K/V segments, padded batches with per-sequence lengths) and HOT-Step's DiT
trainer geometries (windowed and full self-attention, cross-attention with a
short encoder sequence).  Per-batch key lengths are fixed tuples, not draws.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

MASKS = ("full", "causal", "ttt", "window")


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    mask: str  # "full" | "causal" | "ttt" | "window"
    ttt_step: int = 0
    seed: int = 0
    window: tuple | None = None       # (left, right) extents of the window mask
    seq_lengths: tuple | None = None  # per-batch key lengths (padding), None = all keys
    add_mask: bool = False            # one additive bf16 mask [Sq, Skv] for all entries

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def describe(self) -> dict:
        d = {"workload": self.name, "B": self.B, "Hq": self.Hq, "Hkv": self.Hkv, "Sq": self.Sq,
             "Skv": self.Skv, "D": self.D, "mask": self.mask}
        if self.mask == "ttt":
            d["ttt_step"] = self.ttt_step
        if self.window is not None:
            d["window"] = list(self.window)
        if self.seq_lengths is not None:
            d["seq_lengths"] = list(self.seq_lengths)
        if self.add_mask:
            d["add_mask"] = "bf16 [Sq, Skv]: 0.5 N(0,1), 10% -inf, key 0 finite"
        return d


def ttt_workload(step: int, S: int = 8192, B: int = 1, Hq: int = 32, Hkv: int = 8, D: int = 128,
                 seed: int = 3) -> Workload:
    """EAGLE3 Training-Time-Test draft attention at TTT step ``step``: the
    queries are one segment of S rows, the K/V cache holds step+1 segments."""
    return Workload(f"eagle3_ttt_step{step}", B, Hq, Hkv, S, (step + 1) * S, D, "ttt", step, seed)


# The named workloads (shapes only).
TINY = Workload("tiny_causal_B1_H2_S128_D64", 1, 2, 2, 128, 128, 64, "causal", 0, 0)
SWEEP = tuple(
    Workload(f"sweep_causal_B8_H1_S{S}_D{D}", 8, 1, 1, S, S, D, "causal", 0, 1)
    for D in (16, 32, 64) for S in (256, 1024, 4096))
LONG_GQA = Workload("long_causal_gqa_B1_Hq32_Hkv4_S16384_D128", 1, 32, 4, 16384, 16384, 128,
                    "causal", 0, 2)
TTT_STEPS = tuple(ttt_workload(t) for t in range(7))
DIT_SELF = Workload("dit_full_self_B2_H16_S12288_D64", 2, 16, 16, 12288, 12288, 64, "full", 0, 4)
DIT_CROSS = Workload("dit_full_cross_B2_H16_Sq12288_Skv512_D64", 2, 16, 16, 12288, 512, 64,
                     "full", 0, 4)

# Windowed self-attention of the DiT geometry (HOT-Step's trainer has windowed,
# full and cross attention layers; the window extent is not given there: a band
# of +-1024 keys is taken here) and an LLM-style causal sliding window on the
# long GQA shape.
DIT_WINDOW = Workload("dit_window_self_B2_H16_S12288_D64_w1024", 2, 16, 16, 12288, 12288, 64,
                      "window", 0, 4, window=(1024, 1024))
SWA_GQA = Workload("swa_causal_gqa_B1_Hq32_Hkv4_S16384_D128_w4096", 1, 32, 4, 16384, 16384, 128,
                   "window", 0, 2, window=(4095, 0))
# Padded batches (SpecForge's seq_lengths): causal GQA and a TTT step.
VARLEN_GQA = Workload("varlen_causal_gqa_B4_Hq32_Hkv4_S8192_D128", 4, 32, 4, 8192, 8192, 128,
                      "causal", 0, 5, seq_lengths=(8192, 6000, 3100, 1000))
VARLEN_TTT = Workload("varlen_eagle3_ttt_step2_B2_Hq32_Hkv8_S8192_D128", 2, 32, 8, 8192, 3 * 8192,
                      128, "ttt", 2, 6, seq_lengths=(8192, 5000))

# Full self-attention with an additive bias table (HOT-Step section 3: its ops
# accept an arbitrary additive mask, the form in which its DiT trainer passes masks).
DIT_ADDMASK = Workload("dit_addmask_self_B2_H16_S4096_D64", 2, 16, 16, 4096, 4096, 64, "full", 0,
                       4, add_mask=True)

ALL = ((TINY,) + SWEEP + (LONG_GQA,) + TTT_STEPS + (DIT_SELF, DIT_CROSS) +
       (DIT_WINDOW, SWA_GQA, VARLEN_GQA, VARLEN_TTT, DIT_ADDMASK))

# Smaller cases of the same kernels for hardware-counter captures (inputs
# still larger than the 129 MB L2 once outputs are counted).
PROFILE = (Workload("profile_causal_gqa_B1_Hq32_Hkv4_S4096_D128", 1, 32, 4, 4096, 4096, 128,
                    "causal", 0, 2),)


def by_name(name: str) -> Workload:
    for w in ALL + PROFILE:
        if w.name == name:
            return w
    raise KeyError(name)


def _draw(shape, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_inputs(w: Workload, seed: int | None = None, with_dout: bool = True) -> dict:
    """Contiguous [B, H, S, D] bf16 CPU tensors q, k, v (and dout)."""
    s = w.seed if seed is None else seed
    out = {
        "q": _draw((w.B, w.Hq, w.Sq, w.D), s * 16 + 0),
        "k": _draw((w.B, w.Hkv, w.Skv, w.D), s * 16 + 1),
        "v": _draw((w.B, w.Hkv, w.Skv, w.D), s * 16 + 2),
    }
    if with_dout:
        out["dout"] = _draw((w.B, w.Hq, w.Sq, w.D), s * 16 + 3)
    if w.seq_lengths is not None:
        out["seq_lengths"] = torch.tensor(w.seq_lengths, dtype=torch.int32)
    if w.add_mask:
        # an additive bias like a relative-position table with holes: 0.5 N(0, 1),
        # about 10% of the pairs hidden (-inf), key 0 always open (no empty row)
        g = torch.Generator(device="cpu")
        g.manual_seed(s * 16 + 4)
        m = torch.randn(w.Sq, w.Skv, generator=g) * 0.5
        m[torch.rand(w.Sq, w.Skv, generator=g) < 0.1] = float("-inf")
        m[:, 0] = 0.0
        out["add_mask"] = m.to(torch.bfloat16)
    return out


def zero_k(inputs: dict) -> dict:
    """Copy of ``inputs`` with K set to zero (uniform attention weights)."""
    d = dict(inputs)
    d["k"] = torch.zeros_like(inputs["k"])
    return d


# ------------------------------------------------- soft-target log-softmax loss
@dataclass(frozen=True)
class LossWorkload:
    """The SpecForge post's loss benchmark shapes ("In-place Gradient
    Calculation", table of (B, T, V)): fp32 logits and soft targets over a
    vocabulary of V, one position mask per (b, t)."""
    name: str
    B: int
    T: int
    V: int
    seed: int = 7

    @property
    def rows(self) -> int:
        return self.B * self.T

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "T": self.T, "V": self.V}


LOSS = tuple(LossWorkload(f"logsoftmax_loss_B{B}_T{T}_V{V}", B, T, V)
             for B, T, V in ((1, 1024, 32000), (1, 4096, 32000), (1, 4096, 64000),
                             (1, 8192, 32000), (1, 8192, 64000), (1, 16384, 32000)))


def make_loss_inputs(w: LossWorkload, rows: slice | None = None) -> dict:
    """fp32 CPU tensors: logits [B, T, V] ~ 2 N(0, 1); target [B, T, V] = u / sum(u)
    with u ~ Exp(1) (a point drawn uniformly from the probability simplex, the
    shape of a teacher's soft distribution); mask [B, T] in {0, 1}, about 10%
    zeros (padding positions).  Each tensor has its own generator seeded
    seed * 16 + index."""
    g = [torch.Generator(device="cpu") for _ in range(3)]
    for i, gi in enumerate(g):
        gi.manual_seed(w.seed * 16 + 8 + i)
    logits = torch.randn(w.B, w.T, w.V, generator=g[0], dtype=torch.float32) * 2.0
    u = torch.empty(w.B, w.T, w.V, dtype=torch.float32).exponential_(generator=g[1])
    target = u / u.sum(dim=-1, keepdim=True)
    mask = (torch.rand(w.B, w.T, generator=g[2]) >= 0.1).to(torch.float32)
    return {"logits": logits, "target": target, "mask": mask}
