"""Mask-aware FLOP and byte counts (host logic for the benchmark).

FLOPs follow the usual count for attention: the forward does two dense
contractions per visible (q, kv) pair (Q K^T and P V), 2*D multiply-adds each,
so F_fwd = 4 * D * N_vis.  The backward does five (S recompute, dP, dV, dK,
dQ), so F_bwd = 2.5 * F_fwd.  Extra contractions that a two-pass
deterministic schedule executes are not counted.  N_vis is the exact number
of visible pairs, summed over batch and q heads (not rounded to tiles).

Visible pairs per (b, h), in closed form:
  full:   Sq * Skv
  causal: sum_q min(q + 1, Skv)                                (kv <= q)
  ttt(t): sum_{q >= t} (q - t + 1)  +  t * Sq                  (shifted causal
          part of segment 0 plus one diagonal key per appended segment)
These closed forms are checked against the oracle's brute-force count.
"""
from __future__ import annotations


def visible_pairs_per_head(mask: str, Sq: int, Skv: int, t: int = 0) -> int:
    if mask == "full":
        return Sq * Skv
    if mask == "causal":
        # rows q < Skv see q+1 keys, rows q >= Skv see Skv keys
        m = min(Sq, Skv)
        return m * (m + 1) // 2 + max(0, Sq - Skv) * Skv
    if mask == "ttt":
        n = max(0, Sq - t)  # rows q >= t see q - t + 1 keys of segment 0
        return n * (n + 1) // 2 + t * Sq
    raise ValueError(mask)


def visible_pairs(w) -> int:
    return w.B * w.Hq * visible_pairs_per_head(w.mask, w.Sq, w.Skv, w.ttt_step)


def flops_fwd(w) -> float:
    return 4.0 * w.D * visible_pairs(w)


def flops_bwd(w) -> float:
    return 2.5 * flops_fwd(w)


def flops_fwd_bwd(w) -> float:
    return 3.5 * flops_fwd(w)


def bytes_fwd(w) -> int:
    """Algorithmic HBM bytes of one forward: read Q, K, V; write O, LSE."""
    return w.B * (w.Hq * w.Sq * w.D * 2 * 2 + w.Hkv * w.Skv * w.D * 2 * 2 + w.Hq * w.Sq * 4)


def bytes_bwd(w) -> int:
    """Algorithmic HBM bytes of one backward: read Q, O, dO, K, V, LSE;
    write dQ, dK, dV (and the Delta row statistic)."""
    return w.B * (w.Hq * w.Sq * w.D * 2 * 4 + w.Hkv * w.Skv * w.D * 2 * 4 + w.Hq * w.Sq * 4 * 2)
