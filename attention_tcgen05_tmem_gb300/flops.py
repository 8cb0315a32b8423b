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
With a window mask or per-batch key lengths the count is the exact sum over
rows of the visible key interval (plus the t diagonals of rows below the
length for TTT).  All of them are checked against the oracle's brute-force
count.  An additive mask does not change the count: its -inf entries are
data, and the kernels compute every pair the mask kind admits.
"""
from __future__ import annotations

import numpy as np


def visible_pairs_rows(mask: str, Sq: int, Skv: int, t: int = 0, window=None, length=None,
                       r0: int = 0, r1: int | None = None) -> int:
    """Visible pairs of query rows [r0, r1) of one head: the row's visible key
    interval [lo, hi] of the tiled part, plus the t suffix diagonals of TTT
    rows below the key length."""
    r1 = Sq if r1 is None else r1
    q = np.arange(r0, r1, dtype=np.int64)
    kv_main = Sq if mask == "ttt" else Skv
    L = kv_main if length is None else min(max(int(length), 0), kv_main)
    lo = np.zeros_like(q)
    if mask == "full":
        hi = np.full_like(q, L - 1)
    elif mask == "causal":
        hi = np.minimum(q, L - 1)
    elif mask == "ttt":
        hi = np.minimum(q - t, L - 1)
    elif mask == "window":
        wl, wr = window
        lo = np.maximum(q - wl, 0)
        hi = np.minimum(q + wr, L - 1)
    else:
        raise ValueError(mask)
    n = int(np.maximum(hi - lo + 1, 0).sum())
    if mask == "ttt":
        n += t * int((q < L).sum())
    return n


def visible_pairs_per_head(mask: str, Sq: int, Skv: int, t: int = 0, window=None,
                           length=None) -> int:
    if window is not None or length is not None:
        return visible_pairs_rows(mask, Sq, Skv, t, window, length)
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


def _lengths(w):
    return w.seq_lengths if w.seq_lengths is not None else (None,) * w.B


def visible_pairs(w) -> int:
    if w.window is None and w.seq_lengths is None:
        return w.B * w.Hq * visible_pairs_per_head(w.mask, w.Sq, w.Skv, w.ttt_step)
    return w.Hq * sum(visible_pairs_per_head(w.mask, w.Sq, w.Skv, w.ttt_step, w.window, L)
                      for L in _lengths(w))


def diagonal_pairs(w) -> int:
    """TTT suffix-diagonal pairs (one per appended segment and row below the
    key length), summed over batch and q heads."""
    if w.mask != "ttt":
        return 0
    return w.Hq * sum(w.ttt_step * (w.Sq if L is None else min(max(L, 0), w.Sq))
                      for L in _lengths(w))


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
