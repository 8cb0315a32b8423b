"""fp64 CPU oracle for masked training attention (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never links,
loads or calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over the
(b, h) pairs); this module only compiles it with gcc and marshals numpy
arrays.  Every function follows the plain definition of attention:

* SpecForge long-context post, "EAGLE3 Training": softmax(Q K^T / sqrt(d_k)) V.
* SpecForge post, "Flex Attention": the eagle3 ``mask_mod`` =
  or(causal_mask, suffix_mask), read with shift_left = t (the number of
  appended TTT segments), Q_LEN = Sq and KV_LEN = (t+1) Sq; its padding terms
  take optional per-batch key lengths ``seq_lengths``.
* HOT-Step flash-attn-training, section 4 (self-attention over a window): the
  window mask, read as the band q - left <= kv <= q + right; section 3: an
  optional additive mask [B or 1, Sq, Skv] added to the scaled scores
  (-inf hides a pair), shared by every head.
* CS336 README, "Flash Attention (Triton)": LSE saved by the forward; the
  backward recomputes P from it.
* HOT-Step flash-attn-training, section 6 trap 9: a row with no visible key
  has O = 0 and LSE = 0.

Parity is pinned (finite differences, brute force, invariants, the EAGLE3
concatenated-score construction, torch fp64 sdpa, closed forms) by
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MASK_FULL = 0
MASK_CAUSAL = 1
MASK_TTT = 2
MASK_WINDOW = 3
MASK_NAMES = {"full": MASK_FULL, "causal": MASK_CAUSAL, "ttt": MASK_TTT, "window": MASK_WINDOW}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so with gcc (-O3 -fopenmp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-std=c99", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            L = ctypes.c_long
            lib.oracle_visible.restype = ctypes.c_int
            lib.oracle_visible.argtypes = [ctypes.c_int, ctypes.c_int] + [L] * 7
            lib.oracle_mask.restype = None
            lib.oracle_mask.argtypes = [ctypes.c_int, ctypes.c_int] + [L] * 5 + [ctypes.c_void_p]
            # mask, t, wl, wr, lens, additive mask, its batch stride
            geom = [ctypes.c_int, ctypes.c_int, L, L, ctypes.c_void_p, dp, L]
            lib.oracle_fwd.restype = ctypes.c_int
            lib.oracle_fwd.argtypes = [ctypes.c_int] * 3 + [L, L, ctypes.c_int] + geom + [
                ctypes.c_double] + [dp] * 5
            lib.oracle_bwd.restype = ctypes.c_int
            lib.oracle_bwd.argtypes = [ctypes.c_int] * 3 + [L, L, ctypes.c_int] + geom + [
                ctypes.c_double] + [dp] * 7
            lib.oracle_fwd_rows.restype = ctypes.c_int
            lib.oracle_fwd_rows.argtypes = lib.oracle_fwd.argtypes + [L, L]
            lib.oracle_bwd_rows.restype = ctypes.c_int
            lib.oracle_bwd_rows.argtypes = lib.oracle_bwd.argtypes + [L, L]
            lib.oracle_count_visible.restype = ctypes.c_longlong
            lib.oracle_count_visible.argtypes = [ctypes.c_int, ctypes.c_int] + [L] * 5
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_num_threads.argtypes = []
            _lib = lib
    return _lib


def _mask_id(mask) -> int:
    return MASK_NAMES[mask] if isinstance(mask, str) else int(mask)


def _f64(a) -> np.ndarray:
    """Contiguous fp64 numpy copy of a numpy array or a CPU torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_scale(D: int) -> float:
    return 1.0 / float(np.sqrt(D))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _window(window):
    """(left, right) extents of the window mask; (0, 0) when unused."""
    if window is None:
        return 0, 0
    wl, wr = window
    return int(wl), int(wr)


def _len(length) -> int:
    return -1 if length is None else int(length)


def visible(mask, t: int, Sq: int, Skv: int, q: int, kv: int, window=None, length=None) -> bool:
    """Visibility of key kv to query q.  window=(left, right) for the window
    mask; length = the batch entry's key length (seq_lengths[b]), None = all."""
    wl, wr = _window(window)
    return bool(_load().oracle_visible(_mask_id(mask), t, wl, wr, _len(length), Sq, Skv, q, kv))


def mask(mask, t: int, Sq: int, Skv: int, window=None, length=None) -> np.ndarray:
    """Dense [Sq, Skv] uint8 visibility bitmap of one batch entry."""
    out = np.zeros((Sq, Skv), dtype=np.uint8)
    wl, wr = _window(window)
    _load().oracle_mask(_mask_id(mask), t, wl, wr, _len(length), Sq, Skv, out.ctypes.data)
    return out


def count_visible(mask, t: int, Sq: int, Skv: int, window=None, length=None) -> int:
    wl, wr = _window(window)
    return int(_load().oracle_count_visible(_mask_id(mask), t, wl, wr, _len(length), Sq, Skv))


def _dims(q, k):
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    if Bk != B or Dk != D:
        raise ValueError("q/k shape mismatch")
    return B, Hq, Hkv, Sq, Skv, D


def _lens(seq_lengths, B):
    """int32 [B] array of per-batch key lengths (kept alive by the caller), or None."""
    if seq_lengths is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(seq_lengths, dtype=np.int32).reshape(-1))
    if a.shape[0] != B:
        raise ValueError("seq_lengths needs one entry per batch")
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _add(add_mask, B, Sq, Skv):
    """fp64 [Bm, Sq, Skv] copy of an additive mask (Bm = 1 or B), a pointer to it
    and its batch stride."""
    if add_mask is None:
        return None, None, 0
    a = _f64(add_mask)
    if a.ndim == 2:
        a = a[None]
    if a.shape[1:] != (Sq, Skv) or a.shape[0] not in (1, B):
        raise ValueError("additive mask must be [Sq, Skv], [1, Sq, Skv] or [B, Sq, Skv]")
    a = np.ascontiguousarray(a)
    return a, _ptr(a), (0 if a.shape[0] == 1 else Sq * Skv)


def fwd(q, k, v, mask="causal", t: int = 0, scale: float | None = None, rows=None,
        window=None, seq_lengths=None, add_mask=None):
    """Returns (O [B,Hq,Sq,D], LSE [B,Hq,Sq]) in fp64.  rows=(begin, end)
    restricts the work to those query rows (others stay zero); window=(left,
    right) for the window mask; seq_lengths = per-batch key lengths."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, Hkv, Sq, Skv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else float(scale)
    r0, r1 = (0, Sq) if rows is None else rows
    wl, wr = _window(window)
    keep, lens = _lens(seq_lengths, B)
    akeep, aptr, asb = _add(add_mask, B, Sq, Skv)
    o = np.zeros((B, Hq, Sq, D))
    lse = np.zeros((B, Hq, Sq))
    rc = _load().oracle_fwd_rows(B, Hq, Hkv, Sq, Skv, D, _mask_id(mask), t, wl, wr, lens, aptr,
                                 asb, scale, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), r0, r1)
    del keep, akeep
    if rc != 0:
        raise ValueError(f"oracle_fwd rejected the problem (code {rc})")
    return o, lse


def bwd(q, k, v, do, mask="causal", t: int = 0, scale: float | None = None, rows=None,
        window=None, seq_lengths=None, add_mask=None):
    """Returns (dQ, dK, dV) in fp64; dK/dV summed over each kv head's q heads.
    rows=(begin, end) restricts the work to those query rows: dQ of those
    rows and their contributions to dK/dV."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, Hkv, Sq, Skv, D = _dims(q, k)
    scale = default_scale(D) if scale is None else float(scale)
    r0, r1 = (0, Sq) if rows is None else rows
    wl, wr = _window(window)
    keep, lens = _lens(seq_lengths, B)
    akeep, aptr, asb = _add(add_mask, B, Sq, Skv)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rc = _load().oracle_bwd_rows(B, Hq, Hkv, Sq, Skv, D, _mask_id(mask), t, wl, wr, lens, aptr, asb,
                                 scale, _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk),
                                 _ptr(dv), r0, r1)
    del keep, akeep
    if rc != 0:
        raise ValueError(f"oracle_bwd rejected the problem (code {rc})")
    return dq, dk, dv
