"""Thin ctypes binding over ``libattn_train.so`` (include/attn_train.h).

Argument marshalling only: torch tensors become (pointer, strides) views,
the current torch CUDA stream becomes the ``void* stream`` argument, and a
non-OK status becomes an exception.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU or PyTorch fallback, and calling
anything here without the built library raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libattn_train.so")

MASKS = {"full": 0, "causal": 1, "ttt": 2, "window": 3}
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_ALIGNMENT",
          4: "ATTN_ERR_WORKSPACE", 5: "ATTN_ERR_CUDA", 6: "ATTN_ERR_DEVICE_TIMEOUT",
          7: "ATTN_ERR_DEVICE_CHECK"}

# Entry points of include/attn_train.h (checked against the header by the tests).
EXPORTS = ("attn_train_supports", "attn_train_describe", "attn_train_workspace_size",
           "attn_train_fwd",
           "attn_train_fwd_workspace_size", "attn_train_fwd_ws", "attn_train_bwd",
           "attn_train_bwd_passes", "attn_train_bwd_noalloc", "attn_train_last_error", "attn_train_device_status", "attn_train_set_wait_budget_ns",
           "attn_train_mask_pattern", "attn_train_probe_mma", "attn_train_selftest_wait_timeout",
           "attn_train_selftest_debug_check",
           "attn_train_logsoftmax_loss_fwd", "attn_train_logsoftmax_loss_bwd",
           "attn_train_step_host_arena_size", "attn_train_host_session_arena_size",
           "attn_train_step_host", "attn_train_host_session_create",
           "attn_train_host_session_create_slots", "attn_train_host_session_step",
           "attn_train_host_session_join", "attn_train_host_session_destroy")


class AttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_h", ctypes.c_int64), ("stride_s", ctypes.c_int64)]


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("Sq", ctypes.c_int), ("Skv", ctypes.c_int), ("D", ctypes.c_int),
                ("mask", ctypes.c_int), ("ttt_step", ctypes.c_int), ("scale", ctypes.c_float),
                ("out_dtype", ctypes.c_int), ("window_left", ctypes.c_int),
                ("window_right", ctypes.c_int), ("seq_lengths", ctypes.c_void_p),
                ("add_mask", ctypes.c_void_p), ("add_mask_sb", ctypes.c_int64),
                ("add_mask_sq", ctypes.c_int64)]


OUT_DTYPES = {"bf16": 0, "fp32": 1}


class HostIO(ctypes.Structure):
    """attn_host_io: host addresses of one step's inputs and outputs."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "dout", "o", "lse", "dq", "dk", "dv")]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load the library (build it first with ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing "
                               "(run __graft_entry__.build())")
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(Problem)
        T = Tensor
        vp = ctypes.c_void_p
        st = ctypes.c_int
        sig = {
            "attn_train_supports": (st, [P]),
            "attn_train_workspace_size": (st, [P, ctypes.POINTER(ctypes.c_size_t)]),
            "attn_train_fwd": (st, [P, T, T, T, T, vp, vp]),
            "attn_train_fwd_workspace_size": (st, [P, ctypes.POINTER(ctypes.c_size_t)]),
            "attn_train_fwd_ws": (st, [P, T, T, T, T, vp, vp, ctypes.c_size_t, vp]),
            "attn_train_bwd": (st, [P, T, T, T, T, T, vp, T, T, T, vp, ctypes.c_size_t, vp]),
            "attn_train_bwd_passes": (st, [P, ctypes.c_uint, T, T, T, T, T, vp, T, T, T, vp,
                                           ctypes.c_size_t, vp]),
            "attn_train_bwd_noalloc": (st, [P, T, T, T, T, T, vp, T, T, T, vp]),
            "attn_train_last_error": (ctypes.c_char_p, []),
            "attn_train_device_status": (st, [vp]),
            "attn_train_set_wait_budget_ns": (st, [ctypes.c_uint64]),
            "attn_train_mask_pattern": (st, [P, vp, vp, vp]),
            "attn_train_probe_mma": (st, [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp]),
            "attn_train_selftest_wait_timeout": (st, [vp]),
            "attn_train_selftest_debug_check": (st, [vp]),
            "attn_train_logsoftmax_loss_fwd": (st, [ctypes.c_int64, ctypes.c_int64, vp,
                                                    ctypes.c_int64, vp, ctypes.c_int64, vp,
                                                    vp, vp, vp, vp, vp]),
            "attn_train_logsoftmax_loss_bwd": (st, [ctypes.c_int64, ctypes.c_int64, vp,
                                                    ctypes.c_int64, vp, ctypes.c_int64, vp,
                                                    vp, vp, vp, vp]),
            "attn_train_step_host_arena_size": (st, [P, ctypes.c_int,
                                                     ctypes.POINTER(ctypes.c_size_t)]),
            "attn_train_step_host": (st, [P, ctypes.POINTER(HostIO), ctypes.c_int, vp,
                                          ctypes.c_size_t, vp]),
            "attn_train_host_session_create": (st, [P, ctypes.c_int, vp, ctypes.c_size_t,
                                                    ctypes.POINTER(vp)]),
            "attn_train_describe": (st, [P, ctypes.c_char_p, ctypes.c_size_t,
                                         ctypes.POINTER(ctypes.c_size_t)]),
            "attn_train_host_session_arena_size": (st, [P, ctypes.c_int, ctypes.c_int,
                                                        ctypes.POINTER(ctypes.c_size_t)]),
            "attn_train_host_session_create_slots": (st, [P, ctypes.c_int, ctypes.c_int, vp,
                                                          ctypes.c_size_t, ctypes.POINTER(vp)]),
            "attn_train_host_session_step": (st, [vp, ctypes.POINTER(HostIO), vp]),
            "attn_train_host_session_join": (st, [vp, vp]),
            "attn_train_host_session_destroy": (st, [vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        msg = load().attn_train_last_error().decode(errors="replace")
        raise AttnError(status, msg)


def _lens_ptr(seq_lengths, host=False) -> int:
    """Address of an int32 [B] tensor of key lengths (0 = none); a CUDA tensor,
    or a CPU one for the host-memory step (host=True)."""
    if seq_lengths is None:
        return 0
    import torch
    where = "CPU" if host else "CUDA"
    if (seq_lengths.dtype != torch.int32 or seq_lengths.is_cuda == host
            or not seq_lengths.is_contiguous()):
        raise ValueError(f"seq_lengths must be a contiguous int32 {where} tensor")
    return seq_lengths.data_ptr()


def _add_mask(add_mask, host=False):
    """(address, batch stride, row stride) of a bf16 additive mask [Sq, Skv]
    or [B, Sq, Skv] with contiguous keys; a 2-D or batch-1 mask serves every entry.
    A CUDA tensor, or a CPU one for the host-memory step (host=True)."""
    if add_mask is None:
        return 0, 0, 0
    import torch
    where = "CPU" if host else "CUDA"
    if add_mask.dtype != torch.bfloat16 or add_mask.is_cuda == host or add_mask.stride(-1) != 1:
        raise ValueError(f"add_mask must be a bf16 {where} tensor with contiguous keys")
    sb = 0 if add_mask.dim() == 2 or add_mask.shape[0] == 1 else add_mask.stride(0)
    return add_mask.data_ptr(), sb, add_mask.stride(-2)


def problem(B, Hq, Hkv, Sq, Skv, D, mask="causal", ttt_step=0, scale=0.0, out="bf16",
            window=None, seq_lengths=None, add_mask=None, host=False) -> Problem:
    """window=(left, right) for the window mask; seq_lengths = int32 [B] key
    lengths; add_mask = bf16 additive mask; both device tensors, or CPU tensors
    with host=True (the problem of step_host).  The caller keeps the tensors
    alive while the problem is used."""
    m = MASKS[mask] if isinstance(mask, str) else int(mask)
    wl, wr = (0, 0) if window is None else (int(window[0]), int(window[1]))
    am, amsb, amsq = _add_mask(add_mask, host)
    return Problem(B, Hq, Hkv, Sq, Skv, D, m, ttt_step, float(scale), OUT_DTYPES[out], wl, wr,
                   _lens_ptr(seq_lengths, host), am, amsb, amsq)


def problem_for(q, k, mask="causal", ttt_step=0, scale=None, out="bf16", window=None,
                seq_lengths=None, add_mask=None) -> Problem:
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    return problem(B, Hq, Hkv, Sq, Skv, D, mask, ttt_step, 0.0 if scale is None else scale, out,
                   window, seq_lengths, add_mask)


def _torch_out_dtype(out):
    import torch
    return torch.float32 if out == "fp32" else torch.bfloat16


def view(t) -> Tensor:
    """[B, H, S, D] torch tensor -> attn_tensor (D must be contiguous)."""
    if t.dim() != 4:
        raise ValueError("expected a [B, H, S, D] tensor")
    if t.stride(3) != 1:
        raise ValueError("the head dimension must be contiguous")
    return Tensor(t.data_ptr(), t.stride(0), t.stride(1), t.stride(2))


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(int(stream))
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def supports(p: Problem) -> bool:
    return load().attn_train_supports(ctypes.byref(p)) == 0


def check_supported(p: Problem):
    _check(load().attn_train_supports(ctypes.byref(p)))


def describe(p: Problem) -> dict:
    """attn_train_describe: the kernels, tiles, grids and pipeline depths the
    entry points use for this problem (a host-side plan, no device work)."""
    import json
    lib = load()
    n = ctypes.c_size_t(0)
    lib.attn_train_describe(ctypes.byref(p), None, 0, ctypes.byref(n))
    if n.value == 0:
        _check(lib.attn_train_describe(ctypes.byref(p), None, 0, ctypes.byref(n)))
    buf = ctypes.create_string_buffer(n.value)
    _check(lib.attn_train_describe(ctypes.byref(p), buf, n.value, ctypes.byref(n)))
    return json.loads(buf.value.decode())


def workspace_size(p: Problem) -> int:
    n = ctypes.c_size_t(0)
    _check(load().attn_train_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    return int(n.value)


def fwd_workspace_size(p: Problem) -> int:
    """attn_train_fwd_workspace_size: 0 unless the forward splits its key range
    (small grids) on the current device."""
    n = ctypes.c_size_t(0)
    _check(load().attn_train_fwd_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    return int(n.value)


def fwd_raw(p: Problem, q, k, v, o, lse, stream=None):
    """attn_train_fwd on caller-owned tensors (o, lse are written)."""
    _check(load().attn_train_fwd(ctypes.byref(p), view(q), view(k), view(v), view(o),
                                 ctypes.c_void_p(lse.data_ptr()), _stream(stream)))


def fwd_ws_raw(p: Problem, q, k, v, o, lse, workspace, stream=None):
    """attn_train_fwd_ws on caller-owned tensors; workspace None = no split."""
    ws = ctypes.c_void_p(workspace.data_ptr() if workspace is not None else 0)
    n = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().attn_train_fwd_ws(ctypes.byref(p), view(q), view(k), view(v), view(o),
                                    ctypes.c_void_p(lse.data_ptr()), ws, n, _stream(stream)))


def bwd_raw(p: Problem, q, k, v, o, dout, lse, dq, dk, dv, workspace, stream=None):
    """attn_train_bwd on caller-owned tensors (dq, dk, dv are written)."""
    _check(load().attn_train_bwd(ctypes.byref(p), view(q), view(k), view(v), view(o), view(dout),
                                 ctypes.c_void_p(lse.data_ptr()), view(dq), view(dk), view(dv),
                                 ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                 _stream(stream)))


BWD_PREP, BWD_DKDV, BWD_DQ, BWD_TTT, BWD_ALL = 1, 2, 4, 8, 15


def bwd_passes_raw(p: Problem, passes: int, q, k, v, o, dout, lse, dq, dk, dv, workspace,
                   stream=None):
    """attn_train_bwd_passes: enqueue only the backward passes in `passes`."""
    _check(load().attn_train_bwd_passes(ctypes.byref(p), passes, view(q), view(k), view(v),
                                        view(o), view(dout), ctypes.c_void_p(lse.data_ptr()),
                                        view(dq), view(dk), view(dv),
                                        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                        _stream(stream)))


def bwd_noalloc_raw(p: Problem, q, k, v, o, dout, lse, dq, dk, dv, stream=None):
    """attn_train_bwd_noalloc: the backward using the library's built-in
    scratch instead of a workspace (for callers that cannot allocate)."""
    _check(load().attn_train_bwd_noalloc(ctypes.byref(p), view(q), view(k), view(v), view(o),
                                         view(dout), ctypes.c_void_p(lse.data_ptr()), view(dq),
                                         view(dk), view(dv), _stream(stream)))


HOST_MAX_SLOTS = 16  # ATTN_HOST_MAX_SLOTS


def step_host_arena_size(p: Problem, kv_heads_per_chunk: int = 0, slots: int = 2) -> int:
    """Device arena bytes of attn_train_step_host (two slots) or of a host
    session with `slots` slots (kv_heads_per_chunk 0 = one chunk per step)."""
    n = ctypes.c_size_t(0)
    if slots == 2:
        _check(load().attn_train_step_host_arena_size(ctypes.byref(p), int(kv_heads_per_chunk),
                                                      ctypes.byref(n)))
    else:
        _check(load().attn_train_host_session_arena_size(ctypes.byref(p), int(kv_heads_per_chunk),
                                                         int(slots), ctypes.byref(n)))
    return int(n.value)


_HOST_IO = ("q", "k", "v", "dout", "o", "lse", "dq", "dk", "dv")


def _host_io(host: dict) -> HostIO:
    for n in _HOST_IO:
        t = host[n]
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous CPU tensor")
    return HostIO(*(host[n].data_ptr() for n in _HOST_IO))


def step_host_raw(p: Problem, host: dict, arena, kv_heads_per_chunk: int = 0, stream=None):
    """attn_train_step_host: one forward + backward from host memory.  `host`
    maps q, k, v, dout (inputs) and o, lse, dq, dk, dv (outputs) to dense CPU
    tensors (pinned for overlapped copies); `arena` is a CUDA uint8 tensor of
    at least step_host_arena_size bytes.  Returns once enqueued: the outputs
    are valid after the stream is synchronized."""
    io = _host_io(host)
    _check(load().attn_train_step_host(ctypes.byref(p), ctypes.byref(io), int(kv_heads_per_chunk),
                                       ctypes.c_void_p(arena.data_ptr()), arena.numel(),
                                       _stream(stream)))


class HostSession:
    """attn_train_host_session_*: steps of one problem from host memory whose
    copies overlap the neighbouring steps' kernels.  Keep `p` (and its host
    key lengths / mask tensors) and the arena alive while the session is used.
    `slots` (2 to HOST_MAX_SLOTS) device slots let the copies run that many
    chunks minus one ahead of or behind the kernels; the arena must hold
    step_host_arena_size(p, kv_heads_per_chunk, slots) bytes."""

    def __init__(self, p: Problem, arena, kv_heads_per_chunk: int = 0, slots: int = 2):
        self._h = ctypes.c_void_p(0)  # no session yet (close() is safe if creation fails)
        self._lib = load()
        self.p = p
        self.arena = arena
        h = ctypes.c_void_p(0)
        args = (ctypes.c_void_p(arena.data_ptr()), arena.numel(), ctypes.byref(h))
        if slots == 2:
            _check(self._lib.attn_train_host_session_create(ctypes.byref(p),
                                                            int(kv_heads_per_chunk), *args))
        else:
            _check(self._lib.attn_train_host_session_create_slots(
                ctypes.byref(p), int(kv_heads_per_chunk), int(slots), *args))
        self._h = h

    def step(self, host: dict, stream=None):
        """Enqueue one step; outputs are valid after join() and a stream sync."""
        io = _host_io(host)
        _check(self._lib.attn_train_host_session_step(self._h, ctypes.byref(io), _stream(stream)))

    def join(self, stream=None):
        _check(self._lib.attn_train_host_session_join(self._h, _stream(stream)))

    def close(self):
        if self._h:
            self._lib.attn_train_host_session_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        self.close()


def device_status(stream=None):
    _check(load().attn_train_device_status(_stream(stream)))


def set_wait_budget_ns(ns: int):
    _check(load().attn_train_set_wait_budget_ns(int(ns)))


# ------------------------------------------------------------ conveniences
def canary() -> bool:
    """ATTN_TRAIN_CANARY=1: the conveniences below fill the outputs they
    allocate with NaN and the workspace with 0xff bytes (NaN as fp32) instead of
    leaving them uninitialised, so that an element a kernel fails to write shows
    up as NaN rather than as a plausible stale value (a debugging aid; the test
    suite turns it on)."""
    return os.environ.get("ATTN_TRAIN_CANARY", "0") == "1"


def _alloc(shape, dtype, device):
    import torch
    if canary():
        return torch.full(shape, float("nan"), dtype=dtype, device=device)
    return torch.empty(shape, dtype=dtype, device=device)


def _alloc_workspace(nbytes, device):
    import torch
    if canary():
        return torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=device)
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def fwd(q, k, v, mask="causal", ttt_step=0, scale=None, stream=None, out="bf16", window=None,
        seq_lengths=None, add_mask=None, split=True):
    """Allocates O (bf16 or fp32), LSE and, when the forward splits its key range
    (attn_train_fwd_workspace_size > 0), its workspace with torch, runs the
    forward; returns (o, lse).  split=False runs attn_train_fwd (no split)."""
    import torch
    p = problem_for(q, k, mask, ttt_step, scale, out, window, seq_lengths, add_mask)
    o = _alloc(q.shape, _torch_out_dtype(out), q.device)
    lse = _alloc((q.shape[0], q.shape[1], q.shape[2]), torch.float32, q.device)
    n = fwd_workspace_size(p) if split else 0
    if n > 0:
        fwd_ws_raw(p, q, k, v, o, lse, _alloc_workspace(n, q.device), stream)
    else:
        fwd_raw(p, q, k, v, o, lse, stream)
    return o, lse


def bwd(q, k, v, o, lse, dout, mask="causal", ttt_step=0, scale=None, stream=None, workspace=None,
        window=None, seq_lengths=None, add_mask=None):
    """Allocates dQ, dK, dV (same dtype as o: bf16 or fp32) and the workspace
    unless given; returns (dq, dk, dv)."""
    import torch
    out = "fp32" if o.dtype == torch.float32 else "bf16"
    p = problem_for(q, k, mask, ttt_step, scale, out, window, seq_lengths, add_mask)
    dq = _alloc(q.shape, o.dtype, q.device)
    dk = _alloc(k.shape, o.dtype, q.device)
    dv = _alloc(v.shape, o.dtype, q.device)
    if workspace is None:
        workspace = _alloc_workspace(workspace_size(p), q.device)
    bwd_raw(p, q, k, v, o, dout, lse, dq, dk, dv, workspace, stream)
    return dq, dk, dv


def mask_pattern(Sq, Skv, mask, ttt_step=0, device="cuda", with_tiles=True, window=None,
                 seq_length=None):
    """Device view of the mask for one batch entry of key length seq_length
    (None = every key): (bits[6, Sq, Skv] uint8, tiles or None); planes 0-2 are
    the forward, dK/dV and dQ schedules the kernels run for this problem,
    planes 3-5 the same passes in the general form."""
    import torch
    lens = None if seq_length is None else torch.tensor([seq_length], dtype=torch.int32,
                                                        device=device)
    p = problem(1, 1, 1, Sq, Skv, 64, mask, ttt_step, window=window, seq_lengths=lens)
    bits = torch.zeros(6, Sq, Skv, dtype=torch.uint8, device=device)
    tiles = None
    if with_tiles:
        kv_main = Sq if p.mask == 2 else Skv
        tiles = torch.zeros(math.ceil(Sq / 128), math.ceil(kv_main / 128), dtype=torch.uint8,
                            device=device)
    _check(load().attn_train_mask_pattern(ctypes.byref(p), ctypes.c_void_p(bits.data_ptr()),
                                          ctypes.c_void_p(tiles.data_ptr() if tiles is not None else 0),
                                          _stream(None)))
    return bits, tiles


def probe_mma(mode: int, a, b, D: int):
    """One-tile tcgen05 probe; returns the fp32 product (see attn_train.h)."""
    import torch
    c = torch.zeros(128, 128 if mode == 0 else D, dtype=torch.float32, device=a.device)
    _check(load().attn_train_probe_mma(mode, D, ctypes.c_void_p(a.data_ptr()),
                                       ctypes.c_void_p(b.data_ptr()), ctypes.c_void_p(c.data_ptr()),
                                       _stream(None)))
    return c


def selftest_wait_timeout():
    _check(load().attn_train_selftest_wait_timeout(_stream(None)))


def selftest_debug_check():
    """A device-side check that fails on purpose (libraries built with
    -DATTN_DEBUG; AttnError ATTN_ERR_UNSUPPORTED otherwise)."""
    _check(load().attn_train_selftest_debug_check(_stream(None)))


# ------------------------------------------------- soft-target log-softmax loss
def _rows2d(t, name):
    """[..., V] fp32 CUDA tensor -> (rows, V, row stride) with the last dim contiguous."""
    import torch
    if t.dtype != torch.float32 or not t.is_cuda:
        raise ValueError(f"{name} must be a float32 CUDA tensor")
    if t.stride(-1) != 1:
        raise ValueError(f"{name}: the vocabulary dimension must be contiguous")
    V = t.shape[-1]
    rows = t.numel() // V
    ld = t.stride(-2) if t.dim() > 1 else V
    if t.dim() > 2 and t.stride(0) != t.shape[1] * ld:
        raise ValueError(f"{name}: leading dimensions must be dense (flattenable to rows)")
    return rows, V, ld


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def logsoftmax_loss_fwd_raw(logits, target, mask, row_loss, row_lse, row_tsum, loss=None,
                            stream=None):
    rows, V, ldl = _rows2d(logits, "logits")
    rt, Vt, ldt = _rows2d(target, "target")
    if (rt, Vt) != (rows, V):
        raise ValueError("logits and target shapes differ")
    _check(load().attn_train_logsoftmax_loss_fwd(rows, V, _ptr(logits), ldl, _ptr(target), ldt,
                                                 _ptr(mask), _ptr(row_loss), _ptr(row_lse),
                                                 _ptr(row_tsum), _ptr(loss), _stream(stream)))


def logsoftmax_loss_bwd_raw(logits, target, mask, row_lse, row_tsum, grad_loss=None, stream=None):
    rows, V, ldl = _rows2d(logits, "logits")
    rt, Vt, ldt = _rows2d(target, "target")
    if (rt, Vt) != (rows, V):
        raise ValueError("logits and target shapes differ")
    _check(load().attn_train_logsoftmax_loss_bwd(rows, V, _ptr(logits), ldl, _ptr(target), ldt,
                                                 _ptr(mask), _ptr(row_lse), _ptr(row_tsum),
                                                 _ptr(grad_loss), _stream(stream)))


def logsoftmax_loss(logits, target, mask=None, stream=None):
    """Forward: allocates the row statistics and the mean; returns
    (loss [1], row_loss, row_lse, row_tsum), all fp32 on the logits' device."""
    import torch
    rows = logits.numel() // logits.shape[-1]
    f = dict(dtype=torch.float32, device=logits.device)
    row_loss, row_lse, row_tsum = (torch.empty(rows, **f) for _ in range(3))
    loss = torch.empty(1, **f)
    m = None if mask is None else mask.reshape(-1).to(torch.float32).contiguous()
    logsoftmax_loss_fwd_raw(logits, target, m, row_loss, row_lse, row_tsum, loss, stream)
    return loss, row_loss, row_lse, row_tsum
