"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/attn_train.h declares, and rejects malformed or
unsupported problems with the right status before touching the device
(HOT-Step flash-attn-training, section 2: unsupported shapes must fail hard,
never fall back)."""
import ctypes
import os
import re

import pytest

from attention_tcgen05_tmem_gb300 import binding
from attention_tcgen05_tmem_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_train.h")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return binding.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_train_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(binding.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def _p(**kw):
    base = dict(B=1, Hq=4, Hkv=2, Sq=256, Skv=256, D=64, mask="causal", ttt_step=0, scale=0.0)
    base.update(kw)
    return binding.problem(**base)


def _status(lib, p):
    return lib.attn_train_supports(ctypes.byref(p))


def test_supports_accepts_the_workloads(lib):
    from attention_tcgen05_tmem_gb300 import synth
    for w in synth.ALL:
        p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step,
                            window=w.window)
        assert _status(lib, p) == 0, (w.name, lib.attn_train_last_error())


@pytest.mark.parametrize("kw,status", [
    (dict(D=80), 2), (dict(D=256), 2), (dict(D=0), 1), (dict(Hq=6, Hkv=4), 1),
    (dict(B=0), 1), (dict(Sq=-1), 1), (dict(mask=7), 2),
    (dict(mask="ttt", ttt_step=2, Skv=256), 1), (dict(mask="ttt", ttt_step=-1), 1),
    (dict(scale=float("nan")), 1),
    (dict(mask="window", window=(-1, 4)), 1), (dict(mask="window", window=(3, -2)), 1),
    (dict(mask="causal", window=(3, 0)), 1),
])
def test_supports_rejects(lib, kw, status):
    p = _p(**kw)
    assert _status(lib, p) == status
    assert lib.attn_train_last_error()


def test_additive_mask_rules(lib):
    p = _p(Skv=256)
    p.add_mask, p.add_mask_sq = 0x10000, 256
    assert _status(lib, p) == 0
    p.add_mask = 0x10008
    assert _status(lib, p) == 3          # not 16-byte aligned
    p.add_mask, p.add_mask_sq = 0x10000, 260
    assert _status(lib, p) == 3          # row stride not a multiple of 8
    p.add_mask_sq = 248
    assert _status(lib, p) == 1          # row stride below Skv
    q = _p(mask="ttt", ttt_step=1, Skv=512)
    q.add_mask, q.add_mask_sq = 0x10000, 512
    assert _status(lib, q) == 2          # not with TTT


def test_misaligned_seq_lengths_are_rejected(lib):
    p = _p()
    p.seq_lengths = 0x1002
    assert _status(lib, p) == 3
    p.seq_lengths = 0x1004
    assert _status(lib, p) == 0
    assert _status(lib, _p(mask="window", window=(0, 0))) == 0


def test_workspace_size(lib):
    p = _p(B=2, Hq=3, Hkv=1, Sq=100)
    assert binding.workspace_size(p) == ((2 * 3 * 100 * 4 + 255) // 256) * 256
    p = binding.problem(1, 32, 4, 16384, 16384, 128, "causal")
    assert binding.workspace_size(p) == 32 * 16384 * 4  # linear in S
    # TTT step t: Delta plus per-row weight and score gradient of each diagonal
    p = binding.problem(1, 32, 8, 8192, 7 * 8192, 128, "ttt", 6)
    assert binding.workspace_size(p) == 32 * 8192 * 4 * (1 + 2 * 6)


def _t(ptr=0x1000, sb=4 * 256 * 64, sh=256 * 64, ss=64):
    return binding.Tensor(ptr, sb, sh, ss)


@pytest.mark.parametrize("which,tensor,status", [
    ("q", _t(ptr=0), 1),            # null
    ("q", _t(ptr=0x1008), 3),       # misaligned pointer
    ("k", _t(ss=68), 3),            # row stride not a multiple of 16 bytes
    ("v", _t(ss=32), 1),            # rows overlap
    ("o", _t(sh=-64), 1),           # negative stride
])
def test_fwd_rejects_bad_tensors_on_host(lib, which, tensor, status):
    p = _p()
    args = {n: _t() for n in ("q", "k", "v", "o")}
    args[which] = tensor
    st = lib.attn_train_fwd(ctypes.byref(p), args["q"], args["k"], args["v"], args["o"],
                            ctypes.c_void_p(0x2000), None)
    assert st == status, lib.attn_train_last_error()


def test_fwd_rejects_null_lse(lib):
    p = _p()
    st = lib.attn_train_fwd(ctypes.byref(p), _t(), _t(), _t(), _t(), None, None)
    assert st == 1


def test_bwd_rejects_small_workspace(lib):
    p = _p()
    t = _t()
    st = lib.attn_train_bwd(ctypes.byref(p), t, t, t, t, t, ctypes.c_void_p(0x2000), t, t, t,
                            ctypes.c_void_p(0x10000), 16, None)
    assert st == 4
    st = lib.attn_train_bwd(ctypes.byref(p), t, t, t, t, t, ctypes.c_void_p(0x2000), t, t, t,
                            None, 1 << 20, None)
    assert st == 4
    st = lib.attn_train_bwd(ctypes.byref(p), t, t, t, t, t, ctypes.c_void_p(0x2000), t, t, t,
                            ctypes.c_void_p(0x10010), 1 << 20, None)
    assert st == 3


def test_unsupported_head_dim_fails_before_the_device(lib):
    p = _p(D=96)
    st = lib.attn_train_fwd(ctypes.byref(p), _t(), _t(), _t(), _t(), ctypes.c_void_p(0x2000), None)
    assert st == 2
    assert b"head dim" in lib.attn_train_last_error()


def test_binding_raises_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        binding._lib_saved = binding._lib
        try:
            binding._lib = None
            binding.load(str(tmp_path / "missing.so"))
        finally:
            binding._lib = binding._lib_saved
