"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/attn_train.h declares, and rejects malformed or
unsupported problems with the right status before touching the device
(HOT-Step flash-attn-training, section 2: unsupported shapes must fail hard,
never fall back)."""
import ctypes
import os
import re

import pytest
import torch

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


def _up(n):
    return (n + 255) // 256 * 256


def test_step_host_arena_size(lib):
    """Arena = 2 x [key lengths][mask copy], the chunk workspace, 2 slots; a slot
    holds one chunk's q, k, v, dout, o, lse, dq, dk, dv."""
    # B=2, 2 kv heads of 2 q heads each, 1 kv head per chunk -> 4 chunks, 2 slots
    p = binding.problem(2, 4, 2, 100, 100, 64, "causal", out="bf16", host=True)
    nq, nk, nl = 2 * 100 * 64, 100 * 64, 2 * 100
    slot = _up(nq * 2) * 4 + _up(nk * 2) * 4 + _up(nl * 4)  # q, dout, o, dq; k, v, dk, dv; lse
    ws = _up(nl * 4)  # Delta of one chunk
    assert binding.step_host_arena_size(p, 1) == ws + 2 * slot
    # fp32 outputs, one chunk (the whole problem): still two slots (a session's
    # next step takes the other one)
    p = binding.problem(1, 4, 2, 100, 100, 64, "causal", out="fp32", host=True)
    nq, nk, nl = 4 * 100 * 64, 2 * 100 * 64, 4 * 100
    slot = 2 * _up(nq * 2) + 2 * _up(nk * 2) + 2 * _up(nq * 4) + 2 * _up(nk * 4) + _up(nl * 4)
    assert binding.step_host_arena_size(p, 2) == _up(nl * 4) + 2 * slot
    # chunk <= 0: the whole step is one chunk (all batch entries)
    p = binding.problem(1, 32, 4, 16384, 16384, 128, "causal", out="bf16", host=True)
    assert binding.step_host_arena_size(p, 0) == binding.step_host_arena_size(p, 4)
    p = binding.problem(2, 4, 2, 100, 100, 64, "causal", out="bf16", host=True)
    nq, nk, nl = 2 * 4 * 100 * 64, 2 * 2 * 100 * 64, 2 * 4 * 100
    slot = _up(nq * 2) * 4 + _up(nk * 2) * 4 + _up(nl * 4)
    assert binding.step_host_arena_size(p, 0) == _up(nl * 4) + 2 * slot
    # host key lengths and mask get arena space of their own
    lens = torch.tensor([100, 50], dtype=torch.int32)
    am = torch.zeros(100, 104, dtype=torch.bfloat16)[:, :100]
    p0 = binding.problem(2, 2, 2, 100, 100, 64, "full", host=True)
    p1 = binding.problem(2, 2, 2, 100, 100, 64, "full", seq_lengths=lens, add_mask=am, host=True)
    mask_ws = _up(100 * 104 * 2)  # the backward's transposed copy of the mask
    assert (binding.step_host_arena_size(p1, 1) - binding.step_host_arena_size(p0, 1)
            == 2 * (_up(2 * 4) + _up((99 * 104 + 100) * 2)) + mask_ws)


def test_host_session_arena_size_grows_by_one_slot_per_slot(lib):
    """n slots: n chunk slots and n copies of the key lengths and mask; the
    two-slot form equals attn_train_step_host_arena_size."""
    lens = torch.tensor([100, 50], dtype=torch.int32)
    am = torch.zeros(100, 104, dtype=torch.bfloat16)[:, :100]
    p = binding.problem(2, 4, 2, 100, 100, 64, "full", seq_lengths=lens, add_mask=am, out="fp32",
                        host=True)
    nq, nk, nl = 2 * 100 * 64, 100 * 64, 2 * 100  # one kv head of one batch entry
    slot = 2 * _up(nq * 2) + 2 * _up(nk * 2) + 2 * _up(nq * 4) + 2 * _up(nk * 4) + _up(nl * 4)
    stat = _up(2 * 4) + _up((99 * 104 + 100) * 2)
    two = binding.step_host_arena_size(p, 1)
    assert binding.step_host_arena_size(p, 1, 2) == two
    for n in (3, 8, binding.HOST_MAX_SLOTS):
        assert binding.step_host_arena_size(p, 1, n) == two + (n - 2) * (slot + stat)
    for bad in (0, 1, binding.HOST_MAX_SLOTS + 1):
        with pytest.raises(binding.AttnError, match="slots"):
            binding.step_host_arena_size(p, 1, bad)


def test_describe_reports_the_plan(lib):
    """attn_train_describe: one JSON object with the kernels each pass runs, their
    grids and pipeline depths, consistent with the schedule the kernels use."""
    p = binding.problem(1, 32, 4, 16384, 16384, 128, "causal", out="fp32")
    d = binding.describe(p)
    assert d["head_dim"] == 128 and d["mask"] == "causal" and d["outputs"] == "fp32"
    assert d["fwd"]["kernel"] == "fwd_kernel<128,0,0,0>" and d["fwd"]["ctas"] == 64 * 32
    assert d["fwd"]["split_key_tiles"] == 0 and not d["fwd"]["merge_pass"]
    assert d["bwd_dkdv"]["ctas"] == 128 * 4 and d["bwd_dq"]["ctas"] == 128 * 32
    assert d["fwd"]["smem_bytes"] <= 227 * 1024 and d["bwd_dq"]["smem_bytes"] <= 227 * 1024
    assert "ttt_suffix" not in d and "mask_transpose" not in d
    # a TTT step: the scores pre-pass and the suffix-key pass (8 segments per pass at t = 6)
    d = binding.describe(binding.problem(1, 32, 8, 8192, 7 * 8192, 128, "ttt", 6, out="fp32"))
    assert d["fwd"]["ttt_scores_prepass"] and d["bwd_prep"]["kernel"] == "bwd_prep_kernel<128,1>"
    assert d["ttt_suffix"] == {"kernel": "ttt_diag_bwd_kernel<128,8>", "key_rows": 8 * 8192}
    # a small grid takes the key-range split (the S = 4096 sweep: 9 key tiles per chunk)
    d = binding.describe(binding.problem(8, 1, 1, 4096, 4096, 64, "causal"))
    assert d["fwd"]["kernel"] == "fwd_kernel<64,0,0,1>" and d["fwd"]["merge_pass"]
    assert d["fwd"]["split_key_tiles"] == 9
    # general masks: window at D <= 64 rotates three score buffers; an additive mask
    # adds the transpose pass
    d = binding.describe(binding.problem(2, 16, 16, 12288, 12288, 64, "window", window=(1024, 1024)))
    assert d["general_mask"] and d["fwd"]["score_buffers"] == 3
    am = torch.zeros(300, 304, dtype=torch.bfloat16)[:, :300]
    d = binding.describe(binding.problem(2, 2, 2, 300, 300, 64, "full", add_mask=am, host=True))
    assert d["additive_mask"] and d["mask_transpose"] == {"kernel": "mask_transpose_kernel"}
    assert d["fwd"]["kernel"] == "fwd_kernel<64,1,1,0>"


def test_describe_buffer_protocol(lib):
    p = binding.problem(1, 2, 2, 128, 128, 64, "causal")
    need = ctypes.c_size_t(0)
    assert lib.attn_train_describe(ctypes.byref(p), None, 0, ctypes.byref(need)) == 1
    assert need.value > 1
    small = ctypes.create_string_buffer(need.value - 1)
    assert lib.attn_train_describe(ctypes.byref(p), small, need.value - 1, None) == 1
    assert b"needed" in lib.attn_train_last_error()
    buf = ctypes.create_string_buffer(need.value)
    assert lib.attn_train_describe(ctypes.byref(p), buf, need.value, None) == 0
    assert len(buf.value) + 1 == need.value
    # invalid problems are refused like attn_train_supports refuses them
    bad = binding.problem(1, 2, 2, 128, 128, 96, "causal")
    assert lib.attn_train_describe(ctypes.byref(bad), buf, need.value, None) == 2


def test_plain_c_client(lib, tmp_path):
    """The header is plain C: a C99 program includes it, links the library and
    calls the host-side entry points (validation, sizes, error messages)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    libdir = os.path.dirname(binding.LIB_PATH)
    exe = str(tmp_path / "c_abi_client")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                    os.path.join(here, "c_abi_client.c"), "-o", exe, "-L", libdir,
                    "-lattn_train", "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "c abi ok" in r.stdout


def test_size_limits(lib):
    # the mask arithmetic's unbounded extent is 2^30: longer sequences are refused
    p = binding.problem(1, 1, 1, 1 << 30, 128, 16, "full")
    assert lib.attn_train_supports(ctypes.byref(p)) == 2
    assert b"2^30" in lib.attn_train_last_error()
    p = binding.problem(1, 1, 1, 128, (1 << 30) + 5, 16, "full")
    assert lib.attn_train_supports(ctypes.byref(p)) == 2
    # the additive mask's transpose grid bounds Sq
    p = binding.problem(1, 1, 1, 5_000_000, 128, 64, "full")
    p.add_mask, p.add_mask_sb, p.add_mask_sq = 0x10000, 0, 128
    assert lib.attn_train_supports(ctypes.byref(p)) == 2
    p.add_mask = None
    assert lib.attn_train_supports(ctypes.byref(p)) == 0
    # row-wise passes: B*Hq*Sq rows at 16 per block must fit one launch
    p = binding.problem(65536, 64, 64, 1 << 20, 128, 16, "full")
    assert lib.attn_train_supports(ctypes.byref(p)) == 2


def test_step_host_validation(lib):
    p = binding.problem(1, 4, 2, 128, 128, 64, "causal", host=True)
    need = binding.step_host_arena_size(p, 0)
    io = binding.HostIO(*([0x10000] * 9))
    step = lib.attn_train_step_host
    assert step(ctypes.byref(p), ctypes.byref(io), 3, ctypes.c_void_p(0x100000), need, None) == 1
    assert b"kv_heads_per_chunk" in lib.attn_train_last_error()
    assert step(ctypes.byref(p), None, 0, ctypes.c_void_p(0x100000), need, None) == 1
    bad = binding.HostIO(*([0x10000] * 8 + [0]))
    assert step(ctypes.byref(p), ctypes.byref(bad), 0, ctypes.c_void_p(0x100000), need, None) == 1
    assert step(ctypes.byref(p), ctypes.byref(io), 0, None, need, None) == 4
    assert step(ctypes.byref(p), ctypes.byref(io), 0, ctypes.c_void_p(0x100010), need, None) == 3
    assert step(ctypes.byref(p), ctypes.byref(io), 0, ctypes.c_void_p(0x100000), need - 1,
                None) == 4
    assert b"arena too small" in lib.attn_train_last_error()
    # the problem itself is validated as for the device entry points
    q = binding.problem(1, 4, 3, 128, 128, 64, "causal", host=True)
    assert step(ctypes.byref(q), ctypes.byref(io), 0, ctypes.c_void_p(0x100000), need, None) == 1
    # a host mask needs no 16-byte alignment (it is copied to an aligned arena offset)
    am = torch.zeros(130, 136, dtype=torch.bfloat16)[1:129, 4:132]
    p2 = binding.problem(1, 4, 2, 128, 128, 64, "full", add_mask=am, host=True)
    assert binding.step_host_arena_size(p2, 0) > 0


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


def test_forward_split_workspace_sizes():
    """attn_train_fwd_workspace_size is a pure function of the problem: non-zero
    for small grids with long rows (the single-head sweep at S = 4096: 128
    query-tile pairs, the longest walking 32 key tiles), zero where splitting
    does not pay (S <= 1024: short rows), for TTT masks and for grids that fill
    a GB300 (the long GQA workload)."""
    from attention_tcgen05_tmem_gb300 import build as lib_build
    lib_build.build()
    from attention_tcgen05_tmem_gb300 import synth

    def size(w):
        p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step, 0.0, "fp32")
        return binding.fwd_workspace_size(p)

    sweep = {w.name: size(w) for w in synth.SWEEP}
    assert all(v == 0 for n, v in sweep.items() if "_S4096_" not in n)
    assert all(v > 0 for n, v in sweep.items() if "_S4096_" in n)
    # S = 4096, D = 64: 16 pairs x 8 heads, 4 chunks each of 256 rows x (64 + 2) floats
    assert size(synth.by_name("sweep_causal_B8_H1_S4096_D64")) == 16 * 8 * 4 * 256 * 66 * 4
    assert size(synth.LONG_GQA) == 0 and size(synth.DIT_CROSS) == 0
    assert all(size(w) == 0 for w in synth.TTT_STEPS)


def test_forward_split_workspace_checks():
    """A too-short or misaligned forward workspace is refused on the host."""
    from attention_tcgen05_tmem_gb300 import build as lib_build
    lib_build.build()
    lib = binding.load()
    p = binding.problem(1, 1, 1, 4096, 4096, 64, "causal", 0, 0.0, "fp32")
    n = binding.fwd_workspace_size(p)
    t = binding.Tensor(0x1000, 1 << 24, 1 << 22, 64)
    lse = ctypes.c_void_p(0x2000)
    st = lib.attn_train_fwd_ws(ctypes.byref(p), t, t, t, t, lse, ctypes.c_void_p(0x10000), n - 256,
                               None)
    assert st == 4 and b"too small" in lib.attn_train_last_error()
    st = lib.attn_train_fwd_ws(ctypes.byref(p), t, t, t, t, lse, ctypes.c_void_p(0x10010), n, None)
    assert st == 3 and b"256-byte" in lib.attn_train_last_error()


def test_forward_split_workspace_is_bounded_independently_of_s():
    """Whatever the sequence length, the split's partial results fill at most
    four 256-row slots per SM of a GB300 (608 slots of D + 2 floats per row: at
    most 81 MB at D = 128)."""
    from attention_tcgen05_tmem_gb300 import build as lib_build
    lib_build.build()
    worst = 0
    for mask in ("causal", "full"):
        for D in (16, 64, 128):
            for H in (1, 4, 16, 64):
                for S in (512, 4096, 16384, 131072):
                    for Skv in ((S,) if mask == "causal" else (S, 1 << 20)):
                        p = binding.problem(1, H, H, S, Skv, D, mask, 0, 0.0, "fp32")
                        n = binding.fwd_workspace_size(p)
                        worst = max(worst, n / (256 * (D + 2) * 4))
    assert 0 < worst <= 4 * 152


def test_debug_selftest_is_refused_by_the_normal_build():
    from attention_tcgen05_tmem_gb300 import build as lib_build
    lib_build.build()
    lib = binding.load()
    assert lib.attn_train_selftest_debug_check(None) == 2
    assert b"ATTN_DEBUG" in lib.attn_train_last_error()
