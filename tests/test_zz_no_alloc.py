"""The allocation-free backward (attn_train_bwd_noalloc) against the regular
one (attn_train_bwd with a caller-provided workspace).

Some callers cannot allocate device memory: an operator plugged into a host
framework that owns all device memory and passes only inputs and outputs,
or code on a path where cudaMalloc's implicit device synchronization is not
allowed.  For them the library keeps its backward workspace in a fixed 4 MiB
array compiled into the library.  These tests call that entry point through
the C ABI several times in a row (different problems, so a stale scratch from
one call would show in the next) and require the same bits as the regular
entry point, which runs the same kernels on the same inputs.  One problem
fills the array to its last byte.  Problems whose workspace exceeds the array
must be refused on the host.  This file is named so that pytest collects it
last.
"""
import ctypes

import pytest
import torch

from attention_tcgen05_tmem_gb300 import binding, synth
from tests.gpu_util import device

SCRATCH_BYTES = 4 << 20
ATTN_ERR_WORKSPACE = 4

PROBLEMS = [
    synth.Workload("noalloc_causal_gqa", 1, 8, 2, 700, 700, 128, "causal", 0, 21),
    synth.Workload("noalloc_ttt_t2", 1, 4, 2, 300, 900, 64, "ttt", 2, 22),
    # B * Hq * Sq = 1,048,576 rows: Delta takes the whole 4 MiB array
    synth.Workload("noalloc_full_array", 1, 64, 8, 16384, 16384, 16, "causal", 0, 23),
]


def _regular_and_noalloc(w, dev):
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, w.mask, w.ttt_step, out="fp32")
    ref = binding.bwd(q, k, v, o, lse, do, w.mask, w.ttt_step)
    p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step, 0.0, "fp32")
    got = tuple(torch.full_like(t, float("nan")) for t in ref)
    binding.bwd_noalloc_raw(p, q, k, v, o, do, lse, *got)
    binding.device_status()
    return ref, got


@pytest.mark.gpu
def test_noalloc_backward_equals_regular_backward_on_calls_in_a_row():
    dev = device()
    assert binding.workspace_size(binding.problem(1, 64, 8, 16384, 16384, 16, "causal", 0, 0.0,
                                                  "fp32")) == SCRATCH_BYTES
    for w in PROBLEMS + PROBLEMS[:1]:  # calls in a row, the first problem again at the end
        ref, got = _regular_and_noalloc(w, dev)
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            assert torch.equal(a, b), f"{w.name} {name}: no-alloc result differs"


def _noalloc_status(p):
    from attention_tcgen05_tmem_gb300 import build as lib_build
    lib_build.build()
    lib = binding.load()
    # stand-in addresses that are not 16-byte aligned: a problem that passes the
    # workspace check is still refused on the host (alignment) before any launch
    t = binding.Tensor(0x1001, 1 << 20, 1 << 16, 128)
    st = lib.attn_train_bwd_noalloc(ctypes.byref(p), t, t, t, t, t, ctypes.c_void_p(0x2000),
                                    t, t, t, None)
    return st, lib.attn_train_last_error()


def test_noalloc_rejects_problems_beyond_the_built_in_scratch():
    # one query row past the limit: 64 x 16385 rows of Delta = 4,194,560 bytes
    p = binding.problem(1, 64, 8, 16385, 16385, 16, "causal", 0, 0.0, "fp32")
    assert binding.workspace_size(p) > SCRATCH_BYTES
    st, msg = _noalloc_status(p)
    assert st == ATTN_ERR_WORKSPACE
    assert b"built-in scratch holds 4194304 bytes" in msg
    assert b"4194560" in msg


def test_noalloc_rejects_ttt_workspace_above_the_array_below_a_million_rows():
    # EAGLE3 TTT step 6 shape: 262,144 rows (a quarter of 1,048,576) but the
    # suffix diagonals add 12 floats per row: 13 MiB of workspace
    p = binding.problem(1, 32, 8, 8192, 7 * 8192, 128, "ttt", 6, 0.0, "fp32")
    need = binding.workspace_size(p)
    assert 1 * 32 * 8192 < 1 << 20 and need > SCRATCH_BYTES
    st, msg = _noalloc_status(p)
    assert st == ATTN_ERR_WORKSPACE
    assert str(need).encode() in msg


def test_noalloc_accepts_ttt_step_one_of_the_eagle3_workload():
    # step 1: (1 + 2) x 262,144 rows x 4 bytes = 3 MiB fits; the workspace check
    # passes and the call fails only later (the stand-in tensors' alignment, or
    # no device on a machine without a GPU)
    p = binding.problem(1, 32, 8, 8192, 2 * 8192, 128, "ttt", 1, 0.0, "fp32")
    assert binding.workspace_size(p) <= SCRATCH_BYTES
    st, _ = _noalloc_status(p)
    assert st != ATTN_ERR_WORKSPACE
