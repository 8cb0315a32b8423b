"""The allocation-free backward (attn_train_bwd_noalloc) against the regular
one (attn_train_bwd with a caller-provided workspace).

Some callers cannot allocate device memory: an operator plugged into a host
framework that owns all device memory and passes only inputs and outputs,
or code on a path where cudaMalloc's implicit device synchronization is not
allowed.  For them the library keeps its backward scratch in a fixed array
compiled into the library.  These tests call that entry point through the C
ABI twice in a row (two different problems, so a stale scratch from the first
call would show in the second) and check each result against the regular
entry point's within the parity tolerance.  This file is named so that pytest
collects it last.
"""
import ctypes

import pytest
import torch

from attention_tcgen05_tmem_gb300 import binding, synth
from tests.gpu_util import compare, device

PROBLEMS = [
    synth.Workload("noalloc_causal_gqa", 1, 8, 2, 700, 700, 128, "causal", 0, 21),
    synth.Workload("noalloc_ttt_t2", 1, 4, 2, 300, 900, 64, "ttt", 2, 22),
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
def test_noalloc_backward_matches_regular_backward_twice():
    dev = device()
    for w in PROBLEMS:  # two calls in a row
        ref, got = _regular_and_noalloc(w, dev)
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            compare(f"{w.name} {name}", a, b.double().cpu().numpy())


def test_noalloc_rejects_problems_beyond_the_built_in_scratch():
    from attention_tcgen05_tmem_gb300 import build as lib_build
    lib_build.build()
    lib = binding.load()
    # 2 x 32 x 16400 rows > 1,048,576: rejected on the host before any GPU work
    p = binding.problem(2, 32, 4, 16400, 16400, 128, "causal", 0, 0.0, "fp32")
    t = binding.Tensor(0x1000, 1 << 20, 1 << 16, 128)
    st = lib.attn_train_bwd_noalloc(ctypes.byref(p), t, t, t, t, t, ctypes.c_void_p(0x2000),
                                    t, t, t, None)
    assert st == 4
    assert b"built-in scratch" in lib.attn_train_last_error()
