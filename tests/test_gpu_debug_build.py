"""The -DATTN_DEBUG build (libattn_train_debug.so): its device-side checks of
tile coordinates, work items and workspace slots never fire on valid
problems -- the kernels give the same bits as the normal build -- and a check
that fails on purpose is reported as ATTN_ERR_DEVICE_CHECK with its site,
after which the library works again.  The debug library runs in a child
process (a process loads one build)."""
import os
import subprocess
import sys

import numpy as np
import pytest

from attention_tcgen05_tmem_gb300 import binding, synth
from tests.gpu_util import device

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W = synth.Workload
CASES = [W("dbg_causal_gqa_ragged", 2, 4, 2, 333, 333, 128, "causal", seed=61),
         W("dbg_ttt_t3", 1, 4, 2, 257, 1028, 64, "ttt", 3, 62),
         W("dbg_window_varlen", 2, 2, 1, 640, 640, 32, "window", seed=63, window=(100, 20),
           seq_lengths=(640, 250)),
         W("dbg_addmask", 1, 2, 2, 300, 300, 16, "full", seed=64, add_mask=True),
         W("dbg_split", 1, 1, 1, 4096, 4096, 64, "causal", seed=65)]

RUN = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
from attention_tcgen05_tmem_gb300 import binding, synth, build
if sys.argv[3] == "debug":
    binding.load(build.DEBUG_LIB)
from tests import test_gpu_debug_build as t
out = {}
for w in t.CASES:
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
    lens = x["seq_lengths"].cuda() if "seq_lengths" in x else None
    am = None
    if "add_mask" in x:
        am = torch.zeros(w.Sq, w.Skv + (-w.Skv % 8), dtype=torch.bfloat16, device="cuda")[:, :w.Skv]
        am.copy_(x["add_mask"].cuda())
    kw = dict(window=w.window, seq_lengths=lens, add_mask=am)
    o, lse = binding.fwd(q, k, v, w.mask, w.ttt_step, out="fp32", **kw)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, w.mask, w.ttt_step, **kw)
    binding.device_status()
    for n, tt in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        out[w.name + "/" + n] = tt.cpu().numpy()
if sys.argv[3] == "debug":
    binding.selftest_debug_check()
    try:
        binding.device_status()
        raise SystemExit("the failed check was not reported")
    except binding.AttnError as e:
        assert e.status == 7 and "site 99" in str(e), e
    binding.device_status()  # cleared: the library works again
np.savez(sys.argv[2], **out)
"""


def _run(tmp_path, which):
    path = str(tmp_path / f"{which}.npz")
    subprocess.run([sys.executable, "-c", RUN, ROOT, path, which], check=True, cwd=ROOT,
                   timeout=1200)
    return np.load(path)


@pytest.mark.gpu
@pytest.mark.timeout(1500)
def test_debug_build_checks_stay_silent_and_change_no_bit(tmp_path):
    device()
    from attention_tcgen05_tmem_gb300 import build as lib_build
    lib_build.build_debug()
    normal, debug = _run(tmp_path, "normal"), _run(tmp_path, "debug")
    assert sorted(normal.files) == sorted(debug.files)
    for n in normal.files:
        assert np.array_equal(normal[n], debug[n]), n
