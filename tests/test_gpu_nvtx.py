"""ATTN_TRAIN_NVTX=1 wraps every launch in an NVTX range and launches the
backward's passes one at a time; the results must be bit-identical to a run
without it (the flag is read once per process, so the NVTX run is a child
process)."""
import os
import subprocess
import sys

import numpy as np
import pytest

from attention_tcgen05_tmem_gb300 import binding, synth
from tests.gpu_util import device

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W = synth.Workload("nvtx_ttt_t2", 1, 4, 2, 300, 900, 64, "ttt", 2, 31)

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, sys.argv[1])
from attention_tcgen05_tmem_gb300 import binding, synth
w = synth.Workload("nvtx_ttt_t2", 1, 4, 2, 300, 900, 64, "ttt", 2, 31)
x = synth.make_inputs(w)
q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "dout"))
o, lse = binding.fwd(q, k, v, w.mask, w.ttt_step, out="fp32")
dq, dk, dv = binding.bwd(q, k, v, o, lse, do, w.mask, w.ttt_step)
binding.device_status()
np.savez(sys.argv[2], **{n: t.cpu().numpy() for n, t in
                         (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))})
"""


@pytest.mark.gpu
def test_nvtx_mode_gives_identical_results(tmp_path):
    dev = device()
    x = synth.make_inputs(W)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, W.mask, W.ttt_step, out="fp32")
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, W.mask, W.ttt_step)
    binding.device_status()
    path = str(tmp_path / "nvtx.npz")
    env = dict(os.environ, ATTN_TRAIN_NVTX="1")
    subprocess.run([sys.executable, "-c", CHILD, ROOT, path], check=True, env=env, timeout=600)
    got = np.load(path)
    for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert np.array_equal(got[n], t.cpu().numpy()), n
