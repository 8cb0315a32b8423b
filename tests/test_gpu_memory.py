"""Memory is linear in S: besides its inputs and outputs, one forward +
backward needs exactly the backward workspace (the fp32 Delta row statistic,
B*Hq*Sq*4 bytes); the S x S score matrix is never stored (SpecForge post:
Flex attention's memory saving in long-context training; CS336 README:
naive attention's O(N^2) score matrix is what flash attention avoids).  The
forward here runs unsplit; the key-range split used for grids under one wave
adds a workspace bounded independently of S (tests/test_abi_cpu.py)."""
import gc

import pytest
import torch

from attention_tcgen05_tmem_gb300 import binding, synth
from tests.gpu_util import device


@pytest.mark.gpu
def test_extra_memory_is_the_workspace_and_linear_in_s():
    dev = device()
    extra = {}
    for S in (4096, 8192, 16384):
        w = synth.Workload(f"mem_S{S}", 1, 8, 1, S, S, 128, "causal", 0, 31)
        x = synth.make_inputs(w)
        q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
        # tensors of earlier tests still awaiting collection must not be freed while
        # this one measures
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        o, lse = binding.fwd(q, k, v, "causal", out="fp32", split=False)
        dq, dk, dv = binding.bwd(q, k, v, o, lse, do, "causal")
        torch.cuda.synchronize()
        binding.device_status()
        peak = torch.cuda.max_memory_allocated() - base
        outputs = sum(t.numel() * t.element_size() for t in (o, lse, dq, dk, dv))
        extra[S] = peak - outputs
        ws = binding.workspace_size(binding.problem_for(q, k, "causal", out="fp32"))
        assert extra[S] == ws == w.B * w.Hq * S * 4, (S, extra[S], ws)
        del o, lse, dq, dk, dv, q, k, v, do
    assert extra[8192] / extra[4096] <= 2.05 and extra[16384] / extra[8192] <= 2.05
