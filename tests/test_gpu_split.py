"""The forward's key-range split (attn_train_fwd_ws on grids under one wave):
each query-tile pair's key tiles are cut into chunks, one CTA per chunk
writes partial O rows with their running max and sum, and a merge pass
combines them by log-sum-exp in chunk order.  It must match the fp64 oracle
like the unsplit forward, agree with the unsplit forward to rounding, give the
same bits run after run, leave NaN when its work is skipped, and give the same
bits whether a host-memory step runs the problem whole or in GQA-group chunks.
"""
import numpy as np
import pytest
import torch

import oracle
from attention_tcgen05_tmem_gb300 import binding, synth
from tests.gpu_util import LSE_ATOL, compare, device

W = synth.Workload
CASES = [
    W("split_causal_d64", 1, 1, 1, 4096, 4096, 64, "causal", seed=51),
    W("split_causal_gqa_d128", 1, 4, 2, 2000, 2000, 128, "causal", seed=52),
    W("split_full_cross_d128", 1, 2, 1, 300, 5000, 128, "full", seed=53),
    W("split_window_d32", 1, 2, 1, 2000, 2000, 32, "window", seed=54, window=(1500, 200)),
    W("split_varlen_d16", 2, 2, 2, 1500, 1500, 16, "causal", seed=55, seq_lengths=(1500, 0)),
    W("split_addmask_d64", 1, 1, 1, 1300, 1300, 64, "full", seed=56, add_mask=True),
]


def _inputs(w, dev):
    x = synth.make_inputs(w)
    t = {n: x[n].to(dev) for n in ("q", "k", "v", "dout")}
    lens = x["seq_lengths"].to(dev) if "seq_lengths" in x else None
    am = None
    if "add_mask" in x:
        pad = -w.Skv % 8
        am = torch.zeros(w.Sq, w.Skv + pad, dtype=torch.bfloat16, device=dev)[:, :w.Skv]
        am.copy_(x["add_mask"].to(dev))
    kw = dict(window=w.window, seq_lengths=lens, add_mask=am)
    rkw = dict(window=w.window, seq_lengths=w.seq_lengths, add_mask=x.get("add_mask"))
    return x, t, kw, rkw


def _problem(w, out, kw):
    return binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step, 0.0, out,
                           w.window, kw["seq_lengths"], kw["add_mask"])


@pytest.mark.gpu
@pytest.mark.parametrize("out", ["fp32", "bf16"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_split_forward_parity(w, out):
    dev = device()
    x, t, kw, rkw = _inputs(w, dev)
    assert binding.fwd_workspace_size(_problem(w, out, kw)) > 0  # the case does split
    o, lse = binding.fwd(t["q"], t["k"], t["v"], w.mask, w.ttt_step, out=out, **kw)
    binding.device_status()
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], w.mask, w.ttt_step, **rkw)
    compare("O", o, ro)
    compare("LSE", lse, rl, atol=LSE_ATOL, rel_l2=1e-3)
    # the backward on the split forward's O and LSE
    dq, dk, dv = binding.bwd(t["q"], t["k"], t["v"], o, lse, t["dout"], w.mask, w.ttt_step, **kw)
    binding.device_status()
    rdq, rdk, rdv = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], w.mask, w.ttt_step, **rkw)
    compare("dQ", dq, rdq)
    compare("dK", dk, rdk)
    compare("dV", dv, rdv)


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_split_equals_unsplit_to_rounding_and_repeats_bitwise(w):
    dev = device()
    _, t, kw, _ = _inputs(w, dev)
    o1, l1 = binding.fwd(t["q"], t["k"], t["v"], w.mask, out="fp32", **kw)
    o2, l2 = binding.fwd(t["q"], t["k"], t["v"], w.mask, out="fp32", **kw)
    o0, l0 = binding.fwd(t["q"], t["k"], t["v"], w.mask, out="fp32", split=False, **kw)
    binding.device_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # P is rounded to bf16 relative to each chunk's own running max, and the fp32 sums
    # are grouped by chunk: O differs at the level of a bf16 rounding of P (half the
    # parity bar), LSE (fp32 sums of unrounded P) at the level of fp32 rounding
    assert (o1 - o0).abs().max().item() < 1e-2
    assert (l1 - l0).abs().max().item() < 1e-4


@pytest.mark.gpu
def test_split_forward_skipped_work_is_nan():
    dev = device()
    w = CASES[1]
    _, t, kw, _ = _inputs(w, dev)
    p = _problem(w, "fp32", kw)
    ws = torch.zeros(binding.fwd_workspace_size(p), dtype=torch.uint8, device=dev)
    o = torch.full(t["q"].shape, 7.0, dtype=torch.float32, device=dev)
    lse = torch.full((w.B, w.Hq, w.Sq), 7.0, dtype=torch.float32, device=dev)
    binding.selftest_wait_timeout()  # sets the device error word
    binding.fwd_ws_raw(p, t["q"], t["k"], t["v"], o, lse, ws)
    torch.cuda.synchronize(dev)
    assert torch.isnan(o).all() and torch.isnan(lse).all()
    with pytest.raises(binding.AttnError):
        binding.device_status()


@pytest.mark.gpu
def test_split_forward_rejects_a_short_workspace():
    dev = device()
    w = CASES[0]
    _, t, kw, _ = _inputs(w, dev)
    p = _problem(w, "fp32", kw)
    n = binding.fwd_workspace_size(p)
    ws = torch.zeros(n - 256, dtype=torch.uint8, device=dev)
    o = torch.empty(t["q"].shape, dtype=torch.float32, device=dev)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)
    with pytest.raises(binding.AttnError) as ei:
        binding.fwd_ws_raw(p, t["q"], t["k"], t["v"], o, lse, ws)
    assert ei.value.status == 4


@pytest.mark.gpu
@pytest.mark.parametrize("chunk", [0, 1])
def test_host_step_chunks_split_like_the_whole_problem(chunk):
    """A host-memory step cut into one-kv-head chunks splits every chunk's
    forward like the whole problem's, so the outputs equal the device path's."""
    dev = device()
    w = CASES[1]
    x, t, kw, _ = _inputs(w, dev)
    o, lse = binding.fwd(t["q"], t["k"], t["v"], w.mask, out="fp32", **kw)
    dq, dk, dv = binding.bwd(t["q"], t["k"], t["v"], o, lse, t["dout"], w.mask, **kw)
    binding.device_status()
    io = {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v", "dout")}
    for n, like in (("o", "q"), ("dq", "q"), ("dk", "k"), ("dv", "v")):
        io[n] = torch.full(x[like].shape, float("nan"), dtype=torch.float32).pin_memory()
    io["lse"] = torch.full((w.B, w.Hq, w.Sq), float("nan"), dtype=torch.float32).pin_memory()
    p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, 0, 0.0, "fp32", host=True)
    arena = torch.empty(binding.step_host_arena_size(p, chunk), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    binding.step_host_raw(p, io, arena, chunk, stream.cuda_stream)
    stream.synchronize()
    binding.device_status()
    for n, ref in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert np.array_equal(io[n].numpy(), ref.cpu().numpy()), n
