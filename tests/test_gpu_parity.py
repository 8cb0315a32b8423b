"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs, element by element, at sizes the oracle finishes in
seconds that still span several tiles and ragged tails; plus bitwise
determinism of the backward, strided layouts, and the bounded-wait error
path."""
import numpy as np
import pytest
import torch

import oracle
from attention_tcgen05_tmem_gb300 import binding, synth
from tests.gpu_util import LSE_ATOL, compare, device


def run_both(w: synth.Workload, check_bwd=True, out="fp32", stress=False):
    dev = device()
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    lens = x["seq_lengths"].to(dev) if "seq_lengths" in x else None
    am = None
    if "add_mask" in x:
        # device copy with a row stride padded to a multiple of 8 keys
        pad = -w.Skv % 8
        am = torch.zeros(w.Sq, w.Skv + pad, dtype=torch.bfloat16, device=dev)[:, :w.Skv]
        am.copy_(x["add_mask"].to(dev))
    kw = dict(window=w.window, seq_lengths=lens, add_mask=am)
    rkw = dict(window=w.window, seq_lengths=w.seq_lengths, add_mask=x.get("add_mask"))
    o, lse = binding.fwd(q, k, v, w.mask, w.ttt_step, out=out, **kw)
    binding.device_status()
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], w.mask, w.ttt_step, **rkw)
    compare("O", o, ro, stress=stress)
    compare("LSE", lse, rl, atol=LSE_ATOL, rel_l2=1e-3)
    if not check_bwd:
        return
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, w.mask, w.ttt_step, **kw)
    binding.device_status()
    rdq, rdk, rdv = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], w.mask, w.ttt_step, **rkw)
    assert np.abs(rdq).max() > 1e-3  # non-vacuous (HOT-Step trap 7)
    compare("dQ", dq, rdq, stress=stress)
    compare("dK", dk, rdk, stress=stress)
    compare("dV", dv, rdv, stress=stress)


def W(name, B, Hq, Hkv, Sq, Skv, D, mask, t=0, seed=11, window=None, lens=None, add=False):
    return synth.Workload(name, B, Hq, Hkv, Sq, Skv, D, mask, t, seed, window, lens, add)


CASES = [
    synth.TINY,
    W("causal_one_tile_d128", 1, 1, 1, 128, 128, 128, "causal"),
    W("causal_ragged_gqa_d128", 2, 4, 2, 333, 333, 128, "causal"),
    W("causal_ragged_d64", 1, 3, 3, 517, 517, 64, "causal"),
    W("causal_d32", 2, 2, 1, 640, 640, 32, "causal"),
    W("causal_d16", 2, 2, 2, 384, 384, 16, "causal"),
    W("causal_gqa8_d128", 1, 8, 1, 512, 512, 128, "causal"),
    W("causal_sq_lt_skv", 1, 2, 1, 200, 350, 64, "causal"),
    W("causal_sq_gt_skv", 1, 2, 1, 350, 200, 64, "causal"),
    W("full_self_ragged_d64", 1, 2, 2, 300, 300, 64, "full"),
    W("full_cross_d64", 2, 2, 2, 400, 129, 64, "full"),
    W("full_cross_d128", 1, 4, 2, 256, 512, 128, "full"),
    W("ttt_t0", 1, 4, 2, 256, 256, 128, "ttt", 0),
    W("ttt_t1_ragged", 1, 4, 2, 300, 600, 128, "ttt", 1),
    W("ttt_t3", 1, 4, 1, 257, 1028, 128, "ttt", 3),
    W("ttt_t4", 1, 4, 2, 200, 1000, 128, "ttt", 4),
    W("ttt_t5", 1, 4, 2, 200, 1200, 128, "ttt", 5),
    W("ttt_t5_ragged_d64", 1, 4, 1, 333, 1998, 64, "ttt", 5),
    W("ttt_t6_d64", 1, 2, 1, 200, 1400, 64, "ttt", 6),
    W("ttt_t2_tiny", 1, 2, 1, 5, 15, 32, "ttt", 2),
    # window masks: causal sliding, symmetric, one-sided ahead, narrow (rows that see
    # nothing when Sq > Skv), across head dims
    W("window_causal_gqa_d128", 1, 4, 2, 700, 700, 128, "window", window=(200, 0)),
    W("window_sym_d64", 2, 2, 2, 1000, 1000, 64, "window", window=(130, 130)),
    W("window_ahead_d32", 1, 2, 1, 520, 520, 32, "window", window=(0, 300)),
    W("window_narrow_sq_gt_skv_d64", 1, 2, 1, 450, 300, 64, "window", window=(5, 5)),
    W("window_d16", 2, 2, 2, 384, 384, 16, "window", window=(64, 64)),
    W("window_wide_equals_full_d128", 1, 2, 2, 300, 300, 128, "window", window=(400, 400)),
    # per-batch key lengths (padding), including an empty and a one-key batch entry
    W("varlen_causal_gqa_d128", 3, 4, 2, 600, 600, 128, "causal", lens=(600, 333, 1)),
    W("varlen_full_cross_d64", 2, 2, 2, 500, 300, 64, "full", lens=(300, 129)),
    W("varlen_window_d64", 2, 2, 1, 640, 640, 64, "window", window=(100, 20), lens=(640, 250)),
    W("varlen_ttt_t2_d128", 2, 4, 2, 384, 1152, 128, "ttt", 2, lens=(384, 200)),
    W("varlen_empty_entry_d64", 2, 2, 2, 256, 256, 64, "causal", lens=(0, 256)),
    # additive masks (bf16 bias with -inf holes) on the full, causal and window kinds
    W("addmask_full_d64", 2, 2, 2, 300, 300, 64, "full", add=True),
    W("addmask_causal_gqa_d128", 1, 4, 2, 333, 333, 128, "causal", add=True),
    W("addmask_cross_ragged_d64", 2, 2, 1, 250, 190, 64, "full", add=True),
    W("addmask_window_d32", 1, 2, 2, 400, 400, 32, "window", window=(64, 64), add=True),
    W("addmask_varlen_d128", 2, 2, 2, 256, 256, 128, "causal", lens=(256, 100), add=True),
    W("addmask_d16", 1, 2, 2, 384, 384, 16, "full", add=True),
    # degenerate extents: one query row, TTT at D = 16
    W("sq1_full_cross_d64", 2, 2, 1, 1, 257, 64, "full"),
    W("ttt_t1_d16", 1, 2, 2, 130, 260, 16, "ttt", 1),
]


@pytest.mark.gpu
@pytest.mark.parametrize("out", ["fp32", "bf16"])
@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_parity(w, out):
    run_both(w, out=out)


SWEEP_SMALL = [w for w in synth.SWEEP if w.Sq <= 1024]


@pytest.mark.gpu
@pytest.mark.parametrize("w", SWEEP_SMALL, ids=[c.name for c in SWEEP_SMALL])
def test_parity_sweep(w):
    run_both(w)


DET_CASES = [W("det_window", 1, 4, 2, 600, 600, 64, "window", seed=5, window=(150, 40)),
             W("det_varlen_ttt", 2, 4, 2, 384, 1152, 128, "ttt", 2, seed=5, lens=(384, 250)),
             W("det_addmask", 1, 4, 2, 384, 384, 128, "causal", seed=5, add=True)]


@pytest.mark.gpu
@pytest.mark.parametrize("w", DET_CASES, ids=[c.name for c in DET_CASES])
def test_general_mask_backward_is_bitwise_deterministic(w):
    dev = device()
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    kw = dict(window=w.window,
              seq_lengths=x["seq_lengths"].to(dev) if "seq_lengths" in x else None,
              add_mask=x["add_mask"].to(dev) if "add_mask" in x else None)
    o, lse = binding.fwd(q, k, v, w.mask, w.ttt_step, out="fp32", **kw)
    o2, lse2 = binding.fwd(q, k, v, w.mask, w.ttt_step, out="fp32", **kw)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    r1 = binding.bwd(q, k, v, o, lse, do, w.mask, w.ttt_step, **kw)
    r2 = binding.bwd(q, k, v, o, lse, do, w.mask, w.ttt_step, **kw)
    binding.device_status()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


STRESS_CASES = [W("stress_d64_full", 2, 8, 8, 2048, 2048, 64, "full", seed=6),
                W("stress_d64_addmask", 2, 8, 8, 2048, 2048, 64, "full", seed=6, add=True),
                W("stress_d32_window", 2, 8, 4, 2048, 2048, 32, "window", seed=6,
                  window=(300, 300))]


@pytest.mark.gpu
@pytest.mark.parametrize("w", STRESS_CASES, ids=[c.name for c in STRESS_CASES])
def test_forward_repeated_runs_are_bitwise_equal(w):
    """Many CTAs, many key tiles, several runs: a forward that read its O
    accumulator before the last P V products landed (a pipeline ordering bug)
    would show up as outputs that differ between runs."""
    dev = device()
    x = synth.make_inputs(w)
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    am = None
    if "add_mask" in x:
        pad = -w.Skv % 8
        am = torch.zeros(w.Sq, w.Skv + pad, dtype=torch.bfloat16, device=dev)[:, :w.Skv]
        am.copy_(x["add_mask"].to(dev))
    kw = dict(window=w.window, add_mask=am)
    o0, lse0 = binding.fwd(q, k, v, w.mask, out="fp32", **kw)
    for _ in range(5):
        o, lse = binding.fwd(q, k, v, w.mask, out="fp32", **kw)
        assert torch.equal(o, o0) and torch.equal(lse, lse0)
    binding.device_status()


@pytest.mark.gpu
def test_backward_is_bitwise_deterministic():
    dev = device()
    w = W("det", 1, 8, 2, 700, 700, 128, "causal", seed=5)
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, "causal")
    o2, lse2 = binding.fwd(q, k, v, "causal")
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    r1 = binding.bwd(q, k, v, o, lse, do, "causal")
    r2 = binding.bwd(q, k, v, o, lse, do, "causal")
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


@pytest.mark.gpu
def test_strided_bshd_layout():
    dev = device()
    w = W("bshd", 2, 4, 2, 300, 300, 64, "causal", seed=6)
    x = synth.make_inputs(w)
    # store as [B, S, H, D] and hand the library permuted [B, H, S, D] views
    q, k, v, do = (x[n].permute(0, 2, 1, 3).contiguous().to(dev).permute(0, 2, 1, 3)
                   for n in ("q", "k", "v", "dout"))
    assert q.stride(2) != w.D
    o, lse = binding.fwd(q, k, v, "causal")
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, "causal")
    binding.device_status()
    ro, _ = oracle.fwd(x["q"], x["k"], x["v"], "causal")
    rdq, rdk, rdv = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], "causal")
    compare("O", o, ro)
    compare("dQ", dq, rdq)
    compare("dK", dk, rdk)
    compare("dV", dv, rdv)


@pytest.mark.gpu
@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_gqa_32_heads_per_kv_head(out):
    """32 query heads summed into each dK / dV row (gradients ~5x the workloads')."""
    run_both(W("gqa32_causal_d64", 1, 32, 1, 200, 200, 64, "causal"), out=out, stress=True)


@pytest.mark.gpu
def test_single_key():
    """Skv = 1: every row's only key has weight 1, so O = V and LSE = c q.k; then
    dP = dO.v = Delta, so dS and dQ are 0 and dK = 0, dV = sum of dO."""
    dev = device()
    w = W("skv1", 1, 2, 2, 129, 1, 128, "full", seed=14)
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, "full", out="fp32")
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, "full")
    binding.device_status()
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], "full")
    rdq, rdk, rdv = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], "full")
    compare("O", o, ro)
    compare("LSE", lse, rl, atol=LSE_ATOL, rel_l2=1e-3)
    assert torch.equal(o.cpu(), x["v"].float().expand(1, 2, 129, 128))
    assert float(dq.abs().max()) < 1e-4 and float(dk.abs().max()) < 1e-3
    compare("dV", dv, rdv)


@pytest.mark.gpu
def test_explicit_scale():
    """A caller-chosen softmax scale (not 1/sqrt(D)) reaches every pass."""
    dev = device()
    w = W("scale", 1, 4, 2, 300, 300, 128, "causal", seed=12)
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, "causal", scale=0.3, out="fp32")
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, "causal", scale=0.3)
    binding.device_status()
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], "causal", scale=0.3)
    rdq, rdk, rdv = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], "causal", scale=0.3)
    compare("O", o, ro, stress=True)
    compare("LSE", lse, rl, atol=LSE_ATOL, rel_l2=1e-3)
    compare("dQ", dq, rdq, stress=True)
    compare("dK", dk, rdk, stress=True)
    compare("dV", dv, rdv, stress=True)


RESCALE_CASES = [W("rescale_window_d64", 1, 2, 2, 1024, 1024, 64, "window", seed=13,
                   window=(700, 100)),
                 W("rescale_full_d128", 1, 2, 1, 512, 1024, 128, "full", seed=13),
                 W("rescale_causal_d32", 1, 2, 2, 768, 768, 32, "causal", seed=13)]


@pytest.mark.gpu
@pytest.mark.parametrize("w", RESCALE_CASES, ids=[c.name for c in RESCALE_CASES])
def test_growing_scores_rescale_often(w):
    """Key norms that grow along the key axis (x 1 .. x 6) make each row's score
    maximum rise tile after tile, so the forward's lazy O rescale (and, at D <= 64
    with a general mask, its wait for the previous P V) runs on most tiles."""
    dev = device()
    x = synth.make_inputs(w)
    grow = torch.linspace(1.0, 6.0, w.Skv).view(1, 1, w.Skv, 1)
    x["k"] = (x["k"].float() * grow).to(torch.bfloat16)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, w.mask, window=w.window, out="fp32")
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, w.mask, window=w.window)
    binding.device_status()
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], w.mask, window=w.window)
    rdq, rdk, rdv = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], w.mask, window=w.window)
    compare("O", o, ro, stress=True)
    compare("LSE", lse, rl, atol=LSE_ATOL, rel_l2=1e-3)
    compare("dQ", dq, rdq, stress=True)
    compare("dK", dk, rdk, stress=True)
    compare("dV", dv, rdv, stress=True)


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
def test_additive_mask_hides_whole_rows_and_keys(D):
    """A per-batch additive mask that hides entire query rows (O = 0, LSE = 0,
    dQ = 0 exactly: the rows see no key) and entire keys (dK = dV = 0 exactly),
    over several tiles and a ragged tail."""
    dev = device()
    B, H, Sq, Skv = 2, 2, 300, 270
    w = W("hide", B, H, H, Sq, Skv, D, "full", seed=15)
    x = synth.make_inputs(w)
    g = torch.Generator().manual_seed(15)
    m = (0.5 * torch.randn(B, Sq, Skv, generator=g)).to(torch.bfloat16)
    hidden_rows = {0: [0, 129, 299], 1: [7, 200]}
    hidden_keys = {0: [5, 128, 269], 1: [0, 131]}
    for b_, rows in hidden_rows.items():
        m[b_, rows, :] = float("-inf")
    for b_, keys in hidden_keys.items():
        m[b_, :, keys] = float("-inf")
    pad = -Skv % 8
    am = torch.zeros(B, Sq, Skv + pad, dtype=torch.bfloat16, device=dev)[:, :, :Skv]
    am.copy_(m.to(dev))
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, "full", out="fp32", add_mask=am)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, "full", add_mask=am)
    binding.device_status()
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], "full", add_mask=m)
    rdq, rdk, rdv = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], "full", add_mask=m)
    compare("O", o, ro)
    compare("LSE", lse, rl, atol=LSE_ATOL, rel_l2=1e-3)
    compare("dQ", dq, rdq)
    compare("dK", dk, rdk)
    compare("dV", dv, rdv)
    for b_, rows in hidden_rows.items():
        assert torch.all(o[b_, :, rows] == 0) and torch.all(lse[b_, :, rows] == 0)
        assert torch.all(dq[b_, :, rows] == 0)
    for b_, keys in hidden_keys.items():
        assert torch.all(dk[b_, :, keys] == 0) and torch.all(dv[b_, :, keys] == 0)


@pytest.mark.gpu
def test_scores_in_the_thousands():
    """q and k scaled by 20: scores reach about 2000, each row's weights are close
    to one-hot and the running max jumps by far more than the rescale threshold."""
    dev = device()
    w = W("huge", 1, 4, 2, 384, 384, 128, "causal", seed=16)
    x = synth.make_inputs(w)
    x["q"] = (x["q"].float() * 20).to(torch.bfloat16)
    x["k"] = (x["k"].float() * 20).to(torch.bfloat16)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, "causal", out="fp32")
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, "causal")
    binding.device_status()
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], "causal")
    rdq, rdk, rdv = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], "causal")
    assert float(np.abs(rl).max()) > 1000  # the scores really are large
    compare("O", o, ro, stress=True)
    # |LSE| up to ~2100: fp32 keeps it to ~2^-24 |LSE| ~ 1.3e-4, inside the 1e-3 bar
    compare("LSE", lse, rl, atol=LSE_ATOL, rel_l2=1e-3)
    compare("dQ", dq, rdq, stress=True)
    compare("dK", dk, rdk, stress=True)
    compare("dV", dv, rdv, stress=True)


@pytest.mark.gpu
def test_zero_keys_give_uniform_weights():
    # K = 0: every visible key has the same weight; O = mean of visible V rows
    dev = device()
    w = W("zk", 1, 2, 1, 256, 1024, 64, "ttt", 3, seed=8)
    x = synth.zero_k(synth.make_inputs(w))
    o, lse = binding.fwd(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), "ttt", 3)
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], "ttt", 3)
    compare("O", o, ro)
    compare("LSE", lse, rl, atol=LSE_ATOL, rel_l2=1e-3)


@pytest.mark.gpu
def test_unseen_keys_get_exactly_zero_gradient():
    # TTT step t: segment-0 keys kv > S-1-t are seen by no query (HOT-Step trap 8)
    dev = device()
    S, t = 300, 4
    w = W("unseen", 1, 2, 1, S, (t + 1) * S, 128, "ttt", t, seed=9)
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    o, lse = binding.fwd(q, k, v, "ttt", t)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, "ttt", t)
    binding.device_status()
    assert torch.all(dk[:, :, S - t:S] == 0) and torch.all(dv[:, :, S - t:S] == 0)
    assert torch.any(dk[:, :, :S - t] != 0)


@pytest.mark.gpu
def test_device_wait_timeout_is_reported_and_cleared():
    dev = device()
    binding.selftest_wait_timeout()
    with pytest.raises(binding.AttnError) as ei:
        binding.device_status()
    assert ei.value.status == 6
    # the word is cleared: the library works again
    run_both(synth.TINY, check_bwd=False)
    del dev


@pytest.mark.gpu
@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_skipped_work_leaves_nan_not_stale_memory(out):
    """While the device error word is set, every attention kernel returns
    without computing.  Its outputs must then read NaN -- not whatever the
    buffers held before -- also for a caller that does not ask
    attn_train_device_status first.  Clearing the word makes the library work
    again."""
    dev = device()
    w = W("skip_gqa_ragged", 2, 4, 2, 333, 333, 128, "causal", seed=9)
    x = synth.make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, 0, 0.0, out)
    odt = torch.float32 if out == "fp32" else torch.bfloat16
    # buffers holding finite stale values
    o, dq = (torch.full(q.shape, 7.0, dtype=odt, device=dev) for _ in range(2))
    dk, dv = (torch.full(k.shape, 7.0, dtype=odt, device=dev) for _ in range(2))
    lse = torch.full((w.B, w.Hq, w.Sq), 7.0, dtype=torch.float32, device=dev)
    ws = torch.zeros(binding.workspace_size(p), dtype=torch.uint8, device=dev)
    binding.selftest_wait_timeout()  # sets the device error word
    binding.fwd_raw(p, q, k, v, o, lse)
    binding.bwd_raw(p, q, k, v, o, do, lse, dq, dk, dv, ws)
    torch.cuda.synchronize(dev)
    for name, t in (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk), ("dV", dv)):
        assert torch.isnan(t).all(), f"{name}: skipped work left non-NaN values"
    with pytest.raises(binding.AttnError) as ei:
        binding.device_status()
    assert ei.value.status == 6
    run_both(w, out=out)  # the word is cleared: correct results again

