"""attn_train_step_host (one forward + backward from pinned host memory,
pipelined over chunks of GQA groups) against the device-memory entry points
on the same inputs: every output must be bitwise equal, for every chunk size
(the kernels never mix heads, and the device path is checked against the
oracle by the parity tests)."""
import pytest
import torch

from attention_tcgen05_tmem_gb300 import binding, synth

pytestmark = pytest.mark.gpu

W = synth.Workload
CASES = [
    W("hs_causal_gqa_ragged", 2, 8, 2, 300, 300, 128, "causal", seed=41),
    W("hs_full_cross_d64", 2, 6, 3, 200, 136, 64, "full", seed=42),
    W("hs_ttt_step2_gqa", 1, 4, 2, 256, 768, 64, "ttt", ttt_step=2, seed=43),
    W("hs_window_varlen", 3, 4, 4, 384, 384, 32, "window", window=(100, 20), seed=44,
      seq_lengths=(384, 130, 0)),
    W("hs_addmask_d64", 2, 4, 2, 250, 190, 64, "full", seed=45, add_mask=True),
]


def _device_reference(w, x, dev, out):
    lens = x["seq_lengths"].to(dev) if "seq_lengths" in x else None
    am = None
    if "add_mask" in x:
        pad = -w.Skv % 8
        am = torch.zeros(w.Sq, w.Skv + pad, dtype=torch.bfloat16, device=dev)[:, :w.Skv]
        am.copy_(x["add_mask"].to(dev))
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "dout"))
    kw = dict(mask=w.mask, ttt_step=w.ttt_step, window=w.window, seq_lengths=lens, add_mask=am)
    o, lse = binding.fwd(q, k, v, out=out, **kw)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, **kw)
    torch.cuda.synchronize()
    return {"o": o.cpu(), "lse": lse.cpu(), "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}


def _host_step(w, x, dev, out, chunk, arena=None):
    odt = torch.float32 if out == "fp32" else torch.bfloat16
    io = {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v", "dout")}
    io["o"] = torch.full(x["q"].shape, float("nan"), dtype=odt).pin_memory()
    io["dq"] = torch.full(x["q"].shape, float("nan"), dtype=odt).pin_memory()
    io["dk"] = torch.full(x["k"].shape, float("nan"), dtype=odt).pin_memory()
    io["dv"] = torch.full(x["v"].shape, float("nan"), dtype=odt).pin_memory()
    io["lse"] = torch.full((w.B, w.Hq, w.Sq), float("nan"), dtype=torch.float32).pin_memory()
    lens = x["seq_lengths"].contiguous() if "seq_lengths" in x else None
    am = None
    if "add_mask" in x:
        pad = -w.Skv % 8
        am = torch.zeros(w.Sq, w.Skv + pad, dtype=torch.bfloat16)[:, :w.Skv]
        am.copy_(x["add_mask"])
    p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step, 0.0, out,
                        w.window, lens, am, host=True)
    if arena is None:
        arena = torch.empty(binding.step_host_arena_size(p, chunk), dtype=torch.uint8,
                            device=dev)
    stream = torch.cuda.current_stream(dev)
    binding.step_host_raw(p, io, arena, chunk, stream.cuda_stream)
    stream.synchronize()
    binding.device_status()
    return {n: io[n] for n in ("o", "lse", "dq", "dk", "dv")}


@pytest.mark.parametrize("out", ["fp32", "bf16"])
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_step_host_matches_device_path(w, out):
    dev = torch.device("cuda:0")
    x = synth.make_inputs(w)
    ref = _device_reference(w, x, dev, out)
    for chunk in sorted({0, 1, w.Hkv}):
        got = _host_step(w, x, dev, out, chunk)
        for n in ref:
            assert torch.equal(got[n], ref[n]), (w.name, out, chunk, n)


def test_step_host_back_to_back_calls_reuse_arena():
    """Two steps on different inputs through one arena (filled with garbage
    first): each step's outputs depend only on its own inputs."""
    dev = torch.device("cuda:0")
    w1 = W("hs_a", 1, 8, 2, 512, 512, 128, "causal", seed=46)
    w2 = W("hs_b", 1, 8, 2, 512, 512, 128, "causal", seed=47)
    x1, x2 = synth.make_inputs(w1), synth.make_inputs(w2)
    ref1 = _device_reference(w1, x1, dev, "fp32")
    ref2 = _device_reference(w2, x2, dev, "fp32")
    p = binding.problem(1, 8, 2, 512, 512, 128, "causal", out="fp32", host=True)
    arena = torch.full((binding.step_host_arena_size(p, 1),), 0xFF, dtype=torch.uint8, device=dev)
    got1 = _host_step(w1, x1, dev, "fp32", 1, arena)
    got2 = _host_step(w2, x2, dev, "fp32", 1, arena)
    for n in ref2:
        assert torch.equal(got1[n], ref1[n]), n
        assert torch.equal(got2[n], ref2[n]), n


@pytest.mark.parametrize("slots,chunk", [(2, 0), (2, 1), (4, 0), (4, 1)])
@pytest.mark.parametrize("w", [CASES[0], CASES[3], CASES[4]], ids=lambda w: w.name)
def test_session_steps_overlap_and_match(w, chunk, slots):
    """A session of several steps on different inputs with one join at the end:
    the copies of each step overlap its neighbours' kernels and rotate through
    the arena's slots (more steps than slots, so every slot is reused), yet
    every step's outputs equal the device path's."""
    _session_matches(w, chunk, slots, 3 if slots == 2 else slots + 2)


def test_session_with_the_most_slots():
    """ATTN_HOST_MAX_SLOTS slots, eight chunks per step (two batch entries of
    four kv heads): six steps (48 chunks) wrap the slot rotation twice."""
    _session_matches(CASES[3].with_(B=2, seq_lengths=(384, 130)), 1, binding.HOST_MAX_SLOTS, 6)


def test_session_rejects_slot_counts_outside_the_range():
    dev = torch.device("cuda:0")
    w = CASES[0]
    p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, host=True)
    arena = torch.empty(binding.step_host_arena_size(p, 0, 3), dtype=torch.uint8, device=dev)
    for bad in (1, binding.HOST_MAX_SLOTS + 1):
        with pytest.raises(binding.AttnError, match="slots"):
            binding.HostSession(p, arena, 0, bad)
    # an arena sized for three slots is too small for four
    with pytest.raises(binding.AttnError, match="arena too small"):
        binding.HostSession(p, arena, 0, 4)


def _session_matches(w, chunk, slots, n_steps):
    dev = torch.device("cuda:0")
    xs = [synth.make_inputs(w, seed=w.seed + 100 * i) for i in range(n_steps)]
    for x in xs[1:]:  # a session's mask is fixed; q, k, v, dO differ per step
        if "add_mask" in x:
            x["add_mask"] = xs[0]["add_mask"]
    refs = [_device_reference(w, x, dev, "fp32") for x in xs]
    lens = xs[0]["seq_lengths"].contiguous() if "seq_lengths" in xs[0] else None
    am = None
    if "add_mask" in xs[0]:
        pad = -w.Skv % 8
        am = torch.zeros(w.Sq, w.Skv + pad, dtype=torch.bfloat16)[:, :w.Skv]
        am.copy_(xs[0]["add_mask"])
    for x in xs[1:]:  # key lengths come from the shape
        if lens is not None:
            assert torch.equal(x["seq_lengths"], lens)
    p = binding.problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.mask, w.ttt_step, 0.0, "fp32",
                        w.window, lens, am, host=True)
    arena = torch.full((binding.step_host_arena_size(p, chunk, slots),), 0xFF, dtype=torch.uint8,
                       device=dev)
    sess = binding.HostSession(p, arena, chunk, slots)
    ios = []
    for x in xs:
        io = {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v", "dout")}
        for n, shape in (("o", x["q"].shape), ("dq", x["q"].shape), ("dk", x["k"].shape),
                         ("dv", x["v"].shape), ("lse", (w.B, w.Hq, w.Sq))):
            io[n] = torch.full(shape, float("nan"), dtype=torch.float32).pin_memory()
        ios.append(io)
    stream = torch.cuda.current_stream(dev)
    for io in ios:
        sess.step(io, stream.cuda_stream)
    sess.join(stream.cuda_stream)
    stream.synchronize()
    binding.device_status()
    sess.close()
    for i, (io, ref) in enumerate(zip(ios, refs)):
        for n in ref:
            assert torch.equal(io[n], ref[n]), (i, n)
