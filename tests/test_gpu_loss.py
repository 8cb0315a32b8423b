"""GPU parity of the soft-target log-softmax loss (SpecForge long-context post,
"In-place Gradient Calculation") against the fp64 oracle: the mean loss, the
row statistics and the in-place gradient, on ragged and strided rows, plus
bitwise determinism and a sampled check at the page's largest shape."""
import numpy as np
import pytest
import torch

from attention_tcgen05_tmem_gb300 import binding, synth
from oracle import softmax_loss as sl
from tests.gpu_util import device

# fp32 accumulation over up to 64000 entries, ex2.approx (~2^-22 relative)
RTOL = 2e-5


def _close(name, got, want, rtol=RTOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    scale = max(np.abs(want).max(), 1e-30)
    err = np.abs(got - want).max() / scale
    assert err <= rtol, f"{name}: max |diff| / max |ref| = {err:.3g} > {rtol}"


def _run(w, ld_pad=0):
    dev = device()
    x = synth.make_loss_inputs(w)
    V = w.V
    if ld_pad:
        # rows inside a wider buffer (row stride V + ld_pad)
        buf = torch.zeros(w.B, w.T, V + ld_pad, dtype=torch.float32, device=dev)
        logits = buf[..., :V]
        logits.copy_(x["logits"].to(dev))
    else:
        logits = x["logits"].to(dev).contiguous()
    target = x["target"].to(dev)
    mask = x["mask"].to(dev)
    loss, row_loss, row_lse, row_tsum = binding.logsoftmax_loss(logits, target, mask)
    grad_loss = torch.tensor([0.75], device=dev)
    binding.logsoftmax_loss_bwd_raw(logits, target, mask.reshape(-1), row_lse, row_tsum, grad_loss)
    torch.cuda.synchronize()
    ref_loss, ref_row, ref_lse = sl.forward(x["logits"], x["target"], x["mask"])
    ref_grad = sl.backward(x["logits"], x["target"], x["mask"], grad_loss=0.75)
    _close("loss", [loss.item()], [ref_loss])
    _close("row_loss", row_loss.cpu(), ref_row)
    _close("row_lse", row_lse.cpu(), ref_lse)
    _close("row_tsum", row_tsum.cpu(), x["target"].double().sum(-1).reshape(-1))
    _close("grad", logits.cpu(), ref_grad)
    m = x["mask"].reshape(-1) == 0
    if m.any():
        assert torch.all(logits.reshape(-1, V)[m.to(dev)] == 0)


CASES = [synth.LossWorkload("loss_tiny_ragged", 1, 7, 11), synth.LossWorkload("loss_b2", 2, 33, 1000),
         synth.LossWorkload("loss_v32000", 1, 130, 32000), synth.LossWorkload("loss_v64001", 1, 40, 64001)]


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_loss_parity(w):
    _run(w)


@pytest.mark.gpu
def test_loss_strided_rows():
    _run(synth.LossWorkload("loss_strided", 2, 17, 999), ld_pad=13)


@pytest.mark.gpu
def test_loss_is_bitwise_deterministic():
    dev = device()
    x = synth.make_loss_inputs(synth.LossWorkload("det", 1, 64, 32000))
    out = []
    for _ in range(2):
        logits = x["logits"].to(dev)
        target, mask = x["target"].to(dev), x["mask"].to(dev)
        loss, _, lse, tsum = binding.logsoftmax_loss(logits, target, mask)
        binding.logsoftmax_loss_bwd_raw(logits, target, mask.reshape(-1), lse, tsum)
        out.append((loss.clone(), logits.clone()))
    assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1])


@pytest.mark.gpu
@pytest.mark.timeout(1200)
def test_loss_full_size_sampled():
    # the page's largest shape; the oracle checks 48 rows spread over it and the
    # mean against the device's own rows
    w = synth.LOSS[-1]
    dev = device()
    x = synth.make_loss_inputs(w)
    logits = x["logits"].to(dev)
    target, mask = x["target"].to(dev), x["mask"].to(dev)
    loss, row_loss, row_lse, row_tsum = binding.logsoftmax_loss(logits, target, mask)
    binding.logsoftmax_loss_bwd_raw(logits, target, mask.reshape(-1), row_lse, row_tsum)
    torch.cuda.synchronize()
    N = w.rows
    rows = np.linspace(0, N - 1, 48).astype(int)
    xl = x["logits"].reshape(N, w.V)[rows]
    xt = x["target"].reshape(N, w.V)[rows]
    xm = x["mask"].reshape(N)[rows]
    _, ref_row, ref_lse = sl.forward(xl, xt, xm)
    # the sampled rows' gradient with the full problem's 1/N
    ref_grad = sl.backward(xl, xt, xm, grad_loss=len(rows) / N)
    _close("row_loss", row_loss.cpu()[rows], ref_row)
    _close("row_lse", row_lse.cpu()[rows], ref_lse)
    _close("grad", logits.reshape(N, w.V)[torch.from_numpy(rows).to(dev)].cpu(), ref_grad)
    mean = (x["mask"].reshape(-1).double() * row_loss.cpu().double()).sum().item() / N
    assert abs(loss.item() - mean) <= 1e-6 * abs(mean)


@pytest.mark.gpu
def test_loss_extreme_logits():
    """Logits of magnitude ~250 (exp of them overflows fp32 without the running
    max) and one-hot targets: the forward's online max / sum and the backward's
    exp(x - lse) stay finite and match the oracle."""
    dev = device()
    w = synth.LossWorkload("loss_extreme", 1, 64, 5000)
    x = synth.make_loss_inputs(w)
    x["logits"] = x["logits"] * 100.0
    hot = torch.zeros_like(x["target"])
    idx = torch.arange(w.T) * 37 % w.V
    hot[0, torch.arange(w.T), idx] = 1.0
    x["target"] = hot
    logits = x["logits"].to(dev).contiguous()
    target, mask = x["target"].to(dev), x["mask"].to(dev)
    loss, row_loss, row_lse, row_tsum = binding.logsoftmax_loss(logits, target, mask)
    binding.logsoftmax_loss_bwd_raw(logits, target, mask.reshape(-1), row_lse, row_tsum)
    torch.cuda.synchronize()
    assert torch.isfinite(logits).all() and torch.isfinite(row_loss).all()
    ref_loss, ref_row, ref_lse = sl.forward(x["logits"], x["target"], x["mask"])
    ref_grad = sl.backward(x["logits"], x["target"], x["mask"])
    # exp(x - lse) with |x|, |lse| ~ 900 in fp32: lse (and x log2(e)) carry an absolute
    # error of about one fp32 ulp of |x| (2^-24 |x| ~ 5e-5), which exp turns into the
    # same relative error of the gradient; the bar adds four such ulps
    rtol = RTOL + 4 * 2.0 ** -24 * float(x["logits"].abs().max())
    _close("loss", [loss.item()], [ref_loss])
    _close("row_lse", row_lse.cpu(), ref_lse)
    _close("row_loss", row_loss.cpu(), ref_row, rtol)
    _close("grad", logits.cpu(), ref_grad, rtol)
