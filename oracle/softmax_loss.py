"""fp64 CPU oracle for the soft-target log-softmax loss (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the product never calls it and it shares
no code with the CUDA path.

What it computes (SpecForge long-context post, "In-place Gradient
Calculation": the EAGLE3 loss of one TTT step over logits [B, T, V], soft
target probabilities [B, T, V] and a position mask [B, T, 1]):

    out_logp = log_softmax(logits, dim=V)
    loss     = -mean over (b, t) of  mask[b, t] * sum_v target[b, t, v] * out_logp[b, t, v]

Rows are the B*T positions, so the mean divides by N = B*T whatever the
mask.  The backward of that loss with respect to the logits, for an upstream
scalar gradient G, is

    dlogits[r, v] = -(G * mask[r] / N) * (target[r, v] - softmax(logits[r])_v * sum_u target[r, u])

which the page writes with grad_output = G * mask / N per row:
grad = -(target * grad_output - softmax * sum(target * grad_output)).  The
row statistics the page keeps between the passes (running max m and sum d,
so that ln d + m = logsumexp) are returned as well.
"""
from __future__ import annotations

import numpy as np


def _f64(a):
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def row_stats(logits):
    """Per row: (m = max_v x, d = sum_v exp(x - m)), the page's two row statistics."""
    x = _f64(logits)
    m = x.max(axis=-1)
    d = np.exp(x - m[..., None]).sum(axis=-1)
    return m, d


def log_softmax(logits):
    x = _f64(logits)
    m, d = row_stats(x)
    return x - (m + np.log(d))[..., None]


def forward(logits, target, mask=None):
    """Returns (loss, row_loss, lse): the mean loss, the per-row
    -sum_v target * log_softmax (before the mask) and the per-row
    logsumexp m + ln d.  logits, target: [N, V] (or [B, T, V]); mask: [N] or None."""
    x = _f64(logits)
    p = _f64(target)
    V = x.shape[-1]
    x2 = x.reshape(-1, V)
    p2 = p.reshape(-1, V)
    N = x2.shape[0]
    mk = np.ones(N) if mask is None else _f64(mask).reshape(-1)
    logp = log_softmax(x2)
    row_loss = -(p2 * logp).sum(axis=-1)
    m, d = row_stats(x2)
    loss = float((mk * row_loss).sum() / N)
    return loss, row_loss, m + np.log(d)


def backward(logits, target, mask=None, grad_loss: float = 1.0):
    """dLoss/dlogits times grad_loss, same shape as logits."""
    x = _f64(logits)
    p = _f64(target)
    V = x.shape[-1]
    x2 = x.reshape(-1, V)
    p2 = p.reshape(-1, V)
    N = x2.shape[0]
    mk = np.ones(N) if mask is None else _f64(mask).reshape(-1)
    g = grad_loss * mk / N  # the page's per-row grad_output
    soft = np.exp(log_softmax(x2))
    tsum = p2.sum(axis=-1)
    grad = -(p2 * g[:, None] - soft * (tsum * g)[:, None])
    return grad.reshape(x.shape)
