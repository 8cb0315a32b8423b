"""Pins for the soft-target log-softmax loss oracle (SpecForge long-context
post, "In-place Gradient Calculation") against things other than itself:
torch's log_softmax with autograd (the page's PyTorch definition of the loss,
run through a library routine and its automatic gradient), torch's
cross_entropy for one-hot targets, a closed form for uniform logits, scipy's
logsumexp for the row statistics, central finite differences, and the
invariants of the gradient (rows sum to zero, masked rows are zero)."""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle import softmax_loss as sl


def _case(N, V, seed, mask_frac=0.25):
    g = np.random.default_rng(seed)
    x = g.standard_normal((N, V)) * 2.0
    u = g.exponential(size=(N, V))
    p = u / u.sum(axis=1, keepdims=True)  # soft targets: rows of a probability simplex
    mask = (g.random(N) >= mask_frac).astype(np.float64)
    return x, p, mask


@pytest.mark.parametrize("B,T,V", [(1, 7, 11), (2, 5, 64), (1, 33, 1000)])
def test_against_torch_log_softmax_autograd(B, T, V):
    x, p, mask = _case(B * T, V, 1)
    x, p, mask = x.reshape(B, T, V), p.reshape(B, T, V), mask.reshape(B, T, 1)
    tx = torch.tensor(x, requires_grad=True)
    logp = torch.nn.LogSoftmax(dim=2)(tx)
    ref = -torch.sum(torch.from_numpy(mask) * torch.from_numpy(p) * logp, 2).mean()
    ref.backward(torch.tensor(0.7, dtype=torch.float64))
    loss, _, _ = sl.forward(x, p, mask)
    grad = sl.backward(x, p, mask, grad_loss=0.7)
    assert abs(loss - ref.item()) < 1e-12
    np.testing.assert_allclose(grad, tx.grad.numpy(), rtol=0, atol=1e-14)


def test_one_hot_targets_equal_cross_entropy():
    N, V = 40, 257
    g = np.random.default_rng(2)
    x = g.standard_normal((N, V)) * 3
    y = g.integers(0, V, N)
    p = np.zeros((N, V))
    p[np.arange(N), y] = 1.0
    loss, row_loss, _ = sl.forward(x, p)
    ce = torch.nn.functional.cross_entropy(torch.from_numpy(x), torch.from_numpy(y),
                                           reduction="none").numpy()
    np.testing.assert_allclose(row_loss, ce, rtol=0, atol=1e-12)
    assert abs(loss - ce.mean()) < 1e-12


def test_uniform_logits_closed_form():
    N, V = 9, 500
    _, p, mask = _case(N, V, 3)
    x = np.full((N, V), 1.25)
    loss, row_loss, lse = sl.forward(x, p, mask)
    np.testing.assert_allclose(row_loss, p.sum(1) * np.log(V), rtol=1e-14, atol=0)
    assert abs(loss - (mask * p.sum(1)).sum() * np.log(V) / N) < 1e-12
    np.testing.assert_allclose(lse, 1.25 + np.log(V), rtol=1e-14, atol=0)


def test_row_statistics_are_logsumexp():
    x, _, _ = _case(20, 300, 4)
    m, d = sl.row_stats(x)
    np.testing.assert_allclose(m + np.log(d), logsumexp(x, axis=1), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(m, x.max(axis=1))


def test_finite_differences():
    x, p, mask = _case(4, 6, 5, mask_frac=0.3)
    grad = sl.backward(x, p, mask)
    h = 1e-6
    num = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            num[i, j] = (sl.forward(xp, p, mask)[0] - sl.forward(xm, p, mask)[0]) / (2 * h)
    # central difference error: rounding ~ eps |L| / h ~ 1e-10, truncation ~ h^2 ~ 1e-12
    np.testing.assert_allclose(grad, num, rtol=1e-7, atol=5e-10)


def test_gradient_invariants():
    x, p, mask = _case(50, 128, 6, mask_frac=0.4)
    # targets that do not sum to one (a soft target may be unnormalised)
    p = p * np.random.default_rng(7).uniform(0.5, 1.5, (50, 1))
    grad = sl.backward(x, p, mask, grad_loss=2.0)
    np.testing.assert_allclose(grad.sum(axis=1), 0.0, rtol=0, atol=1e-15)
    assert np.all(grad[mask == 0] == 0)
    assert np.abs(grad[mask == 1]).max() > 1e-4
