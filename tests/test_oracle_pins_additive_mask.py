"""Pins for the oracle's additive mask (HOT-Step flash-attn-training, section
3: its ops accept an arbitrary additive mask shaped [S_kv, S], or [S_kv, S, 1, B]
with broadcast):
torch fp64 sdpa with a float attn_mask and autograd (per-batch and broadcast
masks, -inf entries, GQA, combined with the causal kind), the closed form of a
constant bias (softmax unchanged, LSE shifted by the bias), and rows that the
mask hides completely (O = 0, LSE = 0, no gradient)."""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _bias(Bm, Sq, Skv, seed, ninf=0.2):
    g = np.random.default_rng(seed)
    m = g.standard_normal((Bm, Sq, Skv)) * 0.7
    m[g.random((Bm, Sq, Skv)) < ninf] = -np.inf
    m[..., 0] = 0.3  # keep every row non-empty (sdpa returns NaN on empty rows)
    return m


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,kind,Bm", [
    (2, 2, 2, 19, 19, 8, "full", 2),
    (2, 4, 2, 24, 31, 16, "full", 1),
    (1, 4, 1, 21, 21, 4, "causal", 1),
    (2, 2, 1, 17, 17, 8, "causal", 2),
])
def test_additive_mask_against_torch_sdpa(B, Hq, Hkv, Sq, Skv, D, kind, Bm):
    q = _rand((B, Hq, Sq, D), 80)
    k = _rand((B, Hkv, Skv, D), 81)
    v = _rand((B, Hkv, Skv, D), 82)
    do = _rand((B, Hq, Sq, D), 83)
    scale = 1.0 / math.sqrt(D)
    m = _bias(Bm, Sq, Skv, 84)
    o, lse = oracle.fwd(q, k, v, kind, 0, scale, add_mask=m)
    dq, dk, dv = oracle.bwd(q, k, v, do, kind, 0, scale, add_mask=m)
    full = np.broadcast_to(m, (B, Sq, Skv)).copy()
    if kind == "causal":
        full = np.where(np.tril(np.ones((Sq, Skv), bool)), full, -np.inf)
    tm = torch.from_numpy(full)[:, None]  # [B, 1, Sq, Skv], broadcast over heads
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=tm, scale=scale,
                                                           enable_gqa=Hq != Hkv)
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=0, atol=1e-10)
    (out * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-10)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            s = q[b, h] @ k[b, h // G].T * scale + full[b]
            np.testing.assert_allclose(lse[b, h], logsumexp(s, axis=1), rtol=0, atol=1e-12)


def test_constant_bias_shifts_only_the_lse():
    q, k, v = _rand((1, 2, 9, 4), 90), _rand((1, 2, 13, 4), 91), _rand((1, 2, 13, 4), 92)
    o0, l0 = oracle.fwd(q, k, v, "full", 0, 0.5)
    o1, l1 = oracle.fwd(q, k, v, "full", 0, 0.5, add_mask=np.full((9, 13), 2.5))
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l0 + 2.5, rtol=0, atol=1e-13)


def test_rows_hidden_by_the_mask():
    q, k, v, do = (_rand(s, 93 + i) for i, s in enumerate([(1, 1, 6, 4), (1, 1, 6, 4),
                                                           (1, 1, 6, 4), (1, 1, 6, 4)]))
    m = np.zeros((6, 6))
    m[2] = -np.inf
    m[4, :] = -np.inf
    o, lse = oracle.fwd(q, k, v, "full", 0, 0.5, add_mask=m)
    dq, dk, dv = oracle.bwd(q, k, v, do, "full", 0, 0.5, add_mask=m)
    for r in (2, 4):
        assert np.all(o[0, 0, r] == 0) and lse[0, 0, r] == 0 and np.all(dq[0, 0, r] == 0)
    # the hidden rows contribute nothing to dK, dV: drop them and compare
    keep = [0, 1, 3, 5]
    _, dk2, dv2 = oracle.bwd(q[:, :, keep], k, v, do[:, :, keep], "full", 0, 0.5,
                             add_mask=m[keep])
    np.testing.assert_allclose(dk, dk2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, dv2, rtol=0, atol=1e-14)
