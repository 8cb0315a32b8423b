"""Pins for the oracle's window mask and per-batch key lengths.

The window mask is the band of the HOT-Step page's self-attention over a window
(section 4), read as q - left <= kv <= q + right; the key lengths are the
padding terms of the SpecForge post's eagle3 mask_mod ("Flex Attention":
kv < seq_lengths[b] in the causal part, kv % Q_LEN < seq_lengths[b] in the
suffix part), applied as the same key bound to the other masks.

Each pin builds its expectation another way than the oracle's predicate:
numpy's diagonal-offset triangles for the band, closed-form pair counts,
torch fp64 sdpa on explicitly built masks or on truncated keys, the EAGLE3
concatenated-score construction with the padding terms, finite differences.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _band(Sq, Skv, wl, wr, length=None):
    """Band mask from numpy's triangles: kv - q <= wr (tril, offset wr) and
    kv - q >= -wl (triu, offset -wl), keys below the length."""
    ones = np.ones((Sq, Skv), dtype=np.uint8)
    m = np.tril(ones, wr) & np.triu(ones, -wl)
    if length is not None:
        m[:, length:] = 0
    return m


# ------------------------------------------------------------- mask pins
@pytest.mark.parametrize("Sq,Skv,wl,wr", [(9, 9, 2, 0), (9, 9, 3, 3), (7, 12, 0, 4), (12, 7, 5, 1),
                                          (6, 6, 0, 0), (5, 5, 10, 10)])
def test_window_mask_is_the_band(Sq, Skv, wl, wr):
    got = oracle.mask("window", 0, Sq, Skv, window=(wl, wr))
    np.testing.assert_array_equal(got, _band(Sq, Skv, wl, wr))


@pytest.mark.parametrize("mask,wl,wr,L", [("window", 3, 1, 6), ("causal", 0, 0, 4), ("full", 0, 0, 0),
                                          ("full", 0, 0, 9)])
def test_key_length_cuts_columns(mask, wl, wr, L):
    S = 9
    got = oracle.mask(mask, 0, S, S, window=(wl, wr), length=L)
    base = {"window": _band(S, S, wl, wr), "causal": np.tril(np.ones((S, S), np.uint8)),
            "full": np.ones((S, S), np.uint8)}[mask].copy()
    base[:, L:] = 0
    np.testing.assert_array_equal(got, base)


def test_ttt_key_length_follows_the_padding_terms():
    # S = 4, t = 2, seq_length 3: segment-0 keys 0..2 only (causal part shrunk by
    # 2 diagonals), suffix diagonal i of row q only for q < 3
    S, t, L = 4, 2, 3
    want = np.zeros((S, 3 * S), np.uint8)
    for q in range(S):
        for kv in range(S):
            want[q, kv] = int(kv <= q - t and kv < L)
        for i in (1, 2):
            want[q, i * S + q] = int(q < L)
    np.testing.assert_array_equal(oracle.mask("ttt", t, S, 3 * S, length=L), want)


@pytest.mark.parametrize("S,w", [(1, 0), (10, 0), (10, 3), (10, 9), (10, 25), (257, 64)])
def test_window_pair_counts_closed_form(S, w):
    def sum_min(S, w):  # sum over q in [0, S) of min(q, w)
        return S * (S - 1) // 2 if w >= S - 1 else w * S - w * (w + 1) // 2
    assert oracle.count_visible("window", 0, S, S, window=(w, 0)) == S + sum_min(S, w)
    assert oracle.count_visible("window", 0, S, S, window=(w, w)) == S + 2 * sum_min(S, w)


# --------------------------------------------------------- sdpa pins
def _sdpa_masked(q, k, v, m, scale, gqa):
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=torch.from_numpy(m.astype(bool)), scale=scale, enable_gqa=gqa)
    return tq, tk, tv, out


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,wl,wr", [
    (1, 2, 2, 24, 24, 8, 5, 0),
    (2, 4, 2, 31, 31, 16, 7, 7),
    (1, 8, 2, 20, 20, 4, 3, 9),
    (1, 2, 1, 16, 40, 8, 2, 30),
])
def test_window_against_torch_sdpa_fp64(B, Hq, Hkv, Sq, Skv, D, wl, wr):
    q = _rand((B, Hq, Sq, D), 30)
    k = _rand((B, Hkv, Skv, D), 31)
    v = _rand((B, Hkv, Skv, D), 32)
    do = _rand((B, Hq, Sq, D), 33)
    scale = 1.0 / math.sqrt(D)
    m = _band(Sq, Skv, wl, wr)
    assert m.any(axis=1).all()  # sdpa gives NaN on empty rows; those are pinned below
    o, lse = oracle.fwd(q, k, v, "window", 0, scale, window=(wl, wr))
    dq, dk, dv = oracle.bwd(q, k, v, do, "window", 0, scale, window=(wl, wr))
    tq, tk, tv, out = _sdpa_masked(q, k, v, m, scale, Hq != Hkv)
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=0, atol=1e-10)
    (out * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-10)
    G = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            s = np.where(m.astype(bool), q[b, h] @ k[b, h // G].T * scale, -np.inf)
            np.testing.assert_allclose(lse[b, h], logsumexp(s, axis=1), rtol=0, atol=1e-12)


@pytest.mark.parametrize("mask,wl,wr", [("causal", 0, 0), ("full", 0, 0), ("window", 6, 2)])
def test_key_lengths_equal_truncated_keys(mask, wl, wr):
    # each batch entry equals sdpa over its first L_b keys only
    B, Hq, Hkv, S, D = 3, 4, 2, 21, 8
    lens = [21, 13, 1]
    q = _rand((B, Hq, S, D), 40)
    k = _rand((B, Hkv, S, D), 41)
    v = _rand((B, Hkv, S, D), 42)
    do = _rand((B, Hq, S, D), 43)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.fwd(q, k, v, mask, 0, scale, window=(wl, wr), seq_lengths=lens)
    dq, dk, dv = oracle.bwd(q, k, v, do, mask, 0, scale, window=(wl, wr), seq_lengths=lens)
    for b, L in enumerate(lens):
        full = {"causal": np.tril(np.ones((S, S), np.uint8)), "full": np.ones((S, S), np.uint8),
                "window": _band(S, S, wl, wr)}[mask]
        m = full[:, :L]
        rows = m.any(axis=1)
        tq, tk, tv, out = _sdpa_masked(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L],
                                       m, scale, True)
        ref = out.detach().numpy()[0]
        np.testing.assert_allclose(o[b][:, rows], ref[:, rows], rtol=0, atol=1e-10)
        assert np.all(o[b][:, ~rows] == 0) and np.all(lse[b][:, ~rows] == 0)
        g = torch.from_numpy(do[b:b + 1]) * torch.from_numpy(rows[None, None, :, None].astype(float))
        torch.nan_to_num(out).mul(g).sum().backward()
        np.testing.assert_allclose(dq[b][:, rows], tq.grad.numpy()[0][:, rows], rtol=0, atol=1e-10)
        assert np.all(dq[b][:, ~rows] == 0)
        np.testing.assert_allclose(dk[b][:, :L], tk.grad.numpy()[0], rtol=0, atol=1e-10)
        np.testing.assert_allclose(dv[b][:, :L], tv.grad.numpy()[0], rtol=0, atol=1e-10)
        assert np.all(dk[b][:, L:] == 0) and np.all(dv[b][:, L:] == 0)


# ------------------------------------------- EAGLE3 construction with padding
def _eagle3_padded(q, k, v, t, L, scale):
    """The SpecForge construction (causal scores of segment 0 plus one diagonal
    dot product per appended segment, one softmax) with its padding terms:
    segment-0 keys at or past L and the diagonals of rows at or past L drop out.
    Rows left with nothing give O = 0, LSE = 0."""
    S = q.shape[-2]
    k0, v0 = k[:, :S], v[:, :S]
    s0 = q @ k0.transpose(-1, -2) * scale
    qi = torch.arange(S)[:, None]
    ki = torch.arange(S)[None, :]
    s0 = s0.masked_fill(~((ki <= qi - t) & (ki < L)), float("-inf"))
    parts = [s0]
    for i in range(1, t + 1):
        d = (q * k[:, i * S:(i + 1) * S]).sum(-1) * scale
        d = d.masked_fill(~(torch.arange(S) < L), float("-inf"))
        parts.append(d[..., None])
    w = torch.cat(parts, dim=-1)
    empty = torch.isinf(w).all(dim=-1)
    w_safe = w.masked_fill(empty[..., None], 0.0)
    lse = torch.logsumexp(w_safe, dim=-1).masked_fill(empty, 0.0)
    p = torch.softmax(w_safe, dim=-1).masked_fill(empty[..., None], 0.0)
    out = p[..., :S] @ v0
    for i in range(1, t + 1):
        out = out + p[..., S + i - 1, None] * v[:, i * S:(i + 1) * S]
    return out, lse


@pytest.mark.parametrize("S,t,D,L", [(8, 2, 4, 5), (10, 3, 8, 10), (7, 4, 4, 2), (6, 1, 8, 0)])
def test_ttt_key_lengths_against_eagle3_construction(S, t, D, L):
    H = 2
    q = _rand((1, H, S, D), 50)
    k = _rand((1, H, (t + 1) * S, D), 51)
    v = _rand((1, H, (t + 1) * S, D), 52)
    do = _rand((1, H, S, D), 53)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.fwd(q, k, v, "ttt", t, scale, seq_lengths=[L])
    dq, dk, dv = oracle.bwd(q, k, v, do, "ttt", t, scale, seq_lengths=[L])
    tq, tk, tv = (torch.tensor(x[0], requires_grad=True) for x in (q, k, v))
    oe, le = _eagle3_padded(tq, tk, tv, t, L, scale)
    np.testing.assert_allclose(o[0], oe.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], le.detach().numpy(), rtol=0, atol=1e-12)
    (oe * torch.from_numpy(do[0])).sum().backward()
    np.testing.assert_allclose(dq[0], tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk[0], tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv[0], tv.grad.numpy(), rtol=0, atol=1e-11)


# ------------------------------------------------------ finite differences
def test_finite_differences_window_with_key_lengths():
    B, Hq, Hkv, S, D = 2, 2, 1, 7, 3
    lens = [5, 7]
    q = _rand((B, Hq, S, D), 60)
    k = _rand((B, Hkv, S, D), 61)
    v = _rand((B, Hkv, S, D), 62)
    do = _rand((B, Hq, S, D), 63)
    scale = 0.6
    kw = dict(window=(2, 1), seq_lengths=lens)
    dq, dk, dv = oracle.bwd(q, k, v, do, "window", 0, scale, **kw)

    def L(qq, kk, vv):
        o, _ = oracle.fwd(qq, kk, vv, "window", 0, scale, **kw)
        return float((o * do).sum())

    h = 1e-6
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            up = L(*args)
            args[which][idx] -= 2 * h
            dn = L(*args)
            num[idx] = (up - dn) / (2 * h)
        np.testing.assert_allclose(grad, num, rtol=1e-7, atol=1e-8)


def test_window_rows_that_see_nothing():
    # window (0, 0) on Sq > Skv: rows past Skv see no key -> O = 0, LSE = 0, dQ = 0
    q = _rand((1, 1, 6, 4), 70)
    k = _rand((1, 1, 4, 4), 71)
    v = _rand((1, 1, 4, 4), 72)
    do = _rand((1, 1, 6, 4), 73)
    o, lse = oracle.fwd(q, k, v, "window", 0, 0.5, window=(0, 0))
    dq, _, _ = oracle.bwd(q, k, v, do, "window", 0, 0.5, window=(0, 0))
    assert np.all(o[0, 0, 4:] == 0) and np.all(lse[0, 0, 4:] == 0) and np.all(dq[0, 0, 4:] == 0)
    # rows 0..3 see exactly their own key: O = V row, LSE = scaled self score
    np.testing.assert_allclose(o[0, 0, :4], v[0, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0, :4], 0.5 * (q[0, 0, :4] * k[0, 0]).sum(-1), rtol=0,
                               atol=1e-14)


# ------------------------------------------------ mask-aware pair counts
@pytest.mark.parametrize("mask,Sq,Skv,t,window,length", [
    ("window", 300, 300, 0, (40, 0), None), ("window", 300, 300, 0, (17, 17), 211),
    ("window", 200, 450, 0, (0, 90), None), ("window", 450, 200, 0, (90, 3), 150),
    ("causal", 300, 300, 0, None, 123), ("causal", 200, 350, 0, None, 300),
    ("full", 100, 77, 0, None, 50), ("ttt", 64, 192, 2, None, 40), ("ttt", 64, 256, 3, None, 0),
])
def test_pair_counts_with_window_and_lengths(mask, Sq, Skv, t, window, length):
    from attention_tcgen05_tmem_gb300 import flops
    want = oracle.count_visible(mask, t, Sq, Skv, window=window, length=length)
    assert flops.visible_pairs_per_head(mask, Sq, Skv, t, window, length) == want
    # and the per-row sums that the CPU-baseline sample uses
    got = sum(flops.visible_pairs_rows(mask, Sq, Skv, t, window, length, r, r + 1)
              for r in range(Sq))
    assert got == want
