"""Pins for the fp64 oracle against things other than itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped scale, a
wrong sign, a transposed operand, a wrong mask shift, a wrong GQA head map, a
wrong Delta) fails at least one of them:

* hand-derived TTT mask fixtures (tests/golden, from the SpecForge post's
  eagle3 mask_mod) and closed-form visible-pair counts;
* the EAGLE3 construction of the SpecForge post ("EAGLE3 Training"): causal
  scores concatenated with one diagonal dot product per appended segment,
  one softmax, then P0 V0 + sum_i p_i v_i -- forward, and its torch fp64
  autograd for the backward;
* torch.nn.functional.scaled_dot_product_attention in fp64 on the CPU
  (library special case; its own causal flag and GQA head map);
* central finite differences of L = sum(O * dO) (backward vs forward);
* a pure-Python scalar loop on tiny inputs (brute force);
* invariants (rows of P sum to 1, zero gradient on keys nobody sees,
  sum_kv dS = 0 through dQ with K = I) and closed forms.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from attention_tcgen05_tmem_gb300 import flops, synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape)


def _read_mask_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([int(c) for c in line])
    return np.array(rows, dtype=np.uint8)


# ---------------------------------------------------------------- mask pins
@pytest.mark.parametrize("fixture,S,t", [("ttt_mask_S4_t2.txt", 4, 2), ("ttt_mask_S3_t1.txt", 3, 1)])
def test_ttt_mask_matches_hand_fixture(fixture, S, t):
    want = _read_mask_fixture(fixture)
    got = oracle.mask("ttt", t, S, (t + 1) * S)
    assert want.shape == got.shape
    np.testing.assert_array_equal(got, want)


def test_ttt_step0_is_causal_and_causal_is_lower_triangle():
    S = 9
    np.testing.assert_array_equal(oracle.mask("ttt", 0, S, S), np.tril(np.ones((S, S), np.uint8)))
    np.testing.assert_array_equal(oracle.mask("causal", 0, S, S), np.tril(np.ones((S, S), np.uint8)))
    np.testing.assert_array_equal(oracle.mask("full", 0, 5, 7), np.ones((5, 7), np.uint8))


@pytest.mark.parametrize("mask,Sq,Skv,t", [("full", 7, 5, 0), ("causal", 13, 13, 0),
                                           ("causal", 9, 5, 0), ("causal", 5, 9, 0),
                                           ("ttt", 11, 11, 0), ("ttt", 11, 44, 3),
                                           ("ttt", 3, 21, 6)])
def test_visible_pair_closed_form(mask, Sq, Skv, t):
    assert flops.visible_pairs_per_head(mask, Sq, Skv, t) == oracle.count_visible(mask, t, Sq, Skv)


def test_ttt_row_counts_reading():
    # every row j >= t sees j+1 keys; rows j < t see only their t diagonals
    S, t = 10, 3
    m = oracle.mask("ttt", t, S, (t + 1) * S)
    for j in range(S):
        assert m[j].sum() == (j + 1 if j >= t else t)


# -------------------------------------------------- EAGLE3 construction pin
def _eagle3_construction(q, k, v, t, scale):
    """SpecForge post, "EAGLE3 Training": causal scores against segment 0
    (the causal part shrunk by t diagonals), concatenated with the per-row
    dot product against each appended segment i = 1..t, one softmax over the
    concatenation, output = P0 V0 + sum_i p_i v_i.  torch fp64, differentiable.
    q: [H, S, D]; k, v: [H, (t+1) S, D] (one kv head per q head here)."""
    H, S, D = q.shape
    k0, v0 = k[:, :S], v[:, :S]
    w0 = q @ k0.transpose(1, 2) * scale
    rows = torch.arange(S)[:, None]
    cols = torch.arange(S)[None, :]
    w0 = w0.masked_fill(~(cols <= rows - t), float("-inf"))
    parts = [w0]
    for i in range(1, t + 1):
        ki = k[:, i * S:(i + 1) * S]
        parts.append(((q * ki).sum(-1) * scale)[..., None])
    w = torch.cat(parts, dim=-1)
    lse = torch.logsumexp(w, dim=-1)
    p = torch.softmax(w, dim=-1)
    out = p[..., :S] @ v0
    for i in range(1, t + 1):
        vi = v[:, i * S:(i + 1) * S]
        out = out + p[..., S + i - 1, None] * vi
    return out, lse


@pytest.mark.parametrize("S,t,D", [(8, 1, 4), (12, 3, 8), (7, 6, 5), (16, 2, 16)])
def test_eagle3_construction_forward(S, t, D):
    H = 2
    q = _rand((1, H, S, D), 1)
    k = _rand((1, H, (t + 1) * S, D), 2)
    v = _rand((1, H, (t + 1) * S, D), 3)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.fwd(q, k, v, "ttt", t, scale)
    oe, le = _eagle3_construction(torch.from_numpy(q[0]), torch.from_numpy(k[0]),
                                  torch.from_numpy(v[0]), t, scale)
    np.testing.assert_allclose(o[0], oe.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], le.numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("S,t,D", [(8, 2, 4), (6, 4, 8)])
def test_eagle3_construction_backward(S, t, D):
    H = 2
    q = _rand((1, H, S, D), 4)
    k = _rand((1, H, (t + 1) * S, D), 5)
    v = _rand((1, H, (t + 1) * S, D), 6)
    do = _rand((1, H, S, D), 7)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = oracle.bwd(q, k, v, do, "ttt", t, scale)
    tq, tk, tv = (torch.tensor(x[0], requires_grad=True) for x in (q, k, v))
    out, _ = _eagle3_construction(tq, tk, tv, t, scale)
    (out * torch.from_numpy(do[0])).sum().backward()
    np.testing.assert_allclose(dq[0], tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk[0], tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv[0], tv.grad.numpy(), rtol=0, atol=1e-11)


# ------------------------------------------------------- torch sdpa pin
def _sdpa(q, k, v, mask, t, scale, Hq, Hkv):
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    Sq, Skv = q.shape[2], k.shape[2]
    kw = dict(scale=scale, enable_gqa=(Hq != Hkv))
    if mask == "causal" and Sq == Skv:
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, **kw)
    elif mask == "full":
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, **kw)
    else:
        m = torch.from_numpy(oracle.mask(mask, t, Sq, Skv).astype(bool))
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, **kw)
    return tq, tk, tv, out


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,mask,t", [
    (1, 2, 2, 16, 16, 8, "causal", 0),
    (2, 4, 2, 33, 33, 16, "causal", 0),
    (1, 8, 2, 20, 20, 4, "causal", 0),
    (2, 2, 1, 17, 9, 8, "full", 0),
    (1, 4, 4, 40, 40, 32, "full", 0),
    (1, 4, 2, 12, 36, 8, "ttt", 2),
    (1, 6, 3, 9, 63, 16, "ttt", 6),
])
def test_against_torch_sdpa_fp64(B, Hq, Hkv, Sq, Skv, D, mask, t):
    q = _rand((B, Hq, Sq, D), 10)
    k = _rand((B, Hkv, Skv, D), 11)
    v = _rand((B, Hkv, Skv, D), 12)
    do = _rand((B, Hq, Sq, D), 13)
    scale = 0.37 if D == 16 else 1.0 / math.sqrt(D)
    o, lse = oracle.fwd(q, k, v, mask, t, scale)
    dq, dk, dv = oracle.bwd(q, k, v, do, mask, t, scale)
    tq, tk, tv, out = _sdpa(q, k, v, mask, t, scale, Hq, Hkv)
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=0, atol=1e-10)
    (out * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-10)
    # LSE = logsumexp of the masked scaled scores (scipy's routine)
    from scipy.special import logsumexp
    G = Hq // Hkv
    vis = oracle.mask(mask, t, Sq, Skv).astype(bool)
    for b in range(B):
        for h in range(Hq):
            s = q[b, h] @ k[b, h // G].T * scale
            s = np.where(vis, s, -np.inf)
            np.testing.assert_allclose(lse[b, h], logsumexp(s, axis=1), rtol=0, atol=1e-12)


# --------------------------------------------------- finite differences
@pytest.mark.parametrize("mask,Hq,Hkv,Sq,Skv,D,t", [("causal", 2, 1, 6, 6, 4, 0),
                                                   ("ttt", 2, 1, 5, 15, 3, 2),
                                                   ("full", 1, 1, 4, 7, 3, 0)])
def test_finite_differences(mask, Hq, Hkv, Sq, Skv, D, t):
    q = _rand((1, Hq, Sq, D), 20)
    k = _rand((1, Hkv, Skv, D), 21)
    v = _rand((1, Hkv, Skv, D), 22)
    do = _rand((1, Hq, Sq, D), 23)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = oracle.bwd(q, k, v, do, mask, t, scale)

    def L(qq, kk, vv):
        o, _ = oracle.fwd(qq, kk, vv, mask, t, scale)
        return float((o * do).sum())

    h = 1e-6
    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            a_p = arr.copy()
            a_m = arr.copy()
            a_p[idx] += h
            a_m[idx] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which] = a_p
            args_m[which] = a_m
            num[idx] = (L(*args_p) - L(*args_m)) / (2 * h)
        assert np.abs(grad).max() > 1e-3  # non-vacuous (HOT-Step trap 7)
        err = np.abs(num - grad).max() / np.abs(grad).max()
        assert err < 1e-7, (which, err)


# --------------------------------------------------------- brute force
def _brute(q, k, v, do, mask, t, scale):
    """Scalar Python loops over one (b, h) with the predicate evaluated per
    pair through oracle.visible (pinned above)."""
    Sq, D = len(q), len(q[0])
    Skv = len(k)
    O = [[0.0] * D for _ in range(Sq)]
    LSE = [0.0] * Sq
    dQ = [[0.0] * D for _ in range(Sq)]
    dK = [[0.0] * D for _ in range(Skv)]
    dV = [[0.0] * D for _ in range(Skv)]
    for i in range(Sq):
        vis = [j for j in range(Skv) if oracle.visible(mask, t, Sq, Skv, i, j)]
        if not vis:
            continue
        s = {j: scale * sum(q[i][d] * k[j][d] for d in range(D)) for j in vis}
        mx = max(s.values())
        tot = sum(math.exp(x - mx) for x in s.values())
        LSE[i] = mx + math.log(tot)
        p = {j: math.exp(s[j] - LSE[i]) for j in vis}
        for d in range(D):
            O[i][d] = sum(p[j] * v[j][d] for j in vis)
        delta = sum(do[i][d] * O[i][d] for d in range(D))
        for j in vis:
            dp = sum(do[i][d] * v[j][d] for d in range(D))
            ds = p[j] * (dp - delta)
            for d in range(D):
                dQ[i][d] += scale * ds * k[j][d]
                dK[j][d] += scale * ds * q[i][d]
                dV[j][d] += p[j] * do[i][d]
    return O, LSE, dQ, dK, dV


@pytest.mark.parametrize("mask,Sq,Skv,t", [("causal", 12, 12, 0), ("full", 6, 10, 0), ("ttt", 8, 24, 2)])
def test_brute_force_tiny(mask, Sq, Skv, t):
    D = 5
    q = _rand((1, 1, Sq, D), 30)
    k = _rand((1, 1, Skv, D), 31)
    v = _rand((1, 1, Skv, D), 32)
    do = _rand((1, 1, Sq, D), 33)
    scale = 0.6
    o, lse = oracle.fwd(q, k, v, mask, t, scale)
    dq, dk, dv = oracle.bwd(q, k, v, do, mask, t, scale)
    bo, bl, bdq, bdk, bdv = _brute(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                                   do[0, 0].tolist(), mask, t, scale)
    for a, b in ((o[0, 0], bo), (lse[0, 0], bl), (dq[0, 0], bdq), (dk[0, 0], bdk), (dv[0, 0], bdv)):
        np.testing.assert_allclose(a, np.array(b), rtol=0, atol=1e-12)


# ------------------------------------------------ invariants, closed forms
@pytest.mark.parametrize("mask,Sq,Skv,t", [("causal", 10, 10, 0), ("ttt", 6, 24, 3), ("full", 5, 8, 0)])
def test_rows_of_p_sum_to_one_via_identity_v(mask, Sq, Skv, t):
    # with V = I (D = Skv) the output row is the weight row P itself
    q = _rand((1, 1, Sq, Skv), 40)
    k = _rand((1, 1, Skv, Skv), 41)
    v = np.eye(Skv)[None, None]
    o, lse = oracle.fwd(q, k, v, mask, t, 0.5)
    P = o[0, 0]
    vis = oracle.mask(mask, t, Sq, Skv).astype(bool)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(P[~vis] == 0.0)
    assert np.all(P[vis] > 0.0)


def test_zero_grad_on_keys_nobody_sees():
    # TTT: segment-0 keys kv > S-1-t are seen by no query
    S, t, D = 9, 3, 4
    q = _rand((1, 2, S, D), 50)
    k = _rand((1, 1, (t + 1) * S, D), 51)
    v = _rand((1, 1, (t + 1) * S, D), 52)
    do = _rand((1, 2, S, D), 53)
    _, dk, dv = oracle.bwd(q, k, v, do, "ttt", t)
    assert np.all(dk[0, 0, S - t:S] == 0.0) and np.all(dv[0, 0, S - t:S] == 0.0)
    assert np.abs(dk[0, 0, :S - t]).min(axis=1).max() > 0


def test_sum_of_ds_is_zero():
    # with K = 1 (all ones, one column) dQ[q] = scale * sum_kv dS[q, kv] = 0
    Sq, Skv = 11, 11
    q = _rand((1, 1, Sq, 1), 60)
    k = np.ones((1, 1, Skv, 1))
    v = _rand((1, 1, Skv, 1), 62)
    do = _rand((1, 1, Sq, 1), 63)
    dq, _, _ = oracle.bwd(q, k, v, do, "causal", 0, 1.0)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)


def test_closed_forms():
    D = 6
    q = _rand((1, 1, 1, D), 70)
    k = _rand((1, 1, 1, D), 71)
    v = _rand((1, 1, 1, D), 72)
    o, lse = oracle.fwd(q, k, v, "full", 0, 0.3)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 0], 0.3 * float(q[0, 0, 0] @ k[0, 0, 0]), atol=1e-14)
    # causal row 0 is V_0
    q = _rand((1, 1, 8, D), 73)
    k = _rand((1, 1, 8, D), 74)
    v = _rand((1, 1, 8, D), 75)
    o, _ = oracle.fwd(q, k, v, "causal", 0)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15)
    # K = 0: uniform weights over the visible keys
    for mask, t, Sq, Skv in (("causal", 0, 8, 8), ("full", 0, 5, 9), ("ttt", 3, 7, 28)):
        q = _rand((1, 1, Sq, D), 76)
        v = _rand((1, 1, Skv, D), 77)
        o, lse = oracle.fwd(q, np.zeros((1, 1, Skv, D)), v, mask, t)
        vis = oracle.mask(mask, t, Sq, Skv).astype(bool)
        for j in range(Sq):
            n = vis[j].sum()
            if mask == "ttt":
                assert n == (j + 1 if j >= t else t)
            np.testing.assert_allclose(o[0, 0, j], v[0, 0, vis[j]].mean(axis=0), atol=1e-13)
            np.testing.assert_allclose(lse[0, 0, j], math.log(n), atol=1e-13)


def test_gqa_group_sum_order_and_mapping():
    # dK of a kv head equals the sum of per-head results computed with Hkv=Hq
    B, Hq, Hkv, S, D = 1, 4, 2, 10, 4
    q = _rand((B, Hq, S, D), 80)
    k = _rand((B, Hkv, S, D), 81)
    v = _rand((B, Hkv, S, D), 82)
    do = _rand((B, Hq, S, D), 83)
    dq, dk, dv = oracle.bwd(q, k, v, do, "causal")
    kr = np.repeat(k, Hq // Hkv, axis=1)  # contiguous groups: kv head = h // G
    vr = np.repeat(v, Hq // Hkv, axis=1)
    dq2, dk2, dv2 = oracle.bwd(q, kr, vr, do, "causal")
    np.testing.assert_allclose(dq, dq2, atol=1e-14)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, 2, S, D).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, 2, S, D).sum(2), atol=1e-13)


@pytest.mark.parametrize("mask,Sq,Skv,t", [("causal", 7, 3, 0), ("causal", 3, 7, 0),
                                           ("full", 4, 1, 0), ("ttt", 5, 5, 0), ("ttt", 5, 35, 6),
                                           ("ttt", 2, 14, 6)])
def test_no_row_is_fully_masked(mask, Sq, Skv, t):
    # HOT-Step trap 9 defines O = 0, LSE = 0 for a row that sees no key.  For
    # the three masks no valid problem has such a row (causal always sees
    # kv = 0, TTT rows j < t still see their t diagonals), so the convention
    # is unreachable through the API; this pins that claim.
    assert oracle.mask(mask, t, Sq, Skv).sum(axis=1).min() >= 1


def test_inputs_are_seeded_and_bf16():
    w = synth.TINY
    a = synth.make_inputs(w)
    b = synth.make_inputs(w)
    for key in ("q", "k", "v", "dout"):
        assert a[key].dtype == torch.bfloat16
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["q"], a["k"][:, :, : w.Sq])
    assert a["q"].shape == (1, 2, 128, 64)


@pytest.mark.parametrize("mask,t,Sq,Skv", [("causal", 0, 40, 40), ("full", 0, 33, 50),
                                            ("ttt", 2, 20, 60)])
def test_row_restricted_oracle(mask, t, Sq, Skv):
    """rows=(r0, r1) restricts the oracle to those query rows: the forward's rows
    equal the full forward's; the backward's dQ rows equal the full dQ's, and its
    dK/dV equal the full backward with dO zeroed outside the rows (a zero dO row
    has dP = 0 and Delta = 0, so its dS and its dV terms vanish)."""
    g = np.random.default_rng(17)
    q = g.standard_normal((1, 4, Sq, 16))
    k = g.standard_normal((1, 2, Skv, 16))
    v = g.standard_normal((1, 2, Skv, 16))
    do = g.standard_normal((1, 4, Sq, 16))
    r0, r1 = Sq // 3, Sq - 2
    o, lse = oracle.fwd(q, k, v, mask, t)
    o_r, lse_r = oracle.fwd(q, k, v, mask, t, rows=(r0, r1))
    np.testing.assert_array_equal(o_r[:, :, r0:r1], o[:, :, r0:r1])
    np.testing.assert_array_equal(lse_r[:, :, r0:r1], lse[:, :, r0:r1])
    assert not o_r[:, :, :r0].any() and not o_r[:, :, r1:].any()
    dq, _, _ = oracle.bwd(q, k, v, do, mask, t)
    dq_r, dk_r, dv_r = oracle.bwd(q, k, v, do, mask, t, rows=(r0, r1))
    np.testing.assert_allclose(dq_r[:, :, r0:r1], dq[:, :, r0:r1], rtol=0, atol=1e-13)
    do_band = np.zeros_like(do)
    do_band[:, :, r0:r1] = do[:, :, r0:r1]
    _, dk_b, dv_b = oracle.bwd(q, k, v, do_band, mask, t)
    np.testing.assert_allclose(dk_r, dk_b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv_r, dv_b, rtol=0, atol=1e-13)
