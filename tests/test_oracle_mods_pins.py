"""Pins of the oracle's score modifiers ("04 · FA4 (CuTeDSL) and engineering interfaces",
section 7): softcap s' = c tanh(s / c) on the scaled score, and ALiBi, a linear position bias
(the pages give no formula; the reading taken is -slope_h |i + Lk - Lq - j|, the distance
between the query's bottom-right-aligned position and the key), applied after the softcap and
before the visibility mask."""
import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import oracle


def f64(*shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed), dtype=torch.float64)


def test_no_modifier_equals_plain_attention():
    q, k, v = f64(30, 4, 16, seed=1), f64(40, 2, 16, seed=2), f64(40, 2, 16, seed=3)
    o0, l0 = oracle.attn_fwd(q, k, v, [0, 30], [0, 40], 0.3, True, 7, -1)
    o1, l1 = oracle.attn_fwd_mods(q, k, v, [0, 30], [0, 40], 0.3, True, 7, -1)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    # a very large cap leaves the scores unchanged (tanh(x) ~ x)
    o2, l2 = oracle.attn_fwd_mods(q, k, v, [0, 30], [0, 40], 0.3, True, 7, -1, softcap=1e9)
    assert np.allclose(o2, o0, atol=1e-12) and np.allclose(l2, l0, atol=1e-12)


def test_softcap_two_keys_closed_form_and_saturation():
    # d = 1, scale 1, q = 1, keys 0 and a, values 0 and 1: O = sigma(c tanh(a / c))
    c = 2.0
    for a in (0.5, 3.0, 40.0):
        q = torch.ones(1, 1, 1, dtype=torch.float64)
        k = torch.tensor([[[0.0]], [[a]]], dtype=torch.float64)
        v = torch.tensor([[[0.0]], [[1.0]]], dtype=torch.float64)
        o, l = oracle.attn_fwd_mods(q, k, v, [0, 1], [0, 2], 1.0, False, softcap=c)
        s1 = c * math.tanh(a / c)
        assert abs(o[0, 0, 0] - 1 / (1 + math.exp(-s1))) < 1e-14
        assert abs(l[0, 0] - math.log(1 + math.exp(s1))) < 1e-14
    # saturation: however large the score, it never exceeds the cap
    assert o[0, 0, 0] <= 1 / (1 + math.exp(-c)) + 1e-15


def test_alibi_matches_torch_sdpa_with_a_float_bias():
    Lq, Lk, Hq, Hkv, d, scale = 13, 21, 4, 2, 16, 0.35
    q, k, v = f64(Lq, Hq, d, seed=4), f64(Lk, Hkv, d, seed=5), f64(Lk, Hkv, d, seed=6)
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])
    o, l = oracle.attn_fwd_mods(q, k, v, [0, Lq], [0, Lk], scale, True, alibi_slopes=slopes)
    pos = torch.arange(Lq, dtype=torch.float64)[:, None] + (Lk - Lq)
    dist = (pos - torch.arange(Lk, dtype=torch.float64)[None, :]).abs()
    bias = -torch.tensor(slopes)[:, None, None] * dist[None]
    causal = torch.arange(Lk)[None, :] <= torch.arange(Lq)[:, None] + (Lk - Lq)
    bias = bias.masked_fill(~causal[None], float("-inf"))
    ref = F.scaled_dot_product_attention(q.transpose(0, 1)[None], k.transpose(0, 1)[None],
                                         v.transpose(0, 1)[None], attn_mask=bias[None],
                                         scale=scale, enable_gqa=True)[0].transpose(0, 1)
    s = torch.einsum("ihd,jhd->hij", q, k.repeat_interleave(2, 1)) * scale + bias
    assert np.allclose(o, ref.numpy(), atol=1e-12)
    assert np.allclose(l, torch.logsumexp(s, -1).numpy(), atol=1e-12)


def test_alibi_uniform_scores_closed_form():
    # q = 0: every score is 0, so P_j is proportional to exp(-m |pos - j|)
    Lk, m = 9, 0.7
    q = torch.zeros(1, 1, 4, dtype=torch.float64)
    k = f64(Lk, 1, 4, seed=7)
    v = torch.arange(Lk, dtype=torch.float64)[:, None, None].expand(Lk, 1, 4).contiguous()
    o, l = oracle.attn_fwd_mods(q, k, v, [0, 1], [0, Lk], 1.0, False, alibi_slopes=[m])
    w = np.exp(-m * np.abs((Lk - 1) - np.arange(Lk)))
    assert abs(o[0, 0, 0] - (w * np.arange(Lk)).sum() / w.sum()) < 1e-12
    assert abs(l[0, 0] - math.log(w.sum())) < 1e-12


def test_softcap_then_alibi_order():
    # with both: the bias is added to the capped score (the cap does not bound the bias)
    c, m = 1.0, 3.0
    q = torch.ones(1, 1, 1, dtype=torch.float64)
    k = torch.tensor([[[50.0]], [[50.0]]], dtype=torch.float64)
    v = torch.tensor([[[0.0]], [[1.0]]], dtype=torch.float64)
    o, l = oracle.attn_fwd_mods(q, k, v, [0, 1], [0, 2], 1.0, False, softcap=c, alibi_slopes=[m])
    # query position 1: scores c tanh(50) - m and c tanh(50) - 0
    s0, s1 = c * math.tanh(50.0) - m, c * math.tanh(50.0)
    assert abs(o[0, 0, 0] - math.exp(s1) / (math.exp(s0) + math.exp(s1))) < 1e-14
