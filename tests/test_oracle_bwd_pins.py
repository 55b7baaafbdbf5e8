"""Pins of the oracle's backward pass (gradients of sum(O * dO)).

Source: "Attention kernels: FlashAttention and PagedAttention", section 四.3 (the backward
recomputes S and P = exp(S - LSE) and forms dV = P^T dO, dS, dQ, dK) and the FA4 engineering
page, section 2 (preprocess D = rowsum(dO * O)).  The gradient is pinned against central
finite differences of the forward oracle, against torch's fp64 autograd of
scaled_dot_product_attention, and by identities it must satisfy.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle


def f64(*shape, seed):
    return torch.randn(*shape, generator=torch.Generator().manual_seed(seed), dtype=torch.float64)


def loss(q, k, v, g, cu_q, cu_k, scale, causal, wl, wr):
    o, _ = oracle.attn_fwd(q, k, v, cu_q, cu_k, scale, causal, wl, wr)
    return float((o * g.numpy()).sum())


@pytest.mark.parametrize("lq,lk,Hq,Hkv,causal,wl,wr", [
    ([7, 5], [7, 5], 2, 1, True, -1, -1),
    ([6], [9], 4, 2, True, 2, -1),
    ([5, 3], [5, 3], 2, 2, False, 1, 2),
])
def test_gradient_matches_central_differences(lq, lk, Hq, Hkv, causal, wl, wr):
    d, scale, eps = 8, 0.4, 1e-5
    cu_q = np.cumsum([0] + lq).astype(np.int32)
    cu_k = np.cumsum([0] + lk).astype(np.int32)
    q, k, v = f64(cu_q[-1], Hq, d, seed=1), f64(cu_k[-1], Hkv, d, seed=2), f64(cu_k[-1], Hkv, d, seed=3)
    g = f64(cu_q[-1], Hq, d, seed=4)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, g, cu_q, cu_k, scale, causal, wl, wr)
    rng = np.random.default_rng(5)
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.clone(), x.clone()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": q, "k": k, "v": v}
            num = (loss(*[xp if n == name else args[n] for n in ("q", "k", "v")], g, cu_q, cu_k, scale, causal, wl, wr)
                   - loss(*[xm if n == name else args[n] for n in ("q", "k", "v")], g, cu_q, cu_k, scale, causal, wl, wr)) / (2 * eps)
            assert abs(num - grad[idx]) <= 1e-7 * (1 + abs(num)), (name, idx, num, grad[idx])


def test_gradient_matches_torch_fp64_autograd():
    Lq, Lk, Hq, Hkv, d, scale = 11, 14, 4, 2, 16, 0.3
    q, k, v = f64(Lq, Hq, d, seed=6), f64(Lk, Hkv, d, seed=7), f64(Lk, Hkv, d, seed=8)
    g = f64(Lq, Hq, d, seed=9)
    mask = torch.tensor([[bool(oracle.allowed(i, j, Lq, Lk, True, 5, -1)) for j in range(Lk)]
                         for i in range(Lq)])
    qt, kt, vt = (x.clone().transpose(0, 1).requires_grad_() for x in (q, k, v))
    o = F.scaled_dot_product_attention(qt[None], kt[None], vt[None], attn_mask=mask, scale=scale,
                                       enable_gqa=True)[0]
    (o * g.transpose(0, 1)).sum().backward()
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, g, [0, Lq], [0, Lk], scale, True, 5, -1)
    assert np.allclose(dq, qt.grad.transpose(0, 1).numpy(), atol=1e-12)
    assert np.allclose(dk, kt.grad.transpose(0, 1).numpy(), atol=1e-12)
    assert np.allclose(dv, vt.grad.transpose(0, 1).numpy(), atol=1e-12)


def test_D_is_rowsum_of_dout_times_out():
    q, k, v, g = f64(20, 2, 8, seed=10), f64(20, 2, 8, seed=11), f64(20, 2, 8, seed=12), f64(20, 2, 8, seed=13)
    o, _ = oracle.attn_fwd(q, k, v, [0, 20], [0, 20], 0.5, True)
    _, _, _, D = oracle.attn_bwd(q, k, v, g, [0, 20], [0, 20], 0.5, True)
    assert np.allclose(D, (o * g.numpy()).sum(-1).T, atol=1e-13)


def test_key_gradients_sum_to_zero_and_constant_v_has_no_qk_gradient():
    # sum_j dS_ij = 0 for every row, so sum_j dK_j = 0 over a sequence's keys
    q, k, v, g = f64(16, 4, 8, seed=14), f64(16, 2, 8, seed=15), f64(16, 2, 8, seed=16), f64(16, 4, 8, seed=17)
    cu = [0, 9, 16]
    dq, dk, dv, _ = oracle.attn_bwd(q, k, v, g, cu, cu, 0.5, True)
    for b in range(2):
        assert np.abs(dk[cu[b]:cu[b + 1]].sum(0)).max() < 1e-12
    assert np.abs(dk).max() > 1e-3  # not trivially zero
    # V constant along keys: O does not depend on Q or K
    vc = torch.ones(16, 2, 8, dtype=torch.float64) * torch.arange(8, dtype=torch.float64)
    dq, dk, dv, _ = oracle.attn_bwd(q, k, vc, g, cu, cu, 0.5, True)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
