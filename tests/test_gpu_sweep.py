"""Seeded random configurations of every forward entry point against the fp64 oracle.

Each seed draws a batch (1-5 sequences, empty and one-token ones among them), a head pairing
(GQA ratios 1, 2, 3, 4, 8, 64, 128), d in {64, 128}, causal or not, an optional window and lengths up to
a few hundred tokens, then runs with those: the bf16 prefill, the FP8 forward (d = 128, small
batches), the paged decode (page sizes 16-256, automatic and fixed split counts) and the
chunked prefill over a paged cache (with or without rotary embedding).  Tolerances are those
of the dedicated tests: tests.parity for bf16 results, the realised e4m3 bound for FP8, and the
appended cache rows bit-exact or within one bf16 ulp where rotated.
"""
import random

import numpy as np
import pytest
import torch

from exact_attention_70_gb300 import synth
from oracle import oracle
from tests.fp8_exact import fp8_forward_bound
from tests.parity import compare

pytestmark = pytest.mark.gpu

SEEDS = range(96)
HEADS = [(1, 1), (2, 1), (4, 2), (6, 2), (8, 8), (16, 2), (12, 4), (32, 4), (64, 1), (128, 2),
         (128, 1), (8, 2)]


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_70_gb300 import build as attn_build
    attn_build.build()
    from exact_attention_70_gb300 import binding
    binding.load()
    return binding


def draw(seed):
    rnd = random.Random(5000 + seed)
    B = rnd.randint(1, 5)
    Hq, Hkv = rnd.choice(HEADS)
    d = rnd.choice([64, 128])
    causal = rnd.random() < 0.6
    lq = [rnd.choice([0, 1, rnd.randint(1, 64), rnd.randint(1, 700)]) for _ in range(B)]
    if rnd.random() < 0.5:
        lk = list(lq)
    elif causal:
        lk = [q + rnd.randint(0, 400) for q in lq]
    else:
        lk = [rnd.choice([0, rnd.randint(1, 900)]) for _ in lq]
    if Hq >= 64:  # (128 query rows per token and head group: keep the oracle's work small)
        lq = [min(q, 160) for q in lq]
        lk = [min(x, 400) for x in lk]
    if rnd.random() < 0.6:
        window = (-1, -1)
    else:
        window = (rnd.choice([-1, rnd.randint(0, 300)]),
                  0 if causal else rnd.choice([-1, rnd.randint(0, 300)]))
    return rnd, dict(B=B, Hq=Hq, Hkv=Hkv, d=d, causal=causal, lq=lq, lk=lk, window=window)


@pytest.mark.parametrize("seed", SEEDS)
def test_random_configuration(attn, seed):
    rnd, k = draw(seed)
    dev = "cuda"
    name = f"sweep{seed} {k}"
    # bf16 prefill
    c = synth.prefill_case(k["lq"], k["Hq"], k["Hkv"], k["d"], k["causal"], seed=6000 + seed,
                           lengths_k=k["lk"], window=k["window"], name=name)
    out, lse = attn.attn_fwd(c.q.to(dev), c.k.to(dev), c.v.to(dev), c.cu_seqlens_q.to(dev),
                             c.cu_seqlens_k.to(dev), c.max_seqlen_q, c.max_seqlen_k,
                             c.softmax_scale, c.causal, c.window_left, c.window_right)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0, name
    o_ref, l_ref = oracle.attn_fwd(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                   c.softmax_scale, c.causal, c.window_left, c.window_right)
    compare(out.cpu(), lse.cpu().T, o_ref, l_ref.T, name)
    # FP8 forward on the same shapes (d = 128; small batches keep the bound's cost down)
    if k["d"] == 128 and sum(k["lq"]) * k["Hq"] <= 4000:
        c8 = synth.fp8_case(k["lq"], k["Hq"], k["Hkv"], 128, k["causal"], seed=7000 + seed,
                            lengths_k=k["lk"], window=k["window"])
        args = [x.to(dev) for x in (c8.q8, c8.k8, c8.v8t, c8.q_scale, c8.k_scale, c8.v_scale,
                                    c8.cu_seqlens_q, c8.cu_seqlens_k)]
        o8, l8 = attn.attn_fwd_fp8(*args, c8.max_seqlen_q, c8.max_seqlen_k, c8.softmax_scale,
                                   c8.causal, c8.window_left, c8.window_right)
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0, name
        r_o, r_l = oracle.fp8_attn_fwd(c8.q8, c8.k8, c8.v8t, c8.q_scale, c8.k_scale, c8.v_scale,
                                       c8.cu_seqlens_q, c8.cu_seqlens_k, c8.softmax_scale,
                                       c8.causal, c8.window_left, c8.window_right)
        q, kk, v = oracle.fp8_dequantize(c8.q8, c8.k8, c8.v8t, c8.q_scale, c8.k_scale,
                                         c8.v_scale, c8.cu_seqlens_k)
        bound, _ = fp8_forward_bound(q, kk, v, c8.cu_seqlens_q.numpy(), c8.cu_seqlens_k.numpy(),
                                     c8.softmax_scale, c8.causal, c8.window_left,
                                     c8.window_right, None)
        err = np.abs(o8.float().cpu().numpy() - r_o)
        assert np.all(err <= bound + 1e-6), (name, float((err / (bound + 1e-6)).max()))
        fin = np.isfinite(r_l)
        l8 = l8.cpu().numpy()
        assert np.array_equal(fin, np.isfinite(l8)), name
        if fin.any():
            assert np.abs(l8[fin] - r_l[fin]).max() <= 1e-3, name
    # paged decode with the same heads
    page = rnd.choice([16, 32, 64, 128, 256])
    dc = synth.decode_case([rnd.randint(1, 3000) for _ in range(k["B"])], k["Hq"], k["Hkv"],
                           k["d"], page, seed=8000 + seed)
    do, dl = attn.attn_decode_kvcache(dc.q.to(dev), dc.k_cache.to(dev), dc.v_cache.to(dev),
                                      dc.cache_seqlens.to(dev), dc.block_table.to(dev),
                                      dc.softmax_scale, rnd.choice([0, 1, 3, 7]))
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0, name
    d_o, d_l = oracle.decode(dc.q, dc.k_cache, dc.v_cache, dc.cache_seqlens, dc.block_table,
                             dc.softmax_scale)
    compare(do.cpu(), dl.cpu(), d_o, d_l, "decode " + name)
    # chunked prefill over a paged cache: this batch's query lengths (at least one token
    # each) after a cached prefix, optionally rotated
    ql = [max(1, q) for q in k["lq"]]
    ctx = [rnd.choice([0, rnd.randint(1, 600)]) for _ in ql]
    rot = rnd.choice([0, 0, 32, k["d"]])
    kc = synth.kvcache_case(ql, ctx, k["Hq"], k["Hkv"], k["d"], page, seed=9000 + seed,
                            rotary_dim=rot, rotary_interleaved=rnd.random() < 0.5,
                            causal=k["causal"], window=k["window"], poison_unused=True)
    dev_ = lambda t: t.to(dev) if t is not None else None
    k_cache, v_cache = kc.k_cache.to(dev), kc.v_cache.to(dev)
    ko, kl = attn.attn_fwd_kvcache(dev_(kc.q), dev_(kc.k_new), dev_(kc.v_new), k_cache, v_cache,
                                   dev_(kc.cache_seqlens), dev_(kc.block_table),
                                   dev_(kc.cu_seqlens_q), kc.max_seqlen_q, kc.softmax_scale,
                                   kc.causal, kc.window_left, kc.window_right,
                                   dev_(kc.rotary_cos), dev_(kc.rotary_sin),
                                   kc.rotary_interleaved)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0, name
    ko_ref, kl_ref, kc_ref, vc_ref = oracle.kvcache_prefill(
        kc.q, kc.k_new, kc.v_new, kc.k_cache, kc.v_cache, kc.cache_seqlens, kc.block_table,
        kc.cu_seqlens_q, kc.softmax_scale, kc.causal, kc.window_left, kc.window_right,
        kc.rotary_cos, kc.rotary_sin, kc.rotary_interleaved)
    compare(ko.cpu(), kl.cpu().T, ko_ref, kl_ref.T, "kvcache " + name)
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16).astype(np.int32)
    assert np.array_equal(bits(v_cache), vc_ref.astype(np.int32)), name
    dk = np.abs(bits(k_cache) - kc_ref.astype(np.int32))
    assert dk.max() <= (1 if rot else 0), name


def close_grad(gpu, ref, what):
    """The backward tests' relative bound (max error 2 % of the largest, mean 0.5 % of the
    mean) with absolute floors for gradients that vanish exactly: with one visible key per row
    dS = P (dP - D) is zero in exact arithmetic, while the kernel forms dP and D as fp32 sums of
    d products dO_i v_i of N(0, 1) values (rarely above 25 in size), so their cancellation can
    leave about 2^-24 d 25 = 2e-4 in dS, and dK = scale dS q of a single-key row about a tenth
    of that times |q|.  Floors of 1e-4 (max) and 1e-5 (mean) cover that residue and stay far
    below any real gradient error (gradients here are of order 0.1-1)."""
    g = gpu.float().cpu().numpy().astype(np.float64)
    assert g.shape == np.shape(ref), what
    if g.size == 0:  # (a side without rows)
        return
    err = np.abs(g - ref)
    assert np.all(np.isfinite(g)), what
    assert err.max() <= 2e-2 * np.abs(ref).max() + 1e-4, (what, err.max())
    assert err.mean() <= 5e-3 * np.abs(ref).mean() + 1e-5, (what, err.mean())


@pytest.mark.parametrize("seed", range(48))
def test_random_modifiers_and_backward(attn, seed):
    rnd, k = draw(seed + 1000)
    dev = "cuda"
    name = f"sweep-mb{seed} {k}"
    c = synth.prefill_case(k["lq"], k["Hq"], k["Hkv"], k["d"], k["causal"], seed=10000 + seed,
                           lengths_k=k["lk"], window=k["window"], name=name)
    q, kk, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    cq, ck = c.cu_seqlens_q.to(dev), c.cu_seqlens_k.to(dev)
    # softcap and ALiBi
    cap = rnd.choice([0.0, 5.0, 30.0, 100.0])
    slopes = None
    if rnd.random() < 0.6:
        slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / k["Hq"]) for h in range(k["Hq"])],
                              dtype=torch.float32)
    mo, ml = attn.attn_fwd_mods(q, kk, v, cq, ck, c.max_seqlen_q, c.max_seqlen_k, c.softmax_scale,
                                c.causal, c.window_left, c.window_right, softcap=cap,
                                alibi_slopes=slopes.to(dev) if slopes is not None else None)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0, name
    r_o, r_l = oracle.attn_fwd_mods(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                    c.softmax_scale, c.causal, c.window_left, c.window_right,
                                    softcap=cap,
                                    alibi_slopes=slopes.double().numpy() if slopes is not None else None)
    compare(mo.cpu(), ml.cpu().T, r_o, r_l.T, "mods " + name)
    # backward of the plain attention
    out, lse = attn.attn_fwd(q, kk, v, cq, ck, c.max_seqlen_q, c.max_seqlen_k, c.softmax_scale,
                             c.causal, c.window_left, c.window_right)
    dout = synth.randn_bf16(tuple(c.q.shape), 10000 + seed, 9)
    dq, dk, dv = attn.attn_bwd(q, kk, v, out, dout.to(dev), lse, cq, ck, c.max_seqlen_q,
                               c.max_seqlen_k, c.softmax_scale, c.causal, c.window_left,
                               c.window_right)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0, name
    rdq, rdk, rdv, _ = oracle.attn_bwd(c.q, c.k, c.v, dout, c.cu_seqlens_q, c.cu_seqlens_k,
                                       c.softmax_scale, c.causal, c.window_left, c.window_right)
    close_grad(dq, rdq, "dq " + name)
    close_grad(dk, rdk, "dk " + name)
    close_grad(dv, rdv, "dv " + name)
