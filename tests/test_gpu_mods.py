"""Score modifiers (attn_fwd_mods: softcap, ALiBi) versus the fp64 oracle, full rows, with
the parity tolerances of the plain forward pass."""
import numpy as np
import pytest
import torch

from exact_attention_70_gb300 import synth
from oracle import oracle
from tests.parity import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_70_gb300 import build as attn_build
    attn_build.build()
    from exact_attention_70_gb300 import binding
    binding.load()
    return binding


CASES = [
    # (lengths_q, lengths_k, Hq, Hkv, d, causal, window, softcap, alibi)
    ([300, 77], None, 4, 2, 128, True, (-1, -1), 30.0, False),
    ([300, 77], None, 4, 2, 128, True, (-1, -1), 0.0, True),
    ([500], None, 8, 2, 128, True, (-1, -1), 5.0, True),
    ([200, 129], None, 4, 4, 64, False, (-1, -1), 2.0, True),
    ([400], [600], 4, 1, 128, True, (100, 0), 20.0, True),   # bottom-right, window
    ([260], None, 6, 2, 128, False, (40, 40), 0.0, True),    # g = 3
    ([333], None, 4, 2, 128, True, (-1, -1), 64.0, False),   # largest cap of the polynomial form
    ([333], None, 4, 2, 128, True, (-1, -1), 100.0, True),   # exp2 + reciprocal form
    ([190, 70], None, 4, 4, 64, True, (-1, -1), 0.5, False),  # scores deep in saturation
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_modifiers_match_oracle(attn, idx):
    lq, lk, Hq, Hkv, d, causal, window, cap, alibi = CASES[idx]
    c = synth.prefill_case(lq, Hq, Hkv, d, causal, seed=800 + idx, lengths_k=lk, window=window,
                           name=f"mods{idx}")
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32) \
        if alibi else None
    dev = "cuda"
    out, lse = attn.attn_fwd_mods(c.q.to(dev), c.k.to(dev), c.v.to(dev), c.cu_seqlens_q.to(dev),
                                  c.cu_seqlens_k.to(dev), c.max_seqlen_q, c.max_seqlen_k,
                                  c.softmax_scale, c.causal, c.window_left, c.window_right,
                                  softcap=cap, alibi_slopes=slopes.to(dev) if alibi else None)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    o_ref, l_ref = oracle.attn_fwd_mods(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                        c.softmax_scale, c.causal, c.window_left, c.window_right,
                                        softcap=cap,
                                        alibi_slopes=slopes.double().numpy() if alibi else None)
    compare(out.cpu(), lse.cpu().T, o_ref, l_ref.T, c.name)


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_modifiers_repeatable_with_fresh_buffers(attn, idx):
    """The same call, repeated with every input re-uploaded to new device buffers and other
    allocations in between, gives bitwise the same O and LSE, each time within the parity
    tolerances: catches results that depend on timing or on what memory held before."""
    lq, lk, Hq, Hkv, d, causal, window, cap, alibi = CASES[idx]
    c = synth.prefill_case(lq, Hq, Hkv, d, causal, seed=800 + idx, lengths_k=lk, window=window,
                           name=f"mods{idx}")
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32)
    o_ref, l_ref = oracle.attn_fwd_mods(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                        c.softmax_scale, c.causal, c.window_left, c.window_right,
                                        softcap=cap, alibi_slopes=slopes.double().numpy())
    dev = "cuda"
    first = None
    for rep in range(12):
        filler = torch.randn(1 << (14 + rep % 4), device=dev)  # moves the allocator around
        args = [x.to(dev) for x in (c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k)]
        out, lse = attn.attn_fwd_mods(*args, c.max_seqlen_q, c.max_seqlen_k, c.softmax_scale,
                                      c.causal, c.window_left, c.window_right, softcap=cap,
                                      alibi_slopes=slopes.to(dev))
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0
        o, l = out.cpu(), lse.cpu()
        compare(o, l.T, o_ref, l_ref.T, f"{c.name} rep {rep}")
        if first is None:
            first = (o, l)
        else:
            assert torch.equal(o, first[0]) and torch.equal(l, first[1]), f"rep {rep} differs"
        del filler


@pytest.mark.parametrize("cap", [0.5, 2.0, 30.0, 64.0, 100.0, 1e4])
def test_softcap_map_on_the_device(attn, cap):
    """The kernel's softcap map, evaluated by the device code itself (attn_selftest_softcap),
    against c tanh(scale s / c) in fp64: tanh u = 1 - 2 / (e^(2u) + 1) from the hardware exp2
    and reciprocal stays within a few fp32 ulps of 1, times c, saturation included."""
    scale = 128 ** -0.5
    g = torch.Generator().manual_seed(int(cap * 10))
    s = torch.cat([torch.linspace(-3000.0, 3000.0, 1 << 16),
                   torch.randn(1 << 16, generator=g) * 4 * cap / scale,
                   torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e-4, -1e-4, 3e30, -3e30])])
    out = attn.attn_selftest_softcap(s.cuda(), scale, cap).cpu().double()
    ref = cap * torch.tanh(scale * s.double() / cap)
    err = (out - ref).abs().max().item()
    assert err <= cap * 2e-6, (cap, err)
    assert torch.all(out.abs() <= cap * (1 + 2 ** -21))
