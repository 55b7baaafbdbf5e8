"""FP8 quantizer (attn_quantize_fp8) against the oracle's quantizer: codes and scales are
integer or single-rounding results of the same IEEE fp32 operations, so they must match bit
for bit.  End to end, quantize + FP8 forward must track the bf16 attention of the original
inputs within the FP8 error budget (the oracle pins' bounds)."""
import numpy as np
import pytest
import torch

from exact_attention_70_gb300 import binding, synth
from oracle import oracle

pytestmark = pytest.mark.gpu


def signs_for(seed):
    g = torch.Generator().manual_seed(seed)
    return torch.where(torch.rand(128, generator=g) < 0.5, -1.0, 1.0).float()


CASES = [
    dict(lq=[5, 130, 300], Hq=4, Hkv=2, rotate=False),
    dict(lq=[5, 130, 300], Hq=4, Hkv=2, rotate=True),
    dict(lq=[256, 0, 129], lk=[100, 0, 513], Hq=6, Hkv=2, rotate=True),
    dict(lq=[1000], Hq=2, Hkv=1, rotate=False),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_quantizer_is_bit_exact(i):
    k = CASES[i]
    c = synth.prefill_case(k["lq"], k["Hq"], k["Hkv"], 128, True, seed=400 + i,
                           lengths_k=k.get("lk"))
    sg = signs_for(i) if k["rotate"] else None
    dev = "cuda"
    out = binding.attn_quantize_fp8(c.q.to(dev), c.k.to(dev), c.v.to(dev),
                                    c.cu_seqlens_k.to(dev), c.max_seqlen_k,
                                    signs=None if sg is None else sg.to(dev))
    torch.cuda.synchronize()
    q8, qs, k8, ks, v8t, vs = (x.cpu() for x in out)
    kb = ks.shape[1]
    ref = oracle.fp8_quantize(c.q, c.k, c.v, c.cu_seqlens_k,
                              signs=None if sg is None else sg.numpy(), key_blocks=kb)
    names = ("q8", "q_scale", "k8", "k_scale", "v8t", "v_scale")
    for name, got, want in zip(names, (q8, qs, k8, ks, v8t, vs), ref):
        assert got.shape == want.shape, name
        assert torch.equal(got, want), (name, (got != want).sum().item())


def test_quantize_then_fp8_forward_tracks_bf16_attention():
    c = synth.prefill_case([300, 700], 8, 2, 128, True, seed=450)
    dev = "cuda"
    sg = signs_for(7).to(dev)
    q8, qs, k8, ks, v8t, vs = binding.attn_quantize_fp8(c.q.to(dev), c.k.to(dev), c.v.to(dev),
                                                        c.cu_seqlens_k.to(dev), c.max_seqlen_k,
                                                        signs=sg)
    o, lse = binding.attn_fwd_fp8(q8, k8, v8t, qs, ks, vs, c.cu_seqlens_q.to(dev),
                                  c.cu_seqlens_k.to(dev), c.max_seqlen_q, c.max_seqlen_k,
                                  c.softmax_scale, True)
    torch.cuda.synchronize()
    assert binding.attn_get_device_status() == 0
    ref, ref_l = oracle.attn_fwd(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                 c.softmax_scale, causal=True)
    err = np.abs(o.float().cpu().numpy() - ref)
    vmax = float(c.v.float().abs().max())
    assert err.max() <= 2 ** -4 * vmax + 2 ** -3 * vmax and err.mean() < 0.01
    assert np.abs(lse.cpu().numpy() - ref_l).mean() < 0.01
