"""FP8 quantizer (attn_quantize_fp8) against the oracle's quantizer: codes and scales are
integer or single-rounding results of the same IEEE fp32 operations, so they must match bit
for bit; both are also checked against the quantizer's exact fp64 definition (nearest e4m3
code of the exactly rotated, exactly scaled block, up to fp32-level midpoint ties).  End to
end, quantize + FP8 forward is held to the FP8 forward's realised rounding bound against the
exact attention of the quantized inputs, and to that bound plus the quantization's own exact
effect against the bf16 attention of the original inputs (triangle inequality).
"""
import numpy as np
import pytest
import torch

from exact_attention_70_gb300 import binding, synth
from oracle import oracle
from tests.fp8_exact import check_codes, fp8_forward_bound

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
    # the kernel's blocks against the exact definition: Q per 128 packed tokens and head, K per
    # 128 keys of a sequence and kv head (rotated when signs are given), V per (sequence, kv head)
    sgn = None if sg is None else sg.numpy()
    qf, kf, vf = (x.double().numpy() for x in (c.q, c.k, c.v))
    for h in range(qf.shape[1]):
        for blk in range(qs.shape[1]):
            t0, t1 = 128 * blk, min(qf.shape[0], 128 * blk + 128)
            if t1 > t0:
                check_codes(qf[t0:t1, h], q8[t0:t1, h].numpy(), qs[h, blk], sgn)
    cu = c.cu_seqlens_k.tolist()
    kb0 = oracle.key_block_offsets(c.cu_seqlens_k)
    for b in range(len(cu) - 1):
        for h in range(kf.shape[1]):
            for i in range((cu[b + 1] - cu[b] + 127) // 128):
                t0, t1 = cu[b] + 128 * i, min(cu[b + 1], cu[b] + 128 * i + 128)
                check_codes(kf[t0:t1, h], k8[t0:t1, h].numpy(), ks[h, kb0[b] + i], sgn)
            if cu[b + 1] > cu[b]:
                col = 128 * int(kb0[b])
                n = cu[b + 1] - cu[b]
                check_codes(vf[cu[b]:cu[b + 1], h], v8t[h, :, col:col + n].numpy().T, vs[b, h])


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
    o = o.float().cpu().numpy()
    q8, qs, k8, ks, v8t, vs = (x.cpu() for x in (q8, qs, k8, ks, v8t, vs))
    # stage 2: the FP8 forward against the exact attention of the quantized inputs
    oq, lq = oracle.fp8_attn_fwd(q8, k8, v8t, qs, ks, vs, c.cu_seqlens_q, c.cu_seqlens_k,
                                 c.softmax_scale, causal=True)
    qd, kd, vd = oracle.fp8_dequantize(q8, k8, v8t, qs, ks, vs, c.cu_seqlens_k)
    bound, _ = fp8_forward_bound(qd, kd, vd, c.cu_seqlens_q.numpy(), c.cu_seqlens_k.numpy(),
                                 c.softmax_scale, True, -1, -1)
    assert np.all(np.abs(o - oq) <= bound + 1e-6)
    # the whole chain against the bf16 attention of the original inputs
    ref, ref_l = oracle.attn_fwd(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                 c.softmax_scale, causal=True)
    assert np.all(np.abs(o - ref) <= np.abs(oq - ref) + bound + 1e-6)
    assert np.abs(lse.cpu().numpy() - lq).max() <= 1e-3
    # and the quantization itself stays small (rotation on): mean error well under 1 %
    assert np.abs(oq - ref).mean() < 0.01 and np.abs(lq - ref_l).mean() < 0.01
