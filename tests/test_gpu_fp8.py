"""FP8 (e4m3) forward against the oracle on the dequantized inputs.

Tolerance: the only approximation the kernel adds to the exact attention of the dequantized
inputs is the e4m3 rounding of 16 P~ before the second product (plus fp32 accumulation and the
bf16 rounding of O).  tests.fp8_exact.fp8_forward_bound turns the e4m3 grid into a per-element
bound from the exact scores of each row: 2^-4 (P|V|)_i for keys in e4m3's normal range, a
subnormal term for the rest, 2^-9 |O| for the output rounding.  Every element must lie within
it, and the mean error within the standard deviation that independent uniform roundings would
give (plus the output rounding).  LSE comes from the unrounded P~: 1e-3.
"""
import numpy as np
import pytest
import torch

from exact_attention_70_gb300 import binding, synth
from oracle import oracle
from tests.fp8_exact import fp8_forward_bound

pytestmark = pytest.mark.gpu


def run(c):
    dev = "cuda"
    out, lse = binding.attn_fwd_fp8(c.q8.to(dev), c.k8.to(dev), c.v8t.to(dev),
                                    c.q_scale.to(dev), c.k_scale.to(dev), c.v_scale.to(dev),
                                    c.cu_seqlens_q.to(dev), c.cu_seqlens_k.to(dev),
                                    c.max_seqlen_q, c.max_seqlen_k, c.softmax_scale, c.causal,
                                    c.window_left, c.window_right)
    torch.cuda.synchronize()
    assert binding.attn_get_device_status() == 0
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(c, out, lse, ref_o, ref_l, rows=None):
    q, k, v = oracle.fp8_dequantize(c.q8, c.k8, c.v8t, c.q_scale, c.k_scale, c.v_scale,
                                    c.cu_seqlens_k)
    bound, sigma = fp8_forward_bound(q, k, v, c.cu_seqlens_q.numpy(), c.cu_seqlens_k.numpy(),
                                     c.softmax_scale, c.causal, c.window_left, c.window_right,
                                     rows)
    if rows is not None:
        out = out[rows[0], rows[1]]
        lse = lse[rows[1], rows[0]]
    err = np.abs(out - ref_o)
    assert np.all(err <= bound + 1e-6), (err.max(), (err / (bound + 1e-6)).max())
    assert err.mean() <= sigma.mean() + 2.0 ** -9 * np.abs(ref_o).mean() + 1e-6, (
        err.mean(), sigma.mean())
    fin = np.isfinite(ref_l)
    assert np.array_equal(fin, np.isfinite(lse))
    if fin.any():  # (a batch with no keys has no finite LSE)
        assert np.abs(lse[fin] - ref_l[fin]).max() <= 1e-3
    return float((err / (bound + 1e-6)).max())


CASES = [
    dict(lq=[256], Hq=2, Hkv=2, causal=True),
    dict(lq=[5, 130, 300], Hq=8, Hkv=2, causal=True),
    dict(lq=[100, 257], lk=[300, 64], Hq=4, Hkv=4, causal=False),
    dict(lq=[400], Hq=4, Hkv=1, causal=True, window=(64, 0)),
    dict(lq=[190, 77], Hq=4, Hkv=2, causal=False, window=(32, 16)),
    dict(lq=[129, 0, 255], Hq=6, Hkv=2, causal=True),
    dict(lq=[64, 200], lk=[500, 700], Hq=4, Hkv=2, causal=True),
    dict(lq=[300, 129], Hq=4, Hkv=2, causal=True, full_range=True),   # subnormals, +-448
    dict(lq=[200], lk=[450], Hq=2, Hkv=1, causal=False, full_range=True),
    # 48 sequences of 0..289 tokens: more items than CTAs, so the persistent CTAs walk several
    # (empty ones among them)
    dict(lq=[(37 * i) % 290 for i in range(48)], Hq=4, Hkv=2, causal=True),
    # queries but no keys anywhere: items with no key block (O = 0, LSE = -inf)
    dict(lq=[50, 70], lk=[0, 0], Hq=4, Hkv=2, causal=False),
    # long items (48 or more key blocks on average), where the O rescales of a tile meet
    # P V products still in flight
    dict(lq=[300, 129], lk=[6200, 6300], Hq=2, Hkv=1, causal=False, full_range=True),
    dict(lq=[200, 64], lk=[12500, 12300], Hq=2, Hkv=1, causal=True),
    dict(lq=[400], lk=[9000], Hq=2, Hkv=1, causal=False, window=(7000, 100)),
    dict(lq=[(37 * i) % 290 for i in range(8)], lk=[6200 + 50 * i for i in range(8)], Hq=2,
         Hkv=1, causal=False),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_fp8_forward_matches_oracle(i):
    k = CASES[i]
    c = synth.fp8_case(k["lq"], k["Hq"], k["Hkv"], 128, k["causal"], seed=300 + i,
                       lengths_k=k.get("lk"), window=k.get("window", (-1, -1)),
                       full_range=k.get("full_range", False))
    out, lse = run(c)
    ref_o, ref_l = oracle.fp8_attn_fwd(c.q8, c.k8, c.v8t, c.q_scale, c.k_scale, c.v_scale,
                                       c.cu_seqlens_q, c.cu_seqlens_k, c.softmax_scale,
                                       c.causal, c.window_left, c.window_right)
    check(c, out, lse, ref_o, ref_l)


def test_fp8_forward_full_size_sampled_rows():
    c = synth.fp8_bench_case()
    out, lse = run(c)
    g = torch.Generator().manual_seed(9)
    n = 256
    tok = torch.randint(0, c.q8.shape[0], (n,), generator=g).numpy()
    head = torch.randint(0, c.q8.shape[1], (n,), generator=g).numpy()
    tok[:4] = [0, 127, 128, 4095]
    ref_o, ref_l = oracle.fp8_attn_fwd(c.q8, c.k8, c.v8t, c.q_scale, c.k_scale, c.v_scale,
                                       c.cu_seqlens_q, c.cu_seqlens_k, c.softmax_scale,
                                       c.causal, rows=(tok, head))
    check(c, out, lse, ref_o, ref_l, rows=(tok, head))


def test_fp8_short_key_tables_raise_the_bounds_flag():
    c = synth.fp8_case([300], 2, 1, 128, True, seed=5)
    dev = "cuda"
    ks = c.k_scale[:, :2].contiguous()        # 300 keys need three blocks
    vt = c.v8t[:, :, :256].contiguous()
    binding.attn_fwd_fp8(c.q8.to(dev), c.k8.to(dev), vt.to(dev), c.q_scale.to(dev), ks.to(dev),
                         c.v_scale.to(dev), c.cu_seqlens_q.to(dev), c.cu_seqlens_k.to(dev),
                         c.max_seqlen_q, c.max_seqlen_k, c.softmax_scale, True)
    torch.cuda.synchronize()
    assert binding.attn_get_device_status() == -6      # ATTN_ERR_DEVICE_BOUNDS
