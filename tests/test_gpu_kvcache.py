"""Chunked prefill against a paged cache (attn_fwd_kvcache) versus the fp64 oracle.

The CUDA path appends the new keys (rotated) and values into the cache, rotates the queries
and runs the paged prefill kernel.  Compared with the oracle on the same seeded inputs:
O and LSE with the parity tolerances, the appended cache rows bit-exact (values, and keys
without rotation) or within one bf16 ulp (rotated keys: the kernel rotates in fp32, the
oracle in fp64, and the two can round to neighbouring bf16 values at a tie), every other
cache slot untouched.
"""
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


def run_gpu(attn, c):
    dev = lambda t: t.cuda() if t is not None else None
    kc, vc = c.k_cache.cuda(), c.v_cache.cuda()
    out, lse = attn.attn_fwd_kvcache(
        dev(c.q), dev(c.k_new), dev(c.v_new), kc, vc, dev(c.cache_seqlens), dev(c.block_table),
        dev(c.cu_seqlens_q), c.max_seqlen_q, c.softmax_scale, c.causal, c.window_left,
        c.window_right, dev(c.rotary_cos), dev(c.rotary_sin), c.rotary_interleaved)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu(), kc.cpu(), vc.cpu()


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16).astype(np.int32)


def check_cache(c, kc_gpu, vc_gpu, kc_ref, vc_ref):
    # values are copied: bit-exact; untouched slots (incl. NaN poison) keep their bits
    assert np.array_equal(bits(vc_gpu), vc_ref.astype(np.int32))
    dk = np.abs(bits(kc_gpu) - kc_ref.astype(np.int32))
    if c.rotary_cos is None:
        assert dk.max() == 0
    else:
        # neighbouring bf16 bit patterns of the same sign differ by 1
        assert dk.max() <= 1 and (dk != 0).mean() < 1e-3, (dk.max(), (dk != 0).mean())


def oracle_all(c):
    return oracle.kvcache_prefill(c.q, c.k_new, c.v_new, c.k_cache, c.v_cache, c.cache_seqlens,
                                  c.block_table, c.cu_seqlens_q, c.softmax_scale, c.causal,
                                  c.window_left, c.window_right, c.rotary_cos, c.rotary_sin,
                                  c.rotary_interleaved)


CASES = [
    # (q_lens, ctx_lens, Hq, Hkv, d, page_size, rotary_dim, interleaved, causal, window, poison)
    ([4, 1, 1], [8, 11, 5], 4, 2, 128, 16, 0, False, True, (-1, -1), True),  # the pages' figure
    ([300, 77, 1], [0, 500, 1000], 8, 2, 128, 64, 128, False, True, (-1, -1), True),
    ([129, 256], [1000, 33], 32, 8, 128, 256, 64, False, True, (-1, -1), False),
    ([200], [3000], 4, 4, 64, 128, 64, True, True, (300, 0), True),
    ([1, 2, 3, 130], [127, 128, 129, 0], 16, 1, 128, 32, 32, False, True, (-1, -1), True),
    ([500], [0], 4, 2, 128, 16, 0, False, False, (-1, -1), False),       # non-causal
    ([64, 200], [640, 7], 8, 8, 64, 16, 16, True, True, (100, 0), True),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_kvcache_prefill_matches_oracle(attn, idx):
    ql, cl, Hq, Hkv, d, ps, rot, inter, causal, window, poison = CASES[idx]
    c = synth.kvcache_case(ql, cl, Hq, Hkv, d, ps, seed=400 + idx, rotary_dim=rot,
                           rotary_interleaved=inter, causal=causal, window=window,
                           poison_unused=poison, name=f"kv{idx}")
    out, lse, kc, vc = run_gpu(attn, c)
    assert attn.attn_get_device_status() == 0
    o_ref, l_ref, kc_ref, vc_ref = oracle_all(c)
    compare(out, lse.T, o_ref, l_ref.T, c.name)
    check_cache(c, kc, vc, kc_ref, vc_ref)


def test_kvcache_prefill_large_sampled(attn):
    # 4 sequences, 2-8K cached tokens, 512-2048 new ones, page 256, rotary over all of d
    g = torch.Generator().manual_seed(450)
    ctx = torch.randint(2048, 8193, (4,), generator=g).tolist()
    ql = torch.randint(512, 2049, (4,), generator=g).tolist()
    c = synth.kvcache_case(ql, ctx, 32, 8, 128, 256, seed=451, rotary_dim=128, name="kv_large")
    out, lse, kc, vc = run_gpu(attn, c)
    assert attn.attn_get_device_status() == 0
    total_q, Hq = c.q.shape[:2]
    rg = torch.Generator().manual_seed(452)
    rt = torch.randint(0, total_q, (2048,), generator=rg)
    cu = c.cu_seqlens_q.tolist()
    edges = torch.tensor([x for b in range(4) for x in (cu[b], cu[b + 1] - 1)])
    rt = torch.cat([rt, edges]).numpy()
    rh = torch.randint(0, Hq, (len(rt),), generator=rg).numpy()
    o_ref, l_ref, kc_ref, vc_ref = oracle.kvcache_prefill(
        c.q, c.k_new, c.v_new, c.k_cache, c.v_cache, c.cache_seqlens, c.block_table,
        c.cu_seqlens_q, c.softmax_scale, c.causal, -1, -1, c.rotary_cos, c.rotary_sin, False,
        rows_t=rt, rows_h=rh)
    compare(out[rt, rh], lse[rh, rt], o_ref, l_ref, c.name)
    check_cache(c, kc, vc, kc_ref, vc_ref)


def test_kvcache_bad_page_id_is_reported(attn):
    c = synth.kvcache_case([50], [100], 4, 4, 128, 64, seed=460)
    c.block_table[0, 2] = c.k_cache.shape[0] + 7  # the page of positions 128-149
    run_gpu(attn, c)
    assert attn.attn_get_device_status() == -6
    assert attn.attn_get_device_status() == 0
