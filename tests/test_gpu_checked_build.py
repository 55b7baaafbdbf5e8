"""The bounds-checking debug build (kernels compiled with -DATTN_CHECK_BOUNDS): on valid inputs
its extra checks of store indices and TMA coordinates must stay silent (status ATTN_OK) and its
results must match the oracle, like the regular build's."""
import numpy as np
import pytest
import torch

from exact_attention_70_gb300 import build as attn_build
from exact_attention_70_gb300 import binding, synth
from oracle import oracle
from tests.parity import compare, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    regular_lib, regular_path = binding._lib, attn_build.LIB
    path = attn_build.build(check_bounds=True)
    binding._lib = None
    attn_build.LIB = path
    try:
        binding.load()
        yield binding
    finally:
        binding._lib = regular_lib
        attn_build.LIB = regular_path


def test_checked_prefill_ragged_gqa_window(checked):
    for i, (lq, lk, Hq, Hkv, d, causal, window) in enumerate([
            ([1, 130, 257, 600], None, 6, 2, 128, True, (-1, -1)),     # g = 3, ragged tiles
            ([300, 40], [100, 0], 4, 4, 64, True, (-1, -1)),           # a sequence without keys
            ([700, 300], None, 8, 8, 128, False, (100, 50))]):         # window on both sides
        c = synth.prefill_case(lq, Hq, Hkv, d, causal, seed=700 + i, lengths_k=lk, window=window)
        dev = to_dev(c)
        out, lse = checked.attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"],
                                    dev["cu_seqlens_k"], c.max_seqlen_q, c.max_seqlen_k,
                                    c.softmax_scale, causal, window[0], window[1])
        torch.cuda.synchronize()
        assert checked.attn_get_device_status() == 0
        o_ref, l_ref = oracle.attn_fwd(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                       c.softmax_scale, causal, window[0], window[1])
        compare(out.cpu(), lse.cpu().T, o_ref, l_ref.T, f"checked{i}")


def test_checked_decode_and_chunked_prefill(checked):
    c = synth.decode_case([20, 300, 4097], 8, 2, 128, 16, seed=710, max_pages=300)
    for b, L in enumerate([20, 300, 4097]):
        c.block_table[b, (L + 15) // 16:] = -1
    dev = to_dev(c)
    out, lse = checked.attn_decode_kvcache(dev["q"], dev["k_cache"], dev["v_cache"],
                                           dev["cache_seqlens"], dev["block_table"],
                                           c.softmax_scale, 0)
    torch.cuda.synchronize()
    assert checked.attn_get_device_status() == 0
    o_ref, l_ref = oracle.decode(c.q, c.k_cache, c.v_cache, c.cache_seqlens, c.block_table,
                                 c.softmax_scale)
    compare(out.cpu(), lse.cpu(), o_ref, l_ref, "checked decode")
    k = synth.kvcache_case([3, 200], [100, 700], 8, 2, 128, 64, seed=711, rotary_dim=64)
    d = to_dev(k)
    out, lse = checked.attn_fwd_kvcache(d["q"], d["k_new"], d["v_new"], d["k_cache"],
                                        d["v_cache"], d["cache_seqlens"], d["block_table"],
                                        d["cu_seqlens_q"], k.max_seqlen_q, k.softmax_scale, True,
                                        -1, -1, d["rotary_cos"], d["rotary_sin"], False)
    torch.cuda.synchronize()
    assert checked.attn_get_device_status() == 0
    o_ref, l_ref, _, _ = oracle.kvcache_prefill(k.q, k.k_new, k.v_new, k.k_cache, k.v_cache,
                                                k.cache_seqlens, k.block_table, k.cu_seqlens_q,
                                                k.softmax_scale, True, -1, -1, k.rotary_cos,
                                                k.rotary_sin, False)
    compare(out.cpu(), lse.cpu().T, o_ref, l_ref.T, "checked chunked")
