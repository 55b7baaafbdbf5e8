"""The allocation-free decode entry point against the regular one and the oracle.

attn_decode_kvcache_noalloc serves callers that cannot allocate device memory (no allocator
hook behind their interface, all HBM already reserved, or no tolerance for cudaMalloc's
possible synchronisation): it keeps the split partials in the library's own 32 MiB device
array instead of a caller workspace.  It runs the same kernels with the same resolved split
count as attn_decode_kvcache, so its outputs must be bitwise equal to the regular call's.
This file is collected last so that a failure here leaves every other test already run.
"""
import pytest
import torch

from exact_attention_70_gb300 import synth
from oracle import oracle
from tests.parity import compare, to_dev

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


def _both(attn, case, splits):
    d = to_dev(case)
    args = (d["q"], d["k_cache"], d["v_cache"], d["cache_seqlens"], d["block_table"],
            case.softmax_scale, splits)
    o_ref, l_ref = attn.attn_decode_kvcache(*args)
    o_new, l_new = attn.attn_decode_kvcache_noalloc(*args)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    return o_new.cpu(), l_new.cpu(), o_ref.cpu(), l_ref.cpu()


def test_noalloc_matches_regular_entry_point_on_two_calls_in_a_row(attn):
    # The second problem needs more partial rows (batch x heads x splits) than the first, so
    # the first call's partials sit inside the region the second call must rewrite; a slot
    # the second call failed to write would hand it the first call's stale values.
    first = synth.decode_case([77, 2048, 65], 8, 2, 128, 64, seed=901, name="noalloc-a")
    second = synth.decode_case([1, 300, 4097, 20000], 32, 8, 128, 256, seed=900,
                               name="noalloc-b")
    rows = []
    for case, splits in ((first, 7), (second, 0)):
        o_new, l_new, o_ref, l_ref = _both(attn, case, splits)
        assert torch.equal(o_new, o_ref) and torch.equal(l_new, l_ref), case.name
        o_or, l_or = oracle.decode(case.q, case.k_cache, case.v_cache, case.cache_seqlens,
                                   case.block_table, case.softmax_scale)
        compare(o_new, l_new, o_or, l_or, case.name)
        B, Hq = case.q.shape[:2]
        S = splits or attn.attn_decode_num_splits(
            B, Hq, case.k_cache.shape[2], case.block_table.shape[1], case.page_size,
            torch.cuda.get_device_properties(0).multi_processor_count)
        assert S > 1
        rows.append(B * Hq * S)
    assert rows[1] > rows[0]


def test_noalloc_rejects_requests_beyond_its_scratch(attn):
    # 1024 x 64 heads x 16 splits of fp32 partials need far more than 32 MiB
    case = synth.decode_case([64] * 4, 64, 8, 128, 64, seed=902)
    d = to_dev(case)
    q = d["q"].repeat(256, 1, 1)
    sl = d["cache_seqlens"].repeat(256)
    bt = d["block_table"].repeat(256, 1)
    with pytest.raises(attn.AttnError) as e:
        attn.attn_decode_kvcache_noalloc(q, d["k_cache"], d["v_cache"], sl, bt,
                                         case.softmax_scale, 16)
    assert e.value.code == -3


def test_noalloc_checks_table_shapes_before_calling(attn):
    case = synth.decode_case([64, 100], 8, 2, 128, 64, seed=903)
    d = to_dev(case)
    with pytest.raises(ValueError):
        attn.attn_decode_kvcache_noalloc(d["q"], d["k_cache"], d["v_cache"],
                                         d["cache_seqlens"][:1], d["block_table"],
                                         case.softmax_scale)
    with pytest.raises(ValueError):
        attn.attn_decode_kvcache_noalloc(d["q"], d["k_cache"], d["v_cache"],
                                         d["cache_seqlens"], d["block_table"][:1].contiguous(),
                                         case.softmax_scale)
