"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

from exact_attention_70_gb300 import synth
from oracle import oracle
from tests.parity import compare, sample_rows, to_dev

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


def run_fwd(attn, case):
    d = to_dev(case)
    out, lse = attn.attn_fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                             case.max_seqlen_q, case.max_seqlen_k, case.softmax_scale,
                             case.causal, case.window_left, case.window_right)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    return out.cpu(), lse.cpu()


def check_fwd_full(attn, case):
    out, lse = run_fwd(attn, case)
    o_ref, l_ref = oracle.attn_fwd(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                                   case.softmax_scale, case.causal, case.window_left,
                                   case.window_right)
    # out is [total_q, Hq, d] while lse is [Hq, total_q]: compare row-aligned
    return compare(out, lse.T, o_ref, l_ref.T, case.name)


def check_fwd_sampled(attn, case, per_head=512, seed=7):
    out, lse = run_fwd(attn, case)
    rt, rh = sample_rows(case, per_head, seed)
    o_ref, l_ref = oracle.attn_fwd_rows(case.q, case.k, case.v, case.cu_seqlens_q,
                                        case.cu_seqlens_k, case.softmax_scale, rt, rh,
                                        case.causal, case.window_left, case.window_right)
    return compare(out[rt, rh], lse[rh, rt], o_ref, l_ref, case.name)


# ---- prefill -------------------------------------------------------------------------------

def test_config1_single_head_noncausal(attn):
    check_fwd_full(attn, synth.config_case(1))


PREFILL_SMALL = [
    # (lengths_q, lengths_k, Hq, Hkv, d, causal, window)
    ([300], None, 2, 2, 128, True, (-1, -1)),
    ([1, 2, 127, 128, 129, 255, 256, 257, 600], None, 4, 4, 128, True, (-1, -1)),
    ([513, 77, 1000], None, 8, 2, 128, True, (-1, -1)),
    ([700, 129], None, 8, 1, 128, True, (-1, -1)),
    ([333, 64], None, 16, 2, 128, True, (-1, -1)),
    ([250, 31], None, 6, 2, 128, True, (-1, -1)),     # group of 3: 42 tokens per tile
    ([400], None, 32, 1, 64, False, (-1, -1)),        # group of 32: 4 tokens per tile
    ([384, 200], None, 4, 4, 64, False, (-1, -1)),
    ([900], None, 4, 2, 128, True, (37, 0)),
    ([700, 300], None, 4, 4, 128, False, (100, 50)),
    ([600], None, 2, 2, 64, False, (0, 0)),
    ([5, 200, 130], [300, 250, 130], 4, 2, 128, True, (-1, -1)),   # bottom-right, Lk > Lq
    ([300, 40], [100, 0], 4, 4, 128, True, (-1, -1)),              # Lk < Lq; a sequence with no keys
    ([260], [700], 4, 4, 128, False, (-1, -1)),
    ([1000], None, 8, 8, 128, True, (300, 0)),
    # 48 sequences of 0..289 tokens: ~600 work items over the persistent CTAs, several claimed
    # by each, empty sequences among them
    ([(37 * i) % 290 for i in range(48)], None, 8, 2, 128, True, (-1, -1)),
    # queries but no keys anywhere: every work item is claimed and has no key block
    ([50, 70], [0, 0], 4, 2, 128, True, (-1, -1)),
]


@pytest.mark.parametrize("idx", range(len(PREFILL_SMALL)))
def test_prefill_small_full_oracle(attn, idx):
    lq, lk, Hq, Hkv, d, causal, window = PREFILL_SMALL[idx]
    case = synth.prefill_case(lq, Hq, Hkv, d, causal, seed=100 + idx, lengths_k=lk,
                              window=window, name=f"small{idx}")
    check_fwd_full(attn, case)


def test_config2_causal_prefill(attn):
    check_fwd_sampled(attn, synth.config_case(2))


def test_config3_varlen_gqa(attn):
    check_fwd_sampled(attn, synth.config_case(3))


def test_config5_sliding_window(attn):
    check_fwd_sampled(attn, synth.config_case(5))


def test_prefill_is_deterministic(attn):
    case = synth.prefill_case([777, 1500], 8, 2, 128, True, seed=5)
    o1, l1 = run_fwd(attn, case)
    o2, l2 = run_fwd(attn, case)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


SINGLE_KEY_CASES = [
    # (lengths, Hq, Hkv, d): causal, so the first token of each sequence sees exactly one key
    ([300, 77], 4, 2, 128),
    ([500], 8, 2, 128),
    ([200, 129], 4, 4, 64),
    ([1000, 17, 513], 32, 4, 128),
    ([130, 260], 6, 2, 128),
]


@pytest.mark.parametrize("idx", range(len(SINGLE_KEY_CASES)))
@pytest.mark.parametrize("mods", [False, True])
def test_single_visible_key_rows_are_exact(attn, idx, mods):
    """A row that sees one key has P = (1) whatever the running maximum, so O is that key's V
    row bit for bit and LSE is its logit: pins the row maximum and the normalisation (a wrong
    reference maximum shows up here as bf16 rounding of P away from 1)."""
    lengths, Hq, Hkv, d = SINGLE_KEY_CASES[idx]
    c = synth.prefill_case(lengths, Hq, Hkv, d, True, seed=1500 + idx, name=f"single{idx}")
    dev = to_dev(c)
    cap = 20.0 if mods else 0.0
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)], dtype=torch.float32)
    if mods:
        out, lse = attn.attn_fwd_mods(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"],
                                      dev["cu_seqlens_k"], c.max_seqlen_q, c.max_seqlen_k,
                                      c.softmax_scale, True, -1, -1, softcap=cap,
                                      alibi_slopes=slopes.cuda())
    else:
        out, lse = attn.attn_fwd(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"],
                                 dev["cu_seqlens_k"], c.max_seqlen_q, c.max_seqlen_k,
                                 c.softmax_scale, True)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    out, lse = out.float().cpu(), lse.cpu().double()
    g = Hq // Hkv
    cu = c.cu_seqlens_q.tolist()
    for b in range(len(cu) - 1):
        t = cu[b]
        for h in range(Hq):
            v_row = c.v[t, h // g].float()
            assert torch.equal(out[t, h], v_row), f"seq {b} head {h}: O is not V of its one key"
            x = float((c.q[t, h].double() * c.k[t, h // g].double()).sum()) * c.softmax_scale
            if mods:
                x = cap * math.tanh(x / cap)  # the ALiBi bias of the key at distance 0 is 0
            assert abs(float(lse[h, t]) - x) < 1e-5, f"seq {b} head {h}: LSE {float(lse[h, t])} vs {x}"


def test_bounded_wait_reports_timeout_and_context_survives(attn):
    # a wait on a barrier that nothing completes runs out (20 ms limit) and is reported
    assert attn.attn_selftest_wait_timeout() == 0
    assert attn.attn_get_device_status() == -5
    assert attn.attn_get_device_status() == 0  # cleared
    # the context is still usable: a small prefill still matches the oracle
    case = synth.prefill_case([300, 77], 4, 2, 128, True, seed=9)
    check_fwd_full(attn, case)


def test_prefill_bad_cu_seqlens_is_reported(attn):
    case = synth.prefill_case([100, 100], 2, 2, 64, True, seed=6)
    d = to_dev(case)
    bad = torch.tensor([0, 150, 120], dtype=torch.int32, device="cuda")  # decreasing
    attn.attn_fwd(d["q"], d["k"], d["v"], bad, bad, 150, 150, None, True)
    assert attn.attn_get_device_status() == -6
    assert attn.attn_get_device_status() == 0  # cleared


# ---- decode --------------------------------------------------------------------------------

def run_decode(attn, case, num_splits=None):
    d = to_dev(case)
    ns = case.num_splits if num_splits is None else num_splits
    out, lse = attn.attn_decode_kvcache(d["q"], d["k_cache"], d["v_cache"], d["cache_seqlens"],
                                        d["block_table"], case.softmax_scale, ns)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def check_decode(attn, case, num_splits=None):
    out, lse = run_decode(attn, case, num_splits)
    assert attn.attn_get_device_status() == 0
    o_ref, l_ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.cache_seqlens,
                                 case.block_table, case.softmax_scale)
    return compare(out, lse, o_ref, l_ref, case.name)


DECODE_SMALL = [
    # (lengths, Hq, Hkv, d, page_size)
    ([1, 63, 64, 65, 1000, 4097], 8, 2, 128, 256),
    ([17, 300, 2048], 4, 4, 128, 16),
    ([100, 129, 555], 8, 8, 128, 32),
    ([64, 1, 999], 32, 8, 128, 64),
    ([3000, 10], 16, 1, 128, 128),
    ([700, 5], 32, 1, 64, 64),     # 32 heads per kv head: two row groups
    ([250, 1500], 4, 2, 64, 256),
]


@pytest.mark.parametrize("idx", range(len(DECODE_SMALL)))
@pytest.mark.parametrize("splits", [0, 1, 2, 3, 7, 16])
def test_decode_small(attn, idx, splits):
    lens, Hq, Hkv, d, ps = DECODE_SMALL[idx]
    case = synth.decode_case(lens, Hq, Hkv, d, ps, seed=200 + idx, name=f"dec{idx}")
    check_decode(attn, case, splits)


def test_decode_ignores_garbage_past_the_end(attn):
    lens = [1, 70, 300]
    case = synth.decode_case(lens, 8, 2, 128, 256, seed=300)
    # poison every cache slot past each sequence's end (same pages, later slots)
    for b, L in enumerate(lens):
        last = case.block_table[b, (L - 1) // 256]
        case.k_cache[last, L % 256 or 256:] = float("nan")
        case.v_cache[last, L % 256 or 256:] = float("nan")
    for splits in (1, 4):
        check_decode(attn, case, splits)


def test_decode_empty_sequence(attn):
    case = synth.decode_case([0, 50], 4, 4, 128, 64, seed=301, max_pages=2)
    out, lse = run_decode(attn, case, 2)
    assert attn.attn_get_device_status() == 0
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    o_ref, l_ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.cache_seqlens,
                                 case.block_table, case.softmax_scale)
    compare(out, lse, o_ref, l_ref, "empty")


def test_decode_bad_page_id_is_reported(attn):
    case = synth.decode_case([100], 4, 4, 128, 64, seed=302)
    case.block_table[0, 1] = case.k_cache.shape[0] + 5
    run_decode(attn, case, 1)
    assert attn.attn_get_device_status() == -6


def test_config4_paged_decode(attn):
    case = synth.config_case(4)
    out, lse = run_decode(attn, case)
    assert attn.attn_get_device_status() == 0
    g = torch.Generator().manual_seed(44)
    B, Hq = case.q.shape[:2]
    rb = torch.randint(0, B, (768,), generator=g).numpy()
    rh = torch.randint(0, Hq, (768,), generator=g).numpy()
    rb = np.concatenate([rb, np.arange(B)])
    rh = np.concatenate([rh, np.arange(B) % Hq])
    o_ref, l_ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.cache_seqlens,
                                 case.block_table, case.softmax_scale, 0, rb, rh)
    compare(out[rb, rh], lse[rb, rh], o_ref, l_ref, "cfg4")


PADDED_TABLES = [
    # (lengths, Hq, Hkv, d, page_size, max_pages): every table entry past a sequence's
    # ceil(L / page_size) pages is -1, and the table sits at the end of a buffer whose next
    # entries are -1 too, so any read past a sequence's own pages raises BOUNDS
    ([20, 40, 33, 47], 8, 2, 128, 16, 3),   # 3 pages x 16 = 48 keys: not a multiple of 64
    ([1, 17, 100, 250], 8, 2, 128, 32, 9),  # 9 x 32 = 288 keys
    ([5, 64, 129, 30], 32, 8, 64, 16, 13),  # 13 x 16 = 208 keys, d = 64
    ([200, 3], 4, 4, 128, 64, 5),
]


def _padded_table_case(idx):
    lens, Hq, Hkv, d, ps, mp = PADDED_TABLES[idx]
    case = synth.decode_case(lens, Hq, Hkv, d, ps, seed=310 + idx, max_pages=mp,
                             name=f"padded{idx}")
    for b, L in enumerate(lens):
        case.block_table[b, (L + ps - 1) // ps:] = -1
    return case


def _table_at_buffer_end(bt):
    buf = torch.full((bt.numel() + 64,), -1, dtype=torch.int32, device="cuda")
    view = buf[:bt.numel()].view(bt.shape)
    view.copy_(bt)
    return view


@pytest.mark.parametrize("idx", range(len(PADDED_TABLES)))
@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("entry", ["regular", "noalloc"])
def test_decode_reads_only_the_sequences_own_pages(attn, idx, splits, entry):
    case = _padded_table_case(idx)
    d = to_dev(case)
    bt = _table_at_buffer_end(d["block_table"])
    fn = attn.attn_decode_kvcache if entry == "regular" else attn.attn_decode_kvcache_noalloc
    out, lse = fn(d["q"], d["k_cache"], d["v_cache"], d["cache_seqlens"], bt,
                  case.softmax_scale, splits)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    o_ref, l_ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.cache_seqlens,
                                 case.block_table, case.softmax_scale)
    compare(out.cpu(), lse.cpu(), o_ref, l_ref, case.name)
