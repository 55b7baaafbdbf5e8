"""Pins of the oracle's row-selection modes against its full-row modes.

The large-workload parity tests ask the oracle for a chosen set of (token, head) or
(sequence, head) rows only, because the full result would take hours on the host.  Those row
modes look rows up on their own (a binary search for the sequence that holds a packed token,
their own output indexing), so they are pinned here: every row of a small case, requested in a
shuffled order, must equal the matching row of the full result bit for bit.  The cases put
tokens on and next to every sequence boundary, include empty sequences, sequences without keys,
Lk != Lq, GQA groups of 3 and 8 and sliding windows, so that an off-by-one in the sequence
search, a row/head transpose or a wrong output slot fails here.

The full-row modes themselves are pinned in the other oracle test files (hand-worked values,
torch fp64 SDPA, closed forms, invariants).
"""
import numpy as np
import pytest

from oracle import oracle
from exact_attention_70_gb300 import synth

# (lengths_q, lengths_k, Hq, Hkv, d, causal, window)
PREFILL = [
    ([1, 0, 5, 130, 7, 0, 64], None, 6, 2, 16, True, (-1, -1)),            # g = 3
    ([3, 0, 40, 1, 129], [5, 2, 40, 0, 200], 8, 1, 16, True, (-1, -1)),   # g = 8, Lk != Lq
    ([17, 90, 2], [30, 60, 9], 8, 1, 32, False, (6, 3)),                  # window both sides
    ([0, 77, 1, 33], None, 6, 2, 16, True, (9, 0)),                       # causal window
    ([50, 50], [0, 70], 4, 4, 16, False, (-1, -1)),                       # a sequence without keys
]


def _all_rows_shuffled(total, H, seed):
    t, h = np.meshgrid(np.arange(total, dtype=np.int64), np.arange(H, dtype=np.int32),
                       indexing="ij")
    t, h = t.ravel(), h.ravel()
    perm = np.random.default_rng(seed).permutation(len(t))
    return t[perm], h[perm]


def _prefill_case(idx):
    lq, lk, Hq, Hkv, d, causal, window = PREFILL[idx]
    return synth.prefill_case(lq, Hq, Hkv, d, causal, seed=300 + idx, lengths_k=lk,
                              window=window, name=f"rows{idx}")


@pytest.mark.parametrize("idx", range(len(PREFILL)))
def test_attn_fwd_rows_equals_full_rows(idx):
    c = _prefill_case(idx)
    out, lse = oracle.attn_fwd(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, c.softmax_scale,
                               c.causal, c.window_left, c.window_right)
    total, Hq = c.q.shape[0], c.q.shape[1]
    rt, rh = _all_rows_shuffled(total, Hq, idx)
    o_r, l_r = oracle.attn_fwd_rows(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                    c.softmax_scale, rt, rh, c.causal, c.window_left,
                                    c.window_right)
    assert np.array_equal(o_r, out[rt, rh])
    assert np.array_equal(l_r, lse[rh, rt])
    # the case really has rows of both kinds (some empty rows in the cases that have them)
    assert np.isfinite(l_r).any()


def test_attn_fwd_rows_rejects_tokens_outside_the_batch():
    c = _prefill_case(0)
    total = c.q.shape[0]
    for t, h in ((total, 0), (-1, 0), (0, c.q.shape[1])):
        with pytest.raises(ValueError):
            oracle.attn_fwd_rows(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                 c.softmax_scale, [t], [h], True)


@pytest.mark.parametrize("idx", range(len(PREFILL)))
def test_attn_fwd_mods_rows_equal_full_rows(idx):
    c = _prefill_case(idx)
    Hq = c.q.shape[1]
    slopes = [2.0 ** (-(h + 1)) for h in range(Hq)]
    args = (c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k, c.softmax_scale, c.causal,
            c.window_left, c.window_right)
    out, lse = oracle.attn_fwd_mods(*args, softcap=2.5, alibi_slopes=slopes)
    rt, rh = _all_rows_shuffled(c.q.shape[0], Hq, 10 + idx)
    o_r, l_r = oracle.attn_fwd_mods(*args, softcap=2.5, alibi_slopes=slopes, rows_t=rt,
                                    rows_h=rh)
    assert np.array_equal(o_r, out[rt, rh])
    assert np.array_equal(l_r, lse[rh, rt])


# (lengths, Hq, Hkv, d, page_size)
DECODE = [
    ([1, 17, 64, 300, 0], 8, 2, 16, 16),
    ([255, 256, 257, 1000], 12, 4, 32, 64),   # g = 3
    ([5, 700], 8, 1, 16, 256),                # g = 8
]


@pytest.mark.parametrize("idx", range(len(DECODE)))
@pytest.mark.parametrize("splits", [0, 3])
def test_decode_rows_equal_full_rows(idx, splits):
    lengths, Hq, Hkv, d, ps = DECODE[idx]
    c = synth.decode_case(lengths, Hq, Hkv, d, ps, seed=320 + idx)
    args = (c.q, c.k_cache, c.v_cache, c.cache_seqlens, c.block_table, c.softmax_scale, splits)
    out, lse = oracle.decode(*args)
    batch = len(lengths)
    rb, rh = _all_rows_shuffled(batch, Hq, 20 + idx)
    o_r, l_r = oracle.decode(*args, rows_b=rb.astype(np.int32), rows_h=rh)
    assert np.array_equal(o_r, out[rb, rh])
    assert np.array_equal(l_r, lse[rb, rh])


@pytest.mark.parametrize("rotary", [0, 16])
def test_kvcache_prefill_rows_equal_full_rows(rotary):
    c = synth.kvcache_case([3, 1, 20, 0, 9], [8, 0, 30, 5, 16], 6, 2, 32, 16, seed=330,
                           rotary_dim=rotary, window=(12, 0))
    args = (c.q, c.k_new, c.v_new, c.k_cache, c.v_cache, c.cache_seqlens, c.block_table,
            c.cu_seqlens_q, c.softmax_scale, c.causal, c.window_left, c.window_right,
            c.rotary_cos, c.rotary_sin, c.rotary_interleaved)
    out, lse, kc, vc = oracle.kvcache_prefill(*args)
    rt, rh = _all_rows_shuffled(c.q.shape[0], c.q.shape[1], 30 + rotary)
    o_r, l_r, kc_r, vc_r = oracle.kvcache_prefill(*args, rows_t=rt, rows_h=rh)
    assert np.array_equal(o_r, out[rt, rh])
    assert np.array_equal(l_r, lse[rh, rt])
    # the append does not depend on which rows are asked for
    assert np.array_equal(kc_r, kc) and np.array_equal(vc_r, vc)


def test_sampled_rows_cover_every_sequence_boundary():
    """The GPU tests' row sampler always includes each sequence's first and last rows and the
    tile-boundary rows, whatever the random draw."""
    from tests.parity import sample_rows
    c = synth.prefill_case([1, 130, 300, 2], 4, 2, 16, True, seed=340)
    rt, rh = sample_rows(c, 3, seed=1)
    cu = c.cu_seqlens_q.tolist()
    for h in range(4):
        got = set(rt[rh == h].tolist())
        for b in range(len(cu) - 1):
            L = cu[b + 1] - cu[b]
            for i in (0, 1, 127, 128, 129, 255, 256, L - 1):
                if 0 <= i < L:
                    assert cu[b] + i in got
