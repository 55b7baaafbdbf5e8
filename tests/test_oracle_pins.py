"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value printed on a page
(``tests/golden``), a closed form, an invariant, or a library routine (torch fp64 SDPA).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import oracle
from exact_attention_70_gb300 import synth


def f64(*shape, seed=0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


# ---- hand-worked and closed-form cases ---------------------------------------------

def test_hand_worked_two_keys(golden):
    ex = golden["hand_worked_two_keys"]
    q = torch.tensor(ex["q"], dtype=torch.float64).view(1, 1, 1)
    k = torch.tensor(ex["k"], dtype=torch.float64).view(2, 1, 1)
    v = torch.tensor(ex["v"], dtype=torch.float64).view(2, 1, 1)
    out, lse = oracle.attn_fwd(q, k, v, [0, 1], [0, 2], ex["scale"])
    assert abs(out[0, 0, 0] - ex["O"]) < 1e-15
    assert abs(lse[0, 0] - ex["LSE"]) < 1e-15
    # the same numbers through split partials: one key per split, merged
    o, l = oracle.merge([0.0, math.log(3.0)], [1.0, 1.0], [[0.0], [1.0]])
    assert abs(o[0] - ex["O"]) < 1e-15 and abs(l - ex["LSE"]) < 1e-15


def test_causal_2x2_first_row_sees_only_itself():
    q, k, v = f64(2, 1, 4, seed=1), f64(2, 1, 4, seed=2), f64(2, 1, 4, seed=3)
    out, lse = oracle.attn_fwd(q, k, v, [0, 2], [0, 2], 0.5, causal=True)
    assert np.allclose(out[0, 0], v[0, 0].numpy(), atol=0, rtol=0)
    assert abs(lse[0, 0] - 0.5 * float(q[0, 0] @ k[0, 0])) < 1e-14


def test_rows_of_P_sum_to_one_and_masked_entries_are_zero():
    # With d == Lk and V the identity, O's row is exactly P's row.
    N = 24
    q, k = f64(N, 1, N, seed=4), f64(N, 1, N, seed=5)
    v = torch.eye(N, dtype=torch.float64).view(N, 1, N)
    for causal, wl in [(False, -1), (True, -1), (True, 5)]:
        P, _ = oracle.attn_fwd(q, k, v, [0, N], [0, N], 0.3, causal=causal, window_left=wl)
        P = P[:, 0, :]
        assert np.all(np.abs(P.sum(axis=1) - 1.0) <= 1e-12)
        assert np.all(P >= 0)
        for i in range(N):
            for j in range(N):
                if not oracle.allowed(i, j, N, N, causal, wl, -1):
                    assert P[i, j] == 0.0


def test_constant_v_reproduces_the_constant():
    N, d = 40, 16
    q, k = f64(N, 2, d, seed=6), f64(N, 2, d, seed=7)
    v = torch.full((N, 2, d), 0.8125, dtype=torch.float64)
    out, _ = oracle.attn_fwd(q, k, v, [0, N], [0, N], 1.0, causal=True)
    assert np.max(np.abs(out - 0.8125)) <= 1e-12


def test_empty_rows_give_zero_and_minus_inf():
    # window_right = -2 is not a legal API value; use Lk = 0 for a sequence with no keys
    q, k, v = f64(3, 1, 8, seed=8), f64(0, 1, 8, seed=9), f64(0, 1, 8, seed=10)
    out, lse = oracle.attn_fwd(q, k, v, [0, 3], [0, 0], 1.0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ---- special case that reduces to a library routine ------------------------------

def _sdpa_reference(q, k, v, scale, causal, wl, wr):
    """torch fp64 SDPA on one sequence with an explicit boolean mask and logsumexp."""
    Lq, Hq, d = q.shape
    Lk, Hkv, _ = k.shape
    mask = torch.zeros(Lq, Lk, dtype=torch.bool)
    for i in range(Lq):
        for j in range(Lk):
            mask[i, j] = oracle.allowed(i, j, Lq, Lk, causal, wl, wr)
    qh, kh, vh = q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1)
    o = F.scaled_dot_product_attention(qh[None], kh[None], vh[None], attn_mask=mask,
                                       scale=scale, enable_gqa=True)[0].transpose(0, 1)
    g = Hq // Hkv
    s = torch.einsum("qhd,khd->hqk", q, k.repeat_interleave(g, dim=1)) * scale
    lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
    return o, lse


@pytest.mark.parametrize("Lq,Lk,Hq,Hkv,d,causal,wl,wr", [
    (64, 64, 4, 4, 32, False, -1, -1),
    (64, 64, 4, 2, 32, True, -1, -1),
    (50, 77, 8, 2, 16, True, -1, -1),
    (96, 96, 4, 1, 32, True, 17, 0),
    (96, 96, 2, 2, 32, False, 9, 5),
    (33, 120, 6, 3, 8, False, 40, 3),
])
def test_against_torch_fp64_sdpa(Lq, Lk, Hq, Hkv, d, causal, wl, wr):
    q, k, v = f64(Lq, Hq, d, seed=11), f64(Lk, Hkv, d, seed=12), f64(Lk, Hkv, d, seed=13)
    scale = d ** -0.5
    out, lse = oracle.attn_fwd(q, k, v, [0, Lq], [0, Lk], scale, causal=causal,
                               window_left=wl, window_right=wr)
    o_ref, lse_ref = _sdpa_reference(q, k, v, scale, causal, wl, wr)
    finite = torch.isfinite(lse_ref).numpy()  # SDPA returns NaN on rows with no key
    assert finite.any()
    o_ref = o_ref.numpy()
    for h in range(Hq):
        rows = finite[h]
        assert np.max(np.abs(out[rows, h] - o_ref[rows, h])) <= 1e-12
        assert np.max(np.abs(lse[h, rows] - lse_ref[h, rows].numpy())) <= 1e-12
        assert np.all(np.isneginf(lse[h, ~rows])) and np.all(out[~rows, h] == 0)


# ---- structural invariants --------------------------------------------------------

def test_varlen_equals_each_sample_alone(golden):
    ex = golden["cu_seqlens"]
    assert synth.cu_from_lengths(ex["lengths"]).tolist() == ex["cu_seqlens"]
    lens = ex["lengths"]
    cu = ex["cu_seqlens"]
    q, k, v = f64(cu[-1], 2, 8, seed=14), f64(cu[-1], 2, 8, seed=15), f64(cu[-1], 2, 8, seed=16)
    out, lse = oracle.attn_fwd(q, k, v, cu, cu, 0.7, causal=True)
    for b, n in enumerate(lens):
        s, e = cu[b], cu[b + 1]
        o1, l1 = oracle.attn_fwd(q[s:e], k[s:e], v[s:e], [0, n], [0, n], 0.7, causal=True)
        assert np.array_equal(out[s:e], o1) and np.array_equal(lse[:, s:e], l1)


def test_gqa_equals_broadcast_kv_heads():
    L, Hq, Hkv, d = 37, 8, 2, 16
    q, k, v = f64(L, Hq, d, seed=17), f64(L, Hkv, d, seed=18), f64(L, Hkv, d, seed=19)
    out, lse = oracle.attn_fwd(q, k, v, [0, L], [0, L], 0.25, causal=True)
    g = Hq // Hkv
    out2, lse2 = oracle.attn_fwd(q, k.repeat_interleave(g, 1), v.repeat_interleave(g, 1),
                                 [0, L], [0, L], 0.25, causal=True)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def _contiguous_from_paged(case):
    """Gather each sequence's keys in logical order (test-side, by plain indexing)."""
    ks, vs, cu = [], [], [0]
    for b, L in enumerate(case.cache_seqlens.tolist()):
        pages = case.block_table[b, : (L + case.page_size - 1) // case.page_size].long()
        kk = case.k_cache[pages].reshape(-1, *case.k_cache.shape[2:])[:L]
        vv = case.v_cache[pages].reshape(-1, *case.v_cache.shape[2:])[:L]
        ks.append(kk)
        vs.append(vv)
        cu.append(cu[-1] + L)
    return torch.cat(ks), torch.cat(vs), cu


def test_paged_equals_contiguous_and_page_order_does_not_matter():
    case = synth.decode_case([1, 17, 64, 100, 257], 8, 2, 32, 16, seed=20)
    out, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.cache_seqlens,
                             case.block_table, case.softmax_scale)
    k, v, cu_k = _contiguous_from_paged(case)
    B = case.q.shape[0]
    o2, l2 = oracle.attn_fwd(case.q, k, v, list(range(B + 1)), cu_k, case.softmax_scale,
                             causal=True)
    assert np.max(np.abs(out - o2)) <= 1e-13 and np.max(np.abs(lse - l2.T)) <= 1e-13
    # move every page to a new physical slot; the table follows
    perm = torch.randperm(case.k_cache.shape[0], generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(len(perm))
    bt2 = inv[case.block_table.long()].to(torch.int32)
    kc2 = torch.empty_like(case.k_cache)
    vc2 = torch.empty_like(case.v_cache)
    kc2[inv] = case.k_cache
    vc2[inv] = case.v_cache
    o3, l3 = oracle.decode(case.q, kc2, vc2, case.cache_seqlens, bt2, case.softmax_scale)
    assert np.array_equal(out, o3) and np.array_equal(lse, l3)


@pytest.mark.parametrize("S", [1, 2, 3, 7, 16])
def test_split_kv_plus_merge_equals_unsplit(S):
    case = synth.decode_case([5, 100, 333, 1024], 4, 2, 16, 32, seed=21)
    o0, l0 = oracle.decode(case.q, case.k_cache, case.v_cache, case.cache_seqlens,
                           case.block_table, case.softmax_scale, num_splits=0)
    o1, l1 = oracle.decode(case.q, case.k_cache, case.v_cache, case.cache_seqlens,
                           case.block_table, case.softmax_scale, num_splits=S)
    assert np.max(np.abs(o0 - o1)) <= 1e-12 and np.max(np.abs(l0 - l1)) <= 1e-12


# ---- worked integer examples from the pages ----------------------------------------

def test_block_table_worked_example(golden):
    ex = golden["block_table"]
    bs, table, t = ex["block_size"], ex["block_table"], ex["token"]
    num_pages, d = 8, 4
    k_cache = torch.zeros(num_pages, bs, 1, d, dtype=torch.float64)
    v_cache = torch.zeros(num_pages, bs, 1, d, dtype=torch.float64)
    for p in range(num_pages):
        for o in range(bs):
            v_cache[p, o, 0, 0] = p
            v_cache[p, o, 0, 1] = o
    # only the physical slot the example names gets a key aligned with q
    k_cache[ex["physical_block"], ex["offset"], 0, 0] = 1.0
    q = torch.zeros(1, 1, d, dtype=torch.float64)
    q[0, 0, 0] = 1.0
    bt = torch.tensor([table], dtype=torch.int32)
    out, _ = oracle.decode(q, k_cache, v_cache, torch.tensor([t + 1], dtype=torch.int32), bt,
                           200.0)
    assert abs(out[0, 0, 0] - ex["physical_block"]) < 1e-12
    assert abs(out[0, 0, 1] - ex["offset"]) < 1e-12
    assert t // bs == ex["logical_block"] and table[t // bs] == ex["physical_block"]


def test_bottom_right_causal_example(golden):
    ex = golden["bottom_right_causal"]
    Lq, Lk = ex["seqlen_q"], ex["seqlen_k"]
    got = [sum(oracle.allowed(i, j, Lq, Lk, True) for j in range(Lk)) for i in range(Lq)]
    assert got == ex["visible_keys_per_row"]


def test_chunked_prefill_figure(golden):
    ex = golden["chunked_prefill_batch"]
    cq, lk = ex["cu_seqlens_q"], ex["seq_lens_k"]
    got = []
    for b in range(len(lk)):
        Lq = cq[b + 1] - cq[b]
        for i in range(Lq):
            got.append(sum(oracle.allowed(i, j, Lq, lk[b], True) for j in range(lk[b])))
    assert got == ex["visible_keys_per_row"]


def _block_pattern(nblk, B, causal, wl):
    N = nblk * B
    rows = []
    for qb in range(nblk):
        row = ""
        for kb in range(nblk):
            vis = [oracle.allowed(i, j, N, N, causal, wl, -1)
                   for i in range(qb * B, qb * B + B) for j in range(kb * B, kb * B + B)]
            if not any(vis):
                row += "."
            elif all(vis):
                row += "F"
            else:
                row += "D" if kb == qb else "E"
        rows.append(row)
    return rows


def test_block_level_causal_and_window_figure(golden):
    ex = golden["block_masks"]
    B = 4
    causal = _block_pattern(8, B, True, -1)
    assert causal == ex["causal"]
    flat = "".join(causal)
    assert len(flat) - flat.count(".") == ex["causal_tiles"]
    assert flat.count("D") == ex["causal_masked"]
    # The figure's window reaches two blocks back: window_left = 2 * B.
    assert _block_pattern(8, B, True, 2 * B) == ex["causal_window"]


# ---- the pages' byte and FLOP accounting --------------------------------------------

def test_standard_attention_accounting_n4096(golden):
    ex = golden["standard_attention_accounting"]
    N, d = ex["N"], ex["d"]
    q = synth.randn_bf16((N, 1, d), 5, 1)
    k = synth.randn_bf16((N, 1, d), 5, 2)
    v = synth.randn_bf16((N, 1, d), 5, 3)
    out, lse, c = oracle.attn_fwd(q, k, v, [0, N], [0, N], d ** -0.5, with_counts=True)
    # S written by GEMM 1 and read by softmax; P written by softmax and read by GEMM 2
    nsq_bytes = 2 * (2 * c.s_elems + 2 * c.p_elems)
    total = c.qkvo_bytes + nsq_bytes
    assert total == ex["bytes_total"]
    assert nsq_bytes == ex["nsquared_traffic_mib"] * 2 ** 20
    assert round(total / 2 ** 20) == ex["bytes_total_mib"]
    assert c.flops == ex["flops"] == 4 * N * N * d
    assert round(c.flops / total, 2) == ex["intensity_flop_per_byte"]
    assert round(total / (ex["a100_hbm_tbs"] * 1e12) * 1e6, 1) == ex["hbm_bound_us"]
    assert round(c.flops / (ex["a100_bf16_tflops"] * 1e12) * 1e6, 1) == ex["compute_bound_us"]
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    fa = golden["flash_attention_traffic"]
    assert oracle.tiled_traffic_bytes(N, d, 128) == fa["Br_128_mib"] * 2 ** 20
    assert oracle.tiled_traffic_bytes(N, d, 256) == fa["Br_256_mib"] * 2 ** 20


def test_causal_accounting_counts_pairs():
    N, d = 300, 8
    q, k, v = f64(N, 1, d, seed=30), f64(N, 1, d, seed=31), f64(N, 1, d, seed=32)
    _, _, c = oracle.attn_fwd(q, k, v, [0, N], [0, N], 1.0, causal=True, with_counts=True)
    assert c.flops == 4 * d * N * (N + 1) // 2


# ---- input widening -------------------------------------------------------------------

def test_bf16_inputs_widen_exactly():
    x = synth.randn_bf16((64, 1, 8), 9, 1)
    xd = x.to(torch.float64)
    o1, l1 = oracle.attn_fwd(x, x, x, [0, 64], [0, 64], 0.5, causal=True)
    o2, l2 = oracle.attn_fwd(xd, xd, xd, [0, 64], [0, 64], 0.5, causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
