"""Pins of the oracle's chunked prefill over a paged cache (KV append, rotary embedding).

Sources: "Attention kernels: FlashAttention and PagedAttention", section 五.1 (chunked prefill:
new tokens' K/V are written into the cache, then read by the same step; the worked figure);
"04 · FA4 (CuTeDSL) and engineering interfaces", sections 6.1-6.2 (block_table,
cache_seqlens, in-place append of new k, v together with rotary embedding, bottom-right
causal).  The pages name the rotary embedding without its formula; the oracle takes the
standard one (each plane (a, b) -> (a cos - b sin, a sin + b cos), rotate-half or interleaved
planes), pinned here by closed forms and by its defining relative-position property.
"""
import math

import numpy as np
import torch

from oracle import oracle


def f64(*shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float64)


def rope_tables(rows, rot, base=10000.0, offset=0.0):
    inv = base ** (-np.arange(0, rot, 2, dtype=np.float64) / rot)
    ang = (np.arange(rows, dtype=np.float64) + offset)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def one_seq_cache(ctx, q_len, Hkv, d, page_size, num_pages, perm_seed=0):
    """Empty cache with a random page order holding one sequence."""
    need = -(-(ctx + q_len) // page_size)
    g = torch.Generator().manual_seed(perm_seed)
    pages = torch.randperm(num_pages, generator=g)[:need].to(torch.int32)
    bt = torch.zeros((1, need), dtype=torch.int32)
    bt[0, :need] = pages
    kc = torch.zeros((num_pages, page_size, Hkv, d), dtype=torch.float64)
    return kc, kc.clone(), bt


def test_bf16_rounding_ties_and_library():
    b = oracle.f64_to_bf16_bits
    assert b(1.0) == 0x3F80
    assert b(1 + 2 ** -8) == 0x3F80            # tie, to even
    assert b(1 + 3 * 2 ** -8) == 0x3F82        # tie, to even
    assert b(1 + 2 ** -8 + 2 ** -30) == 0x3F81  # above the tie
    assert b(-0.0) == 0x8000 and b(float("inf")) == 0x7F80
    assert b(3.4e38) == 0x7F80                  # past the largest finite bf16
    # any fp32 value: agrees with torch's round-to-nearest-even fp32 -> bf16
    g = torch.Generator().manual_seed(3)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-140, 120, (20000,), generator=g).float())
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([b(float(v)) for v in x.tolist()], dtype=np.uint16)
    assert np.array_equal(got, ref)


def run(q, kn, vn, kc, vc, ctx, bt, cu, scale=0.5, causal=True, cos=None, sin=None, inter=False,
        wl=-1, wr=-1):
    return oracle.kvcache_prefill(q, kn, vn, kc, vc, torch.tensor(ctx, dtype=torch.int32), bt,
                                  torch.tensor(cu, dtype=torch.int32), scale, causal, wl, wr,
                                  cos, sin, inter)


def test_rope_quarter_turn_closed_form():
    # d = 2, one plane, angle pi/2 at position 0: key (1, 0) -> (0, 1), (0, 1) -> (-1, 0)
    kc, vc, bt = one_seq_cache(0, 2, 1, 2, 4, 2)
    cos, sin = np.array([[0.0], [0.0]]), np.array([[1.0], [1.0]])
    kn = torch.tensor([[[1.0, 0.0]], [[0.0, 1.0]]], dtype=torch.float64)
    q = torch.zeros((2, 1, 2), dtype=torch.float64)
    _, _, k2, _ = run(q, kn, kn, kc, vc, [0], bt, [0, 2], cos=cos, sin=sin)
    page = int(bt[0, 0])
    assert np.allclose(k2[page, 0, 0], [0.0, 1.0], atol=0) and np.allclose(k2[page, 1, 0], [-1.0, 0.0], atol=0)


def test_rope_rotate_half_versus_interleaved_planes():
    # d = 4, two planes with angles pi/2 (plane 0) and 0 (plane 1); x = (1, 2, 3, 4)
    kc, vc, bt = one_seq_cache(0, 1, 1, 4, 4, 1)
    cos, sin = np.array([[0.0, 1.0]]), np.array([[1.0, 0.0]])
    kn = torch.tensor([[[1.0, 2.0, 3.0, 4.0]]], dtype=torch.float64)
    q = torch.zeros((1, 1, 4), dtype=torch.float64)
    _, _, k_half, _ = run(q, kn, kn, kc, vc, [0], bt, [0, 1], cos=cos, sin=sin, inter=False)
    _, _, k_int, _ = run(q, kn, kn, kc, vc, [0], bt, [0, 1], cos=cos, sin=sin, inter=True)
    page = int(bt[0, 0])
    # rotate-half: planes (x0, x2) by 90 degrees, (x1, x3) unchanged -> (-3, 2, 1, 4)
    assert list(k_half[page, 0, 0]) == [-3.0, 2.0, 1.0, 4.0]
    # interleaved: planes (x0, x1) by 90 degrees, (x2, x3) unchanged -> (-2, 1, 3, 4)
    assert list(k_int[page, 0, 0]) == [-2.0, 1.0, 3.0, 4.0]
    # components past rot_dim are left alone (rot_dim 2 of 4)
    _, _, k_part, _ = run(q, kn, kn, kc, vc, [0], bt, [0, 1], cos=cos[:, :1], sin=sin[:, :1])
    assert list(k_part[page, 0, 0]) == [-2.0, 1.0, 3.0, 4.0]


def test_rope_same_position_keeps_the_score():
    # one query and its own key at the same position: the rotation cancels in <q, k>
    d, rot = 8, 8
    kc, vc, bt = one_seq_cache(5, 1, 1, d, 4, 4)
    cos, sin = rope_tables(16, rot)
    q, kn, vn = f64(1, 1, d, seed=1), f64(1, 1, d, seed=2), f64(1, 1, d, seed=3)
    # a window that leaves only the new key visible
    out, lse, _, _ = run(q, kn, vn, kc, vc, [5], bt, [0, 1], cos=cos, sin=sin, wl=0)
    assert abs(lse[0, 0] - 0.5 * float((q[0, 0] * kn[0, 0]).sum())) < 1e-12
    assert np.allclose(out[0, 0], vn[0, 0].numpy(), atol=1e-15)


def test_rope_scores_depend_only_on_relative_position():
    # shifting every position's angle by the same amount changes nothing
    d, rot, L = 16, 12, 24
    q, kn, vn = f64(L, 2, d, seed=4), f64(L, 1, d, seed=5), f64(L, 1, d, seed=6)
    kc, vc, bt = one_seq_cache(0, L, 1, d, 8, 4)
    c0, s0 = rope_tables(L, rot)
    c1, s1 = rope_tables(L, rot, offset=37.0)
    o0, l0, _, _ = run(q, kn, vn, kc, vc, [0], bt, [0, L], cos=c0, sin=s0)
    o1, l1, _, _ = run(q, kn, vn, kc, vc, [0], bt, [0, L], cos=c1, sin=s1)
    assert np.allclose(o0, o1, atol=1e-12) and np.allclose(l0, l1, atol=1e-12)
    # and the rotation does matter (guards against a no-op)
    on, ln_, _, _ = run(q, kn, vn, kc, vc, [0], bt, [0, L])
    assert np.abs(ln_ - l0).max() > 1e-3


def test_chunk_equals_rows_of_full_prefill_without_rope():
    d, Hq, Hkv, L, ctx = 32, 4, 2, 40, 29
    q, k, v = f64(L, Hq, d, seed=7), f64(L, Hkv, d, seed=8), f64(L, Hkv, d, seed=9)
    o_full, l_full = oracle.attn_fwd(q, k, v, [0, L], [0, L], 0.3, causal=True)
    kc, vc, bt = one_seq_cache(ctx, L - ctx, Hkv, d, 16, 6)
    # cached prefix written in page order by hand (block_table addressing)
    for j in range(ctx):
        kc[bt[0, j // 16], j % 16] = k[j]
        vc[bt[0, j // 16], j % 16] = v[j]
    o, l, _, _ = run(q[ctx:], k[ctx:], v[ctx:], kc, vc, [ctx], bt, [0, L - ctx], scale=0.3)
    assert np.allclose(o, o_full[ctx:], atol=1e-12) and np.allclose(l, l_full[:, ctx:], atol=1e-12)


def test_chunk_equals_rows_of_full_prefill_with_rope_and_window():
    d, Hq, Hkv, L, ctx, rot = 32, 2, 1, 50, 33, 32
    q, k, v = f64(L, Hq, d, seed=10), f64(L, Hkv, d, seed=11), f64(L, Hkv, d, seed=12)
    cos, sin = rope_tables(64, rot)
    kc, vc, bt = one_seq_cache(0, L, Hkv, d, 16, 8)
    # the whole sequence as one chunk over an empty cache
    o_full, l_full, kc1, vc1 = run(q, k, v, kc, vc, [0], bt, [0, L], cos=cos, sin=sin, wl=9)
    # the cache after that step holds every rotated key; keep only the first ctx positions
    kc2, vc2 = kc1.copy(), vc1.copy()
    for j in range(ctx, L):
        kc2[bt[0, j // 16], j % 16] = 0.0
        vc2[bt[0, j // 16], j % 16] = 0.0
    o, l, kc3, _ = run(q[ctx:], k[ctx:], v[ctx:], torch.from_numpy(kc2), torch.from_numpy(vc2), [ctx],
                       bt, [0, L - ctx], cos=cos, sin=sin, wl=9)
    assert np.array_equal(kc3, kc1)
    assert np.allclose(o, o_full[ctx:], atol=1e-12) and np.allclose(l, l_full[:, ctx:], atol=1e-12)


def test_append_writes_only_the_new_positions_bit_exact():
    # bf16 data, three sequences (the pages' chunked-prefill figure: q_len 4/1/1 after
    # 8/11/5 cached tokens), page size 4, random page order
    Hq, Hkv, d, ps = 4, 2, 16, 4
    ctx, ql = [8, 11, 5], [4, 1, 1]
    cu = [0, 4, 5, 6]
    need = [-(-(c + n) // ps) for c, n in zip(ctx, ql)]
    num_pages = sum(need) + 2
    g = torch.Generator().manual_seed(13)
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    bt = torch.zeros((3, max(need)), dtype=torch.int32)
    at = 0
    for b in range(3):
        bt[b, :need[b]] = perm[at:at + need[b]]
        at += need[b]
    kc = torch.randn(num_pages, ps, Hkv, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(num_pages, ps, Hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(6, Hq, d, generator=g).to(torch.bfloat16)
    kn = torch.randn(6, Hkv, d, generator=g).to(torch.bfloat16)
    vn = torch.randn(6, Hkv, d, generator=g).to(torch.bfloat16)
    out, lse, k2, v2 = run(q, kn, vn, kc, vc, ctx, bt, cu, scale=0.25)
    k0 = kc.view(torch.int16).numpy().view(np.uint16)
    v0 = vc.view(torch.int16).numpy().view(np.uint16)
    expect_k, expect_v = k0.copy(), v0.copy()
    for b in range(3):
        for i in range(ql[b]):
            pos = ctx[b] + i
            page, off = int(bt[b, pos // ps]), pos % ps
            expect_k[page, off] = kn[cu[b] + i].view(torch.int16).numpy().view(np.uint16)
            expect_v[page, off] = vn[cu[b] + i].view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(k2, expect_k) and np.array_equal(v2, expect_v)
    # rows see 9, 10, 11, 12 / 12 / 6 keys: each row's LSE equals the one computed by the
    # contiguous oracle over the gathered keys of its sequence
    for b in range(3):
        L = ctx[b] + ql[b]
        idx = [(int(bt[b, j // ps]), j % ps) for j in range(L)]
        kk = torch.from_numpy(np.stack([k2[p, o] for p, o in idx]).view(np.int16)).view(torch.bfloat16)
        vv = torch.from_numpy(np.stack([v2[p, o] for p, o in idx]).view(np.int16)).view(torch.bfloat16)
        o_ref, l_ref = oracle.attn_fwd(q[cu[b]:cu[b + 1]], kk, vv, [0, ql[b]], [0, L], 0.25, causal=True)
        assert np.allclose(out[cu[b]:cu[b + 1]], o_ref, atol=1e-12)
        assert np.allclose(lse[:, cu[b]:cu[b + 1]], l_ref, atol=1e-12)
