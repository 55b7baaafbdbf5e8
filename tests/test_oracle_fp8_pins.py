"""Pins of the oracle's FP8 (e4m3) part against the format's definition and plain identities.

The e4m3 values come from the standard 8-bit float definition (OCP 8-bit floating point,
E4M3); the FP8 forward reads them with block scales ("Attention kernels: FlashAttention and
PagedAttention", section 四.2, FlashAttention-3)."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle


def test_e4m3_table_points():
    # the format's named points: largest normal S.1111.110 = 448, smallest normal
    # S.0001.000 = 2^-6, largest subnormal S.0000.111 = 0.875 * 2^-6, smallest subnormal
    # S.0000.001 = 2^-9, one = S.0111.000, NaN = S.1111.111
    d = oracle.e4m3_to_f64
    assert d([0x7E])[0] == 448.0
    assert d([0x08])[0] == 2.0 ** -6
    assert d([0x07])[0] == 0.875 * 2.0 ** -6
    assert d([0x01])[0] == 2.0 ** -9
    assert d([0x38])[0] == 1.0
    assert d([0x39])[0] == 1.125
    assert d([0xB8])[0] == -1.0
    assert d([0xFE])[0] == -448.0
    assert math.isnan(d([0x7F])[0]) and math.isnan(d([0xFF])[0])
    assert d([0x00])[0] == 0.0 and math.copysign(1.0, d([0x80])[0]) == -1.0


def test_e4m3_grid_structure():
    pos = oracle.e4m3_to_f64(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0)                       # increasing with the code
    assert np.array_equal(oracle.e4m3_to_f64(np.arange(0x80, 0xFF)), -pos)  # sign bit mirrors
    # spacing is 2^(e-10) in binade e >= 1 (8 values per binade) and 2^-9 among subnormals
    for c in range(1, 0x7E):
        e = max((c >> 3) & 15, 1)
        assert pos[c + 1] - pos[c] == 2.0 ** (e - 10)
    assert len(set(oracle.e4m3_to_f64(np.r_[0:0x7F, 0x80:0xFF]).tolist())) == 253


def test_e4m3_encode_round_trip_ties_and_saturation():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.f64_to_e4m3(oracle.e4m3_to_f64([c])[0]) == c
    pos = oracle.e4m3_to_f64(np.arange(0x7F))
    for c in range(0x7E):
        mid = (pos[c] + pos[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.f64_to_e4m3(mid) == even             # ties to the even mantissa
        assert oracle.f64_to_e4m3(np.nextafter(mid, 0)) == c
        assert oracle.f64_to_e4m3(np.nextafter(mid, 1e9)) == c + 1
        assert oracle.f64_to_e4m3(-mid) == 0x80 | even
    assert oracle.f64_to_e4m3(449.0) == 0x7E and oracle.f64_to_e4m3(1e30) == 0x7E
    assert oracle.f64_to_e4m3(-1e30) == 0xFE and oracle.f64_to_e4m3(float("nan")) == 0x7F


def _small_case(seed, lens_q, lens_k, Hq, Hkv, d, int_codes=False):
    g = torch.Generator().manual_seed(seed)
    tq, tk = sum(lens_q), sum(lens_k)
    cu_q = torch.tensor([0] + np.cumsum(lens_q).tolist(), dtype=torch.int32)
    cu_k = torch.tensor([0] + np.cumsum(lens_k).tolist(), dtype=torch.int32)
    kb0 = oracle.key_block_offsets(cu_k)
    nkb = int(kb0[-1]) + 1
    if int_codes:   # codes of -2, -1, 0, 1, 2
        pick = torch.tensor([0xC0, 0xB8, 0x00, 0x38, 0x40], dtype=torch.uint8)
        cq = pick[torch.randint(0, 5, (tq, Hq, d), generator=g)]
        ck = pick[torch.randint(0, 5, (tk, Hkv, d), generator=g)]
        cv = pick[torch.randint(0, 5, (Hkv, d, 128 * nkb), generator=g)]
    else:
        cq = torch.randint(0, 0x7F, (tq, Hq, d), generator=g, dtype=torch.uint8)
        ck = torch.randint(0, 0x7F, (tk, Hkv, d), generator=g, dtype=torch.uint8)
        cv = torch.randint(0, 0x7F, (Hkv, d, 128 * nkb), generator=g, dtype=torch.uint8)
        for c in (cq, ck, cv):
            c ^= (torch.randint(0, 2, c.shape, generator=g, dtype=torch.uint8) << 7)
    qs = torch.rand((Hq, (tq + 127) // 128), generator=g, dtype=torch.float64) + 0.5
    ks = torch.rand((Hkv, nkb), generator=g, dtype=torch.float64) + 0.5
    vs = torch.rand((len(lens_q), Hkv), generator=g, dtype=torch.float64) + 0.5
    return cq, ck, cv, qs, ks, vs, cu_q, cu_k


def test_dequantize_layout_by_brute_force():
    lens_q, lens_k = [3, 140], [130, 5]
    cq, ck, cv, qs, ks, vs, cu_q, cu_k = _small_case(1, lens_q, lens_k, 4, 2, 8)
    q, k, v = oracle.fp8_dequantize(cq, ck, cv, qs, ks, vs, cu_k)
    dec = lambda c: oracle.e4m3_to_f64([int(c)])[0]
    # Q: global 128-token blocks
    for t in (0, 2, 127, 128, 142):
        for h in range(4):
            assert q[t, h, 5] == dec(cq[t, h, 5]) * float(qs[h, t // 128])
    # K and V: per-sequence 128-key blocks; sequence 1 starts at block ceil(130/128) = 2
    blocks = {(0, 0): 0, (0, 127): 0, (0, 128): 1, (0, 129): 1, (1, 0): 2, (1, 4): 2}
    for (b, i), blk in blocks.items():
        t = int(cu_k[b]) + i
        for h in range(2):
            assert k[t, h, 3] == dec(ck[t, h, 3]) * float(ks[h, blk])
            assert v[t, h, 6] == dec(cv[h, 6, 128 * blk + i % 128]) * float(vs[b, h])


def test_fp8_attention_matches_library_on_integer_values():
    # with unit scales and codes of small integers the decoded inputs are exact integers, and
    # the result must equal torch's fp64 scaled_dot_product_attention on them
    lens = [37, 150]
    cq, ck, cv, qs, ks, vs, cu_q, cu_k = _small_case(2, lens, lens, 4, 2, 16, int_codes=True)
    qs[:] = 1.0
    ks[:] = 1.0
    vs[:] = 1.0
    out, lse = oracle.fp8_attn_fwd(cq, ck, cv, qs, ks, vs, cu_q, cu_k, 0.25, causal=True)
    q, k, v = oracle.fp8_dequantize(cq, ck, cv, qs, ks, vs, cu_k)
    assert set(np.unique(q).tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}
    for b in range(2):
        s0, s1 = int(cu_q[b]), int(cu_q[b + 1])
        qt = torch.from_numpy(q[s0:s1]).permute(1, 0, 2)[None]
        kt = torch.from_numpy(k[s0:s1]).permute(1, 0, 2).repeat_interleave(2, 0)[None]
        vt = torch.from_numpy(v[s0:s1]).permute(1, 0, 2).repeat_interleave(2, 0)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                               scale=0.25)
        np.testing.assert_allclose(out[s0:s1], ref[0].permute(1, 0, 2).numpy(), atol=1e-12)


def test_fp8_scales_act_linearly():
    lens = [64, 200]
    cq, ck, cv, qs, ks, vs, cu_q, cu_k = _small_case(3, lens, lens, 2, 1, 16)
    base, lse0 = oracle.fp8_attn_fwd(cq, ck, cv, qs, ks, vs, cu_q, cu_k, 0.05, causal=True)
    # V's scale multiplies O
    out, lse = oracle.fp8_attn_fwd(cq, ck, cv, qs, ks, vs * 3.0, cu_q, cu_k, 0.05, causal=True)
    np.testing.assert_allclose(out, 3.0 * base, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse0, atol=1e-12)
    # doubling every Q scale is the same as doubling the softmax scale
    out2, lse2 = oracle.fp8_attn_fwd(cq, ck, cv, qs * 2.0, ks, vs, cu_q, cu_k, 0.05, causal=True)
    out3, lse3 = oracle.fp8_attn_fwd(cq, ck, cv, qs, ks, vs, cu_q, cu_k, 0.10, causal=True)
    np.testing.assert_allclose(out2, out3, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse2, lse3, rtol=1e-12, atol=1e-12)


# ---- the quantizer (block scales and the optional random-sign Hadamard rotation) ----------

def _bf16_bits(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rotation_is_the_sylvester_hadamard_matrix():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    d = 128
    H = scipy_linalg.hadamard(d)
    for j in (0, 1, 5, 64, 127):
        x = np.zeros((1, d), np.float32)
        x[0, j] = 1.0
        codes, s = oracle.fp8_quantize_rows(_bf16_bits(x), signs=np.ones(d, np.float32))
        # H e_j / sqrt(d) = column j of H over sqrt(d): every entry has magnitude amax -> 448
        assert s == np.float32(np.float32(1.0 / math.sqrt(d)) / np.float32(448.0))
        expect = np.where(H[:, j] > 0, 0x7E, 0xFE)
        assert np.array_equal(codes[0], expect)
    # the signs multiply before the transform: signs = e_j-indicator flips column j
    sg = np.ones(d, np.float32)
    sg[3] = -1.0
    x = np.zeros((1, d), np.float32)
    x[0, 3] = 1.0
    codes, _ = oracle.fp8_quantize_rows(_bf16_bits(x), signs=sg)
    assert np.array_equal(codes[0], np.where(H[:, 3] > 0, 0xFE, 0x7E))


def test_block_quantization_grid_and_extremes():
    g = np.random.default_rng(4)
    x = g.standard_normal((100, 128)).astype(np.float32) * 3.0
    bits = _bf16_bits(x)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    codes, s = oracle.fp8_quantize_rows(bits)
    assert s == np.float32(np.float32(np.abs(xb).max()) / np.float32(448.0))
    i = np.unravel_index(np.abs(xb).argmax(), xb.shape)
    assert codes[i] in (0x7E, 0xFE)                       # the block's largest element
    dec = oracle.e4m3_to_f64(codes)
    rcp = np.float32(448.0) / np.float32(np.abs(xb).max())
    y = np.clip((xb * rcp).astype(np.float64), -448.0, 448.0)  # (beyond 448 saturates)
    pos = oracle.e4m3_to_f64(np.arange(0x7F))
    step = np.array([pos[min(np.searchsorted(pos, abs(v)), 0x7E)] - pos[max(np.searchsorted(pos, abs(v)) - 1, 0)]
                     for v in y.ravel()]).reshape(y.shape)
    assert np.all(np.abs(dec - y) <= step / 2 + 1e-12)  # nearest grid point
    zc, zs = oracle.fp8_quantize_rows(np.zeros((3, 128), np.uint16))
    assert zs == 1.0 and not zc.any()


def test_rotation_preserves_norms_and_attention():
    c = _rotation_case()
    g = np.random.default_rng(11)
    signs = np.where(g.integers(0, 2, 128) > 0, 1.0, -1.0).astype(np.float32)
    # row norms survive the orthogonal rotation (up to the e4m3 rounding)
    q8, qs, k8, ks, v8t, vs = oracle.fp8_quantize(c.q, c.k, c.v, c.cu_seqlens_k, signs=signs)
    q, k, v = oracle.fp8_dequantize(q8, k8, v8t, qs, ks, vs, c.cu_seqlens_k)
    qf = c.q.double().numpy()
    np.testing.assert_allclose(np.linalg.norm(q, axis=2), np.linalg.norm(qf, axis=2), rtol=2 ** -4)
    # and Q K^T: attention on the rotated, quantized inputs tracks the bf16 attention
    out, lse = oracle.fp8_attn_fwd(q8, k8, v8t, qs, ks, vs, c.cu_seqlens_q, c.cu_seqlens_k,
                                   c.softmax_scale, causal=True)
    ref, ref_l = oracle.attn_fwd(c.q, c.k, c.v, c.cu_seqlens_q, c.cu_seqlens_k,
                                 c.softmax_scale, causal=True)
    # (V's own e4m3 rounding allows 2^-4 max|V| per element; a rotation that did not cancel
    # in Q K^T would scramble the scores and move the mean error to order 1)
    vmax = float(np.abs(c.v.double().numpy()).max())
    good = np.abs(out - ref).mean()
    assert np.abs(out - ref).max() <= 2 ** -4 * vmax and good < 0.01
    # (a single score carries the full Q and K rounding, about 2 * 2^-4 of |q||k| scale)
    assert np.abs(lse - ref_l).mean() < 0.01 and np.abs(lse - ref_l).max() < 0.2
    # the control: the same quantizer without the rotation on K (only Q rotated) breaks it
    q8b, qsb, _, _, _, _ = oracle.fp8_quantize(c.q, c.k, c.v, c.cu_seqlens_k, signs=signs)
    _, _, k8u, ksu, _, _ = oracle.fp8_quantize(c.q, c.k, c.v, c.cu_seqlens_k)
    bad, _ = oracle.fp8_attn_fwd(q8b, k8u, v8t, qsb, ksu, vs, c.cu_seqlens_q, c.cu_seqlens_k,
                                 c.softmax_scale, causal=True)
    assert np.abs(bad - ref).mean() > 10 * good
    # with V unrotated and the same rows, quantize -> dequantize returns V to within e4m3 steps
    vf = c.v.double().numpy()
    assert np.all(np.abs(v - vf) <= 2 ** -4 * np.abs(vf) + float(vs.max()) * 2 ** -9)


def _rotation_case():
    from exact_attention_70_gb300 import synth
    return synth.prefill_case([70, 200], 4, 2, 128, True, 21)


def test_quantize_layout_round_trip():
    from exact_attention_70_gb300 import synth
    c = synth.prefill_case([5, 130, 300], 4, 2, 128, True, 22)
    q8, qs, k8, ks, v8t, vs = oracle.fp8_quantize(c.q, c.k, c.v, c.cu_seqlens_k)
    kb0 = oracle.key_block_offsets(c.cu_seqlens_k)
    assert ks.shape == (2, int(kb0[-1])) and v8t.shape == (2, 128, 128 * int(kb0[-1]))
    # padding columns of V^T are code 0
    cu = c.cu_seqlens_k.tolist()
    for b in range(3):
        n = cu[b + 1] - cu[b]
        col = 128 * int(kb0[b])
        assert not v8t[:, :, col + n:128 * int(kb0[b + 1])].any()
    q, k, v = oracle.fp8_dequantize(q8, k8, v8t, qs, ks, vs, c.cu_seqlens_k)
    for got, ref, sc in ((q, c.q, qs), (k, c.k, ks), (v, c.v, vs)):
        r = ref.double().numpy()
        assert np.all(np.abs(got - r) <= 2 ** -4 * np.abs(r) + float(sc.max()) * 2 ** -9)
