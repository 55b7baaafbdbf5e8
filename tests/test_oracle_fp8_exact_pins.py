"""The oracle's FP8 quantizer against the quantizer's exact fp64 definition.

The oracle quantizes in fp32 (the same single IEEE operations a device can do, so a device
quantizer can be compared with it bit for bit).  That makes its codes a statement about fp32
arithmetic; this file pins them to the definition instead: the exact rotation (a matrix
product with the Sylvester Hadamard matrix), the exact block maximum and the exact ratio
448 / max|y|.  Every code must be the nearest e4m3 value of that exact quantity, except where
the quantity sits within the fp32 evaluation error of a rounding midpoint, where either
neighbour is accepted (and such elements must be rare).
"""
import numpy as np
import pytest
import torch

from oracle import oracle
from tests.fp8_exact import check_codes, e4m3_grid


def _bits(x):
    t = torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.double().numpy()


def _blocks():
    g = np.random.default_rng(77)
    yield "normal", g.standard_normal((128, 128)) * 1.7
    yield "ragged rows", g.standard_normal((37, 128))
    heavy = g.standard_normal((128, 128))
    heavy[3, 17] = 60.0                                  # one outlier sets the scale
    yield "outlier", heavy
    yield "wide range", g.standard_normal((64, 128)) * np.exp(g.uniform(-12, 6, (64, 128)))
    yield "single row", g.standard_normal((1, 128)) * 1e-3
    yield "integers", g.integers(-8, 9, (16, 128)).astype(np.float64)


@pytest.mark.parametrize("rotate", [False, True])
def test_quantizer_codes_are_nearest_to_the_exact_definition(rotate):
    g = np.random.default_rng(5)
    signs = np.where(g.integers(0, 2, 128) > 0, 1.0, -1.0).astype(np.float32) if rotate else None
    near_total = elems = 0
    for name, x in _blocks():
        bits, xv = _bits(x)
        codes, scale = oracle.fp8_quantize_rows(bits, signs)
        near_total += check_codes(xv, codes, scale, signs)
        elems += xv.size
    # midpoints within a few fp32 roundings are rare
    assert near_total <= max(4, elems // 1000)


def test_checker_catches_plausible_mistakes():
    """The checker is strict enough to see a wrong rounding, a wrong scale or a dropped sign
    (mistakes planted on the host, in copies of the oracle's output)."""
    g = np.random.default_rng(9)
    bits, xv = _bits(g.standard_normal((32, 128)))
    codes, scale = oracle.fp8_quantize_rows(bits)
    check_codes(xv, codes, scale)
    grid = e4m3_grid()
    # truncation instead of rounding on one element that is not near a midpoint
    z = xv * (448.0 / np.abs(xv).max())
    a = np.abs(z)
    hi = np.searchsorted(grid, a)
    lo = np.maximum(hi - 1, 0)
    frac = (a - grid[lo]) / np.maximum(grid[np.minimum(hi, 0x7E)] - grid[lo], 1e-300)
    i = np.unravel_index(np.argmax(np.where(frac < 0.9, frac, -1)), a.shape)
    assert 0.6 < frac[i] < 0.9
    bad = codes.copy()
    bad[i] = (bad[i] & 0x80) | lo[i]
    with pytest.raises(AssertionError):
        check_codes(xv, bad, scale)
    with pytest.raises(AssertionError):                 # scale off by one part in 2^10
        check_codes(xv, codes, scale * (1 + 2 ** -10))
    bad = codes.copy()
    j = np.unravel_index(np.argmax(np.abs(xv)), xv.shape)
    bad[j] ^= 0x80
    with pytest.raises(AssertionError):
        check_codes(xv, bad, scale)
    # and the rotation: codes of the unrotated block fail against the rotated definition
    signs = np.ones(128, np.float32)
    with pytest.raises(AssertionError):
        check_codes(xv, codes, scale, signs)


def test_all_zero_block():
    bits, xv = _bits(np.zeros((5, 128)))
    codes, scale = oracle.fp8_quantize_rows(bits)
    assert scale == 1.0 and not codes.any()
    check_codes(xv, codes, scale)
