"""The FP8 block quantizer's exact (fp64) definition, for checking codes from either side.

Reading ("Attention kernels: FlashAttention and PagedAttention", section 四.2, FlashAttention-3:
block scales and incoherent processing): one block of rows x (bf16 values) becomes
  y = H diag(signs) x / sqrt(d)   per row, when a rotation is asked for (H: the Sylvester
                                  Walsh-Hadamard matrix), else y = x;
  scale = max|y| / 448;  code = the e4m3 value nearest to y / scale, ties to even.
Here every step is carried out exactly (or to fp64 rounding, far below the fp32 steps of the
implementations): the Hadamard product as a matrix product, the exact block maximum and the
exact ratio 448 / max|y|.  The implementations work in fp32, so a value that lies within a
few fp32 roundings of the midpoint between two e4m3 neighbours may legitimately land on
either; everywhere else the code must be the nearest one.  The e4m3 grid is built here from the
format's definition (sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals
(m/8) 2^-6, largest finite 448), independently of any codec under test.
"""
import numpy as np

U32 = 2.0 ** -24   # unit roundoff of fp32


def e4m3_grid():
    """Non-negative finite e4m3 values, indexed by code 0 .. 0x7E."""
    vals = []
    for c in range(0x7F):
        e, m = (c >> 3) & 15, c & 7
        vals.append(m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, np.float64)


def sylvester(d):
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def exact_block(x, signs=None):
    """x [n, d] fp64 (the bf16 values).  Returns (y_scaled = y * 448 / max|y|, scale_exact,
    err): err [n, d] bounds how far an fp32 evaluation of the same steps may sit from
    y_scaled (a rigorous first-order bound, doubled)."""
    x = np.asarray(x, np.float64)
    n, d = x.shape
    if signs is not None:
        s = np.asarray(signs, np.float64)
        H = sylvester(d)
        y = (x * s[None, :]) @ H.T / np.sqrt(d)
        # fp32 butterflies: log2(d) roundings on sums bounded by the row's L1 norm, then the
        # 1/sqrt(d) constant and the product (two more)
        l1 = np.abs(x).sum(axis=1, keepdims=True) / np.sqrt(d)
        abs_err = (np.log2(d) + 2) * U32 * l1 * np.ones_like(y)
    else:
        y = x.copy()
        abs_err = np.zeros_like(y)
    amax = float(np.abs(y).max()) if y.size else 0.0
    if amax == 0.0:
        return y, 1.0, np.zeros_like(y)
    r = 448.0 / amax
    # the implementation's maximum is one of its y's: off by at most max(abs_err); the
    # reciprocal and the product add one rounding each
    amax_rel = float(abs_err.max()) / amax
    err = r * abs_err + np.abs(y) * r * (amax_rel + 3 * U32)
    return y * r, amax / 448.0, 2.0 * err + 1e-300


def check_codes(x, codes, scale, signs=None):
    """Assert that `codes` (uint8 [n, d]) and `scale` quantize the bf16 block x [n, d] as the
    exact definition says.  Returns the number of elements that sat within the fp32 error of a
    rounding midpoint (where either neighbour is accepted)."""
    z, s_exact, err = exact_block(x, signs)
    grid = e4m3_grid()
    codes = np.asarray(codes).astype(np.int64)
    assert codes.shape == z.shape
    assert not np.any((codes & 0x7F) == 0x7F), "NaN code"
    mag = grid[codes & 0x7F]
    neg = (codes & 0x80) != 0
    # sign: a nonzero code carries the value's sign
    nz = mag > 0
    assert np.all(neg[nz] == (z[nz] < 0)), "sign"
    a = np.minimum(np.abs(z), 448.0)
    hi = np.searchsorted(grid, a)                   # first grid point >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    exact_hit = grid[hi] == a
    d_lo, d_hi = a - grid[lo], grid[hi] - a
    nearest = np.where(exact_hit | (d_hi < d_lo), hi, lo)
    # ties to the even code
    tie = (d_lo == d_hi) & ~exact_hit
    nearest = np.where(tie, np.where(hi % 2 == 0, hi, lo), nearest)
    mid = 0.5 * (grid[lo] + grid[hi])
    near_mid = (np.abs(a - mid) <= err) & ~exact_hit
    got = codes & 0x7F
    ok = (got == nearest) | (near_mid & ((got == lo) | (got == hi)))
    # around a value that rounds to zero the sign of a zero code is free
    assert np.all(ok), (
        f"{int((~ok).sum())} codes are not the nearest e4m3 value of the exact block "
        f"(first at {np.argwhere(~ok)[0].tolist()})")
    # the stored scale is amax / 448 up to the fp32 error of the implementation's maximum
    rel = float(err.max()) / 448.0 + 4 * U32
    assert abs(float(scale) - s_exact) <= rel * s_exact, (float(scale), s_exact)
    return int((near_mid & (got != nearest)).sum())


def fp8_forward_bound(q, k, v, cu_q, cu_k, scale, causal, wl, wr, rows=None):
    """Per-element bound on |O_fp8 - O_ref| for the FP8 forward pass, O_ref being the exact
    attention of the dequantized fp64 inputs q [tq, Hq, d], k, v [tk, Hkv, d].

    The kernel rounds 16 P~ to e4m3, where P~ = exp2(x - m_ref) and m_ref is a block maximum
    of the row at most 4 (log2 units) below the true row maximum m, so 1 <= max P~ <= 16 and
    l~ = sum P~ >= L^ = sum exp2(x - m).  Per key:
      normal range (16 P~ >= 2^-6): |dP~| <= 2^-4 P~, i.e. 2^-4 P_j after normalisation;
      subnormal range: |dP~| <= min(P~, 2^-14), i.e. <= min(P^_j, 2^-14) / L^ normalised,
      which can only happen where P^_j = exp2(x_j - m) < 2^-10.
    So |dO_i| <= 2^-4 (P|V|)_i + sum_{P^_j < 2^-10} min(P^_j, 2^-14) |v_j| / L^, plus the
    bf16 rounding of O (2^-9 |O|) and fp32 accumulation (2^-12 (P|V|)_i, generous).
    Returns (bound, sigma): sigma_i = 2^-4 / sqrt(3) * sqrt(sum_j P_j^2 v_j^2), the standard
    deviation of the first term when the roundings are independent and uniform.
    rows = (tok, head) restricts the result to those rows ([n, d]); else [tq, Hq, d]."""
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    tq, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    cu_q = np.asarray(cu_q, np.int64)
    cu_k = np.asarray(cu_k, np.int64)
    if rows is None:
        tt, hh = np.meshgrid(np.arange(tq), np.arange(Hq), indexing="ij")
        tok, head = tt.ravel(), hh.ravel()
    else:
        tok, head = (np.asarray(a, np.int64) for a in rows)
    bound = np.zeros((len(tok), d))
    sigma = np.zeros((len(tok), d))
    seq = np.searchsorted(cu_q, tok, side="right") - 1
    for n in range(len(tok)):
        b, h = seq[n], head[n]
        i = tok[n] - cu_q[b]
        Lq, Lk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        if Lk == 0:
            continue
        kk = k[cu_k[b]:cu_k[b + 1], h // g]
        vv = np.abs(v[cu_k[b]:cu_k[b + 1], h // g])
        pos = i + Lk - Lq
        j = np.arange(Lk)
        right = 0 if causal else wr
        vis = np.ones(Lk, bool)
        if right >= 0:
            vis &= j <= pos + right
        if wl >= 0:
            vis &= j >= pos - wl
        if not vis.any():
            continue
        x = scale * (kk[vis] @ q[tok[n], h]) / np.log(2.0)   # log2 units
        ph = np.exp2(x - x.max())
        L = ph.sum()
        P = ph / L
        va = vv[vis]
        pv = P @ va
        sub = np.where(ph < 2.0 ** -10, np.minimum(ph, 2.0 ** -14), 0.0) @ va / L
        o = P @ (v[cu_k[b]:cu_k[b + 1], h // g][vis])
        bound[n] = (2.0 ** -4 + 2.0 ** -12) * pv + sub + 2.0 ** -9 * np.abs(o)
        sigma[n] = 2.0 ** -4 / np.sqrt(3.0) * np.sqrt((P ** 2) @ (va ** 2))
    if rows is None:
        bound = bound.reshape(tq, Hq, d)
        sigma = sigma.reshape(tq, Hq, d)
    return bound, sigma
