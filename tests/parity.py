"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle, compare.

Tolerances (bf16 inputs, fp32 accumulation, bf16 P into the second contraction, bf16 O):
O max abs error <= 2e-2 and mean abs error <= 2e-3, LSE max abs error <= 1e-3.  Rows the
oracle reports as empty (no visible key) must come back as O == 0 and LSE == -inf exactly.
"""
import numpy as np
import torch

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_* [..., d]; lse_* matching leading shape.  GPU values as torch (any device)."""
    o_gpu = o_gpu.detach().float().cpu().numpy().astype(np.float64)
    lse_gpu = lse_gpu.detach().float().cpu().numpy().astype(np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    lse_ref = np.asarray(lse_ref, np.float64)
    assert o_gpu.shape == o_ref.shape and lse_gpu.shape == lse_ref.shape, what
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), finite), f"{what}: empty-row pattern differs"
    assert np.all(lse_gpu[~finite] == -np.inf), what
    assert np.all(o_gpu[~finite] == 0.0), f"{what}: empty rows must be zero"
    stats = {}
    if finite.any():
        oe = np.abs(o_gpu[finite] - o_ref[finite])
        le = np.abs(lse_gpu[finite] - lse_ref[finite])
        stats = dict(o_max=float(oe.max()), o_mean=float(oe.mean()), lse_max=float(le.max()))
        assert np.all(np.isfinite(o_gpu[finite])), f"{what}: non-finite output"
        assert stats["o_max"] <= O_MAX, f"{what}: O max err {stats}"
        assert stats["o_mean"] <= O_MEAN, f"{what}: O mean err {stats}"
        assert stats["lse_max"] <= LSE_MAX, f"{what}: LSE max err {stats}"
    return stats


def to_dev(case, device="cuda"):
    import dataclasses
    out = {}
    for f in dataclasses.fields(case):
        v = getattr(case, f.name)
        out[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
    return out


def sample_rows(case, per_head, seed):
    """Seeded (token, head) rows plus the boundary rows of every sequence and of the tiles."""
    g = torch.Generator().manual_seed(seed)
    cu = case.cu_seqlens_q.tolist()
    total = cu[-1]
    Hq = case.q.shape[1]
    toks = set()
    for b in range(len(cu) - 1):
        s, e = cu[b], cu[b + 1]
        L = e - s
        for i in (0, 1, 15, 16, 127, 128, 129, 255, 256, L - 2, L - 1):
            if 0 <= i < L:
                toks.add(s + i)
        wl = case.window_left
        if wl >= 0:
            for i in (wl - 1, wl, wl + 1, wl + 128):
                if 0 <= i < L:
                    toks.add(s + i)
    base = sorted(toks)
    rows_t, rows_h = [], []
    for h in range(Hq):
        pick = torch.randint(0, total, (per_head,), generator=g).tolist()
        for t in sorted(set(pick) | set(base)):
            rows_t.append(t)
            rows_h.append(h)
    return np.array(rows_t, np.int64), np.array(rows_h, np.int32)
