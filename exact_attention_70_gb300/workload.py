"""Algorithmic work of a workload, for the roofline figures the benchmark reports.

Prefill FLOPs count only what the method must do: 4 d FLOP per visible (query row, key) pair
and query head -- 2d for QK^T and 2d for PV ("Attention kernels:
FlashAttention and PagedAttention", section 二.2: 4 N^2 d for a full N x N head).  Skipped
(masked) tiles are not counted.

Decode bytes count what must cross HBM once: every visible K and V row of every kv head, plus
q, out, lse, cache_seqlens and the block_table entries that are read ("Attention kernels ...",
section 五.2: the KV cache is read once per generated token).  The split partials are
overhead and are not counted.
"""
from __future__ import annotations

import numpy as np


def visible_pairs(Lq: int, Lk: int, causal: bool, wl: int = -1, wr: int = -1) -> int:
    """Visible (query, key) pairs of one sequence and head under bottom-right alignment."""
    if Lq <= 0 or Lk <= 0:
        return 0
    i = np.arange(Lq, dtype=np.int64)
    p = i + (Lk - Lq)
    right = 0 if causal else wr
    hi = np.full(Lq, Lk - 1, np.int64) if right < 0 else np.minimum(Lk - 1, p + right)
    lo = np.zeros(Lq, np.int64) if wl < 0 else np.maximum(0, p - wl)
    return int(np.maximum(0, hi - lo + 1).sum())


def prefill_flops(lengths_q, lengths_k, Hq: int, d: int, causal: bool, wl=-1, wr=-1) -> int:
    pairs = sum(visible_pairs(int(a), int(b), causal, wl, wr) for a, b in zip(lengths_q, lengths_k))
    return 4 * d * Hq * pairs


def prefill_case_flops(case) -> int:
    cu_q = case.cu_seqlens_q.tolist()
    cu_k = case.cu_seqlens_k.tolist()
    lq = [cu_q[b + 1] - cu_q[b] for b in range(len(cu_q) - 1)]
    lk = [cu_k[b + 1] - cu_k[b] for b in range(len(cu_k) - 1)]
    return prefill_flops(lq, lk, case.q.shape[1], case.q.shape[2], case.causal,
                         case.window_left, case.window_right)


def prefill_case_bytes(case) -> int:
    """Compulsory HBM bytes of a prefill: Q, K, V read once, O and LSE written once."""
    tq, Hq, d = case.q.shape
    tk, Hkv, _ = case.k.shape
    return 2 * tq * Hq * d * 2 + 2 * tk * Hkv * d * 2 + tq * Hq * 4


def decode_case_bytes(case) -> int:
    batch, Hq, d = case.q.shape
    _, page_size, Hkv, _ = case.k_cache.shape
    lens = [int(x) for x in case.cache_seqlens.tolist()]
    kv = sum(lens) * Hkv * d * 2 * 2
    pages = sum((n + page_size - 1) // page_size for n in lens)
    return kv + 2 * batch * Hq * d * 2 + batch * Hq * 4 + batch * 4 + pages * 4


def decode_case_flops(case) -> int:
    batch, Hq, d = case.q.shape
    return 4 * d * Hq * int(case.cache_seqlens.sum())
