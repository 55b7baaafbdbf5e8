"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws numbers.  Both the CUDA path and the
oracle receive exactly the tensors built here (bf16 bits drawn on the host), so they see
identical inputs.

Recipes (the shapes of the pages' workloads; there is no dataset):
  * Q, K, V entries are iid N(0, 1) drawn in fp32 and rounded to bf16;
  * sequence lengths are drawn uniformly with ``torch.randint`` from a generator seeded with
    ``1000 + config id``;
  * the paged cache's physical pages are a ``torch.randperm`` of the pool, the pool holding
    exactly sum_b ceil(L_b / page_size) pages;
  * large tensors are drawn in fixed-size blocks, block ``i`` from its own generator seeded
    with ``seed * 1_000_003 + stream * 65_537 + i``, so a tensor's bits do not depend on how
    many threads drew it.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import torch

_BLOCK = 1 << 22


def randn_bf16(shape, seed: int, stream: int = 0) -> torch.Tensor:
    """iid N(0,1) rounded to bf16, on the host, reproducible for (shape, seed, stream)."""
    numel = math.prod(shape)
    out = torch.empty(numel, dtype=torch.bfloat16)
    nblk = (numel + _BLOCK - 1) // _BLOCK

    def fill(i):
        s, e = i * _BLOCK, min(numel, (i + 1) * _BLOCK)
        g = torch.Generator().manual_seed(seed * 1_000_003 + stream * 65_537 + i)
        out[s:e].copy_(torch.randn(e - s, generator=g, dtype=torch.float32))

    if nblk <= 2:
        for i in range(nblk):
            fill(i)
    else:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nblk)))
    return out.view(*shape)


@dataclass
class PrefillCase:
    """Packed varlen prefill inputs: q [total_q, Hq, d], k/v [total_k, Hkv, d]."""
    name: str
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    cu_seqlens_q: torch.Tensor
    cu_seqlens_k: torch.Tensor
    max_seqlen_q: int
    max_seqlen_k: int
    softmax_scale: float
    causal: bool
    window_left: int = -1
    window_right: int = -1
    meta: dict = field(default_factory=dict)

    @property
    def batch(self):
        return len(self.cu_seqlens_q) - 1


@dataclass
class DecodeCase:
    """Decode inputs: q [batch, Hq, d]; caches [num_pages, page_size, Hkv, d]."""
    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    cache_seqlens: torch.Tensor
    block_table: torch.Tensor
    page_size: int
    softmax_scale: float
    num_splits: int = 0
    meta: dict = field(default_factory=dict)


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def prefill_case(lengths_q, Hq, Hkv, d, causal, seed, lengths_k=None, window=(-1, -1),
                 scale=None, name="prefill") -> PrefillCase:
    lengths_k = list(lengths_q) if lengths_k is None else list(lengths_k)
    cu_q, cu_k = cu_from_lengths(lengths_q), cu_from_lengths(lengths_k)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    return PrefillCase(
        name=name,
        q=randn_bf16((tq, Hq, d), seed, 1),
        k=randn_bf16((tk, Hkv, d), seed, 2),
        v=randn_bf16((tk, Hkv, d), seed, 3),
        cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
        max_seqlen_q=max([0] + [int(x) for x in lengths_q]),
        max_seqlen_k=max([0] + [int(x) for x in lengths_k]),
        softmax_scale=d ** -0.5 if scale is None else scale, causal=bool(causal),
        window_left=window[0], window_right=window[1],
    )


def decode_case(lengths, Hq, Hkv, d, page_size, seed, max_pages=None, num_splits=0,
                scale=None, name="decode") -> DecodeCase:
    g = torch.Generator().manual_seed(seed)
    pages_per = [(int(n) + page_size - 1) // page_size for n in lengths]
    num_pages = max(1, sum(pages_per))
    max_pages = max([1] + pages_per) if max_pages is None else max_pages
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    bt = torch.zeros((len(lengths), max_pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[off:off + n]
        off += n
    return DecodeCase(
        name=name,
        q=randn_bf16((len(lengths), Hq, d), seed, 1),
        k_cache=randn_bf16((num_pages, page_size, Hkv, d), seed, 2),
        v_cache=randn_bf16((num_pages, page_size, Hkv, d), seed, 3),
        cache_seqlens=torch.tensor([int(n) for n in lengths], dtype=torch.int32),
        block_table=bt, page_size=page_size,
        softmax_scale=d ** -0.5 if scale is None else scale, num_splits=num_splits,
    )


@dataclass
class KvcacheCase:
    """Chunked prefill against a paged cache (new tokens appended in the same call)."""
    name: str
    q: torch.Tensor            # [total_q, Hq, d] bf16
    k_new: torch.Tensor        # [total_q, Hkv, d] bf16
    v_new: torch.Tensor
    k_cache: torch.Tensor      # [num_pages, page_size, Hkv, d] bf16 (prefix + unused slots)
    v_cache: torch.Tensor
    cache_seqlens: torch.Tensor  # [batch] int32, cached tokens before the call
    block_table: torch.Tensor    # [batch, max_pages] int32
    cu_seqlens_q: torch.Tensor   # [batch + 1] int32
    max_seqlen_q: int
    page_size: int
    softmax_scale: float
    causal: bool
    window_left: int
    window_right: int
    rotary_cos: torch.Tensor = None   # [rows, rot / 2] fp32
    rotary_sin: torch.Tensor = None
    rotary_interleaved: bool = False


def rotary_tables(rows, rot_dim, base=10000.0):
    """Standard rotary tables: row p, plane i holds the angle p * base^(-2i / rot_dim)."""
    inv = base ** (-torch.arange(0, rot_dim, 2, dtype=torch.float64) / rot_dim)
    ang = torch.arange(rows, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cos(ang).float(), torch.sin(ang).float()


def kvcache_case(q_lens, ctx_lens, Hq, Hkv, d, page_size, seed, rotary_dim=0,
                 rotary_interleaved=False, causal=True, window=(-1, -1), spare_pages=2,
                 poison_unused=False, scale=None, name="kvcache") -> KvcacheCase:
    """Pages for ctx + q_len tokens per sequence, in a seeded random order; the cache's other
    slots hold random values (or NaN with poison_unused, which must never reach a result)."""
    g = torch.Generator().manual_seed(seed)
    lens = [int(c) + int(n) for c, n in zip(ctx_lens, q_lens)]
    pages_per = [max(1, (L + page_size - 1) // page_size) for L in lens]
    num_pages = sum(pages_per) + spare_pages
    max_pages = max(pages_per)
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    bt = torch.zeros((len(lens), max_pages), dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[off:off + n]
        off += n
    total_q = sum(int(n) for n in q_lens)
    k_cache = randn_bf16((num_pages, page_size, Hkv, d), seed, 4)
    v_cache = randn_bf16((num_pages, page_size, Hkv, d), seed, 5)
    if poison_unused:
        keep = torch.zeros((num_pages, page_size), dtype=torch.bool)
        for b, c in enumerate(ctx_lens):
            for j in range(int(c)):
                keep[bt[b, j // page_size], j % page_size] = True
        k_cache[~keep] = float("nan")
        v_cache[~keep] = float("nan")
    cos = sin = None
    if rotary_dim:
        cos, sin = rotary_tables(max(lens) + 1, rotary_dim)
    return KvcacheCase(
        name=name, q=randn_bf16((total_q, Hq, d), seed, 1),
        k_new=randn_bf16((total_q, Hkv, d), seed, 2), v_new=randn_bf16((total_q, Hkv, d), seed, 3),
        k_cache=k_cache, v_cache=v_cache,
        cache_seqlens=torch.tensor([int(c) for c in ctx_lens], dtype=torch.int32),
        block_table=bt, cu_seqlens_q=cu_from_lengths(q_lens), max_seqlen_q=max(int(n) for n in q_lens),
        page_size=page_size, softmax_scale=d ** -0.5 if scale is None else scale,
        causal=causal, window_left=window[0], window_right=window[1],
        rotary_cos=cos, rotary_sin=sin, rotary_interleaved=rotary_interleaved)


# ---- the five workload configurations ------------------------------------------------

CONFIG_NAMES = {
    1: "single-head non-causal B=1 H=1 N=128 d=64",
    2: "causal prefill B=4 Hq=Hkv=16 N=4096 d=128",
    3: "varlen GQA causal prefill 8 seqs L~U[512,8192] Hq=32 Hkv=4 d=128",
    4: "paged decode batch=64 L~U[1024,32768] page=256 Hq=32 Hkv=8 d=128",
    5: "sliding-window causal prefill B=1 N=32768 Hq=32 Hkv=8 d=128 window=(4096,0)",
}


def config_case(cfg: int):
    seed = 1000 + cfg
    if cfg == 1:
        c = prefill_case([128], 1, 1, 64, False, seed, name="cfg1")
    elif cfg == 2:
        c = prefill_case([4096] * 4, 16, 16, 128, True, seed, name="cfg2")
    elif cfg == 3:
        g = torch.Generator().manual_seed(seed)
        lengths = torch.randint(512, 8192 + 1, (8,), generator=g).tolist()
        c = prefill_case(lengths, 32, 4, 128, True, seed, name="cfg3")
    elif cfg == 4:
        g = torch.Generator().manual_seed(seed)
        lengths = torch.randint(1024, 32768 + 1, (64,), generator=g).tolist()
        c = decode_case(lengths, 32, 8, 128, 256, seed + 7, max_pages=128, name="cfg4")
    elif cfg == 5:
        c = prefill_case([32768], 32, 8, 128, True, seed, window=(4096, 0), name="cfg5")
    else:
        raise ValueError(cfg)
    c.meta["config"] = CONFIG_NAMES[cfg]
    return c


CHUNKED_NAME = ("chunked prefill over a paged cache: 8 seqs, ctx~U[2048,16384] cached + 2048 new "
                "tokens each, Hq=32 Hkv=8 d=128 page=256 rotary=128, causal")


def chunked_case() -> KvcacheCase:
    g = torch.Generator().manual_seed(1100)
    ctx = torch.randint(2048, 16384 + 1, (8,), generator=g).tolist()
    return kvcache_case([2048] * 8, ctx, 32, 8, 128, 256, seed=1101, rotary_dim=128,
                        name="chunked")


# ---- FP8 (e4m3) inputs -------------------------------------------------------------------
#
# Recipe: e4m3 bit patterns drawn directly (no rounding of values happens here): the sign bit
# and the 3 mantissa bits uniform, the 4-bit exponent field uniform in [4, 10], i.e. magnitudes
# log-uniform over [2^-3, 15]; the NaN pattern never occurs.  Scales are uniform in
# [0.15, 0.25] (decoded values then have an RMS near 1).  V^T columns past a sequence's keys
# (the layout's padding) are code 0 (value 0).  The full-range variant draws the exponent field
# uniformly from all 16 values, so zeros, subnormals and +-448 occur (the NaN pattern
# S.1111.111 is replaced by S.1111.110 = +-448), with scales of 2^-6 that keep the logits in
# the range a softmax can resolve.

def e4m3_codes(shape, seed: int, stream: int = 0, full_range: bool = False) -> torch.Tensor:
    """Random e4m3 bit patterns (uint8), reproducible for (shape, seed, stream)."""
    numel = math.prod(shape)
    out = torch.empty(numel, dtype=torch.uint8)
    nblk = (numel + _BLOCK - 1) // _BLOCK

    def fill(i):
        s, e = i * _BLOCK, min(numel, (i + 1) * _BLOCK)
        g = torch.Generator().manual_seed(seed * 1_000_003 + stream * 65_537 + i)
        bits = torch.randint(0, 1 << 30, (e - s,), generator=g, dtype=torch.int64)
        sign = (bits & 1) << 7
        man = (bits >> 1) & 7
        if full_range:
            exp = (bits >> 4) & 15
            man = torch.where((exp == 15) & (man == 7), torch.full_like(man, 6), man)
        else:
            exp = 4 + (bits >> 4) % 7
        out[s:e].copy_((sign | (exp << 3) | man).to(torch.uint8))

    if nblk <= 2:
        for i in range(nblk):
            fill(i)
    else:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nblk)))
    return out.view(*shape)


@dataclass
class Fp8Case:
    name: str
    q8: torch.Tensor        # uint8 [total_q, Hq, d]
    k8: torch.Tensor        # uint8 [total_k, Hkv, d]
    v8t: torch.Tensor       # uint8 [Hkv, d, 128 * key_blocks]
    q_scale: torch.Tensor   # fp32 [Hq, ceil(total_q / 128)]
    k_scale: torch.Tensor   # fp32 [Hkv, key_blocks]
    v_scale: torch.Tensor   # fp32 [batch, Hkv]
    cu_seqlens_q: torch.Tensor
    cu_seqlens_k: torch.Tensor
    max_seqlen_q: int
    max_seqlen_k: int
    softmax_scale: float
    causal: bool
    window_left: int = -1
    window_right: int = -1


def fp8_case(lengths_q, Hq, Hkv, d, causal, seed, lengths_k=None, window=(-1, -1), scale=None,
             name="fp8", full_range=False) -> Fp8Case:
    lengths_k = list(lengths_q) if lengths_k is None else list(lengths_k)
    cu_q, cu_k = cu_from_lengths(lengths_q), cu_from_lengths(lengths_k)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    blocks = [(int(n) + 127) // 128 for n in lengths_k]
    key_blocks = max(1, sum(blocks))
    v8t = e4m3_codes((Hkv, d, 128 * key_blocks), seed, 3, full_range)
    col = 0
    for n, nb in zip(lengths_k, blocks):   # zero the padding columns of each sequence
        v8t[:, :, col + int(n):col + 128 * nb] = 0
        col += 128 * nb
    v8t[:, :, col:] = 0
    g = torch.Generator().manual_seed(seed * 7 + 5)
    lo, span = (2.0 ** -6, 2.0 ** -7) if full_range else (0.15, 0.1)
    return Fp8Case(
        name=name,
        q8=e4m3_codes((tq, Hq, d), seed, 1, full_range),
        k8=e4m3_codes((tk, Hkv, d), seed, 2, full_range),
        v8t=v8t,
        q_scale=lo + span * torch.rand((Hq, (tq + 127) // 128), generator=g),
        k_scale=lo + span * torch.rand((Hkv, key_blocks), generator=g),
        v_scale=lo + span * torch.rand((len(lengths_q), Hkv), generator=g),
        cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
        max_seqlen_q=max([0] + [int(x) for x in lengths_q]),
        max_seqlen_k=max([0] + [int(x) for x in lengths_k]),
        softmax_scale=d ** -0.5 if scale is None else scale, causal=bool(causal),
        window_left=window[0], window_right=window[1],
    )


FP8_NAME = "FP8 e4m3 causal prefill B=4 Hq=Hkv=16 N=4096 d=128"


def fp8_bench_case() -> Fp8Case:
    """The causal prefill workload's shape with FP8 inputs."""
    return fp8_case([4096] * 4, 16, 16, 128, True, seed=1200, name="fp8")
