"""CPU checks of libattn.so: it loads, exports every symbol include/attn.h declares, rejects bad
arguments before touching a device, and its integer tile logic matches brute force over the
oracle's visibility rule (bit-exact)."""
import ctypes
import os
import re

import pytest
import torch

from exact_attention_70_gb300 import build as attn_build
from exact_attention_70_gb300 import binding
from oracle import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    attn_build.build()
    return binding.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "attn_fwd" in names and "attn_decode_kvcache" in names
    for n in names:
        assert hasattr(lib, n), n
        assert ctypes.cast(getattr(lib, n), ctypes.c_void_p).value


def test_status_strings(lib):
    for code in range(-6, 1):
        assert lib.attn_status_string(code)


def test_workspace_sizes(lib):
    # tile list: header + prefix + (pairs of 128-row tiles) x Hkv int4 entries
    b = binding.attn_fwd_workspace_bytes(4, 4096, 16, 16)
    assert b == 256 + 32 + 4 * 16 * 16 * 16
    assert binding.attn_fwd_workspace_bytes(1, 100, 6, 4) == 0  # Hq % Hkv != 0
    # decode partials: O fp32 + LSE fp32 per (b, h, split), 256-byte aligned pieces
    assert binding.attn_decode_workspace_bytes(64, 32, 128, 1) == 0
    assert binding.attn_decode_workspace_bytes(64, 32, 128, 16) == 64 * 32 * 16 * 128 * 4 + 64 * 32 * 16 * 4
    assert binding.attn_decode_workspace_bytes(64, 32, 128, 0) == binding.attn_decode_workspace_bytes(64, 32, 128, 16)


def test_num_splits_heuristic(lib):
    # long sequences: one split per ~2048 keys, capped at 16
    assert binding.attn_decode_num_splits(64, 32, 8, 128, 256, 152) == 16
    # short sequences, few groups: enough splits for several waves of CTAs
    s = binding.attn_decode_num_splits(1, 8, 8, 4, 256, 152)
    assert 1 <= s <= 16 and s * 8 >= 16
    assert binding.attn_decode_num_splits(2, 4, 4, 1, 16, 152) >= 1


def test_bad_arguments_are_rejected_before_any_launch(lib):
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: every call below fails validation first
    f = lib.attn_fwd
    args = dict(q=fake, k=fake, v=fake, out=fake, lse=fake, cuq=fake, cuk=fake, batch=1,
                tq=16, tk=16, mq=16, mk=16, hq=4, hkv=2, d=128, scale=0.1, causal=1, wl=-1,
                wr=-1, ws=fake, wsb=1 << 20, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return f(*a.values())

    assert call(hq=6, hkv=4) == -1            # Hq % Hkv
    assert call(d=96) == -2                   # head_dim not built
    assert call(scale=0.0) == -1
    assert call(scale=float("nan")) == -1
    assert call(wl=-2) == -1
    assert call(q=None) == -1
    assert call(q=P(4098)) == -1              # misaligned
    assert call(ws=None) == -3
    assert call(wsb=16) == -3
    assert call(batch=0) == 0                 # nothing to do
    dec = lib.attn_decode_kvcache
    base = [fake, fake, fake, fake, fake, 256, 0, fake, fake, 2, 8, 2, 128, 4, 8, 0.1, fake,
            1 << 20, None]

    def dcall(i, v):
        a = list(base)
        a[i] = v
        return dec(*a)

    assert dcall(5, 48) == -2                 # page size neither divides nor is a multiple of 64
    assert dcall(5, 8) == -2                  # not a multiple of 16
    assert dcall(6, 65) == -1                 # num_splits out of range
    assert dcall(12, 80) == -2                # head_dim
    assert dcall(10, 3) == -1                 # Hq % Hkv
    assert dcall(0, None) == -1
    assert dcall(9, 0) == 0                   # batch 0


# ---- tile logic vs brute force over the oracle's visibility rule -------------------------

def brute_blocks(i_min, i_max, Lq, Lk, bn, causal, wl, wr):
    need, masked = [], []
    nblk = (Lk + bn - 1) // bn
    for j in range(nblk):
        vis = [oracle.allowed(i, kk, Lq, Lk, causal, wl, wr)
               for i in range(i_min, i_max + 1) for kk in range(j * bn, j * bn + bn)]
        if any(vis):
            need.append(j)
            masked.append(not all(vis))
    return need, masked


@pytest.mark.parametrize("seed", range(6))
def test_block_range_and_mask_match_brute_force(lib, seed):
    g = torch.Generator().manual_seed(seed)
    bn = [4, 8, 16][seed % 3]
    for _ in range(120):
        Lq = int(torch.randint(1, 60, (1,), generator=g))
        Lk = int(torch.randint(0, 70, (1,), generator=g))
        causal = bool(torch.randint(0, 2, (1,), generator=g))
        wl = int(torch.randint(-1, 20, (1,), generator=g))
        wr = int(torch.randint(-1, 20, (1,), generator=g))
        i_min = int(torch.randint(0, Lq, (1,), generator=g))
        i_max = int(torch.randint(i_min, Lq, (1,), generator=g))
        need, masked = brute_blocks(i_min, i_max, Lq, Lk, bn, causal, wl, wr)
        lo, hi = binding.attn_kv_block_range(i_min, i_max, Lq, Lk, bn, causal, wl, wr)
        assert list(range(lo, hi)) == need, (Lq, Lk, causal, wl, wr, i_min, i_max)
        got = [binding.attn_kv_block_masked(j, i_min, i_max, Lq, Lk, bn, causal, wl, wr)
               for j in range(lo, hi)]
        assert got == masked, (Lq, Lk, causal, wl, wr, i_min, i_max)


def test_block_figure_from_the_library(golden):
    ex = golden["block_masks"]
    B, n = 4, 8
    for key, wl in (("causal", -1), ("causal_window", 2 * B)):
        rows = []
        for qb in range(n):
            lo, hi = binding.attn_kv_block_range(qb * B, qb * B + B - 1, n * B, n * B, B, True,
                                                 wl, -1)
            row = ""
            for kb in range(n):
                if not lo <= kb < hi:
                    row += "."
                elif not binding.attn_kv_block_masked(kb, qb * B, qb * B + B - 1, n * B, n * B,
                                                      B, True, wl, -1):
                    row += "F"
                else:
                    row += "D" if kb == qb else "E"
            rows.append(row)
        assert rows == ex[key]


def test_kvcache_arguments_are_rejected_before_any_launch(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    f = lib.attn_fwd_kvcache
    args = dict(q=fake, kn=fake, vn=fake, kc=fake, vc=fake, sl=fake, bt=fake, cuq=fake,
                cos=None, sin=None, rot=0, rows=0, inter=0, out=fake, lse=fake, batch=2, tq=16,
                mq=8, hq=8, hkv=2, d=128, ps=64, mp=4, np_=16, scale=0.1, causal=1, wl=-1, wr=-1,
                ws=fake, wsb=1 << 22, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return f(*a.values())

    assert call(ps=48) == -2                  # page neither divides 128 nor is a multiple
    assert call(ps=8) == -2                   # not a multiple of 16
    assert call(ps=192) == -2                 # multiple of 64 but not of 128
    assert call(rot=24, cos=fake, sin=fake, rows=10) == -2   # rotary_dim not a multiple of 16
    assert call(rot=64) == -1                 # rotary without tables
    assert call(d=96) == -2
    assert call(hq=6, hkv=4) == -1
    assert call(kn=None) == -1
    assert call(q=P(4098)) == -1              # misaligned
    assert call(ws=None) == -3
    assert call(batch=0) == 0
    # workspace: the work list, plus the rotated q with rotary
    base = binding.attn_fwd_workspace_bytes(2, 8, 8, 2)
    assert lib.attn_fwd_kvcache_workspace_bytes(2, 16, 8, 8, 2, 128, 0) == (base + 255) // 256 * 256
    assert lib.attn_fwd_kvcache_workspace_bytes(2, 16, 8, 8, 2, 128, 64) == \
        (base + 255) // 256 * 256 + 16 * 8 * 128 * 2


def test_bwd_arguments_are_rejected_before_any_launch(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    f = lib.attn_bwd
    args = [fake] * 11 + [1, 16, 16, 16, 16, 4, 2, 128, 0.1, 1, -1, -1, fake, 1 << 20, None]

    def call(i, v):
        a = list(args)
        a[i] = v
        return f(*a)

    assert call(17, 3) == -1       # Hq % Hkv
    assert call(18, 96) == -2      # head_dim
    assert call(19, 0.0) == -1     # scale
    assert call(0, None) == -1     # q
    assert call(4, P(4100)) == -1  # misaligned dout
    assert call(23, None) == -3    # workspace
    assert call(11, 0) == 0        # batch 0
    # one side without rows: the other side's gradients must be given (and are zeroed on the
    # device), the empty side's tensors may be NULL
    a = list(args)
    a[12], a[7] = 0, None          # total_q = 0 and no dk
    assert f(*a) == -1
    a = list(args)
    a[13], a[6] = 0, P(4100)       # total_k = 0 and a misaligned dq
    assert f(*a) == -1
    assert lib.attn_bwd_workspace_bytes(1000, 8) == (32000 + 255) // 256 * 256
    assert lib.attn_bwd_workspace_bytes(1001, 8) == (32032 + 255) // 256 * 256


def test_modifier_arguments_are_checked(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    f = lib.attn_fwd_mods
    base = [fake] * 7 + [1, 16, 16, 16, 16, 4, 2, 128, 0.1, 1, -1, -1, 0.0, None, fake, 1 << 20, None]

    def call(i, v):
        a = list(base)
        a[i] = v
        return f(*a)

    assert call(19, -1.0) == -1              # negative softcap
    assert call(19, float("nan")) == -1
    assert call(19, 1e-7) == -1              # below 2^-20
    assert call(19, 2e30) == -1              # above 1e30
    assert call(15, 1e-39) == -1             # subnormal scale (its reciprocal overflows)
    sc = lib.attn_selftest_softcap
    assert sc(fake, fake, 3, 0.1, 30.0, None) == -1   # odd n
    assert sc(fake, fake, 2, 0.1, 1e-7, None) == -1   # softcap out of range
    assert sc(fake, P(4100), 2, 0.1, 30.0, None) == -1  # misaligned out
    assert sc(fake, fake, 0, 0.1, 30.0, None) == 0    # nothing to do
    assert call(20, P(4098)) == -1           # misaligned slopes
    assert call(7, 0) == 0                   # batch 0


def test_fp8_arguments_are_checked(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    f = lib.attn_fwd_fp8
    # q8 k8 v8t q_scale k_scale v_scale out lse cu_q cu_k | batch total_q total_k max_q max_k
    # Hq Hkv d key_blocks | scale causal wl wr stream
    base = [fake] * 10 + [1, 16, 16, 16, 16, 4, 2, 128, 1, 0.1, 1, -1, -1, None]

    def call(i, v):
        a = list(base)
        a[i] = v
        return f(*a)

    assert call(17, 64) == -2               # head_dim 64 is not built for FP8
    assert call(15, 5) == -1                # Hq % Hkv != 0
    assert call(18, 0) == -1                # no key blocks
    assert call(18, -1) == -1
    assert call(19, -0.1) == -1             # scale
    assert call(0, None) == -1              # null q8
    assert call(1, P(4097)) == -1           # misaligned k8
    assert call(3, P(4098)) == -1           # misaligned q_scale
    assert call(21, -2) == -1               # window
    assert call(10, 0) == 0                 # batch 0


def test_quantize_arguments_are_checked(lib):
    P = ctypes.c_void_p
    fake = P(4096)
    f = lib.attn_quantize_fp8
    # q k v cu_k | batch total_q total_k max_k Hq Hkv d key_blocks | signs q8 qs k8 ks v8t vs stream
    base = [fake] * 4 + [1, 16, 16, 16, 4, 2, 128, 2] + [None, fake, fake, fake, fake, fake, fake, None]

    def call(i, v):
        a = list(base)
        a[i] = v
        return f(*a)

    assert call(10, 64) == -2               # head_dim 64 is not built for FP8
    assert call(11, -1) == -1               # key_blocks
    assert call(8, 0) == -1                 # Hq
    assert call(13, None) == -1             # null q8
    assert call(12, P(4098)) == -1          # misaligned signs
    assert call(14, P(4097)) == -1          # misaligned q_scale


def test_bounds_checking_build_exports_every_declared_symbol():
    """The debugging library (kernels compiled with -DATTN_CHECK_BOUNDS) builds and has the
    same interface as the regular one."""
    path = attn_build.build(check_bounds=True)
    assert path != attn_build.LIB
    checked = ctypes.CDLL(path)
    for n in declared_functions():
        assert ctypes.cast(getattr(checked, n), ctypes.c_void_p).value, n
