"""Python face of the fp64 attention oracle (``attn_oracle.c``).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this module.  It never imports the
CUDA package, and the CUDA package never imports it.

Every function takes host arrays (numpy, or CPU torch tensors which are viewed without a
copy of their bits) and returns fp64 numpy arrays.  bf16 inputs are passed as their raw
16-bit patterns and widened to fp64 exactly inside the C code.

Sources (page titles and sections):
  * "Attention kernels: FlashAttention and PagedAttention" (arganzheng.life),
    section 二 (standard attention, its byte and FLOP accounting), 四.3 (LSE),
    六.1 (block-table addressing), 六.3 (merge of split partials), 七 (varlen, causal,
    sliding window);
  * "04 · FA4 (CuTeDSL) and engineering interfaces" (llm-infra-atlas), sections 4-7
    (cu_seqlens, pack_gqa head mapping, paged KV, split-KV, bottom-right causal, window).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

F64, BF16 = 0, 1


class Counts(ctypes.Structure):
    _fields_ = [("flops", ctypes.c_longlong), ("s_elems", ctypes.c_longlong),
                ("p_elems", ctypes.c_longlong), ("qkvo_bytes", ctypes.c_longlong)]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, OpenMP, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, dbl, ll = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_longlong
            lib.oracle_allowed.restype = i32
            lib.oracle_allowed.argtypes = [ll, ll, ll, ll, i32, i32, i32]
            lib.oracle_attn_fwd.restype = i32
            lib.oracle_attn_fwd.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, dbl, i32,
                                            i32, i32, P, P, ll, P]
            lib.oracle_attn_fwd_rows.restype = i32
            lib.oracle_attn_fwd_rows.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, dbl,
                                                 i32, i32, i32, P, P, ll, P, P]
            lib.oracle_merge.restype = i32
            lib.oracle_merge.argtypes = [i32, i32, P, P, P, P, P]
            lib.oracle_decode.restype = i32
            lib.oracle_decode.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32,
                                          dbl, i32, P, P, ll, P, P]
            lib.oracle_tiled_traffic_bytes.restype = ll
            lib.oracle_tiled_traffic_bytes.argtypes = [ll, ll, ll]
            lib.oracle_num_threads.restype = i32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_attn_fwd_mods.restype = i32
            lib.oracle_attn_fwd_mods.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, dbl,
                                                 i32, i32, i32, dbl, P, P, P, ll, P, P]
            lib.oracle_attn_bwd.restype = i32
            lib.oracle_attn_bwd.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32, dbl, i32,
                                            i32, i32, P, P, P, P]
            lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
            lib.oracle_f64_to_bf16.argtypes = [dbl]
            lib.oracle_e4m3_to_f64.restype = dbl
            lib.oracle_e4m3_to_f64.argtypes = [i32]
            lib.oracle_f64_to_e4m3.restype = i32
            lib.oracle_f64_to_e4m3.argtypes = [dbl]
            lib.oracle_fp8_quantize_rows.restype = i32
            lib.oracle_fp8_quantize_rows.argtypes = [P, ll, i32, P, P, P]
            lib.oracle_kvcache_prefill.restype = i32
            lib.oracle_kvcache_prefill.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, i32, P,
                                                   i32, i32, i32, i32, P, P, i32, i32, i32, dbl,
                                                   i32, i32, i32, P, P, ll, P, P]
            _lib = lib
    return _lib


def _host(x, dtype_hint=None):
    """Return (contiguous numpy array, oracle dtype code) for an input tensor."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach()
            if x.device.type != "cpu":
                raise ValueError("the oracle takes host tensors only")
            x = x.contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float64:
                return x.numpy(), F64
            if x.dtype == torch.int32:
                return x.numpy(), None
            if x.dtype == torch.int64:
                return x.numpy(), None
            raise ValueError(f"unsupported dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.uint16:
        return x, BF16
    return x, None


def _i32(x):
    a, _ = _host(x)
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def allowed(i, j, Lq, Lk, causal, window_left=-1, window_right=-1) -> bool:
    """The visibility rule (bottom-right aligned causal / sliding window)."""
    return bool(_load().oracle_allowed(i, j, Lq, Lk, int(causal), window_left, window_right))


def attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale, causal=False,
             window_left=-1, window_right=-1, with_counts=False):
    """Standard attention over every row.  q [total_q, Hq, d]; k, v [total_k, Hkv, d].

    Returns (out [total_q, Hq, d] f64, lse [Hq, total_q] f64[, Counts]).
    """
    qa, dt = _host(q)
    ka, dk = _host(k)
    va, dv = _host(v)
    if not (dt == dk == dv) or dt is None:
        raise ValueError("q, k, v must share one dtype (bf16 or fp64)")
    total_q, Hq, d = qa.shape
    Hkv = ka.shape[1]
    cu_q, cu_k = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    batch = len(cu_q) - 1
    out = np.zeros((total_q, Hq, d), np.float64)
    lse = np.full((Hq, total_q), np.nan, np.float64)
    counts = Counts()
    rc = _load().oracle_attn_fwd(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(cu_q), _ptr(cu_k), batch,
                                 Hq, Hkv, d, float(softmax_scale), int(causal), window_left,
                                 window_right, _ptr(out), _ptr(lse), total_q,
                                 ctypes.byref(counts))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return (out, lse, counts) if with_counts else (out, lse)


def attn_fwd_rows(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale, row_tok, row_head,
                  causal=False, window_left=-1, window_right=-1):
    """Standard attention for chosen (packed token, query head) rows.

    Returns (out [n, d] f64, lse [n] f64).
    """
    qa, dt = _host(q)
    ka, _ = _host(k)
    va, _ = _host(v)
    total_q, Hq, d = qa.shape
    Hkv = ka.shape[1]
    cu_q, cu_k = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    tok = np.ascontiguousarray(np.asarray(row_tok), dtype=np.int64)
    head = np.ascontiguousarray(np.asarray(row_head), dtype=np.int32)
    n = len(tok)
    out = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_attn_fwd_rows(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(cu_q), _ptr(cu_k),
                                      len(cu_q) - 1, Hq, Hkv, d, float(softmax_scale),
                                      int(causal), window_left, window_right, _ptr(tok),
                                      _ptr(head), n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_rows rejected its arguments")
    return out, lse


def merge(m_i, l_i, o_i):
    """Merge split partials (m_i, l_i, O_i normalised) -> (O, LSE)."""
    m = np.ascontiguousarray(m_i, np.float64)
    l = np.ascontiguousarray(l_i, np.float64)
    o = np.ascontiguousarray(o_i, np.float64)
    S, d = o.shape
    out = np.zeros((d,), np.float64)
    lse = np.zeros((1,), np.float64)
    _load().oracle_merge(S, d, _ptr(m), _ptr(l), _ptr(o), _ptr(out), _ptr(lse))
    return out, float(lse[0])


def decode(q, k_cache, v_cache, cache_seqlens, block_table, softmax_scale, num_splits=0,
           rows_b=None, rows_h=None):
    """Decode (one query per sequence) over a paged cache.

    q [batch, Hq, d]; k_cache, v_cache [num_pages, page_size, Hkv, d];
    block_table [batch, max_pages] int32; cache_seqlens [batch] int32.
    Returns (out [n, d], lse [n]) for the chosen (b, h) rows, or ([batch, Hq, d], [batch, Hq]).
    """
    qa, dt = _host(q)
    ka, _ = _host(k_cache)
    va, _ = _host(v_cache)
    batch, Hq, d = qa.shape
    num_pages, page_size, Hkv, _ = ka.shape
    sl = _i32(cache_seqlens)
    bt = _i32(block_table)
    max_pages = bt.shape[1] if bt.ndim == 2 else 0
    if rows_b is None:
        n = batch * Hq
        rb = rh = None
    else:
        rb = np.ascontiguousarray(np.asarray(rows_b), dtype=np.int32)
        rh = np.ascontiguousarray(np.asarray(rows_h), dtype=np.int32)
        n = len(rb)
    out = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_decode(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(sl), _ptr(bt), max_pages,
                               page_size, num_pages, batch, Hq, Hkv, d, float(softmax_scale),
                               int(num_splits), _ptr(rb) if rb is not None else None,
                               _ptr(rh) if rh is not None else None, n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments (bad page index or length)")
    if rows_b is None:
        return out.reshape(batch, Hq, d), lse.reshape(batch, Hq)
    return out, lse


def attn_fwd_mods(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale, causal=False,
                  window_left=-1, window_right=-1, softcap=0.0, alibi_slopes=None,
                  rows_t=None, rows_h=None):
    """attn_fwd with the softcap and ALiBi score modifiers.

    Returns (out, lse): [n, d] and [n] for chosen (token, head) rows, or
    [total_q, Hq, d] and [Hq, total_q] for all rows.
    """
    qa, dt = _host(q)
    ka, _ = _host(k)
    va, _ = _host(v)
    total_q, Hq, d = qa.shape
    Hkv = ka.shape[1]
    cu_q, cu_k = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    sl = None if alibi_slopes is None else np.ascontiguousarray(np.asarray(alibi_slopes, dtype=np.float64))
    if rows_t is None:
        n, rt, rh = total_q * Hq, None, None
    else:
        rt = np.ascontiguousarray(np.asarray(rows_t), dtype=np.int64)
        rh = np.ascontiguousarray(np.asarray(rows_h), dtype=np.int32)
        n = len(rt)
    out = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_attn_fwd_mods(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(cu_q), _ptr(cu_k),
                                      len(cu_q) - 1, Hq, Hkv, d, float(softmax_scale), int(causal),
                                      window_left, window_right, float(softcap),
                                      _ptr(sl) if sl is not None else None,
                                      _ptr(rt) if rt is not None else None,
                                      _ptr(rh) if rh is not None else None, n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_fwd_mods rejected its arguments")
    if rows_t is None:
        return out.reshape(total_q, Hq, d), lse.reshape(total_q, Hq).T.copy()
    return out, lse


def attn_bwd(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, softmax_scale, causal=False,
             window_left=-1, window_right=-1):
    """Gradients of sum(O * dout) for attn_fwd's attention.

    Returns (dq [total_q, Hq, d], dk [total_k, Hkv, d], dv [total_k, Hkv, d],
    D [Hq, total_q] = rowsum(dout * O)), all fp64.
    """
    qa, dt = _host(q)
    ka, _ = _host(k)
    va, _ = _host(v)
    da, _ = _host(dout)
    total_q, Hq, d = qa.shape
    total_k, Hkv = ka.shape[0], ka.shape[1]
    cu_q, cu_k = _i32(cu_seqlens_q), _i32(cu_seqlens_k)
    dq = np.zeros((total_q, Hq, d), np.float64)
    dk = np.zeros((total_k, Hkv, d), np.float64)
    dv = np.zeros((total_k, Hkv, d), np.float64)
    D = np.zeros((Hq, total_q), np.float64)
    rc = _load().oracle_attn_bwd(_ptr(qa), _ptr(ka), _ptr(va), _ptr(da), dt, _ptr(cu_q),
                                 _ptr(cu_k), len(cu_q) - 1, Hq, Hkv, d, float(softmax_scale),
                                 int(causal), window_left, window_right, _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(D))
    if rc != 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    return dq, dk, dv, D


def f64_to_bf16_bits(x: float) -> int:
    """bf16 bit pattern of x rounded to nearest, ties to even (directly from fp64)."""
    return int(_load().oracle_f64_to_bf16(float(x)))


def kvcache_prefill(q, k_new, v_new, k_cache, v_cache, cache_seqlens, block_table,
                    cu_seqlens_q, softmax_scale, causal=True, window_left=-1, window_right=-1,
                    rotary_cos=None, rotary_sin=None, rotary_interleaved=False,
                    rows_t=None, rows_h=None):
    """Chunked prefill against a paged cache, with the new k, v appended (and rotated).

    q [total_q, Hq, d]; k_new, v_new [total_q, Hkv, d]; k_cache, v_cache
    [num_pages, page_size, Hkv, d]; cache_seqlens [batch] = cached tokens before this step;
    block_table [batch, max_pages]; rotary_cos / rotary_sin [rows, rot_dim / 2] or None.
    The caches are not modified: updated copies are returned.
    Returns (out, lse, k_cache_new, v_cache_new) with out [n, d], lse [n] for the chosen
    (token, head) rows, or out [total_q, Hq, d], lse [Hq, total_q] for all rows.
    """
    qa, dt = _host(q)
    kn, _ = _host(k_new)
    vn, _ = _host(v_new)
    kc, _ = _host(k_cache)
    vc, _ = _host(v_cache)
    kc, vc = kc.copy(), vc.copy()
    total_q, Hq, d = qa.shape
    num_pages, page_size, Hkv, _ = kc.shape
    sl = _i32(cache_seqlens)
    bt = _i32(block_table)
    cu = _i32(cu_seqlens_q)
    batch = len(cu) - 1
    if rotary_cos is not None:
        rc_ = np.ascontiguousarray(np.asarray(rotary_cos, dtype=np.float64))
        rs_ = np.ascontiguousarray(np.asarray(rotary_sin, dtype=np.float64))
        rot_rows, rot_dim = rc_.shape[0], 2 * rc_.shape[1]
    else:
        rc_ = rs_ = None
        rot_rows = rot_dim = 0
    if rows_t is None:
        n = total_q * Hq
        rt = rh = None
    else:
        rt = np.ascontiguousarray(np.asarray(rows_t), dtype=np.int64)
        rh = np.ascontiguousarray(np.asarray(rows_h), dtype=np.int32)
        n = len(rt)
    out = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_kvcache_prefill(
        _ptr(qa), _ptr(kn), _ptr(vn), dt, _ptr(kc), _ptr(vc), _ptr(sl), _ptr(bt), bt.shape[1],
        page_size, num_pages, _ptr(cu), batch, Hq, Hkv, d,
        _ptr(rc_) if rc_ is not None else None, _ptr(rs_) if rs_ is not None else None,
        rot_dim, rot_rows, int(rotary_interleaved), float(softmax_scale), int(causal),
        window_left, window_right, _ptr(rt) if rt is not None else None,
        _ptr(rh) if rh is not None else None, n, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_kvcache_prefill rejected its arguments")
    if rows_t is None:
        out = out.reshape(total_q, Hq, d)
        lse = lse.reshape(total_q, Hq).T.copy()
    return out, lse, kc, vc


def tiled_traffic_bytes(N, d, Br) -> int:
    return int(_load().oracle_tiled_traffic_bytes(N, d, Br))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ---- FP8 (e4m3) forward ------------------------------------------------------------------
#
# "Attention kernels: FlashAttention and PagedAttention", section 四.2 (FlashAttention-3): Q, K
# and V go to the 8-bit MMA as e4m3 with block-wise scales, and V is re-laid out so that the
# PV product reads it key-major.  The oracle decodes the codes (the e4m3 definition above),
# applies the scales and runs the plain fp64 attention on the values.  The FP8 kernel rounds P
# to e4m3 before the second product, an approximation of that result whose per-element error is
# at most 2^-4 sum_j P_j |v_j| (keys in e4m3's normal range) plus a subnormal term and the bf16
# rounding of O.
#
# Scale and layout reading (the page fixes neither):
#   q_scale [Hq, ceil(total_q / 128)]   one scale per 128 consecutive packed query tokens;
#   k_scale [Hkv, nkb]                  one scale per 128-key block of a sequence
#                                       (block kb0[b] + (t - k0) // 128);
#   v8t     [Hkv, d, 128 * nkb]         V transposed, key t of sequence b in column
#                                       128 * kb0[b] + (t - k0); the rest is padding;
#   v_scale [batch, Hkv]                one scale per (sequence, kv head);
# with kb0 the exclusive prefix sum of ceil(Lk_b / 128) and nkb >= kb0[batch].

def e4m3_to_f64(codes):
    """Decode e4m3 codes (any integer array) to fp64."""
    lut = np.array([_load().oracle_e4m3_to_f64(c) for c in range(256)], np.float64)
    return lut[np.asarray(codes, dtype=np.int64) & 0xFF]


def f64_to_e4m3(x) -> int:
    """Nearest e4m3 code of x (ties to even, saturating at 448)."""
    return int(_load().oracle_f64_to_e4m3(float(x)))


def key_block_offsets(cu_seqlens_k):
    """kb0: exclusive prefix sum of ceil(Lk_b / 128) (length batch + 1)."""
    cu = _i32(cu_seqlens_k).astype(np.int64)
    nb = (cu[1:] - cu[:-1] + 127) // 128
    return np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)


def fp8_dequantize(q8, k8, v8t, q_scale, k_scale, v_scale, cu_seqlens_k):
    """fp64 Q [total_q, Hq, d], K, V [total_k, Hkv, d] from the FP8 inputs and their scales."""
    def arr(x):
        try:
            import torch
            if isinstance(x, torch.Tensor):
                x = x.detach().cpu()
                if x.dtype == torch.uint8:
                    return x.numpy()
                return x.double().numpy()
        except ImportError:  # pragma: no cover
            pass
        return np.asarray(x)
    q8, k8, v8t = arr(q8), arr(k8), arr(v8t)
    qs, ks, vs = (arr(x).astype(np.float64) for x in (q_scale, k_scale, v_scale))
    total_q, Hq, d = q8.shape
    total_k, Hkv, _ = k8.shape
    cu = _i32(cu_seqlens_k).astype(np.int64)
    kb0 = key_block_offsets(cu)
    q = e4m3_to_f64(q8) * qs.T[np.arange(total_q) // 128][:, :, None]
    k = e4m3_to_f64(k8)
    v = np.zeros((total_k, Hkv, d), np.float64)
    vt = e4m3_to_f64(v8t)
    for b in range(len(cu) - 1):
        k0, k1 = int(cu[b]), int(cu[b + 1])
        if k1 == k0:
            continue
        t = np.arange(k0, k1)
        blk = kb0[b] + (t - k0) // 128
        k[k0:k1] *= ks.T[blk][:, :, None]
        cols = 128 * kb0[b] + (t - k0)
        v[k0:k1] = vt[:, :, cols].transpose(2, 0, 1) * vs[b][None, :, None]
    return q, k, v


def fp8_attn_fwd(q8, k8, v8t, q_scale, k_scale, v_scale, cu_seqlens_q, cu_seqlens_k,
                 softmax_scale, causal=False, window_left=-1, window_right=-1, rows=None):
    """Attention on the dequantized FP8 inputs: every row (out [total_q, Hq, d], lse [Hq,
    total_q]) or, with rows = (tok, head), the chosen rows (out [n, d], lse [n])."""
    q, k, v = fp8_dequantize(q8, k8, v8t, q_scale, k_scale, v_scale, cu_seqlens_k)
    if rows is None:
        return attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale, causal,
                        window_left, window_right)
    return attn_fwd_rows(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale, rows[0], rows[1],
                         causal, window_left, window_right)


def fp8_quantize_rows(rows_bf16_bits, signs=None):
    """One block: rows [n, d] of bf16 bits (uint16) -> (codes uint8 [n, d], scale float)."""
    a = np.ascontiguousarray(rows_bf16_bits, dtype=np.uint16)
    n, d = a.shape
    codes = np.zeros((n, d), np.uint8)
    sc = np.zeros((1,), np.float32)
    sg = None if signs is None else np.ascontiguousarray(signs, dtype=np.float32)
    rc = _load().oracle_fp8_quantize_rows(_ptr(a), n, d, None if sg is None else _ptr(sg),
                                          _ptr(codes), _ptr(sc))
    if rc != 0:
        raise ValueError("oracle_fp8_quantize_rows rejected its arguments")
    return codes, float(sc[0])


def fp8_quantize(q, k, v, cu_seqlens_k, signs=None, key_blocks=None):
    """bf16 Q, K, V -> the FP8 inputs of fp8_attn_fwd, block by block:
    q8, q_scale (128 packed tokens per block and head; Q rotated when signs is given),
    k8, k_scale (128 keys of a sequence per block and kv head; K rotated likewise),
    v8t, v_scale (V transposed into whole 128-key blocks per sequence, one scale per
    (sequence, kv head); columns past a sequence's keys are code 0)."""
    import torch
    qa, _ = _host(q)
    ka, _ = _host(k)
    va, _ = _host(v)
    total_q, Hq, d = qa.shape
    total_k, Hkv, _ = ka.shape
    cu = _i32(cu_seqlens_k).astype(np.int64)
    batch = len(cu) - 1
    kb0 = key_block_offsets(cu)
    nkb = int(kb0[-1]) if key_blocks is None else int(key_blocks)
    nqb = (total_q + 127) // 128
    q8 = np.zeros((total_q, Hq, d), np.uint8)
    qs = np.zeros((Hq, nqb), np.float32)
    for h in range(Hq):
        for blk in range(nqb):
            t0, t1 = 128 * blk, min(total_q, 128 * blk + 128)
            c, s_ = fp8_quantize_rows(qa[t0:t1, h, :], signs)
            q8[t0:t1, h, :] = c
            qs[h, blk] = s_
    k8 = np.zeros((total_k, Hkv, d), np.uint8)
    ks = np.ones((Hkv, max(nkb, 1)), np.float32)
    v8t = np.zeros((Hkv, d, 128 * max(nkb, 1)), np.uint8)
    vs = np.ones((batch, Hkv), np.float32)
    for b in range(batch):
        k0, k1 = int(cu[b]), int(cu[b + 1])
        for h in range(Hkv):
            for i in range((k1 - k0 + 127) // 128):
                t0, t1 = k0 + 128 * i, min(k1, k0 + 128 * i + 128)
                c, s_ = fp8_quantize_rows(ka[t0:t1, h, :], signs)
                k8[t0:t1, h, :] = c
                ks[h, kb0[b] + i] = s_
            if k1 > k0:
                c, s_ = fp8_quantize_rows(va[k0:k1, h, :])
                col = 128 * kb0[b]
                v8t[h, :, col:col + (k1 - k0)] = c.T
                vs[b, h] = s_
    t = torch.from_numpy
    return t(q8), t(qs), t(k8), t(ks), t(v8t), t(vs)
