"""ctypes binding of libattn.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module checks tensor
dtypes and shapes, allocates outputs and workspace with torch when the caller does not pass
them, and forwards raw device pointers and the current CUDA stream.  If the library has not
been built the first call raises ``AttnError`` -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported configuration",
          -3: "workspace missing or too small", -4: "CUDA call failed",
          -5: "a kernel wait exceeded its time limit", -6: "a device-side index was out of range"}


class AttnError(RuntimeError):
    def __init__(self, code, where):
        super().__init__(f"{where}: {STATUS.get(code, code)} ({code})")
        self.code = code


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libattn.so (built by ``__graft_entry__.build()`` / ``exact_attention_70_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise AttnError(-4, f"libattn.so not built (expected at {path})")
            lib = ctypes.CDLL(path)
            P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.attn_fwd.restype = i32
            lib.attn_fwd.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                     f32, i32, i32, i32, P, sz, P]
            lib.attn_fwd_workspace_bytes.restype = sz
            lib.attn_fwd_workspace_bytes.argtypes = [i32, i32, i32, i32]
            lib.attn_decode_kvcache.restype = i32
            lib.attn_decode_kvcache.argtypes = [P, P, P, P, P, i32, i32, P, P, i32, i32, i32, i32,
                                                i32, i32, f32, P, sz, P]
            lib.attn_decode_workspace_bytes.restype = sz
            lib.attn_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
            lib.attn_decode_num_splits.restype = i32
            lib.attn_decode_num_splits.argtypes = [i32, i32, i32, i32, i32, i32]
            lib.attn_get_device_status.restype = i32
            lib.attn_get_device_status.argtypes = [P]
            lib.attn_selftest_wait_timeout.restype = i32
            lib.attn_selftest_wait_timeout.argtypes = [P]
            lib.attn_selftest_softcap.restype = i32
            lib.attn_selftest_softcap.argtypes = [P, P, i32, f32, f32, P]
            lib.attn_fwd_kvcache.restype = i32
            lib.attn_fwd_kvcache.argtypes = [P, P, P, P, P, P, P, P, P, P, i32, i32, i32, P, P,
                                             i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                             ctypes.c_float, i32, i32, i32, P, sz, P]
            lib.attn_quantize_fp8.restype = i32
            lib.attn_quantize_fp8.argtypes = [P] * 4 + [i32] * 8 + [P] * 8
            lib.attn_fwd_fp8.restype = i32
            lib.attn_fwd_fp8.argtypes = [P] * 10 + [i32] * 9 + [f32, i32, i32, i32, P]
            lib.attn_fwd_mods.restype = i32
            lib.attn_fwd_mods.argtypes = [P, P, P, P, P, P, P] + [i32] * 8 + [f32, i32, i32, i32,
                                                                            f32, P, P, sz, P]
            lib.attn_bwd.restype = i32
            lib.attn_bwd.argtypes = [P] * 11 + [i32] * 8 + [f32, i32, i32, i32, P, sz, P]
            lib.attn_bwd_workspace_bytes.restype = sz
            lib.attn_bwd_workspace_bytes.argtypes = [i32, i32]
            lib.attn_fwd_kvcache_workspace_bytes.restype = sz
            lib.attn_fwd_kvcache_workspace_bytes.argtypes = [i32] * 7
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_status_string.argtypes = [i32]
            lib.attn_kv_block_range.restype = i32
            lib.attn_kv_block_range.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32,
                                                ctypes.POINTER(i32), ctypes.POINTER(i32)]
            lib.attn_kv_block_masked.restype = i32
            lib.attn_kv_block_masked.argtypes = [i32] * 9
            _lib = lib
    return _lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_bwd_workspace_bytes(total_q, nheads_q) -> int:
    return int(load().attn_bwd_workspace_bytes(int(total_q), int(nheads_q)))


def attn_fwd_workspace_bytes(batch, max_seqlen_q, nheads_q, nheads_kv) -> int:
    return int(load().attn_fwd_workspace_bytes(batch, max_seqlen_q, nheads_q, nheads_kv))


def attn_decode_workspace_bytes(batch, nheads_q, head_dim, num_splits) -> int:
    return int(load().attn_decode_workspace_bytes(batch, nheads_q, head_dim, num_splits))


def attn_decode_num_splits(batch, nheads_q, nheads_kv, max_pages_per_seq, page_size, num_sms):
    return int(load().attn_decode_num_splits(batch, nheads_q, nheads_kv, max_pages_per_seq,
                                             page_size, num_sms))


def attn_kv_block_range(i_min, i_max, seqlen_q, seqlen_k, block_n, causal, wl, wr):
    lo, hi = ctypes.c_int(), ctypes.c_int()
    rc = load().attn_kv_block_range(i_min, i_max, seqlen_q, seqlen_k, block_n, int(causal), wl,
                                    wr, ctypes.byref(lo), ctypes.byref(hi))
    if rc != 0:
        raise AttnError(-1, "attn_kv_block_range")
    return lo.value, hi.value


def attn_kv_block_masked(j, i_min, i_max, seqlen_q, seqlen_k, block_n, causal, wl, wr) -> bool:
    return bool(load().attn_kv_block_masked(j, i_min, i_max, seqlen_q, seqlen_k, block_n,
                                            int(causal), wl, wr))


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    return int(load().attn_get_device_status(_stream(stream)))


def attn_selftest_wait_timeout(stream=None) -> int:
    """Launch the bounded-wait self-test kernel (its wait runs out after 20 ms)."""
    return int(load().attn_selftest_wait_timeout(_stream(stream)))


def attn_selftest_softcap(scores, softmax_scale: float, softcap: float, stream=None):
    """softcap * tanh(softmax_scale * scores / softcap) as the modifier kernel computes it
    (scores: contiguous device fp32, even length)."""
    _check(scores, "scores", torch.float32, 1)
    out = torch.empty_like(scores)
    rc = load().attn_selftest_softcap(_ptr(scores), _ptr(out), scores.numel(),
                                      float(softmax_scale), float(softcap), _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_selftest_softcap")
    return out


def _workspace(nbytes, device, workspace):
    if nbytes == 0:
        return None
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise AttnError(-3, "workspace")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
             softmax_scale=None, causal=False, window_left=-1, window_right=-1,
             out=None, lse=None, workspace=None, stream=None):
    """Varlen prefill.  q [total_q, Hq, d], k/v [total_k, Hkv, d] bf16; cu_seqlens int32.

    Returns (out [total_q, Hq, d] bf16, lse [Hq, total_q] fp32).
    """
    lib = load()
    _check(q, "q", torch.bfloat16, 3)
    _check(k, "k", torch.bfloat16, 3)
    _check(v, "v", torch.bfloat16, 3)
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    total_q, Hq, d = q.shape
    total_k, Hkv, dk = k.shape
    if v.shape != k.shape or dk != d:
        raise ValueError("k and v must both be [total_k, Hkv, d] with q's d")
    batch = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != batch + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    scale = d ** -0.5 if softmax_scale is None else float(softmax_scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    _check(out, "out", torch.bfloat16, 3)
    _check(lse, "lse", torch.float32, 2)
    nbytes = int(lib.attn_fwd_workspace_bytes(max(batch, 0), int(max_seqlen_q), Hq, Hkv))
    ws = _workspace(nbytes, q.device, workspace)
    rc = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                      _ptr(cu_seqlens_k), batch, total_q, total_k, int(max_seqlen_q),
                      int(max_seqlen_k), Hq, Hkv, d, scale, int(bool(causal)), int(window_left),
                      int(window_right), _ptr(ws), nbytes, _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_fwd")
    return out, lse


def attn_fwd_mods(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                  softmax_scale=None, causal=False, window_left=-1, window_right=-1,
                  softcap=0.0, alibi_slopes=None, out=None, lse=None, workspace=None,
                  stream=None):
    """attn_fwd with softcap (0 = off) and ALiBi slopes (fp32 [Hq] CUDA tensor or None)."""
    lib = load()
    _check(q, "q", torch.bfloat16, 3)
    _check(k, "k", torch.bfloat16, 3)
    _check(v, "v", torch.bfloat16, 3)
    if alibi_slopes is not None:
        _check(alibi_slopes, "alibi_slopes", torch.float32, 1)
    total_q, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    scale = d ** -0.5 if softmax_scale is None else float(softmax_scale)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = int(lib.attn_fwd_workspace_bytes(max(batch, 0), int(max_seqlen_q), Hq, Hkv))
    ws = _workspace(nbytes, q.device, workspace)
    rc = lib.attn_fwd_mods(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                           _ptr(cu_seqlens_k), batch, total_q, total_k, int(max_seqlen_q),
                           int(max_seqlen_k), Hq, Hkv, d, scale, int(bool(causal)),
                           int(window_left), int(window_right), float(softcap),
                           _ptr(alibi_slopes), _ptr(ws), nbytes, _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_mods")
    return out, lse


def attn_quantize_fp8(q, k, v, cu_seqlens_k, max_seqlen_k, signs=None, key_blocks=None,
                      stream=None):
    """bf16 q, k, v (d = 128) -> (q8, q_scale, k8, k_scale, v8t, v_scale) for attn_fwd_fp8.
    signs: fp32 [128] CUDA tensor of +-1 (rotate Q and K) or None.  key_blocks defaults to
    ceil(total_k / 128) + batch."""
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, 3)
    if signs is not None:
        _check(signs, "signs", torch.float32, 1)
    total_q, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    batch = cu_seqlens_k.numel() - 1
    kb = (total_k + 127) // 128 + batch if key_blocks is None else int(key_blocks)
    dev = q.device
    q8 = torch.empty((total_q, Hq, d), dtype=torch.uint8, device=dev)
    qs = torch.empty((Hq, max(1, (total_q + 127) // 128)), dtype=torch.float32, device=dev)
    k8 = torch.empty((total_k, Hkv, d), dtype=torch.uint8, device=dev)
    ks = torch.empty((Hkv, kb), dtype=torch.float32, device=dev)
    v8t = torch.empty((Hkv, d, 128 * kb), dtype=torch.uint8, device=dev)
    vs = torch.empty((max(batch, 1), Hkv), dtype=torch.float32, device=dev)
    rc = lib.attn_quantize_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_k), batch, total_q,
                               total_k, int(max_seqlen_k), Hq, Hkv, d, kb, _ptr(signs), _ptr(q8),
                               _ptr(qs), _ptr(k8), _ptr(ks), _ptr(v8t), _ptr(vs), _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_quantize_fp8")
    return q8, qs, k8, ks, v8t, vs


def attn_fwd_fp8(q8, k8, v8t, q_scale, k_scale, v_scale, cu_seqlens_q, cu_seqlens_k,
                 max_seqlen_q, max_seqlen_k, softmax_scale=None, causal=False, window_left=-1,
                 window_right=-1, out=None, lse=None, stream=None):
    """FP8 (e4m3) forward.  q8 [total_q, Hq, 128], k8 [total_k, Hkv, 128] and v8t [Hkv, 128,
    128 * key_blocks] are uint8 e4m3 codes; q_scale [Hq, ceil(total_q/128)], k_scale [Hkv,
    key_blocks], v_scale [batch, Hkv] fp32.  Returns (out bf16, lse fp32) as attn_fwd."""
    lib = load()
    _check(q8, "q8", torch.uint8, 3)
    _check(k8, "k8", torch.uint8, 3)
    _check(v8t, "v8t", torch.uint8, 3)
    _check(q_scale, "q_scale", torch.float32, 2)
    _check(k_scale, "k_scale", torch.float32, 2)
    _check(v_scale, "v_scale", torch.float32, 2)
    total_q, Hq, d = q8.shape
    total_k, Hkv, _ = k8.shape
    key_blocks = k_scale.shape[1]
    if v8t.shape != (Hkv, d, 128 * key_blocks):
        raise ValueError("v8t must be [Hkv, d, 128 * key_blocks]")
    batch = cu_seqlens_q.numel() - 1
    scale = d ** -0.5 if softmax_scale is None else float(softmax_scale)
    out = torch.empty((total_q, Hq, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q8.device) if lse is None else lse
    rc = lib.attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8t), _ptr(q_scale), _ptr(k_scale),
                          _ptr(v_scale), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                          _ptr(cu_seqlens_k), batch, total_q, total_k, int(max_seqlen_q),
                          int(max_seqlen_k), Hq, Hkv, d, key_blocks, scale, int(bool(causal)),
                          int(window_left), int(window_right), _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_fp8")
    return out, lse


def attn_bwd(q, k, v, out, dout, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
             softmax_scale=None, causal=False, window_left=-1, window_right=-1, dq=None,
             dk=None, dv=None, workspace=None, stream=None):
    """Gradients of sum(out * dout) for attn_fwd.  Returns (dq, dk, dv), bf16."""
    lib = load()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _check(t, n, torch.bfloat16, 3)
    _check(lse, "lse", torch.float32, 2)
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _check(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    total_q, Hq, d = q.shape
    total_k, Hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    scale = d ** -0.5 if softmax_scale is None else float(softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = int(lib.attn_bwd_workspace_bytes(total_q, Hq))
    ws = _workspace(nbytes, q.device, workspace)
    rc = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq),
                      _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, total_q,
                      total_k, int(max_seqlen_q), int(max_seqlen_k), Hq, Hkv, d, scale,
                      int(bool(causal)), int(window_left), int(window_right), _ptr(ws), nbytes,
                      _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_fwd_kvcache(q, k_new, v_new, k_cache, v_cache, cache_seqlens, block_table,
                     cu_seqlens_q, max_seqlen_q, softmax_scale=None, causal=True,
                     window_left=-1, window_right=-1, rotary_cos=None, rotary_sin=None,
                     rotary_interleaved=False, out=None, lse=None, workspace=None, stream=None):
    """Chunked prefill against a paged cache; the new k, v (rotated k) are written into it.

    q [total_q, Hq, d], k_new / v_new [total_q, Hkv, d] bf16; caches
    [num_pages, page_size, Hkv, d] bf16 (updated in place); cache_seqlens [batch],
    block_table [batch, max_pages], cu_seqlens_q [batch + 1] int32; rotary_cos / rotary_sin
    fp32 [rows, rotary_dim / 2] or None.  Returns (out [total_q, Hq, d], lse [Hq, total_q]).
    """
    lib = load()
    _check(q, "q", torch.bfloat16, 3)
    _check(k_new, "k_new", torch.bfloat16, 3)
    _check(v_new, "v_new", torch.bfloat16, 3)
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(cache_seqlens, "cache_seqlens", torch.int32, 1)
    _check(block_table, "block_table", torch.int32, 2)
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    total_q, Hq, d = q.shape
    num_pages, page_size, Hkv, dk = k_cache.shape
    if v_cache.shape != k_cache.shape or dk != d or k_new.shape != (total_q, Hkv, d) or \
            v_new.shape != k_new.shape:
        raise ValueError("inconsistent q / k_new / v_new / cache shapes")
    batch = cu_seqlens_q.numel() - 1
    if cache_seqlens.numel() != batch or block_table.shape[0] != batch:
        raise ValueError("cache_seqlens and block_table must have one row per sequence")
    if rotary_cos is not None:
        _check(rotary_cos, "rotary_cos", torch.float32, 2)
        _check(rotary_sin, "rotary_sin", torch.float32, 2)
        rot_rows, rot_dim = rotary_cos.shape[0], 2 * rotary_cos.shape[1]
    else:
        rot_rows = rot_dim = 0
    scale = d ** -0.5 if softmax_scale is None else float(softmax_scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    nbytes = int(lib.attn_fwd_kvcache_workspace_bytes(max(batch, 0), total_q, int(max_seqlen_q),
                                                      Hq, Hkv, d, rot_dim))
    ws = _workspace(nbytes, q.device, workspace)
    rc = lib.attn_fwd_kvcache(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                              _ptr(cache_seqlens), _ptr(block_table), _ptr(cu_seqlens_q),
                              _ptr(rotary_cos), _ptr(rotary_sin), rot_dim, rot_rows,
                              int(bool(rotary_interleaved)), _ptr(out), _ptr(lse), batch, total_q,
                              int(max_seqlen_q), Hq, Hkv, d, page_size, block_table.shape[1],
                              num_pages, scale, int(bool(causal)), int(window_left),
                              int(window_right), _ptr(ws), nbytes, _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_kvcache")
    return out, lse


def _decode_shapes(q, k_cache, v_cache, cache_seqlens, block_table):
    """Checks shared by both decode entry points: dtypes, ranks, and one table row and one
    length per sequence (a short table or length vector would be read past its end)."""
    _check(q, "q", torch.bfloat16, 3)
    _check(k_cache, "k_cache", torch.bfloat16, 4)
    _check(v_cache, "v_cache", torch.bfloat16, 4)
    _check(cache_seqlens, "cache_seqlens", torch.int32, 1)
    _check(block_table, "block_table", torch.int32, 2)
    batch, Hq, d = q.shape
    num_pages, page_size, Hkv, dk = k_cache.shape
    if v_cache.shape != k_cache.shape or dk != d:
        raise ValueError("k_cache and v_cache must both be [num_pages, page_size, Hkv, d]")
    if cache_seqlens.numel() != batch or block_table.shape[0] != batch:
        raise ValueError("cache_seqlens and block_table must have one row per sequence")
    return batch, Hq, Hkv, d, num_pages, page_size


def _decode_outputs(q, out, lse):
    batch, Hq, _ = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((batch, Hq), dtype=torch.float32, device=q.device)
    _check(out, "out", torch.bfloat16, 3)
    _check(lse, "lse", torch.float32, 2)
    if tuple(out.shape) != tuple(q.shape) or tuple(lse.shape) != (batch, Hq):
        raise ValueError("out must be [batch, Hq, d] and lse [batch, Hq]")
    return out, lse


def attn_decode_kvcache(q, k_cache, v_cache, cache_seqlens, block_table, softmax_scale=None,
                        num_splits=0, out=None, lse=None, workspace=None, stream=None):
    """Decode over a paged cache.  q [batch, Hq, d]; caches [num_pages, page_size, Hkv, d].

    Returns (out [batch, Hq, d] bf16, lse [batch, Hq] fp32).
    """
    lib = load()
    batch, Hq, Hkv, d, num_pages, page_size = _decode_shapes(q, k_cache, v_cache, cache_seqlens,
                                                             block_table)
    scale = d ** -0.5 if softmax_scale is None else float(softmax_scale)
    out, lse = _decode_outputs(q, out, lse)
    nbytes = int(lib.attn_decode_workspace_bytes(batch, Hq, d, int(num_splits)))
    ws = _workspace(nbytes, q.device, workspace)
    rc = lib.attn_decode_kvcache(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens),
                                 _ptr(block_table), page_size, int(num_splits), _ptr(out),
                                 _ptr(lse), batch, Hq, Hkv, d, block_table.shape[1], num_pages,
                                 scale, _ptr(ws), nbytes, _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_decode_kvcache")
    return out, lse


def attn_decode_kvcache_noalloc(q, k_cache, v_cache, cache_seqlens, block_table,
                                softmax_scale=None, num_splits=0, out=None, lse=None,
                                stream=None):
    """Decode over a paged cache without any workspace from the caller.

    For callers that cannot allocate device memory: the split partials live in a 32 MiB
    scratch array owned by the library (see attn_decode_kvcache_noalloc in include/attn.h).
    Calls on one device share that array, so calls whose kernels overlap on the GPU race.
    The outputs are allocated here only when `out` / `lse` are not given.
    """
    lib = load()
    fn = lib.attn_decode_kvcache_noalloc
    if fn.argtypes is None:
        P, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fn.restype = i32
        fn.argtypes = [P, P, P, P, P, i32, i32, P, P, i32, i32, i32, i32, i32, i32, f32, P]
    batch, Hq, Hkv, d, num_pages, page_size = _decode_shapes(q, k_cache, v_cache, cache_seqlens,
                                                             block_table)
    scale = d ** -0.5 if softmax_scale is None else float(softmax_scale)
    out, lse = _decode_outputs(q, out, lse)
    rc = fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens), _ptr(block_table),
            page_size, int(num_splits), _ptr(out), _ptr(lse), batch, Hq, Hkv, d,
            block_table.shape[1], num_pages, scale, _stream(stream))
    if rc != 0:
        raise AttnError(rc, "attn_decode_kvcache_noalloc")
    return out, lse
