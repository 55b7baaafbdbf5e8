"""Backward pass (attn_bwd) versus the fp64 oracle's gradients.

The GPU forward produces out and lse; a seeded bf16 dout drives the GPU backward and the
oracle (which recomputes everything in fp64 from q, k, v, dout).  Tolerance, per gradient
tensor, relative to its own scale: max |err| <= 2e-2 * max |ref| and mean |err| <= 5e-3 *
mean |ref| (observed: at most 0.8e-2 and 0.25e-2).  Sources of difference: P and dS enter the tensor-core products as bf16 (relative
rounding 2^-9 each), dout V^T and the products accumulate in fp32, D uses the bf16 forward
output, and the gradients are rounded to bf16 (2^-9); with hundreds of terms per element the
errors add like a random walk, leaving the typical element a few 1e-3 relative.
"""
import numpy as np
import pytest
import torch

from exact_attention_70_gb300 import synth
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_70_gb300 import build as attn_build
    attn_build.build()
    from exact_attention_70_gb300 import binding
    binding.load()
    return binding


def check_grad(gpu, ref, what):
    g = gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    scale_max, scale_mean = np.abs(ref).max(), np.abs(ref).mean()
    assert np.all(np.isfinite(g)), what
    assert err.max() <= 2e-2 * scale_max + 1e-6, (what, err.max(), scale_max)
    assert err.mean() <= 5e-3 * scale_mean + 1e-7, (what, err.mean(), scale_mean)


def run_case(attn, case, seed):
    dev = "cuda"
    q, k, v = case.q.to(dev), case.k.to(dev), case.v.to(dev)
    cq, ck = case.cu_seqlens_q.to(dev), case.cu_seqlens_k.to(dev)
    out, lse = attn.attn_fwd(q, k, v, cq, ck, case.max_seqlen_q, case.max_seqlen_k,
                             case.softmax_scale, case.causal, case.window_left, case.window_right)
    dout = synth.randn_bf16(tuple(case.q.shape), seed, 9)
    dq, dk, dv = attn.attn_bwd(q, k, v, out, dout.to(dev), lse, cq, ck, case.max_seqlen_q,
                               case.max_seqlen_k, case.softmax_scale, case.causal,
                               case.window_left, case.window_right)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    rdq, rdk, rdv, _ = oracle.attn_bwd(case.q, case.k, case.v, dout, case.cu_seqlens_q,
                                       case.cu_seqlens_k, case.softmax_scale, case.causal,
                                       case.window_left, case.window_right)
    check_grad(dq, rdq, case.name + " dq")
    check_grad(dk, rdk, case.name + " dk")
    check_grad(dv, rdv, case.name + " dv")


CASES = [
    # (lengths_q, lengths_k, Hq, Hkv, d, causal, window)
    ([300], None, 2, 2, 128, True, (-1, -1)),
    ([1, 130, 257], None, 4, 2, 128, True, (-1, -1)),
    ([200, 77], None, 8, 2, 64, False, (-1, -1)),
    ([500], None, 4, 1, 128, True, (100, 0)),
    ([128, 129], None, 6, 2, 128, True, (-1, -1)),     # g = 3: 42 tokens per tile
    ([96], None, 32, 1, 64, False, (-1, -1)),          # g = 32: 4 tokens per tile
    ([40, 300], [200, 300], 4, 4, 128, True, (-1, -1)),  # bottom-right, Lk > Lq
    ([600], None, 2, 2, 128, False, (50, 50)),
]


@pytest.mark.parametrize("idx", range(len(CASES)))
def test_backward_matches_oracle(attn, idx):
    lq, lk, Hq, Hkv, d, causal, window = CASES[idx]
    case = synth.prefill_case(lq, Hq, Hkv, d, causal, seed=500 + idx, lengths_k=lk, window=window,
                              name=f"bwd{idx}")
    run_case(attn, case, 600 + idx)


def test_backward_is_deterministic(attn):
    case = synth.prefill_case([700, 300], 8, 2, 128, True, seed=550)
    dev = "cuda"
    q, k, v = case.q.to(dev), case.k.to(dev), case.v.to(dev)
    cq, ck = case.cu_seqlens_q.to(dev), case.cu_seqlens_k.to(dev)
    out, lse = attn.attn_fwd(q, k, v, cq, ck, case.max_seqlen_q, case.max_seqlen_k,
                             case.softmax_scale, True)
    dout = synth.randn_bf16(tuple(case.q.shape), 551, 9).to(dev)
    a = attn.attn_bwd(q, k, v, out, dout, lse, cq, ck, case.max_seqlen_q, case.max_seqlen_k,
                      case.softmax_scale, True)
    b = attn.attn_bwd(q, k, v, out, dout, lse, cq, ck, case.max_seqlen_q, case.max_seqlen_k,
                      case.softmax_scale, True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_at_the_benchmarked_shape(attn):
    """The causal B=4, H=16, N=4096, d=128 workload the benchmark times, with the benchmark's
    seeded dout, against the full fp64 oracle gradients (about a minute on the host cores)."""
    case = synth.config_case(2)
    run_case(attn, case, 1200)
