#!/usr/bin/env python
"""Benchmark of the hot path on GB300.

One step = one pass of the whole path over one batch: the causal prefill workload
(B=4, Hq=Hkv=16, N=4096, d=128, packed varlen layout) through attn_fwd, then the paged decode
workload (batch 64, cache lengths U[1024, 32768], page 256, Hq=32, Hkv=8, d=128) through
attn_decode_kvcache.  Inputs are resident in HBM when the timed region starts.  The headline
value is the prefill's TFLOPS; the decode's GB/s sits in "decode".  Both carry a roofline
object against the measured peaks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed steps, then K timed steps between a barrier and a device synchronisation;
CUDA events on the launching stream bracket each call, and the reported times are the medians
of the K per-call times (the mean can be pulled by one slow step).  The prefill inputs are
larger than L2; before every decode call a 256 MiB buffer is read through so that the decode
starts from a cold L2 (the read is outside the decode's events; a read leaves clean lines, so no
write-back competes with the decode), and the single-head workload is timed the same way, one
flushed call at a time.

Under torchrun every rank runs its own replica of the workload (weak scaling, no collective
on the data path); rank 0 prints one JSON line with the aggregate over ranks and the maximum
time over ranks.  ``--impl reference`` times the fp64 CPU oracle on bounded samples of the same
workload (the reference arm of this build); only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOPS & decode KV GB/s on 1 GB300, % of roofline"
L2_FLUSH_BYTES = 256 << 20  # twice the GB300's L2


class L2Flush:
    """Evicts L2 by reading a device buffer twice its size (a reduction kernel)."""

    def __init__(self, device):
        import torch
        self.buf = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=device)
        self.out = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self):
        import torch
        torch.sum(self.buf, dim=0, out=self.out)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal GB300 figures, shown as a second denominator beside the measured ones: dense bf16
# tensor-core peak and HBM3e bandwidth from the vendor's specification.
NOMINAL_PEAKS = {"bf16_tflops": 2250.0, "hbm_gbs": 8000.0}
PREFILL_CFG, DECODE_CFG = 2, 4


# ---- helpers ------------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def reduce_max(values, world, device=None):
    """Element-wise max of a list of floats over ranks (identity when world == 1)."""
    if world == 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rate(units_per_rank, ms_per_rank, world):
    """Whole-job throughput of `world` replicas that each process `units_per_rank` units: the
    units of all ranks over the slowest rank's time (ms_per_rank already reduced to the max
    over ranks), in units per second."""
    return world * units_per_rank / (ms_per_rank * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(name):
    """Hash of a kernel's source file and the headers every kernel inlines."""
    h = hashlib.sha256()
    for f in (name, "ptx.cuh", "kernels.h", "tile_math.h"):
        with open(os.path.join(ROOT, "exact_attention_70_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, source):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source still matches."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            t = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None
    if not t or t.get("source_sha") != source_sha(source):
        return None
    return t.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        self.proc = None
        self.path = None
        self.index = None
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            parts = vis.split(",")
            if local_rank < len(parts) and parts[local_rank].strip().isdigit():
                self.index = parts[local_rank].strip()
        elif local_rank >= 0:
            self.index = str(local_rank)

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "10", "-f", self.path]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 9:
                    continue
                rows.append(c)
        os.unlink(self.path)
        if self.index is not None and len({r[0] for r in rows}) > 1:
            rows = [r for r in rows if r[0] == self.index]
        if not rows:
            return {"samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = max([num(r[2]) for r in rows if num(r[2]) is not None] or [0.0])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if s >= 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max([num(r[3]) or 0.0 for r in rows])}


# ---- the CPU oracle (cpu_baseline and the reference arm) ------------------------------------

def oracle_rate(case, seconds, seed=0, n_rows=None):
    """Time the fp64 oracle on seeded rows of a prefill case for about `seconds` of CPU work
    (or on exactly `n_rows` rows, skipping the calibration).

    Returns (TFLOPS-equivalent, threads, sample description, seconds taken, flops done,
    rows)."""
    import numpy as np
    import torch
    from oracle import oracle
    cu = case.cu_seqlens_q.tolist()
    Hq, d = case.q.shape[1], case.q.shape[2]
    g = torch.Generator().manual_seed(seed)

    def rows(n):
        t = torch.randint(0, cu[-1], (n,), generator=g).numpy().astype(np.int64)
        h = torch.randint(0, Hq, (n,), generator=g).numpy().astype(np.int32)
        return t, h

    def pairs_of_row(tok):
        # visible keys of query row i (Lq == Lk in the prefill workloads)
        b = max(i for i in range(len(cu) - 1) if cu[i] <= tok)
        i, L = tok - cu[b], cu[b + 1] - cu[b]
        right = 0 if case.causal else case.window_right
        hi = L - 1 if right < 0 else min(L - 1, i + right)
        lo = 0 if case.window_left < 0 else max(0, i - case.window_left)
        return max(0, hi - lo + 1)

    # calibrate on a small sample and then on one of about a second (fixed costs dominate the
    # first), then run a sample sized for `seconds`
    n = 32 if n_rows is None else n_rows
    for target in ((1.0, seconds) if n_rows is None else ()):
        t, h = rows(n)
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                             case.softmax_scale, t, h, case.causal, case.window_left,
                             case.window_right)
        dt = max(time.perf_counter() - t0, 1e-4)
        n = int(max(32, min(2000000, n * target / dt)))
    t, h = rows(n)
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                         case.softmax_scale, t, h, case.causal, case.window_left,
                         case.window_right)
    dt = time.perf_counter() - t0
    fl = sum(4 * d * pairs_of_row(x) for x in t.tolist())
    return fl / dt / 1e12, oracle.num_threads(), f"{n} seeded (token, head) rows", dt, fl, n


# ---- our implementation ---------------------------------------------------------------------

def median_ms(fn, stream, reps=30, warm=10, flush=None):
    """Median over `reps` calls of fn's CUDA-event time on `stream`, after `warm` untimed calls;
    with `flush` (an L2Flush) L2 is evicted before every call, outside the events."""
    import torch
    for _ in range(warm):
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        if flush is not None:
            flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


EXTRA_WORKLOADS = ("cfg1", "cfg3", "cfg5", "chunked", "mods", "bwd", "fp8")


def build_workload(name, dev):
    """One of the extra workloads, its inputs on the device: a dict with the call, its
    algorithmic work (FLOP, or bytes), the rate's unit ("tflops": work / ms / 1e9), a
    description and whether the call is timed from a cold L2."""
    import torch
    from exact_attention_70_gb300 import binding, synth, workload
    if name in ("cfg1", "cfg2", "cfg3", "cfg5"):
        c = synth.config_case(int(name[3:]))
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        cq, ck = c.cu_seqlens_q.to(dev), c.cu_seqlens_k.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
        ws = torch.empty(binding.attn_fwd_workspace_bytes(c.batch, c.max_seqlen_q, q.shape[1],
                                                          k.shape[1]), dtype=torch.uint8,
                         device=dev)

        def call():
            binding.attn_fwd(q, k, v, cq, ck, c.max_seqlen_q, c.max_seqlen_k, c.softmax_scale,
                             c.causal, c.window_left, c.window_right, out=o, lse=lse,
                             workspace=ws)
        # the single-head workload fits in L2: it is timed from a cold L2, call by call
        return dict(call=call, work=workload.prefill_case_flops(c), unit="tflops",
                    desc=synth.CONFIG_NAMES[int(name[3:])], flush=name == "cfg1")
    if name == "chunked":
        # chunked prefill against the paged cache (append + rotary + attention, one call)
        c = synth.chunked_case()
        t = {f: getattr(c, f).to(dev) for f in ("q", "k_new", "v_new", "k_cache", "v_cache",
                                                 "cache_seqlens", "block_table", "cu_seqlens_q",
                                                 "rotary_cos", "rotary_sin")}
        o = torch.empty_like(t["q"])
        lse = torch.empty((t["q"].shape[1], t["q"].shape[0]), dtype=torch.float32, device=dev)

        def call():
            binding.attn_fwd_kvcache(t["q"], t["k_new"], t["v_new"], t["k_cache"], t["v_cache"],
                                     t["cache_seqlens"], t["block_table"], t["cu_seqlens_q"],
                                     c.max_seqlen_q, c.softmax_scale, c.causal, -1, -1,
                                     t["rotary_cos"], t["rotary_sin"], False, out=o, lse=lse)
        ql = (c.cu_seqlens_q[1:] - c.cu_seqlens_q[:-1]).tolist()
        lk = [int(x) + n for x, n in zip(c.cache_seqlens.tolist(), ql)]
        return dict(call=call, unit="tflops", desc=synth.CHUNKED_NAME, flush=False,
                    work=workload.prefill_flops(ql, lk, t["q"].shape[1], t["q"].shape[2], True))
    if name == "mods":
        # the causal prefill workload with both score modifiers (softcap 30, ALiBi slopes)
        c = synth.config_case(2)
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        cq, ck = c.cu_seqlens_q.to(dev), c.cu_seqlens_k.to(dev)
        Hq = q.shape[1]
        slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / Hq) for h in range(Hq)],
                              dtype=torch.float32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((Hq, q.shape[0]), dtype=torch.float32, device=dev)

        def call():
            binding.attn_fwd_mods(q, k, v, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                  c.softmax_scale, True, softcap=30.0, alibi_slopes=slopes,
                                  out=o, lse=lse)
        return dict(call=call, work=workload.prefill_case_flops(c), unit="tflops", flush=False,
                    desc=synth.CONFIG_NAMES[2] + " with softcap 30 and ALiBi")
    if name == "bwd":
        # backward of the causal prefill workload (gradients of q, k, v)
        c = synth.config_case(2)
        q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
        cq, ck = c.cu_seqlens_q.to(dev), c.cu_seqlens_k.to(dev)
        o, lse = binding.attn_fwd(q, k, v, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                                  c.softmax_scale, True)
        do = synth.randn_bf16(tuple(c.q.shape), 1200, 9).to(dev)
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(binding.attn_bwd_workspace_bytes(q.shape[0], q.shape[1]),
                         dtype=torch.uint8, device=dev)

        def call():
            binding.attn_bwd(q, k, v, o, do, lse, cq, ck, c.max_seqlen_q, c.max_seqlen_k,
                             c.softmax_scale, True, dq=gq, dk=gk, dv=gv, workspace=ws)
        # S, dP, dV, dK, dQ: 10 d per visible pair
        return dict(call=call, work=workload.prefill_case_flops(c) * 10 // 4, unit="tflops",
                    desc="backward of " + synth.CONFIG_NAMES[2], flush=False)
    if name in ("fp8", "quant"):
        # the causal prefill workload's shape with FP8 e4m3 inputs and block scales, and the
        # quantizer that produces such inputs from bf16 (rotation of Q and K on)
        c = synth.fp8_bench_case()
        f8 = [x.to(dev) for x in (c.q8, c.k8, c.v8t, c.q_scale, c.k_scale, c.v_scale,
                                  c.cu_seqlens_q, c.cu_seqlens_k)]
        o = torch.empty((c.q8.shape[0], c.q8.shape[1], c.q8.shape[2]), dtype=torch.bfloat16,
                        device=dev)
        lse = torch.empty((c.q8.shape[1], c.q8.shape[0]), dtype=torch.float32, device=dev)
        cq_ = synth.config_case(2)
        bq, bk, bv = cq_.q.to(dev), cq_.k.to(dev), cq_.v.to(dev)
        bck = cq_.cu_seqlens_k.to(dev)
        sg = torch.where(torch.arange(128, device=dev) % 3 == 0, -1.0, 1.0).float()

        def call():
            binding.attn_fwd_fp8(*f8, c.max_seqlen_q, c.max_seqlen_k, c.softmax_scale,
                                 c.causal, out=o, lse=lse)

        def quant():
            binding.attn_quantize_fp8(bq, bk, bv, bck, cq_.max_seqlen_k, signs=sg)
        # bytes: Q, K, V read as bf16 (V twice: its maximum, then its codes), codes written
        qbytes = (bq.numel() + bk.numel() + 2 * bv.numel()) * 2 + bq.numel() + bk.numel() + bv.numel()
        if name == "quant":
            return dict(call=quant, work=qbytes, unit="gbs", flush=False,
                        desc="FP8 quantizer on " + synth.CONFIG_NAMES[2])
        ql = (c.cu_seqlens_q[1:] - c.cu_seqlens_q[:-1]).tolist()

        def after(stream):
            qms = median_ms(quant, stream)
            return {"quantize_ms": round(qms, 4), "quantize_gbs": round(qbytes / qms / 1e6, 1)}
        return dict(call=call, unit="tflops", desc=synth.FP8_NAME, flush=False, after=after,
                    work=workload.prefill_flops(ql, ql, c.q8.shape[1], c.q8.shape[2], c.causal))
    raise ValueError(name)


def run_workload(args):
    """--workload NAME: only that workload, W untimed and K timed calls (profiler captures)."""
    import torch
    from exact_attention_70_gb300 import binding
    from exact_attention_70_gb300 import build as attn_build
    torch.cuda.set_device(0)
    attn_build.build()
    binding.load()
    dev = torch.device("cuda", 0)
    w = build_workload(args.workload, dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev) if w["flush"] else None
    ms = median_ms(w["call"], stream, reps=args.steps, warm=args.warmup, flush=flush)
    if binding.attn_get_device_status() != 0:
        raise RuntimeError("device status is not ok")
    print(json.dumps({"workload": w["desc"], "ms": round(ms, 4),
                      w["unit"]: round(w["work"] / ms / 1e9, 2), "steps": args.steps,
                      "warmup": args.warmup}))



def run_ours(args, rank, world, local):
    import torch
    from exact_attention_70_gb300 import binding, synth, workload
    from exact_attention_70_gb300 import build as attn_build

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        attn_build.build()
    if world > 1:
        torch.distributed.barrier()
    binding.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    pre = synth.config_case(PREFILL_CFG)
    dec = synth.config_case(DECODE_CFG)
    if args.decode_batch < dec.q.shape[0]:
        # keep only the first sequences and the pages they use (smaller device footprint)
        nb = args.decode_batch
        ps = dec.page_size
        npg = [(int(n) + ps - 1) // ps for n in dec.cache_seqlens[:nb].tolist()]
        used = torch.cat([dec.block_table[b, :n] for b, n in enumerate(npg)]).long()
        remap = torch.zeros(dec.k_cache.shape[0], dtype=torch.long)
        remap[used] = torch.arange(len(used))
        bt = torch.zeros((nb, dec.block_table.shape[1]), dtype=torch.int32)
        for b, n in enumerate(npg):
            bt[b, :n] = remap[dec.block_table[b, :n].long()].to(torch.int32)
        dec.k_cache = dec.k_cache[used].contiguous()
        dec.v_cache = dec.v_cache[used].contiguous()
        dec.q = dec.q[:nb].contiguous()
        dec.cache_seqlens = dec.cache_seqlens[:nb].contiguous()
        dec.block_table = bt
        dec.meta["config"] += f" (first {nb} sequences)"
    p_flops = workload.prefill_case_flops(pre)
    d_bytes = workload.decode_case_bytes(dec)
    q, k, v = pre.q.to(dev), pre.k.to(dev), pre.v.to(dev)
    cuq, cuk = pre.cu_seqlens_q.to(dev), pre.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
    ws_f = torch.empty(binding.attn_fwd_workspace_bytes(pre.batch, pre.max_seqlen_q, q.shape[1],
                                                        k.shape[1]), dtype=torch.uint8, device=dev)
    dq, kc, vc = dec.q.to(dev), dec.k_cache.to(dev), dec.v_cache.to(dev)
    sl, bt = dec.cache_seqlens.to(dev), dec.block_table.to(dev)
    dout = torch.empty_like(dq)
    dlse = torch.empty(dq.shape[:2], dtype=torch.float32, device=dev)
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    splits = binding.attn_decode_num_splits(dq.shape[0], dq.shape[1], kc.shape[2], bt.shape[1],
                                            dec.page_size, n_sms)
    ws_d_bytes = binding.attn_decode_workspace_bytes(dq.shape[0], dq.shape[1], dq.shape[2], 0)
    ws_d = torch.empty(max(ws_d_bytes, 256), dtype=torch.uint8, device=dev)

    do_pre = args.only in ("all", "prefill")
    do_dec = args.only in ("all", "decode")

    def prefill():
        if not do_pre:
            return
        binding.attn_fwd(q, k, v, cuq, cuk, pre.max_seqlen_q, pre.max_seqlen_k,
                         pre.softmax_scale, True, -1, -1, out=out, lse=lse, workspace=ws_f)

    def decode():
        if not do_dec:
            return
        binding.attn_decode_kvcache(dq, kc, vc, sl, bt, dec.softmax_scale, 0, out=dout,
                                    lse=dlse, workspace=ws_d)

    flush = L2Flush(dev)

    for _ in range(args.warmup):
        prefill()
        flush()
        decode()
    torch.cuda.synchronize()
    if binding.attn_get_device_status() != 0:
        raise RuntimeError("device status after warm-up is not ok")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    t_start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        prefill()
        ev[i][1].record(stream)
        flush()  # cold L2 for the decode
        ev[i][2].record(stream)
        decode()
        ev[i][3].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    status = binding.attn_get_device_status()
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    dec_ms = statistics.median(e[2].elapsed_time(e[3]) for e in ev)
    total_ms, pre_ms, dec_ms = reduce_max([total_ms, pre_ms, dec_ms], world, dev)

    # end to end through the public API: pinned host inputs in, results back to the host
    h_q, h_k, h_v = (x.pin_memory() for x in (pre.q, pre.k, pre.v))
    h_cuq, h_cuk = pre.cu_seqlens_q.pin_memory(), pre.cu_seqlens_k.pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h_lse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    h_dq, h_sl, h_bt = dec.q.pin_memory(), dec.cache_seqlens.pin_memory(), dec.block_table.pin_memory()
    h_dout = torch.empty(dout.shape, dtype=dout.dtype, pin_memory=True)
    h_dlse = torch.empty(dlse.shape, dtype=dlse.dtype, pin_memory=True)
    e2e_steps = max(3, min(K, 50))
    # Prefill, pipelined as a serving loop runs it: every step copies its own q, k, v and
    # cu_seqlens in and its out and lse back, on their own streams, so step i + 1's inputs and
    # step i - 1's results move while step i computes (two device buffer sets).  The value is
    # the whole loop's time over its steps.
    e2e_pre = 1e-9
    if do_pre:
        sets = [dict(q=q, k=k, v=v, cuq=cuq, cuk=cuk, out=out, lse=lse),
                dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                     cuq=torch.empty_like(cuq), cuk=torch.empty_like(cuk),
                     out=torch.empty_like(out), lse=torch.empty_like(lse))]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        out_free = [torch.cuda.Event() for _ in range(2)]

        def e2e_prefill_step(i):
            bs = sets[i & 1]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(done[i & 1])  # step i - 2 has read this set's inputs
                for name, src in (("q", h_q), ("k", h_k), ("v", h_v), ("cuq", h_cuq), ("cuk", h_cuk)):
                    bs[name].copy_(src, non_blocking=True)
                in_ready[i & 1].record(s_in)
            stream.wait_event(in_ready[i & 1])
            if i >= 2:
                stream.wait_event(out_free[i & 1])  # step i - 2's results are on the host
            binding.attn_fwd(bs["q"], bs["k"], bs["v"], bs["cuq"], bs["cuk"], pre.max_seqlen_q,
                             pre.max_seqlen_k, pre.softmax_scale, True, -1, -1, out=bs["out"],
                             lse=bs["lse"], workspace=ws_f, stream=stream)
            done[i & 1].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[i & 1])
                h_out.copy_(bs["out"], non_blocking=True)
                h_lse.copy_(bs["lse"], non_blocking=True)
                out_free[i & 1].record(s_out)

        for i in range(2):
            e2e_prefill_step(i)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        s_in.wait_stream(stream)
        for i in range(e2e_steps):
            e2e_prefill_step(i)
        stream.wait_stream(s_out)
        a1.record(stream)
        torch.cuda.synchronize()
        e2e_pre = a0.elapsed_time(a1) / e2e_steps
    # Decode: per step, copy the new queries and the tables in, then the outputs back.
    pe = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps + 2)]
    for i in range(e2e_steps + 2):
        pe[i][0].record(stream)
        for dst, src in ((dq, h_dq), (sl, h_sl), (bt, h_bt)):
            dst.copy_(src, non_blocking=True)
        decode()
        h_dout.copy_(dout, non_blocking=True)
        h_dlse.copy_(dlse, non_blocking=True)
        pe[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_dec = statistics.median(e[0].elapsed_time(e[1]) for e in pe[2:])
    e2e_pre, e2e_dec = reduce_max([e2e_pre, e2e_dec], world, dev)
    h2d_pre = sum(x.numel() * x.element_size() for x in (h_q, h_k, h_v, h_cuq, h_cuk))
    d2h_pre = out.numel() * 2 + lse.numel() * 4
    h2d_dec = sum(x.numel() * x.element_size() for x in (h_dq, h_sl, h_bt))
    d2h_dec = dout.numel() * 2 + dlse.numel() * 4

    # the other workloads, timed alone (parity cases; reported for context)
    extra = {}
    if not args.no_extra:
        for name in EXTRA_WORKLOADS:
            w = build_workload(name, dev)
            ms = median_ms(w["call"], stream, flush=flush if w["flush"] else None)
            extra[name] = {"workload": w["desc"], "ms": round(ms, 4),
                           w["unit"]: round(w["work"] / ms / 1e9, 2)}
            if "after" in w:
                extra[name].update(w["after"](stream))
            del w
    return dict(p_flops=p_flops, d_bytes=d_bytes, total_ms=total_ms, pre_ms=pre_ms,
                dec_ms=dec_ms, e2e_pre=e2e_pre, e2e_dec=e2e_dec, h2d_pre=h2d_pre,
                d2h_pre=d2h_pre, h2d_dec=h2d_dec, d2h_dec=d2h_dec, clocks=clk, splits=splits,
                status=status, extra=extra, pre=pre, dec=dec)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--only", choices=["all", "prefill", "decode"], default="all",
                    help="time one half of the step only (for profiler captures)")
    ap.add_argument("--decode-batch", type=int, default=64,
                    help="use the first B sequences of the decode workload (profiling)")
    ap.add_argument("--workload", choices=["step", "cfg1", "cfg2", "cfg3", "cfg5", "chunked",
                                           "mods", "bwd", "fp8", "quant"], default="step",
                    help="run one workload alone, W + K calls, instead of the timed step "
                         "(for profiler captures; prints that workload's median time only)")
    args = ap.parse_args()
    if args.workload != "step":
        run_workload(args)
        return
    rank, world, local = dist_env()
    peaks, peak_src = load_peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        from exact_attention_70_gb300 import synth
        case = synth.config_case(PREFILL_CFG)
        # every step runs the same number of rows, sized once so that the W + K steps take
        # about 90 s of host time together
        budget = max(0.2, 90.0 / max(1, args.steps + args.warmup))
        _, _, _, _, _, n_rows = oracle_rate(case, budget, seed=10 ** 6)
        rates, times = [], []
        for i in range(args.warmup + args.steps):
            r, cores, sample, dt, _, _ = oracle_rate(case, budget, seed=i, n_rows=n_rows)
            if i >= args.warmup:
                rates.append(r)
                times.append(dt * 1e3)
        value = statistics.median(rates)
        line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(times),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference",
                "config": {"workload": synth.CONFIG_NAMES[PREFILL_CFG], "sample": sample},
                "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores,
                                 "kind": "oracle", "sample": f"{sample} per step"},
                "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    r = run_ours(args, rank, world, local)
    if args.only == "decode":
        r["p_flops"], r["e2e_pre"] = 0, max(r["e2e_pre"], 1e-9)
    if args.only == "prefill":
        r["d_bytes"], r["e2e_dec"] = 0, max(r["e2e_dec"], 1e-9)
    r["pre_ms"], r["dec_ms"] = max(r["pre_ms"], 1e-9), max(r["dec_ms"], 1e-9)
    pre_tflops = job_rate(r["p_flops"], r["pre_ms"], world) / 1e12
    dec_gbs = job_rate(r["d_bytes"], r["dec_ms"], world) / 1e9
    tensor_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    per_gpu_pre = r["p_flops"] / (r["pre_ms"] * 1e-3) / 1e12
    per_gpu_dec = r["d_bytes"] / (r["dec_ms"] * 1e-3) / 1e9
    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, cores, sample, dt, fl, _ = oracle_rate(r["pre"], args.cpu_seconds)
        cpu = {"value": rate, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
               "sample": f"{sample} of the prefill workload, {dt:.1f} s, {fl:.3e} FLOP"}
    launches_per_step = (2 if args.only != "decode" else 0) + (
        (2 if r["splits"] > 1 else 1) if args.only != "prefill" else 0)
    line = {
        "metric": METRIC,
        "value": round(pre_tflops, 3),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(r["total_ms"] / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "prefill " + r["pre"].meta["config"] + " + decode " + r["dec"].meta["config"],
            "prefill_flops_per_step": r["p_flops"],
            "decode_bytes_per_step": r["d_bytes"],
            "decode_num_splits": r["splits"],
            "l2": "prefill inputs larger than L2; 256 MiB read through before each decode call",
            "timing": "median of the timed steps' per-call CUDA-event times",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "tensor", "achieved": round(per_gpu_pre, 2),
            "peak": tensor_peak, "unit": "TFLOP/s",
            "frac": round(per_gpu_pre / tensor_peak, 4),
            "traffic": ncu_traffic("fwd_kernel", "fwd_kernel.cu"),
            "kernel": "fwd_kernel (prepare + persistent launch, CUDA events around attn_fwd)",
            "peak_source": f"{peak_src} bf16 dense burst",
            "nominal_peak": NOMINAL_PEAKS["bf16_tflops"],
            "nominal_frac": round(per_gpu_pre / NOMINAL_PEAKS["bf16_tflops"], 4),
        },
        "decode": {
            "value": round(dec_gbs, 2), "unit": "GB/s", "ms": round(r["dec_ms"], 5),
            "roofline": {
                "bound": "hbm", "achieved": round(per_gpu_dec, 2), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(per_gpu_dec / hbm_peak, 4),
                "traffic": ncu_traffic("decode_split_kernel", "decode_kernel.cu"),
                "kernel": "decode_split_kernel + combine (CUDA events around attn_decode_kvcache)",
                "peak_source": f"{peak_src} copy bandwidth",
                "nominal_peak": NOMINAL_PEAKS["hbm_gbs"],
                "nominal_frac": round(per_gpu_dec / NOMINAL_PEAKS["hbm_gbs"], 4),
            },
            "e2e": {"value": round(job_rate(r["d_bytes"], r["e2e_dec"], world) / 1e9, 2),
                    "unit": "GB/s", "h2d_bytes_per_step": r["h2d_dec"],
                    "d2h_bytes_per_step": r["d2h_dec"],
                    "note": "KV cache resident in HBM; new queries and tables copied in"},
        },
        "prefill_ms": round(r["pre_ms"], 5),
        "e2e": {"value": round(job_rate(r["p_flops"], r["e2e_pre"], world) / 1e12, 3),
                "unit": "TFLOPS", "h2d_bytes_per_step": r["h2d_pre"],
                "d2h_bytes_per_step": r["d2h_pre"],
                "note": "each step copies its inputs in and its results out; copies run on "
                        "their own streams, overlapping the neighbouring steps' attention"},
        "cpu_baseline": cpu,
        "clocks": r["clocks"],
        "gpu_launches": launches_per_step * args.steps,
        "device_status": r["status"],
        "configs": r["extra"],
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
