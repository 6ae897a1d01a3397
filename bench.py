#!/usr/bin/env python
"""Benchmark of the triangle-attention forward on GB300: one JSON line.

A step is one forward pass of the whole path (mask resolution, tile loads,
QK^T, online softmax with -1e9 masking, PV, epilogue with lse/max) over one
batch of the workload.  The default workload is "bf16_long"
(B=1,N=768,H=4,Q=K=768,D=64 bf16, bias bf16, kv_lengths uniform in [0,768]
with all-masked rows); its q/k/v/O (1.2 GB) exceed the 129 MB L2, so no L2
flush is needed between steps.  The other workloads are reported under
"per_config" with an L2 flush before every timed launch.

Metric: effective TFLOP/s = 4*B*N*H*Q*D*sum(K_valid) / time (varlen: 4*H*D
* valid (q,k) pairs / time).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N>1) each rank runs its contiguous range of the workload's
(b, n) slabs with the bias replicated (strong scaling, no data-path
collective); rank 0 prints the line with the max time over ranks.  The main
number is the median over five timed regions of `--steps` launches.
--impl reference times the fp64 CPU oracle on a bounded sample of the
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "fwd effective TFLOP/s and % of GB300 dense-bf16 peak, per config, 1 GPU"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
TIMED_REGIONS = 5
ESIZE = {"f32": 4, "f16": 2, "bf16": 2}


def kernel_source_hash() -> str:
    """SHA-256 over the sources of the tensor-core forward kernels (path + content): tc_*.cu,
    tc_*.cuh, tmem_io.h and internal.h.  The CUDA-core kernels, the backward and the host entry
    points do not change what the measured kernels do, so they are left out."""
    import glob
    import hashlib
    cs = os.path.join(ROOT, "masked_attention_tri_gb300", "csrc")
    files = sorted(glob.glob(os.path.join(cs, "tc_*.cu")) + glob.glob(os.path.join(cs, "tc_*.cuh")) +
                   [os.path.join(cs, "tmem_io.h"), os.path.join(cs, "internal.h")])
    files = [f for f in files if os.path.basename(f) not in ("tc_bwd.cu", "tc_wide.cu")]
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.relpath(f, ROOT).encode())
        h.update(b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu summary (profiles/<kernel>_<workload>.json) taken
    on the current sources, or None when the kernel has changed since the counters were taken."""
    import glob
    cur = kernel_source_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", f"*_{workload}.json"))):
        with open(path) as fh:
            rec = json.load(fh)
        if rec.get("workload") == workload and rec.get("source_sha256") == cur:
            return rec["dram_bytes_per_launch"]
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# Work accounting (effective FLOPs and algorithmic bytes)
# ---------------------------------------------------------------------------

def kv_valid(c) -> torch.Tensor:
    """Per (b,n) count of valid keys: clamp(kv_len,0,K), popcount of the mask, or K."""
    if c.kv_lengths is not None:
        return c.kv_lengths.clamp(0, c.K).to(torch.int64)
    if c.mask is not None:
        return (c.mask.reshape(c.B, c.N, c.K) != 0).sum(-1).to(torch.int64)
    return torch.full((c.B, c.N), c.K, dtype=torch.int64)


def triangle_work(c, slabs=None):
    """(effective flops, algorithmic bytes) of the triangle workload, or of the (b,n) slabs listed."""
    kv = kv_valid(c).reshape(-1)
    if slabs is not None:
        kv = kv[torch.as_tensor(slabs)]
    nslab = kv.numel()
    e, eb = ESIZE[c.dtype], ESIZE[c.bias_dtype]
    flops = 4.0 * c.H * c.Q * c.D * float(kv.sum())
    byts = 2.0 * nslab * c.H * c.Q * c.D * e                      # Q and O
    byts += 2.0 * c.H * c.D * e * float(kv.sum())                 # K and V of valid keys
    byts += float((kv == 0).sum()) * c.H * c.K * c.D * e          # V of all-masked slabs (mean of V)
    byts += c.B * c.H * c.Q * c.K * eb                            # bias, once
    byts += (nslab * c.K) if c.mask is not None else (4 * nslab if c.kv_lengths is not None else 0)
    byts += 8.0 * nslab * c.H * c.Q                               # lse and max
    return flops, byts


def varlen_work(c, window=0):
    """(effective flops, algorithmic bytes) of a packed workload: causal, sliding window (q - window
    < k <= q: sum over q of min(q + 1, window) pairs per sequence) or every pair."""
    L = c.lengths.to(torch.int64)
    if c.mask_mod == "sliding_window":
        W = int(window)
        pairs = float(sum(min(n, W) * (min(n, W) + 1) // 2 + max(n - W, 0) * W for n in L.tolist()))
    elif c.mask_mod == "causal":
        pairs = float((L * (L + 1) // 2).sum())
    else:
        pairs = float((L * L).sum())
    e = ESIZE[c.dtype]
    total = float(L.sum())
    flops = 4.0 * c.H * c.D * pairs
    byts = 4.0 * total * c.H * c.D * e + 8.0 * c.H * total        # Q, K, V, O once; lse, max
    return flops, byts


# ---------------------------------------------------------------------------
# Clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "50"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def gpu_triangle_inputs(c, dev):
    g = lambda t: None if t is None else t.to(dev)  # noqa: E731
    return dict(q=g(c.q), k=g(c.k), v=g(c.v), bias=g(c.bias), mask=g(c.mask), kv_lengths=g(c.kv_lengths))


def make_l2_flusher(dev):
    buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        buf.fill_(1.0)
    return flush


def time_triangle(ta, c, dev, steps, warmup, flush=None, repeats=1, world=1):
    """Device time (ms) per launch: `repeats` timed regions of `steps` back-to-back launches each
    (CUDA events on the launching stream, every region bracketed by a barrier and a synchronize),
    and the median over the regions.  With `flush`, the L2 is flushed before every launch and only
    the launch itself is inside the events."""
    x = gpu_triangle_inputs(c, dev)
    out = torch.empty_like(x["q"])
    lse = torch.empty(c.B, c.N, c.H, c.Q, 1, device=dev, dtype=torch.float32)
    mx = torch.empty_like(lse)

    # The C-ABI call with the pointers resolved once, so host overhead per launch stays small.
    from masked_attention_tri_gb300 import abi
    from masked_attention_tri_gb300.api import _DT, _ptr
    argv = (_ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _DT[x["q"].dtype], _ptr(x["bias"]), _DT[x["bias"].dtype],
            _ptr(None if x["mask"] is None else x["mask"].view(torch.uint8)), _ptr(x["kv_lengths"]),
            c.B, c.N, c.H, c.Q, c.K, c.D, c.scale, _ptr(out), _ptr(lse), _ptr(mx),
            torch.cuda.current_stream(dev).cuda_stream)

    def launch():
        abi.tri_attn_fwd(*argv)

    for _ in range(warmup):
        launch()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    per = []
    for _ in range(repeats):
        barrier(world)
        torch.cuda.synchronize(dev)
        if flush is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                launch()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            per.append(e0.elapsed_time(e1) / steps)
        else:
            tot = 0.0
            for _ in range(steps):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                launch()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                tot += e0.elapsed_time(e1)
            per.append(tot / steps)
        barrier(world)
    return statistics.median(per)


def time_backward(ta, c, dev, steps, warmup, repeats=3, with_dbias=True):
    """Device time (ms) of one backward (dQ, dK, dV, dBias) through the C ABI, with the
    forward's O given (per-row sums dO . O); median of `repeats` timed regions."""
    from masked_attention_tri_gb300 import abi
    from masked_attention_tri_gb300.api import _DT, _ptr
    x = gpu_triangle_inputs(c, dev)
    B, N, H, Q, D = c.q.shape
    K = c.k.shape[3]
    o, lse, _ = ta.triangle_attention(x["q"], x["k"], x["v"], x["bias"], x["mask"], c.scale, True,
                                      kv_lengths=x["kv_lengths"])
    g = torch.Generator("cpu").manual_seed(11)
    d_out = torch.randn(tuple(c.q.shape), generator=g).to(x["q"].dtype).to(dev)
    dq, dk, dv, db = (torch.empty_like(t) for t in (x["q"], x["k"], x["v"], x["bias"]))
    nbytes = abi.tri_attn_bwd_workspace_size(B, N, H, Q, K, D)
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    m8 = None if x["mask"] is None else x["mask"].view(torch.uint8)
    argv = (_ptr(x["q"]), _ptr(x["k"]), _ptr(x["v"]), _DT[x["q"].dtype], _ptr(x["bias"]), _DT[x["bias"].dtype],
            _ptr(m8), _ptr(x["kv_lengths"]), B, N, H, Q, K, D, c.scale, _ptr(lse), _ptr(o), _ptr(d_out), _ptr(dq),
            _ptr(dk), _ptr(dv), _ptr(db) if with_dbias else 0, _ptr(ws), nbytes,
            torch.cuda.current_stream(dev).cuda_stream)
    for _ in range(warmup):
        abi.tri_attn_bwd(*argv)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    per = []
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            abi.tri_attn_bwd(*argv)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        per.append(e0.elapsed_time(e1) / steps)
    return statistics.median(per)


def backward_entry(ta, c, dev, peaks, steps=5, warmup=2, with_dbias=True):
    """The backward of the triangle workload `c`: ms and effective TFLOP/s over its five
    contractions (S, dP, dV, dK, dQ: 10 * B*N*H*Q*K_valid*D, 2.5x the forward's count)."""
    t = time_backward(ta, c, dev, steps, warmup, with_dbias=with_dbias)
    f = 2.5 * triangle_work(c)[0]
    return {"ms": t, "tflops": f / (t * 1e-3) / 1e12,
            "pct_bf16_peak": 100 * f / (t * 1e-3) / (peaks["bf16_tflops"] * 1e12),
            "outputs": "dQ, dK, dV, dBias (summed over N)" if with_dbias else "dQ, dK, dV",
            "path": "per-row sums from the forward's O, per-key-tile gradients on tcgen05 (16-bit, D <= 128)"}


def varlen_backward_entry(ta, c, dev, peaks, steps=5, warmup=2, repeats=3):
    """The backward of the packed workload `c` through `varlen_attention_backward` (its
    BlockMask, the forward's O and lse given): ms per call and effective TFLOP/s over the
    five contractions (2.5x the forward's count)."""
    bm = ta.BlockMask.from_kv_blocks(c.kv_num_blocks.to(dev), c.kv_indices.to(dev), c.full_kv_num_blocks.to(dev),
                                     c.full_kv_indices.to(dev), BLOCK_SIZE=c.block, mask_mod=c.mask_mod)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    cu = c.cu_seqlens.to(dev)
    o, lse, _ = ta.varlen_attention(q, k, v, cu, cu, c.max_seqlen, c.max_seqlen, block_mask=bm, scale=c.scale,
                                    return_aux=True)
    g = torch.Generator("cpu").manual_seed(12)
    d_out = torch.randn(tuple(c.q.shape), generator=g).to(q.dtype).to(dev)

    def call():
        ta.varlen_attention_backward(q, k, v, cu, cu, c.max_seqlen, c.max_seqlen, o, lse, d_out, block_mask=bm,
                                     scale=c.scale)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    per = []
    for _ in range(repeats):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            call()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        per.append(e0.elapsed_time(e1) / steps)
    assert ta.get_status() == 0
    t = statistics.median(per)
    f = 2.5 * varlen_work(c)[0]
    return {"ms": t, "tflops": f / (t * 1e-3) / 1e12,
            "pct_bf16_peak": 100 * f / (t * 1e-3) / (peaks["bf16_tflops"] * 1e12),
            "outputs": "dQ, dK, dV",
            "path": "per-row sums from the forward's O, per-(sequence, head, key block) gradients on tcgen05",
            "timing": "through varlen_attention_backward (argument checks and workspace included)"}


def shard_case(c, world, rank):
    """This rank's contiguous range of (b, n) slabs of a B = 1 workload (the bias replicated)."""
    from masked_attention_tri_gb300.shard import slab_range
    if world == 1:
        return c
    assert c.B == 1, "the benchmark workloads have B = 1"
    n0, n1 = slab_range(c.N, world, rank)
    sl = lambda t: None if t is None else t[:, n0:n1].contiguous()  # noqa: E731
    return synth.TriangleCase(c.name, 1, n1 - n0, c.H, c.Q, c.K, c.D, c.dtype, c.bias_dtype, sl(c.q), sl(c.k),
                              sl(c.v), c.bias, sl(c.mask), sl(c.kv_lengths), c.scale)


def time_varlen(ta, c, dev, steps, warmup, flush, qkv_packed=False, window=0):
    """Device time (ms) per launch of the packed-sequence forward, L2 flushed before each launch.

    qkv_packed: q, k, v read in place from one (total, 3, H, D) buffer
    (NVTE_QKV_INTERLEAVED).  The C-ABI call is made with its pointers resolved
    once (as in `time_triangle`), so the events bracket the kernel and not the
    Python binding's argument checks: the call is enqueued while the L2 flush
    still runs, and the kernel starts right after the first event.
    """
    from masked_attention_tri_gb300 import abi
    from masked_attention_tri_gb300.api import _DT, _ptr
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    cu = c.cu_seqlens.to(dev)
    kn, ki, fn, fi = (t.to(dev) for t in (c.kv_num_blocks, c.kv_indices, c.full_kv_num_blocks, c.full_kv_indices))
    out = torch.empty_like(q)
    lse = torch.empty(c.H, q.shape[0], device=dev, dtype=torch.float32)
    mx = torch.empty_like(lse)
    H, D = c.H, c.D
    if qkv_packed:
        qkv = torch.stack([q, k, v], dim=1).contiguous()
        qq, kk, vv = qkv.unbind(1)
        rs = 3 * H * D
    else:
        qq, kk, vv = q, k, v
        rs = H * D
    mm = {"causal": abi.TA_MASK_CAUSAL, "none": abi.TA_MASK_NONE,
          "sliding_window": abi.TA_MASK_SLIDING_WINDOW}[c.mask_mod]
    argv = (_ptr(qq), _ptr(kk), _ptr(vv), _DT[q.dtype], _ptr(cu), _ptr(cu), len(c.lengths), q.shape[0], k.shape[0],
            c.max_seqlen, c.max_seqlen, H, D, c.scale, _ptr(kn), _ptr(ki), _ptr(fn), _ptr(fi), kn.shape[1],
            kn.shape[2], ki.shape[3], c.block, c.block, mm, window, None, 0, None, abi.TA_F32, rs, rs, rs, _ptr(out),
            _ptr(lse), _ptr(mx),
            torch.cuda.current_stream(dev).cuda_stream)

    def launch():
        abi.tri_attn_varlen_fwd_masked(*argv)

    for _ in range(warmup):
        launch()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    tot = 0.0
    for _ in range(steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        tot += e0.elapsed_time(e1)
    return tot / steps


def e2e_triangle(ta, c, dev, steps, warmup):
    """Same metric through the public API with pinned host buffers; copies inside the timed region.

    Every step copies its inputs host -> device, runs `triangle_attention` and
    copies O, lse and max device -> host.  Steps are pipelined the way a
    server would run them: two sets of device buffers, the input copies of
    step i+1 on one stream, the kernel of step i on the compute stream and the
    result copies of step i-1 on a third, ordered by events.  The timed region
    runs from the first input copy to the last result copy.
    """
    hq, hk, hv, hb = (t.pin_memory() for t in (c.q, c.k, c.v, c.bias))
    hkl = c.kv_lengths.pin_memory() if c.kv_lengths is not None else None
    hm = c.mask.pin_memory() if c.mask is not None else None
    h_in = [t for t in (hq, hk, hv, hb, hkl, hm) if t is not None]
    d_in = [[torch.empty_like(t, device=dev) for t in h_in] for _ in range(2)]
    d_out = [torch.empty_like(hq, device=dev) for _ in range(2)]
    d_lse = [torch.empty(c.B, c.N, c.H, c.Q, 1, device=dev, dtype=torch.float32) for _ in range(2)]
    d_mx = [torch.empty_like(d_lse[0]) for _ in range(2)]
    ho = [torch.empty_like(hq).pin_memory() for _ in range(2)]
    hl = [torch.empty(c.B, c.N, c.H, c.Q, 1, dtype=torch.float32).pin_memory() for _ in range(2)]
    hmx = [torch.empty_like(hl[0]).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = ho[0].numel() * ho[0].element_size() + 2 * hl[0].numel() * 4

    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    s_k = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_done, k_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(k_done[b])  # the kernel of step i-2 has read buffer b
            for d, h in zip(d_in[b], h_in):
                d.copy_(h, non_blocking=True)
            in_done[b].record(s_in)
        s_k.wait_event(in_done[b])
        if started[b]:
            s_k.wait_event(out_done[b])  # the results of step i-2 have left buffer b
        it = iter(d_in[b])
        dq, dk, dv, db = next(it), next(it), next(it), next(it)
        dkl = next(it) if hkl is not None else None
        dm = next(it) if hm is not None else None
        ta.triangle_attention(dq, dk, dv, db, mask=dm, scale=c.scale, return_aux=True, kv_lengths=dkl,
                              out=d_out[b], lse=d_lse[b], mx=d_mx[b])
        k_done[b].record(s_k)
        with torch.cuda.stream(s_out):
            s_out.wait_event(k_done[b])
            ho[b].copy_(d_out[b], non_blocking=True)
            hl[b].copy_(d_lse[b], non_blocking=True)
            hmx[b].copy_(d_mx[b], non_blocking=True)
            out_done[b].record(s_out)
        started[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(warmup, warmup + steps):
        step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / steps, h2d, d2h


def cpu_oracle_sample(c, budget_s: float, max_slabs=None, t_slab=None):
    """Time the oracle (as it stands) on whole (b,n) slabs of the workload; returns
    (effective TFLOP/s, seconds, slabs, threads).  The sample size comes from the time of one
    slab: measured here, or `t_slab` seconds when the caller measured it already."""
    import numpy as np
    import oracle
    threads = oracle.default_threads()
    nslab_total = c.B * c.N
    per = c.H * c.Q

    def rows_of(slabs):
        return np.concatenate([np.arange(s * per, (s + 1) * per, dtype=np.int64) for s in slabs])

    # calibrate on one slab that is not all-masked
    kv = kv_valid(c).reshape(-1)
    order = [int(i) for i in torch.argsort(kv, descending=True)[: max(1, nslab_total)]]
    probe = [order[len(order) // 2]]
    if t_slab is None:
        t0 = time.perf_counter()
        oracle.tri_fwd(c.q, c.k, c.v, c.bias, mask=c.mask, kv_lengths=c.kv_lengths, scale=c.scale,
                       rows=rows_of(probe), threads=threads)
        t1 = time.perf_counter() - t0
    else:
        t1 = t_slab
    n = max(1, min(nslab_total, int(budget_s / max(t1, 1e-6))))
    if max_slabs:
        n = min(n, max_slabs)
    slabs = [int(s) for s in np.linspace(0, nslab_total - 1, n).round().astype(int)]
    slabs = sorted(set(slabs))
    t0 = time.perf_counter()
    oracle.tri_fwd(c.q, c.k, c.v, c.bias, mask=c.mask, kv_lengths=c.kv_lengths, scale=c.scale, rows=rows_of(slabs),
                   threads=threads)
    dt = time.perf_counter() - t0
    flops, _ = triangle_work(c, slabs)
    return flops / dt / 1e12, dt, slabs, threads


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, world, rank):
    """The oracle arm: the fp64 CPU oracle, as it stands, on bounded samples of the workload."""
    if rank != 0:
        return
    c = synth.TRIANGLE_WORKLOADS[args.workload]()
    # The whole run stays near 150 s of oracle work: each step is a sample of
    # 150 / (steps + warmup) seconds (at least one slab), sized from one slab's time.
    budget = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    _, t_slab, _, _ = cpu_oracle_sample(c, 0.0, max_slabs=1)
    vals = []
    times = []
    info = None
    for i in range(args.warmup + args.steps):
        v, dt, slabs, threads = cpu_oracle_sample(c, budget, t_slab=t_slab)
        if i >= args.warmup:
            vals.append(v)
            times.append(dt)
            info = (slabs, threads)
    slabs, threads = info
    value = statistics.mean(vals)
    flops, _ = triangle_work(c, slabs)
    sample = f"{len(slabs)} of {c.B * c.N} (b,n) slabs of {args.workload} (all H*Q rows each), {flops:.3e} effective FLOP"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(c, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(c, world=1):
    """The `config` of the JSON line; both arms print the same dict for the same workload."""
    desc = {
        "bf16_long": "bf16 long: B=1,N=768,H=4,Q=K=768,D=64; q,k,v,bias ~N(0,1) bf16; kv_lengths U[0,768] incl. 0",
        "bf16_pairstack": "bf16 pair-stack: B=1,N=384,H=4,Q=K=384,D=32; bias ~N(0,4) bf16; kv_lengths U[192,384]",
        "fp16_kvlen": "fp16: B=1,N=128,H=2,Q=K=128,D=32; bias fp32; kv_lengths=96",
        "fp16_dense": "fp16: B=1,N=128,H=2,Q=K=128,D=32; bias fp32; dense Bernoulli(0.5) key mask",
        "tiny_fp32": "tiny fp32: B=1,N=32,H=2,Q=K=32,D=32; no mask",
    }.get(c.name, c.name)
    big = 2 * c.B * c.N * c.H * (c.Q + c.K) * c.D * ESIZE[c.dtype] > L2_BYTES
    return {"workload": desc, "B": c.B, "N": c.N, "H": c.H, "Q": c.Q, "K": c.K, "D": c.D,
            "qkv_dtype": c.dtype, "bias_dtype": c.bias_dtype,
            "mask": "kv_lengths" if c.kv_lengths is not None else ("dense" if c.mask is not None else "none"),
            "global_batch": c.B, "parallelism": f"n_split{world}" if world > 1 else "single",
            "l2": "inputs larger than L2 (q,k,v,O vs 129 MB)" if big else "L2 flushed before each launch"}


def run_only(args):
    """Launch one workload `warmup` + `steps` times (L2 flushed before each timed launch) and print
    its time; used as the command under ncu."""
    import masked_attention_tri_gb300 as ta
    from masked_attention_tri_gb300 import build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    flush = make_l2_flusher(dev)
    c = synth.WORKLOADS[args.only]()
    if isinstance(c, synth.VarlenCase):
        window = 512 if c.mask_mod == "sliding_window" else 0  # the window workload's window
        f, _ = varlen_work(c, window=window)
        t = time_varlen(ta, c, dev, args.steps, args.warmup, flush, window=window)
    else:
        f, _ = triangle_work(c)
        t = time_triangle(ta, c, dev, args.steps, args.warmup, flush=flush)
    status = ta.get_status()
    assert status == 0, f"device status {status}"
    print(json.dumps({"only": args.only, "us": 1e3 * t, "tflops": f / (t * 1e-3) / 1e12, "steps": args.steps,
                      "warmup": args.warmup}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bf16_long", choices=sorted(synth.TRIANGLE_WORKLOADS))
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--only-backward", action="store_true",
                    help="time only the backward of the bf16_long workload (one JSON line)")
    ap.add_argument("--backward-no-dbias", action="store_true", help="with --only-backward: skip dBias")
    ap.add_argument("--backward-d", type=int, default=64, choices=(64, 128),
                    help="with --only-backward: the head dimension (128: the same shape with D = 128)")
    ap.add_argument("--backward-varlen", action="store_true",
                    help="with --only-backward: the backward of the bf16_varlen packed sequences instead")
    ap.add_argument("--backward-n", type=int, default=None,
                    help="with --only-backward: the first N of the workload's 768 n rows only (a small case)")
    ap.add_argument("--only", default=None, choices=sorted(synth.WORKLOADS),
                    help="profiling mode: warm-up + timed launches of this one workload, a short JSON line, "
                         "nothing else (no per-config, end-to-end or CPU legs)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.only_backward:
        import masked_attention_tri_gb300 as ta
        dev = torch.device("cuda", 0)
        if args.backward_varlen:
            line = varlen_backward_entry(ta, synth.bf16_varlen(), dev, load_peaks()[0], args.steps, args.warmup)
            line["workload"] = "bf16_varlen backward"
            print(json.dumps(line))
            return
        c = synth.bf16_long() if args.backward_d == 64 else synth.bf16_long_d128()
        name = "bf16_long" if args.backward_d == 64 else "bf16_long_d128"
        if args.backward_n:
            n = args.backward_n
            c.q, c.k, c.v = (t[:, :n].contiguous() for t in (c.q, c.k, c.v))
            c.kv_lengths = c.kv_lengths[:, :n].contiguous()
            c.N = n
        line = backward_entry(ta, c, dev, load_peaks()[0], args.steps, args.warmup,
                              with_dbias=not args.backward_no_dbias)
        line["workload"] = f"{name} backward, first {c.N} of 768 n rows" if args.backward_n else f"{name} backward"
        print(json.dumps(line))
        return
    if args.only:
        run_only(args)
        return

    import masked_attention_tri_gb300 as ta
    from masked_attention_tri_gb300 import build
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    peaks, peak_kind = load_peaks()
    c_all = synth.TRIANGLE_WORKLOADS[args.workload]()
    flops_all, _ = triangle_work(c_all)
    # Each rank runs its contiguous range of (b, n) slabs (the bias replicated); one GPU runs it all.
    c = shard_case(c_all, world, rank)
    flops, byts = triangle_work(c)

    barrier(world)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    sampler.start()
    ms = time_triangle(ta, c, dev, args.steps, args.warmup, repeats=TIMED_REGIONS, world=world)
    clocks = sampler.stop()
    status = ta.get_status()
    barrier(world)
    ms_max = max_over_ranks(ms, world, dev)
    assert status == 0, f"device status {status}"

    value = flops_all / (ms_max * 1e-3) / 1e12
    t_mma = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    bound = "hbm" if t_hbm >= t_mma else "tensor"
    if bound == "hbm":
        achieved = byts / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic(args.workload)}
    else:
        achieved = flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": None}
    roof["peak_source"] = f"{peak_kind} (MEASURED_PEAKS.json burst)" if peak_kind == "measured" else "fallback"
    roof["algorithmic_bytes"] = byts
    roof["effective_flops"] = flops
    roof["two_term_roofline_frac"] = max(t_mma, t_hbm) / (ms * 1e-3)

    barrier(world)
    e2e_ms, h2d, d2h = e2e_triangle(ta, c, dev, max(3, min(args.steps, 50)), 3)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    h2d = int(max_over_ranks(float(h2d), world, dev))
    d2h = int(max_over_ranks(float(d2h), world, dev))

    per_config = {}
    if not args.no_per_config and rank == 0:
        flush = make_l2_flusher(dev)
        for name in ("tiny_fp32", "fp16_kvlen", "fp16_dense", "bf16_pairstack"):
            cc = synth.TRIANGLE_WORKLOADS[name]()
            f, b = triangle_work(cc)
            t = time_triangle(ta, cc, dev, 50, 5, flush=flush)
            per_config[name] = {"us": 1e3 * t, "tflops": f / (t * 1e-3) / 1e12,
                                "pct_bf16_peak": 100 * f / (t * 1e-3) / (peaks["bf16_tflops"] * 1e12),
                                "two_term_roofline_frac": max(f / (peaks["bf16_tflops"] * 1e12),
                                                              b / (peaks["hbm_gbs"] * 1e9)) / (t * 1e-3),
                                "l2": "flushed before each launch"}
        vc = synth.bf16_varlen()
        f, b = varlen_work(vc)
        t = time_varlen(ta, vc, dev, 50, 5, flush)
        per_config["bf16_varlen"] = {"us": 1e3 * t, "tflops": f / (t * 1e-3) / 1e12,
                                     "pct_bf16_peak": 100 * f / (t * 1e-3) / (peaks["bf16_tflops"] * 1e12),
                                     "two_term_roofline_frac": max(f / (peaks["bf16_tflops"] * 1e12),
                                                                   b / (peaks["hbm_gbs"] * 1e9)) / (t * 1e-3),
                                     "lengths": vc.lengths.tolist(), "l2": "flushed before each launch"}
        t = time_varlen(ta, vc, dev, 50, 5, flush, qkv_packed=True)
        per_config["bf16_varlen_qkvpacked"] = {
            "us": 1e3 * t, "tflops": f / (t * 1e-3) / 1e12,
            "pct_bf16_peak": 100 * f / (t * 1e-3) / (peaks["bf16_tflops"] * 1e12),
            "two_term_roofline_frac": max(f / (peaks["bf16_tflops"] * 1e12), b / (peaks["hbm_gbs"] * 1e9)) / (t * 1e-3),
            "layout": "one (total, 3, H, D) buffer read in place", "l2": "flushed before each launch"}
        per_config["bf16_varlen_backward"] = varlen_backward_entry(ta, vc, dev, peaks)
        # The widened rows, measured like the others: a sliding-window BlockMask on the packed
        # sequences (mask_mod sliding_window, window 512, its block lists) and D = 256.
        wc = synth.bf16_varlen_window512()
        f, b = varlen_work(wc, window=512)
        t = time_varlen(ta, wc, dev, 50, 5, flush, window=512)
        per_config["bf16_varlen_window512"] = {
            "us": 1e3 * t, "tflops": f / (t * 1e-3) / 1e12,
            "pct_bf16_peak": 100 * f / (t * 1e-3) / (peaks["bf16_tflops"] * 1e12),
            "two_term_roofline_frac": max(f / (peaks["bf16_tflops"] * 1e12), b / (peaks["hbm_gbs"] * 1e9)) / (t * 1e-3),
            "mask": "sliding window of 512 keys (valid pairs counted)", "l2": "flushed before each launch"}
        dc = synth.bf16_d256()
        f, b = triangle_work(dc)
        t = time_triangle(ta, dc, dev, 20, 3, flush=flush)
        per_config["bf16_d256"] = {"us": 1e3 * t, "tflops": f / (t * 1e-3) / 1e12,
                                   "pct_bf16_peak": 100 * f / (t * 1e-3) / (peaks["bf16_tflops"] * 1e12),
                                   "two_term_roofline_frac": max(f / (peaks["bf16_tflops"] * 1e12),
                                                                 b / (peaks["hbm_gbs"] * 1e9)) / (t * 1e-3),
                                   "path": "tensor cores, 64-key tiles (D in (128, 256])", "l2": "flushed before each launch"}
        per_config["bf16_long"] = {"us": 1e3 * ms, "tflops": flops / (ms * 1e-3) / 1e12,
                                   "pct_bf16_peak": 100 * flops / (ms * 1e-3) / (peaks["bf16_tflops"] * 1e12),
                                   "two_term_roofline_frac": roof["two_term_roofline_frac"],
                                   "l2": "inputs larger than L2"}
        per_config["bf16_long_backward"] = backward_entry(ta, c, dev, peaks)
        c128 = synth.bf16_long_d128()
        per_config["bf16_long_d128_backward"] = backward_entry(ta, c128, dev, peaks)
        del c128

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, slabs, threads = cpu_oracle_sample(c, args.cpu_budget)
        fl, _ = triangle_work(c, slabs)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{len(slabs)} of {c.B * c.N} (b,n) slabs of {args.workload} (all H*Q rows each), "
                         f"{fl:.3e} effective FLOP in {dt:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": c.dtype, "data": "synthetic", "config": workload_config(c_all, world),
            "pct_bf16_peak": 100 * flops_all / (ms_max * 1e-3) / (peaks["bf16_tflops"] * 1e12),
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": flops_all / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps, "timed_regions": TIMED_REGIONS,
            "timing": f"median over {TIMED_REGIONS} timed regions of {args.steps} launches (one launch per step)",
            "clocks": clocks, "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
