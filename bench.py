"""Throughput of attention with an attention sink on GB300, against its roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload extend_varlen] [--no-extra]

Prints ONE JSON line (rank 0).  The headline workload is the varlen chunked
extend with a learnable sink (8 requests, prefix U{0..16384} + chunk
U{512..8192}, Hq 64, Hkv 8, d 64): one step = one attn_sink_fwd call over the
whole batch; the metric is algorithmic attention TFLOP/s (4*d FLOPs per
visible (query, key) pair per head).  The decode workloads (HBM-bound, KV
GB/s) and the training step (forward + backward TFLOP/s) are measured in the
same run and reported under "workloads" with their own rooflines.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the stream the library launches on; L2 is flushed (a 512 MB write) before
every timed step, outside the events.  Multi-GPU (torchrun): every rank runs
an independent replica (the path shards by request; no collective), the time
is the max over ranks and the value the sum of all ranks' work.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum from an ncu capture of that kernel on the workload).
# Keyed by kernel + workload; each entry records the hash of the kernel source
# it was measured on and is reported only while that source is unchanged.
NCU_TRAFFIC = {
    # fwd_kernel<64>: 443.6 MB read + 258.8 MB written per launch
    "fwd_kernel/extend_varlen": {"src": "01113da51d930ad5", "bytes": 702_400_512},
    # fwd_kernel<64>, first 1024 + last 7168 window: 488.6 MB + 267.9 MB
    "fwd_kernel/extend_window": {"src": "01113da51d930ad5", "bytes": 756_435_968},
    # fwd_kernel<64> reading K/V through a page-16 table: 445.6 MB + 258.6 MB
    "fwd_kernel/extend_paged": {"src": "01113da51d930ad5", "bytes": 704_219_904},
    # fwd2_kernel<128> (two query heads per CTA): 998.5 MB + 272.9 MB
    "fwd_kernel/extend_d128": {"src": "01113da51d930ad5", "bytes": 1_271_381_504},
    # bwd_main_kernel<64>: 2.684 GB read + 1.048 GB written per launch
    "bwd_main_kernel/train": {"src": "8450e18315e5943f", "bytes": 3_731_941_632},
    # bwd_main128_kernel on the head-dim-128 training step: 1.910 GB + 0.946 GB
    "bwd_main128_kernel/train_d128": {"src": "8450e18315e5943f", "bytes": 2_856_080_128},
    # decode_split_kernel: 1.943 GB + 0.010 GB
    "decode/decode_sink": {"src": "5bc7ecc88224f35a", "bytes": 1_953_821_440},
    # decode_split_kernel: 1.074 GB + 0.007 GB
    "decode/decode_window": {"src": "5bc7ecc88224f35a", "bytes": 1_080_700_928},
}


def _src_hash(name):
    p = os.path.join(ROOT, "paged_kv_sink_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _traffic(key, src):
    ent = NCU_TRAFFIC.get(key)
    if not ent or ent["src"] != _src_hash(src):
        return None
    return ent["bytes"]


def check_status(ext, what):
    """The kernels report bad inputs and timed-out waits through a sticky device
    status instead of faulting; a timed call that raised one did not do the work
    it is credited with, so the bench fails instead of printing a number."""
    st = ext.device_status()
    if st != 0:
        raise RuntimeError(f"{what}: device status {st:#x} after the timed calls")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            out = dict(FALLBACK_PEAKS)
            for k in out:
                for cand in (k, k.replace("_gbs", "_GBps")):
                    if cand in d and isinstance(d[cand], (int, float)):
                        out[k] = float(d[cand])
            return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Work counts (algorithmic, from the definition)

def fwd_flops(p):
    """4*d FLOPs (QK^T and PV) per visible (query, key) pair per query head."""
    import numpy as np
    total = 0
    for Lq, Lk in zip(p.seqlens_q, p.seqlens_k):
        off = Lk - Lq
        if p.win_last <= 0:
            if p.causal:
                pos = np.arange(Lq) + off
                total += int(np.clip(pos + 1, 0, Lk).sum())
            else:
                total += Lq * Lk
        else:
            pos = np.arange(Lq) + off
            n = np.clip(pos + 1, 0, None)
            first = np.minimum(p.win_first, n)
            last_begin = np.maximum(n - p.win_last, first)
            total += int((first + (n - last_begin)).sum())
    return 4.0 * p.head_dim * p.hq * total


def _visible_counts(seqlens, F, W):
    out = []
    for L in seqlens:
        if W <= 0:
            out.append(L)
        else:
            first = min(F, L)
            last_begin = max(L - W, first)
            out.append(first + (L - last_begin))
    return out


# ---------------------------------------------------------------------------
# Our arm

def _flush_buf(torch, dev):
    return torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)


def max_over_ranks(torch, dist, values, device="cpu"):
    """Element-wise maximum of per-rank values over all ranks (identity at N = 1)."""
    if dist is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def sum_over_ranks(torch, dist, value, device="cpu"):
    """Sum of a per-rank value over all ranks (identity at N = 1)."""
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_rate(work_all_ranks, seconds_max):
    """Whole-job throughput: the work all ranks did over the slowest rank's time."""
    return work_all_ranks / seconds_max


def rank_sync(torch, dist):
    """Barrier across ranks (when there are several) and a device synchronise."""
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()


def time_steps(torch, fn, steps, warmup, flush, sync=None):
    """Per-step device times (CUDA events on the launching stream), L2 flushed
    between steps outside the events; `sync` brackets the timed steps."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if sync is not None:
        sync()
    times = []
    for _ in range(steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if sync is not None:
        sync()
    return times


def bench_extend(torch, ext, dev, p, steps, warmup, flush, peaks, peak_src, sync=None):
    q, k, v = p.q.to(dev), p.k.to(dev), p.v.to(dev)
    sink = p.sink.to(dev)
    cq, ck = p.cu_seqlens_q.to(dev), p.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((p.hq, q.shape[0]), dtype=torch.float32, device=dev)

    def step():
        ext.attn_sink_fwd(q, k, v, sink, cq, ck, p.max_seqlen_q, p.max_seqlen_k, p.win_first, p.win_last,
                          out=out, lse=lse)

    times = time_steps(torch, step, steps, warmup, flush, sync)
    flops = fwd_flops(p)  # visible (query, key) pairs only: keys a window skips are work avoided
    ms = sum(times) / len(times)
    achieved = flops / (ms * 1e-3) / 1e12
    kname = "attn::prefill::fwd2_kernel" if p.head_dim == 128 and (p.hq // p.hkv) % 2 == 0 else "attn::prefill::fwd_kernel"
    roof = {"kernel": kname, "bound": "tensor", "achieved": achieved,
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
            "peak_source": f"bf16 burst, {peak_src}",
            "traffic": _traffic("fwd_kernel/" + p.name.split()[0], "prefill_fwd.cu"),
            "algorithmic_flops_per_launch": flops}
    return ms, flops, roof, times


def e2e_extend(torch, ext, dev, p, steps, warmup):
    """Same metric through the public call with host buffers: attn_sink_fwd_host
    takes the pinned host tensors, copies every request's q/k/v rows to the
    device, runs the forward and copies out/lse back (pipelined against the
    kernels); all of it is inside the timed region, and the step ends when the
    host buffers hold the results."""
    hq_ = [t.pin_memory() for t in (p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)]
    out_h = torch.empty_like(p.q).pin_memory()
    lse_h = torch.empty((p.hq, p.q.shape[0]), dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream()

    def step():
        ext.attn_sink_fwd_host(*hq_, out=out_h, lse=lse_h)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    h2d = sum(t.numel() * t.element_size() for t in hq_)
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
    return ms, h2d, d2h


def bench_decode(torch, ext, dev, dc, steps, warmup, flush, peaks, peak_src):
    t = dict(q=dc.q.to(dev), kc=dc.k_cache.to(dev), vc=dc.v_cache.to(dev), pt=dc.page_table.to(dev),
             sl=dc.seqlens.to(dev), sink=None if dc.sink is None else dc.sink.to(dev))
    out = torch.empty_like(t["q"])
    lse = torch.empty((dc.batch, dc.hq), dtype=torch.float32, device=dev)

    def step():
        ext.attn_sink_decode_paged(t["q"], t["kc"], t["vc"], t["pt"], t["sl"], t["sink"], dc.win_first,
                                   dc.win_last, out=out, lse=lse)

    times = time_steps(torch, step, steps, warmup, flush)
    nvis = _visible_counts(dc.seqlens.tolist(), dc.win_first, dc.win_last)
    kv_bytes = sum(nvis) * 2 * dc.hkv * dc.head_dim * 2
    ms = sum(times) / len(times)
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    del t
    return {"metric": "decode KV GB/s", "value": gbs, "unit": "GB/s", "ms_per_step": ms,
            "kv_bytes": kv_bytes,
            "roofline": {"kernel": "attn::decode::decode_split_kernel + decode_combine_kernel (whole call)",
                         "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": peak_src,
                         "traffic": _traffic(f"decode/{dc.name.split()[0]}", "decode.cu")}}


def bench_train(torch, ext, dev, p, steps, warmup, flush, peaks, peak_src):
    """One training step = attn_sink_fwd + attn_sink_bwd over the whole batch.
    FLOPs: forward 4*d per visible pair per head; backward 2.5x that (five
    GEMMs including the recomputed S), the usual convention."""
    q, k, v = p.q.to(dev), p.k.to(dev), p.v.to(dev)
    sink, dout = p.sink.to(dev), p.dout.to(dev)
    cq, ck = p.cu_seqlens_q.to(dev), p.cu_seqlens_k.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((p.hq, q.shape[0]), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dsink = torch.empty_like(sink)
    stream = torch.cuda.current_stream()
    fwd_ms, bwd_ms = [], []

    def fwd():
        ext.attn_sink_fwd(q, k, v, sink, cq, ck, p.max_seqlen_q, p.max_seqlen_k, out=out, lse=lse)

    def bwd():
        ext.attn_sink_bwd(q, k, v, sink, out, lse, dout, cq, ck, p.max_seqlen_q, p.max_seqlen_k, dq=dq, dk=dk,
                          dv=dv, dsink=dsink)

    for _ in range(warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    for _ in range(steps):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        fwd()
        e[1].record(stream)
        bwd()
        e[2].record(stream)
        torch.cuda.synchronize()
        fwd_ms.append(e[0].elapsed_time(e[1]))
        bwd_ms.append(e[1].elapsed_time(e[2]))
    ff = fwd_flops(p)
    bf = 2.5 * ff
    fm, bm = sum(fwd_ms) / steps, sum(bwd_ms) / steps
    total = (ff + bf) / ((fm + bm) * 1e-3) / 1e12
    main = "bwd_main128_kernel" if p.head_dim == 128 else "bwd_main_kernel"
    bw_ach = bf / (bm * 1e-3) / 1e12
    return {"metric": "attn fwd+bwd TFLOP/s", "value": total, "unit": "TFLOP/s", "ms_per_step": fm + bm,
            "fwd_ms": fm, "bwd_ms": bm, "fwd_tflops": ff / (fm * 1e-3) / 1e12, "bwd_tflops": bw_ach,
            "algorithmic_tflop_per_step": (ff + bf) / 1e12,
            "roofline": {"kernel": f"attn_sink_bwd call ({main} + preprocess + dq convert)",
                         "bound": "tensor", "achieved": bw_ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": bw_ach / peaks["bf16_tflops"], "peak_source": f"bf16 burst, {peak_src}",
                         "traffic": _traffic(f"{main}/" + p.name.split()[0], "bwd.cu"),
                         "algorithmic_flops_per_launch": bf}}


def bench_extend_paged(torch, ext, dev, pe, steps, warmup, flush, peaks, peak_src):
    """The varlen extend through a page table: each step appends the chunk's K/V
    into the cache and runs the paged forward (one attn_sink_fwd_paged call).
    FLOPs as the contiguous extend (4*d per visible pair per query head)."""
    t = dict(q=pe.q.to(dev), kc=pe.k_cache.to(dev), vc=pe.v_cache.to(dev), pt=pe.page_table.to(dev),
             cq=pe.cu_seqlens_q.to(dev), sk=pe.seqlens_k.to(dev), sink=pe.sink.to(dev),
             kn=pe.k_new.to(dev), vn=pe.v_new.to(dev))
    out = torch.empty_like(t["q"])
    lse = torch.empty((pe.hq, pe.q.shape[0]), dtype=torch.float32, device=dev)

    def step():
        ext.attn_sink_fwd_paged(t["q"], t["kc"], t["vc"], t["pt"], t["cq"], t["sk"], pe.max_seqlen_q,
                                pe.max_seqlen_k, t["sink"], t["kn"], t["vn"], pe.win_first, pe.win_last,
                                out=out, lse=lse)

    times = time_steps(torch, step, steps, warmup, flush)
    ms = sum(times) / len(times)

    class _Lens:  # the FLOP count only needs the lengths, windows and head sizes
        seqlens_q = pe.seqlens_q
        seqlens_k = pe.seqlens_k.tolist()
        win_first, win_last, causal = pe.win_first, pe.win_last, pe.causal
        head_dim, hq = pe.q.shape[2], pe.hq

    flops = fwd_flops(_Lens)
    tf = flops / (ms * 1e-3) / 1e12
    del t
    return {"metric": "attn TFLOP/s", "value": tf, "unit": "TFLOP/s", "ms_per_step": ms,
            "algorithmic_tflop_per_step": flops / 1e12, "page_size": pe.page_size,
            "roofline": {"kernel": "attn_sink_fwd_paged call (kv_append_kernel + fwd_kernel, paged loads)",
                         "bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "peak_source": f"bf16 burst, {peak_src}",
                         "traffic": _traffic("fwd_kernel/extend_paged", "prefill_fwd.cu"),
                         "algorithmic_flops_per_launch": flops}}


def bench_decode_append(torch, ext, dev, dc, steps, warmup, flush, peaks, peak_src):
    """Decode with the new token's K/V appended in the same call, launched
    eagerly and replayed from a CUDA graph.  Bytes: the visible K/V as in
    bench_decode (the appended row is one of them)."""
    g = torch.Generator().manual_seed(1)
    kn = torch.randn(dc.batch, dc.hkv, dc.head_dim, generator=g).to(torch.bfloat16).to(dev)
    vn = torch.randn(dc.batch, dc.hkv, dc.head_dim, generator=g).to(torch.bfloat16).to(dev)
    t = dict(q=dc.q.to(dev), kc=dc.k_cache.to(dev), vc=dc.v_cache.to(dev), pt=dc.page_table.to(dev),
             sl=dc.seqlens.to(dev), sink=None if dc.sink is None else dc.sink.to(dev))
    out = torch.empty_like(t["q"])
    lse = torch.empty((dc.batch, dc.hq), dtype=torch.float32, device=dev)

    def step():
        ext.attn_sink_decode_paged_append(t["q"], kn, vn, t["kc"], t["vc"], t["pt"], t["sl"], t["sink"],
                                          dc.win_first, dc.win_last, out=out, lse=lse)

    times = time_steps(torch, step, steps, warmup, flush)
    ms = sum(times) / len(times)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        step()
    times_g = time_steps(torch, graph.replay, steps, warmup, flush)
    ms_g = sum(times_g) / len(times_g)
    nvis = _visible_counts(dc.seqlens.tolist(), dc.win_first, dc.win_last)
    kv_bytes = sum(nvis) * 2 * dc.hkv * dc.head_dim * 2
    gbs = kv_bytes / (ms * 1e-3) / 1e9
    del t
    return {"metric": "decode KV GB/s", "value": gbs, "unit": "GB/s", "ms_per_step": ms,
            "graph_replay_ms_per_step": ms_g, "graph_replay_gbs": kv_bytes / (ms_g * 1e-3) / 1e9,
            "kv_bytes": kv_bytes,
            "roofline": {"kernel": "attn_sink_decode_paged_append call (kv_append + split + combine)",
                         "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "peak_source": peak_src, "traffic": None}}


# ---------------------------------------------------------------------------
# CPU baseline (the oracle as it stands, on a bounded sample)

def _sample_pairs(p, b):
    Lq, Lk = p.seqlens_q[b], p.seqlens_k[b]
    return sum(max(0, min(Lk - Lq + i + 1, Lk)) for i in range(Lq))


def cpu_baseline_extend(p, budget_s=15.0):
    """Sample: every row of the longest request, query heads 0..n-1, n doubled
    until the oracle run takes about a third of the budget."""
    import numpy as np
    from oracle import attn_sink_oracle as orc
    threads = _blas_threads()
    b = int(np.argmax(p.seqlens_q))
    nh = 1
    while True:
        t0 = time.perf_counter()
        orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k, p.win_first, p.win_last,
                     p.causal, p.scale, heads=range(nh), requests=[b])
        elapsed = time.perf_counter() - t0
        if elapsed > budget_s / 3 or nh >= p.hq:
            break
        nh = min(p.hq, nh * 2)
    work = 4.0 * p.head_dim * nh * _sample_pairs(p, b)
    return {"value": work / elapsed / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 numpy oracle, request {b} (all {p.seqlens_q[b]} rows), {nh} of {p.hq} "
                      f"heads ({work/1e9:.1f} GFLOP) in {elapsed:.1f} s"}


def cpu_baseline_decode(dc, budget_s=10.0):
    from oracle import attn_sink_oracle as orc
    threads = _blas_threads()
    n = 1
    while True:
        reqs = list(range(min(n, dc.batch)))
        t0 = time.perf_counter()
        orc.attn_decode_paged(dc.q, dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens, dc.page_size,
                              dc.sink, dc.win_first, dc.win_last, dc.scale, requests=reqs)
        el = time.perf_counter() - t0
        if el > budget_s / 3 or len(reqs) == dc.batch:
            break
        n *= 2
    nvis = _visible_counts(dc.seqlens.tolist()[:len(reqs)], dc.win_first, dc.win_last)
    b = sum(nvis) * 2 * dc.hkv * dc.head_dim * 2
    return {"value": b / el / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 numpy oracle, {len(reqs)} of {dc.batch} requests, all heads, {el:.1f} s"}


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="extend_varlen")
    ap.add_argument("--no-extra", action="store_true", help="skip the decode / training workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU baseline")
    ap.add_argument("--only", default=None,
                    choices=["decode_sink", "decode_window", "train", "extend_paged", "decode_append",
                             "extend_window", "extend_varlen", "extend_d128", "train_d128"],
                    help="run one secondary workload alone and print its line (for profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import torch
    from paged_kv_sink_gb300 import workloads as wl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    if args.impl == "reference":
        if rank != 0:
            return
        return reference_arm(args, wl)

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import paged_kv_sink_gb300 as ext
    ext.lib()
    peaks, peak_src = load_peaks()
    flush = _flush_buf(torch, dev)

    if args.only:
        w = wl.workload("decode_sink" if args.only == "decode_append" else args.only, seed=0)
        if args.only in ("train", "train_d128"):
            r = bench_train(torch, ext, dev, w, args.steps, args.warmup, flush, peaks, peak_src)
        elif args.only == "extend_paged":
            r = bench_extend_paged(torch, ext, dev, w, args.steps, args.warmup, flush, peaks, peak_src)
        elif args.only == "decode_append":
            r = bench_decode_append(torch, ext, dev, w, args.steps, args.warmup, flush, peaks, peak_src)
        elif args.only in ("extend_window", "extend_varlen", "extend_d128"):
            ms, flops, roof, _ = bench_extend(torch, ext, dev, w, args.steps, args.warmup, flush, peaks, peak_src)
            r = {"metric": "attn TFLOP/s (visible pairs)" if args.only == "extend_window" else "attn TFLOP/s",
                 "value": roof["achieved"], "unit": "TFLOP/s", "ms_per_step": ms,
                 "algorithmic_tflop_per_step": flops / 1e12, "roofline": roof}
        else:
            r = bench_decode(torch, ext, dev, w, args.steps, args.warmup, flush, peaks, peak_src)
        check_status(ext, args.only)
        if rank == 0:
            print(json.dumps({"workload": w.name, **r}))
        return

    # Every rank runs the same seeded workload: N replicas with fixed work per GPU.
    p = wl.workload(args.workload, seed=0)
    with ClockSampler(local) as clk:
        ms, flops, roof, times = bench_extend(torch, ext, dev, p, args.steps, args.warmup, flush, peaks,
                                              peak_src, sync=lambda: rank_sync(torch, dist))
    clocks = clk.summary()
    check_status(ext, p.name)
    e2e_ms, h2d, d2h = e2e_extend(torch, ext, dev, p, max(3, args.steps // 4), 2)
    check_status(ext, p.name + " (host buffers)")

    ms_max, e2e_ms = max_over_ranks(torch, dist, [ms, e2e_ms], device=dev)
    flops_all = sum_over_ranks(torch, dist, flops, device=dev)
    value = job_rate(flops_all, ms_max * 1e-3) / 1e12
    e2e_value = job_rate(flops_all, e2e_ms * 1e-3) / 1e12

    extra = {}
    if not args.no_extra:
        for name in ("decode_sink", "decode_window"):
            dc = wl.workload(name, seed=0)
            r = bench_decode(torch, ext, dev, dc, args.steps, args.warmup, flush, peaks, peak_src)
            if rank == 0 and not args.no_cpu and world == 1:
                r["cpu_baseline"] = cpu_baseline_decode(dc)
            check_status(ext, name)
            extra[name] = r
            del dc
        tr = wl.workload("train", seed=0)
        extra["train"] = bench_train(torch, ext, dev, tr, max(3, args.steps // 2), args.warmup, flush, peaks,
                                     peak_src)
        check_status(ext, "train")
        del tr
        pw = wl.workload("extend_window", seed=0)
        ms_w, flops_w, roof_w, _ = bench_extend(torch, ext, dev, pw, max(3, args.steps // 2), args.warmup, flush,
                                                peaks, peak_src)
        check_status(ext, "extend_window")
        extra["extend_window"] = {"metric": "attn TFLOP/s (visible pairs)", "value": roof_w["achieved"],
                                  "unit": "TFLOP/s", "ms_per_step": ms_w,
                                  "algorithmic_tflop_per_step": flops_w / 1e12, "workload": pw.name,
                                  "roofline": roof_w}
        del pw
        pe = wl.workload("extend_paged", seed=0)
        extra["extend_paged"] = bench_extend_paged(torch, ext, dev, pe, max(3, args.steps // 2), args.warmup,
                                                   flush, peaks, peak_src)
        check_status(ext, "extend_paged")
        del pe
        dc = wl.workload("decode_sink", seed=0)
        extra["decode_sink_append"] = bench_decode_append(torch, ext, dev, dc, args.steps, args.warmup, flush,
                                                          peaks, peak_src)
        check_status(ext, "decode_sink_append")
        del dc

    line = {
        "metric": "attn TFLOP/s (prefill, fwd+bwd) & decode KV GB/s, % of GB300 roofline",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the varlen-extend workload)",
        "config": {"workload": p.name, "requests": p.batch, "total_q": int(p.q.shape[0]),
                   "total_k": int(p.k.shape[0]), "hq": p.hq, "hkv": p.hkv, "head_dim": p.head_dim,
                   "causal": True, "l2": "flushed before every timed step (512 MB write)",
                   "algorithmic_tflop_per_step": flops / 1e12},
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "workloads": extra,
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline_extend(p)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def reference_arm(args, wl):
    """The oracle, as it stands, timed on the host cores: each step is a
    bounded sample of the headline workload."""
    p = wl.workload(args.workload)
    from oracle import attn_sink_oracle as orc
    import numpy as np
    b = int(np.argmax(p.seqlens_q))
    work = 4.0 * p.head_dim * _sample_pairs(p, b)
    run = lambda: orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k, p.win_first,
                               p.win_last, p.causal, p.scale, heads=[0], requests=[b])
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = (time.perf_counter() - t0) / args.steps
    value = work / el / 1e12
    sample = f"fp64 numpy oracle, request {b} (all rows), head 0 ({work/1e9:.2f} GFLOP) per step"
    print(json.dumps({
        "impl": "reference",
        "metric": "attn TFLOP/s (prefill, fwd+bwd) & decode KV GB/s, % of GB300 roofline",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": {"workload": p.name},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    main()
