#!/usr/bin/env python3
"""Benchmark of the GQA FlashAttention backward on GB300.

One step = the whole backward hot path on one batch of synthetic input that is
already resident in HBM: gqa_attn_bwd_preprocess (Delta, row statistics,
accumulator zeroing) -> gqa_attn_bwd (main kernel) -> gqa_attn_bwd_postprocess
(fp32 -> fp16 casts) [-> gqa_attn_dsink when the workload has a sink].  The
forward that produces O and LSE runs once, untimed.

Workload: the causal MHA backward B=4, H=8, d=64, fp16 (the Triton
fused-attention table's shape), headline N_CTX=16384, plus a sweep over
N_CTX in {2048..32768}.  TFLOPS use the 2.5 x forward, causal-halved count.

The inputs of a step (Q,K,V,O,dO plus the fp32 dQ accumulator) are larger than
the 129 MB L2, so steps run back to back with no flush in between.

`--impl reference` times the fp64 CPU oracle instead (bounded sample).
Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path has no data exchange); value = all ranks' FLOPs / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE_N = 16384
SWEEP = (2048, 4096, 8192, 16384, 32768)
NOMINAL_DENSE_TFLOPS = 2250.0  # NVIDIA's dense fp16 / bf16 tensor figure for GB300


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Ranks:
    """The replicas' coordination under torchrun (one process per GPU, nothing shared in the data
    path): barrier, the maximum of a time over ranks, teardown.  `backend` is "nccl" on the GPUs
    and "gloo" in the CPU tests of this logic."""

    def __init__(self, backend: str, device):
        import torch.distributed as dist
        self.dist = dist
        self.ws, self.rank, self.local = _dist()
        self.device = device
        if self.ws > 1 and not dist.is_initialized():
            if backend == "nccl":
                dist.init_process_group(backend, device_id=device)
            else:
                dist.init_process_group(backend)

    def barrier(self):
        if self.ws > 1:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.ws == 1:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.ws > 1:
            self.dist.barrier()
            self.dist.destroy_process_group()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []  # (host monotonic time, csv line)
        self.window = None  # host times bracketing the timed region
        self._t = None
        self._first = threading.Event()

    def start(self):
        """Starts sampling and waits (up to 5 s) for the first sample, so the timed region is covered."""
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            self._first.wait(timeout=5.0)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))
            self._first.set()

    def mark(self, t0: float, t1: float):
        """Host times (after a device synchronize) at the start and the end of the timed region."""
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        return self.summary()

    def summary(self):
        """Median SM clock, maximum clock and throttle reasons of the samples in the timed region."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lines = self.lines
        if self.window is not None:
            # samples taken during the timed region (a sample reports the state of its last period)
            inside = [x for x in lines if self.window[0] <= x[0] <= self.window[1] + self.period * 1e-3]
            lines = inside if inside else lines
        scope = "timed region" if self.window is not None and lines is not self.lines else "whole run"
        for _, ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"])
        return dict(sm_mhz=statistics.median(sm), sm_max_mhz=max(smax), reasons=sorted(reasons), samples=len(sm),
                    sample_ms=self.period, scope=scope)


def _src_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gqa_flashattention_backward_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic(kernel_key: str, src_hash: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_sha") == src_hash:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def launches_per_step(p):
    """Kernels one preprocess / main / postprocess pass launches, by the library's rules: the
    preprocess, the key-stationary main kernel and either the dQ cast (an fp32 dQ accumulator:
    Dqk 64 / 128, not deterministic) or the query-stationary dQ pass; with per-head CTAs (group
    mode b) also the dK and dV casts."""
    import gqa_flashattention_backward_gb300._native as nat
    return 3 + (2 if not p.deterministic and p.group_mode == nat.GQA_GROUP_ATOMIC else 0)


def run_gpu(args):
    import torch

    import gqa_flashattention_backward_gb300 as pkg
    from gqa_flashattention_backward_gb300 import _native as nat
    from gqa_flashattention_backward_gb300 import workloads as W

    ws_n, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ranks = Ranks("nccl", dev)
    barrier = ranks.barrier

    nat.load()
    peaks = _peaks()

    inputs_cache = {}

    def case(w):
        """Inputs on the device and the forward's O / LSE of workload w (made once per workload)."""
        if w.name not in inputs_cache:
            q, k, v, do, sink = W.make_inputs(w)
            q, k, v, do = (t.to(dev) for t in (q, k, v, do))
            sink = sink.to(dev) if sink is not None else None
            cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev) if w.cu_seqlens else None
            kw = dict(causal=w.causal, window=w.window, scale=w.resolved_scale, cu_seqlens=cu,
                      max_seqlen=w.max_seqlen if cu is not None else None)
            o, lse = pkg.attention_forward(q, k, v, sink=sink, **kw)
            inputs_cache[w.name] = dict(w=w, q=q, k=k, v=v, do=do, o=o, lse=lse, sink=sink, cu=cu,
                                        max_seqlen=kw["max_seqlen"])
        return inputs_cache[w.name]

    def drop(w):
        inputs_cache.pop(w.name, None)

    def setup(w, red_mode=None, group_mode=nat.GQA_GROUP_TMEM, deterministic=False):
        c = dict(case(w))
        q, k, v, lse = c["q"], c["k"], c["v"], c["lse"]
        p = pkg._params(q, k, v, w.causal, w.window, w.resolved_scale, c["cu"], c["max_seqlen"], group_mode,
                        red_mode, deterministic)
        wsb = nat.alloc_workspace(p, dev)
        out = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                   delta=torch.empty(lse.shape, dtype=torch.float32, device=dev))
        if c["sink"] is not None:
            out["dsink"] = torch.empty(w.Hq, dtype=torch.float32, device=dev)
        c.update(p=p, ws=wsb, out=out)
        return c

    def step(c, ev=None):
        """One backward pass through the C ABI; returns the number of kernels launched."""
        p, o = c["p"], c["out"]
        nat.bwd_preprocess(p, c["o"], c["do"], c["lse"], o["delta"], c["ws"])
        if ev is not None:
            ev[0].record()
        nat.bwd(p, c["q"], c["k"], c["v"], c["do"], o["dq"], o["dk"], o["dv"], c["ws"])
        if ev is not None:
            ev[1].record()
        nat.bwd_postprocess(p, o["dq"], o["dk"], o["dv"], c["ws"])
        n = launches_per_step(p)
        if c["sink"] is not None:
            nat.dsink(p, c["sink"], c["lse"], o["delta"], o["dsink"])
            n += 1
        return n

    def timed(c, steps, warmup, main_events=False, sampler=None):
        for _ in range(warmup):
            step(c)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)] \
            if main_events else [None] * steps
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        launches = 0
        h0 = time.monotonic()
        t0.record()
        for i in range(steps):
            launches += step(c, evs[i])
        t1.record()
        torch.cuda.synchronize()
        if sampler is not None:
            sampler.mark(h0, time.monotonic())
        barrier()
        ms = t0.elapsed_time(t1)
        main_ms = sum(a.elapsed_time(b) for a, b in evs) / steps if main_events else None
        return ms, main_ms, launches

    max_over_ranks = ranks.max

    w = W.mha_causal(args.n_ctx)
    c = setup(w)
    sampler = ClockSampler(local)
    sampler.start()
    total_ms, main_ms, launches = timed(c, args.steps, args.warmup, main_events=True, sampler=sampler)
    clocks = sampler.stop()
    total_ms = max_over_ranks(total_ms)
    ms_step = total_ms / args.steps
    flops_conv = w.flops_convention()
    flops_exact = w.flops_exact()
    value = ws_n * flops_conv / (ms_step * 1e-3) / 1e12

    # roofline of the dominant kernel (the backward main kernel)
    achieved = flops_exact / (main_ms * 1e-3) / 1e12
    src = _src_hash("kv_kernel.cu", "umma.cuh", "common.cuh")
    traffic = _traffic(f"kv_kernel/{w.name}", src)
    roofline = dict(bound="tensor", achieved=round(achieved, 2), peak=peaks["bf16_tflops"], unit="TFLOP/s",
                    frac=round(achieved / peaks["bf16_tflops"], 4), traffic=traffic,
                    peak_nominal=NOMINAL_DENSE_TFLOPS, frac_nominal=round(achieved / NOMINAL_DENSE_TFLOPS, 4),
                    peak_nominal_source="NVIDIA's dense fp16/bf16 tensor figure for GB300 (2.25 PFLOP/s)",
                    kernel="kv_kernel<64,64,fp16>", kernel_ms=round(main_ms, 4),
                    flops_per_launch=flops_exact, peak_source=f"{peaks['source']} bf16 burst (fp16 same rate)")

    # end-to-end through the public API with host buffers: every step uploads its own inputs from pinned
    # host memory and reads its own dQ / dK / dV back.  The uploads, the backward and the read-backs run
    # on three streams with two device buffer sets, so step i+1's upload and step i-1's read-back
    # overlap step i's backward (events order every reuse of a buffer); the serial time is also kept.
    e2e = None
    if not args.no_e2e:
        names_in = ("q", "k", "v", "o", "do", "lse")
        pinned = {n: c[n].cpu().pin_memory() for n in names_in}
        h2d = sum(t.numel() * t.element_size() for t in pinned.values())
        host_out = {n: torch.empty(c["out"][n].shape, dtype=c["out"][n].dtype).pin_memory() for n in ("dq", "dk", "dv")}
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        dbufs = [{n: torch.empty_like(c[n]) for n in names_in} for _ in range(2)]
        douts = [c["out"], {n: torch.empty_like(t) for n, t in c["out"].items()}]
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        in_done = [torch.cuda.Event() for _ in range(2)]
        cmp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        for sl in range(2):
            cmp_done[sl].record(s_cmp)
            out_done[sl].record(s_out)

        link_ev = []  # (upload start, upload end, read-back start, read-back end) per timed step

        def e2e_step(i, evs=None):
            sl = i % 2
            with torch.cuda.stream(s_in):
                s_in.wait_event(cmp_done[sl])  # the backward that last read this input set is done
                if evs is not None:
                    evs[0].record(s_in)
                for n in names_in:
                    dbufs[sl][n].copy_(pinned[n], non_blocking=True)
                in_done[sl].record(s_in)
                if evs is not None:
                    evs[1].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_done[sl])
                s_cmp.wait_event(out_done[sl])  # the read-back of this output set is done
                d = dbufs[sl]
                pkg.attention_backward(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], causal=w.causal,
                                       scale=w.resolved_scale, workspace=c["ws"], out=douts[sl])
                cmp_done[sl].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp_done[sl])
                if evs is not None:
                    evs[2].record(s_out)
                for n in ("dq", "dk", "dv"):
                    host_out[n].copy_(douts[sl][n], non_blocking=True)
                out_done[sl].record(s_out)
                if evs is not None:
                    evs[3].record(s_out)

        def e2e_serial_step():
            for n in names_in:
                dbufs[0][n].copy_(pinned[n], non_blocking=True)
            d = dbufs[0]
            r = pkg.attention_backward(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], causal=w.causal,
                                       scale=w.resolved_scale, workspace=c["ws"], out=douts[0])
            for n in ("dq", "dk", "dv"):
                host_out[n].copy_(r[n], non_blocking=True)

        for i in range(max(1, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        s_cmp.wait_event(t0)
        s_out.wait_event(t0)
        for i in range(args.steps):
            evs = tuple(torch.cuda.Event(enable_timing=True) for _ in range(4))
            link_ev.append(evs)
            e2e_step(i, evs)
        t1.record(s_out)
        torch.cuda.synchronize()
        barrier()
        e_ms = max_over_ranks(t0.elapsed_time(t1)) / args.steps
        up_ms = sum(a.elapsed_time(b) for a, b, _, _ in link_ev)
        down_ms = sum(c_.elapsed_time(d_) for _, _, c_, d_ in link_ev)
        # the same steps one after another on one stream (no overlap), for reference
        e2e_serial_step()
        torch.cuda.synchronize()
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        u0.record()
        for _ in range(args.steps):
            e2e_serial_step()
        u1.record()
        torch.cuda.synchronize()
        s_ms = u0.elapsed_time(u1) / args.steps
        e2e = dict(value=round(ws_n * flops_conv / (e_ms * 1e-3) / 1e12, 2), unit="TFLOPS", ms_per_step=round(e_ms, 3),
                   h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                   copies="pinned host buffers; uploads / backward / read-backs on three streams, double-buffered",
                   h2d_gbs=round(h2d * args.steps / (up_ms * 1e-3) / 1e9, 1),
                   d2h_gbs=round(d2h * args.steps / (down_ms * 1e-3) / 1e9, 1),
                   link_note="GB/s = bytes over the copy streams' event time; the step is bound by the host link "
                             "when (h2d + d2h bytes) / link GB/s exceeds the device step",
                   serial_ms_per_step=round(s_ms, 3),
                   serial_value=round(ws_n * flops_conv / (s_ms * 1e-3) / 1e12, 2))
        del pinned, host_out, dbufs, douts

    # accumulation variants at the headline size (p3's atomic_add / none comparison)
    # accumulation variants: the group reduction of dK/dV ((a) in TMEM, (b) per-head CTAs adding into fp32)
    # crossed with the way every fp32 partial is added (bulk tensor reduce, red.v4, scalar red, or plain
    # stores -- wrong results, the cost floor), and the deterministic mode; [P3]'s atomic_add / none question
    VARIANTS = (("tmem_bulk", dict(red_mode=nat.GQA_RED_BULK)),
                ("tmem_v4", dict(red_mode=nat.GQA_RED_V4)),
                ("tmem_scalar", dict(red_mode=nat.GQA_RED_SCALAR)),
                ("tmem_none", dict(red_mode=nat.GQA_RED_NONE)),
                ("atomic_bulk", dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_BULK)),
                ("atomic_v4", dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_V4)),
                ("atomic_none", dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_NONE)),
                ("deterministic", dict(deterministic=True)))

    def run_variants(wv):
        out = {}
        nst = max(3, args.steps // 4)
        for name, kw in VARIANTS:
            cv = setup(wv, **kw)
            ms, mms, _ = timed(cv, nst, args.warmup, main_events=True)
            stp = ms / nst
            out[name] = dict(tflops_exact=round(wv.flops_exact() / (stp * 1e-3) / 1e12, 2), ms=round(stp, 4),
                             main_kernels_ms=round(mms, 4))
            del cv
        base = out["tmem_none"]["ms"]
        out["overhead_vs_none"] = {n: round(out[n]["ms"] / base - 1.0, 4) for n in ("tmem_bulk", "tmem_v4", "tmem_scalar")}
        out["overhead_vs_none"]["atomic_bulk_vs_atomic_none"] = round(out["atomic_bulk"]["ms"] / out["atomic_none"]["ms"] - 1.0, 4)
        out["group_reduction_atomic_bulk_vs_tmem_bulk"] = round(out["atomic_bulk"]["ms"] / out["tmem_bulk"]["ms"] - 1.0, 4)
        out["group_size"] = wv.Hq // wv.Hkv
        return out

    variants = {}
    if not args.no_variants:
        variants = run_variants(w)

    sweep = {}
    if not args.no_sweep:
        for n in SWEEP:
            ws_ = W.mha_causal(n)
            cs = setup(ws_)
            ms, mms, _ = timed(cs, max(3, args.steps // 2), args.warmup, main_events=True)
            stp = ms / max(3, args.steps // 2)
            sweep[str(n)] = dict(tflops=round(ws_.flops_convention() / (stp * 1e-3) / 1e12, 2),
                                 ms=round(stp, 4), main_kernel_tflops_exact=round(
                                     ws_.flops_exact() / (mms * 1e-3) / 1e12, 2))
            del cs

    # the other workloads, same hot path and launch configuration (preprocess -> bwd -> postprocess [-> dsink]);
    # TFLOP/s on the exact, window-aware count first (the convention count ignores the window)
    configs = {}
    if not args.no_configs:
        for wc in (W.varlen(), W.sink_window(), W.long_context()):
            cc = setup(wc)
            nst = max(3, args.steps // 2)
            ms, mms, _ = timed(cc, nst, args.warmup, main_events=True)
            stp = ms / nst
            te = wc.flops_exact() / (stp * 1e-3) / 1e12
            configs[wc.name] = dict(tflops_exact=round(te, 2), frac_of_peak_exact=round(te / peaks["bf16_tflops"], 4),
                                    ms=round(stp, 4), main_kernels_ms=round(mms, 4),
                                    tflops_convention=round(wc.flops_convention() / (stp * 1e-3) / 1e12, 2),
                                    shape=wc.describe())
            del cc
            if not args.no_variants:
                configs[wc.name]["variants"] = run_variants(wc)

    # the forward (prerequisite of the backward, not part of the step): exact-count TFLOP/s per workload
    forward = {}
    if not args.no_forward:
        for wf in (w, W.varlen(), W.sink_window(), W.long_context()):
            cf = c if wf is w else setup(wf)
            nst = max(3, args.steps // 2)

            def fstep():
                nat.fwd(cf["p"], cf["q"], cf["k"], cf["v"], cf["sink"], cf["o"], cf["lse"], cf["ws"])

            for _ in range(args.warmup):
                fstep()
            torch.cuda.synchronize()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record()
            for _ in range(nst):
                fstep()
            f1.record()
            torch.cuda.synchronize()
            fms = f0.elapsed_time(f1) / nst
            fflops = 2.0 * wf.pairs() * (wf.Dqk + wf.Dv)
            forward[wf.name] = dict(ms=round(fms, 4), tflops_exact=round(fflops / (fms * 1e-3) / 1e12, 2),
                                    frac_of_peak_exact=round(fflops / (fms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4))
            if cf is not c:
                del cf
                drop(wf)

    # small, launch-bound problems: the eager chain of launches against one CUDA-graph replay of it
    graphs = {}
    if not args.no_graph:
        for wg in (W.tiny(), W.shrink(W.sink_window(), name="small_sink_window", B=1, Hq=8, Hkv=2, S=512, window=256)):
            cg = setup(wg)
            kwg = dict(causal=wg.causal, window=wg.window, scale=wg.resolved_scale, sink=cg["sink"])
            gb = pkg.GraphedBackward(cg["q"], cg["k"], cg["v"], cg["o"], cg["lse"], cg["do"], **kwg)
            nst = 50

            def run_many(fn):
                for _ in range(args.warmup):
                    fn()
                torch.cuda.synchronize()
                g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                g0.record()
                for _ in range(nst):
                    fn()
                g1.record()
                torch.cuda.synchronize()
                return g0.elapsed_time(g1) / nst * 1e3

            graphs[wg.name] = dict(shape=wg.describe(), eager_us_per_step=round(run_many(lambda: step(cg)), 2),
                                   graph_us_per_step=round(run_many(gb.replay), 2))
            del cg, gb

    line = None
    if rank == 0:
        cpu = None
        if ws_n == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(args)
        line = dict(metric="GQA attention bwd TFLOPS (1xGB300, causal)", value=round(value, 2), unit="TFLOPS",
                    n_gpus=ws_n, steps=args.steps, warmup=args.warmup, ms_per_step=round(ms_step, 4),
                    higher_is_better=True, scaling="weak", vs_baseline=None, dtype="fp16", data="synthetic",
                    config=_config(w.S, ws_n),
                    mode="dK/dV summed in TMEM; dQ by " + (
                        "bulk tensor reduce" if pkg.preferred_red_mode(w.Dqk) == nat.GQA_RED_BULK
                        else "red.global.add.v4.f32"),
                    flops_per_step_convention=flops_conv, flops_per_step_exact=flops_exact,
                    frac_of_peak_exact=round(flops_exact / (ms_step * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                    roofline=roofline, cpu_baseline=cpu, e2e=e2e, gpu_launches=launches, clocks=clocks,
                    variants=variants, sweep=sweep, configs=configs, forward=forward,
                    graph=graphs)
        print(json.dumps(line), flush=True)
    ranks.close()
    return line


def _config(n_ctx: int, ws_n: int) -> dict:
    """The workload both arms report (the reference arm samples it, see its cpu_baseline)."""
    return dict(workload=f"mha_causal_n{n_ctx}", B=4, Hq=8, Hkv=8, S=n_ctx, D=64, causal=True,
                flop_count="2.5x forward, causal-halved", l2="inputs larger than L2, no flush",
                parallelism=f"replicas x{ws_n}" if ws_n > 1 else "single GPU")


def _oracle_sample(n: int):
    """(workload, timer) for the oracle backward of one (batch, head) of the causal
    d=64 workload at length n; timer() runs it once and returns seconds."""
    from gqa_flashattention_backward_gb300 import workloads as W
    from oracle import oracle as orc

    w = W.shrink(W.mha_causal(n), name=f"oracle_sample_n{n}", B=1, Hq=1, Hkv=1)
    q, k, v, do, _ = W.make_inputs(w)
    f = lambda t: t.double().numpy()  # noqa: E731
    q, k, v, do = f(q), f(k), f(v), f(do)
    pb = orc.Problem(B=1, Hq=1, Hkv=1, S=n, Dqk=64, Dv=64, causal=True, scale=w.resolved_scale)
    o, lse = orc.forward(pb, q, k, v)

    def timer():
        t0 = time.perf_counter()
        orc.backward(pb, q, k, v, o, lse, do)
        return time.perf_counter() - t0

    return w, timer


def _calibrated_sample(target_s: float):
    n = 1024
    while True:
        w, timer = _oracle_sample(n)
        dt = timer()
        if dt * 3.5 > target_s or n >= 16384:
            return n, w, timer, dt
        n *= 2


def _sample_text(n):
    return f"fp64 oracle backward of 1 of the 32 (batch, head) pairs at N_CTX={n} (d=64, causal)"


def cpu_baseline(args, target_s: float = 12.0):
    """The oracle timed on the host cores on a bounded sample of the same workload."""
    n, w, timer, dt = _calibrated_sample(target_s)
    return dict(value=round(w.flops_convention() / dt / 1e12, 6), unit="TFLOPS",
                cores=len(os.sched_getaffinity(0)), kind="oracle", seconds=round(dt, 3), sample=_sample_text(n))


def run_reference(args):
    """Reference arm: the fp64 CPU oracle, each step a bounded sample of the workload."""
    ws_n, rank, _ = _dist()
    if rank != 0:
        return None
    # each step: the oracle backward of one of the workload's 32 (batch, head) pairs at the workload's own
    # N_CTX (about 2 s on 16 Arm cores at 16384), so the line describes the same configuration
    n = args.n_ctx
    w, timer = _oracle_sample(n)
    for _ in range(args.warmup):
        timer()
    tot = sum(timer() for _ in range(args.steps))
    val = round(args.steps * w.flops_convention() / tot / 1e12, 6)
    cores = len(os.sched_getaffinity(0))
    line = dict(impl="reference", metric="GQA attention bwd TFLOPS (1xGB300, causal)", value=val, unit="TFLOPS",
                n_gpus=ws_n, steps=args.steps, warmup=args.warmup, ms_per_step=round(1e3 * tot / args.steps, 3),
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                config=_config(args.n_ctx, ws_n),
                cpu_baseline=dict(kind="oracle", cores=cores, sample=_sample_text(n), value=val, unit="TFLOPS"),
                e2e=dict(value=val, unit="TFLOPS", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)
    return line


PROFILE_WORKLOADS = {
    "tiny": lambda W: W.tiny(),
    "mha_causal_n8192": lambda W: W.mha_causal(8192),
    "mha_causal_n16384": lambda W: W.mha_causal(16384),
    "varlen": lambda W: W.varlen(),
    "sink_window": lambda W: W.sink_window(),
    "long_context": lambda W: W.long_context(),
    # the long-context shape at a quarter of its length: a few hundred MB on the device, for captures
    # that replay a launch many times
    "long_context_s8192": lambda W: W.shrink(W.long_context(), name="long_context_s8192", S=8192),
}


def run_only(args):
    """One workload, one mode, nothing else: the command the ncu captures profile.  `--only NAME:MODE`
    with MODE a backward variant (tmem_bulk (default), tmem_v4, tmem_scalar, tmem_none, atomic_bulk,
    atomic_v4, atomic_none, deterministic) or "forward".  Runs `--warmup` + `--steps` steps and prints
    the mean step time."""
    import torch

    import gqa_flashattention_backward_gb300 as pkg
    from gqa_flashattention_backward_gb300 import _native as nat
    from gqa_flashattention_backward_gb300 import workloads as W

    name, _, mode = args.only.partition(":")
    mode = mode or "tmem_bulk"
    modes = dict(tmem_bulk=dict(red_mode=nat.GQA_RED_BULK), tmem_v4=dict(red_mode=nat.GQA_RED_V4),
                 tmem_scalar=dict(red_mode=nat.GQA_RED_SCALAR), tmem_none=dict(red_mode=nat.GQA_RED_NONE),
                 atomic_bulk=dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_BULK),
                 atomic_v4=dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_V4),
                 atomic_none=dict(group_mode=nat.GQA_GROUP_ATOMIC, red_mode=nat.GQA_RED_NONE),
                 deterministic=dict(deterministic=True), forward=dict())
    if name not in PROFILE_WORKLOADS or mode not in modes:
        raise SystemExit(f"--only {args.only}: workload one of {sorted(PROFILE_WORKLOADS)}, mode one of {sorted(modes)}")
    w = PROFILE_WORKLOADS[name](W)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    nat.load()
    q, k, v, do, sink = (t.to(dev) if t is not None else None for t in W.make_inputs(w))
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev) if w.cu_seqlens else None
    kw = dict(causal=w.causal, window=w.window, scale=w.resolved_scale, cu_seqlens=cu,
              max_seqlen=w.max_seqlen if cu is not None else None)
    o, lse = pkg.attention_forward(q, k, v, sink=sink, **kw)
    ws = nat.alloc_workspace(pkg._params(q, k, v, w.causal, w.window, w.resolved_scale, cu, kw["max_seqlen"],
                                         **modes[mode]), dev)
    out = {}

    def step():
        if mode == "forward":
            pkg.attention_forward(q, k, v, sink=sink, workspace=ws, **kw)
        else:
            pkg.attention_backward(q, k, v, o, lse, do, sink=sink, workspace=ws, out=out, **modes[mode], **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    print(json.dumps(dict(only=args.only, ms_per_step=round(e0.elapsed_time(e1) / max(1, args.steps), 4))), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--n-ctx", type=int, default=HEADLINE_N)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--no-forward", action="store_true", help="skip the forward timings")
    ap.add_argument("--no-graph", action="store_true", help="skip the eager / CUDA-graph comparison")
    ap.add_argument("--only", default=None, help="WORKLOAD[:MODE]: one workload in one mode (for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.only:
        run_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
