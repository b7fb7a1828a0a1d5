#!/usr/bin/env python
"""KVM layer benchmark on GB300: prefill tokens/s at 8k (+ roofline) and decode-step time.

One step = one kvm_prefill over the whole fixed-state 8k workload (B=8, H=12,
N=8192, head_dim 64, chunk 128, window 512, 256 slots incl. 16 sinks, bf16),
inputs resident in HBM.  Inputs (q, k, v: 302 MB) are larger than L2, so no
explicit flush is done between steps.  The prefill runs overlapped (the
library's default): fold-chain segments on one SM partition, the attention of
folded chunks beside them.  A second, untimed-for-the-headline pass runs the
sequential prefill to report each kernel's own duration.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload fixed8k|sqrt8k|long64k]

--workload picks the headline prefill workload (default fixed8k, the line the
metric is quoted on); the other two prefill workloads (sqrt-growth 8k, 64k long
prefill) are timed in the same run and reported under "workloads".

Under torchrun (N > 1) every rank runs its own copy of the workload on its
GPU (the (batch, head) rows are independent: no collective on the data path),
timing is max over ranks, and value = total tokens of all ranks / that time.
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
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from compressed_kv_state_gb300 import workloads as wl  # noqa: E402

METRIC = "KVM layer prefill tokens/s @8k (1 GB300)"
UNIT = "tokens/s"
PREFILL = {"fixed8k": wl.FIXED_8K, "sqrt8k": wl.SQRT_8K, "long64k": wl.LONG_64K}
W = wl.FIXED_8K


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# --------------------------------------------------------------- work model

def attention_work(w):
    """Algorithmic attention work of one prefill: (query, key) pairs of the state
    and of the window, FLOPs (state QK over the d - r non-rotary dims only),
    exponentials, and the FLOPs counted at 4d per pair for every key."""
    C, Wc, d, r = w.chunk, w.window // w.chunk, w.d, w.rope_dims
    n_after = _schedule(w)
    state_pairs = win_pairs = 0
    for p in range(w.N):
        c = p // C
        e = c - Wc - 1
        state_pairs += n_after[e] if e >= 0 else 0
        win_pairs += p - max(0, (c - Wc) * C) + 1
    rows = w.B * w.H
    state_pairs *= rows
    win_pairs *= rows
    flops = state_pairs * (2 * (d - r) + 2 * d) + win_pairs * 4 * d
    return dict(state_pairs=state_pairs, window_pairs=win_pairs, flops=flops,
                flops_4d=(state_pairs + win_pairs) * 4 * d, exps=state_pairs + win_pairs)


def _schedule(w):
    import math
    C = w.chunk
    nchunks = -(-w.N // C)
    E = max(0, nchunks - w.window // C - 1)
    out, n, t = [], 0, 0
    for e in range(E):
        sinks = sum(1 for i in range(C) if e * C + i < w.n_sinks)
        n0 = n + sinks
        t += C
        cap = w.max_slots if w.sched == 0 else w.n_sinks + math.ceil(w.coef * t ** w.expo)
        a = min(max(cap - n0, 0), C - sinks)
        n = n0 + a
        out.append(n)
    return out


def fold_work(w):
    """Similarity FLOPs of the fold chain (each token against every mergeable slot
    once, plus the remaining tokens against the new slots)."""
    C, S, d = w.chunk, w.n_sinks, w.d
    n_prev, fl = 0, 0
    for e, n_after in enumerate(_schedule(w)):
        sinks = sum(1 for i in range(C) if e * C + i < S)
        n0 = n_prev + sinks
        cand = C - sinks
        a = n_after - n0
        fl += 2 * d * (cand * max(0, n0 - S) + (cand - a) * a)
        n_prev = n_after
    return fl * w.B * w.H


def decode_bytes(dw, r_in_chunk, n):
    """Algorithmic HBM bytes of one decode step (all rows): window K, V (bf16),
    the state's read view (key on the d - r non-rotary dims, value), q, out, and
    the new token written into the ring."""
    d, r = dw.d, dw.rope_dims
    per_row = (dw.window + r_in_chunk + 1) * d * 2 * 2 + n * (d - r + d) * 2 + 2 * d * 2 \
        + 2 * d * 2 + 4
    return per_row * dw.B * dw.H


# ------------------------------------------------------------------ clocks

class Clocks:
    """nvidia-smi sampler (every 200 ms) running while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        # The sampler is a child process: it must not outlive this program on any
        # exit path (a profiler waits for the whole process tree), so it is stopped
        # at interpreter exit too, and it ends by itself after max_s seconds.
        import atexit
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["timeout", str(self.max_s), "nvidia-smi", f"--id={self.index}",
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            atexit.register(self._kill)
        except Exception:
            self.proc = None

    max_s = 900

    def _kill(self):
        if self.proc is not None and self.proc.poll() is None:
            self.proc.kill()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        pmax = max(r["power"] for r in rows)
        load = [r for r in rows if r["power"] >= 0.5 * pmax] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() in ("active", "1", "0x1"):
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in load),
                    sm_max_mhz=max(r["smax"] for r in load), reasons=sorted(reasons),
                    samples=len(load), power_w_max=pmax)


# -------------------------------------------------------------- traffic

def _ncu_traffic(kernel_file, workload):
    """DRAM bytes per launch from a committed ncu summary (entry "<file>@<workload>",
    else "<file>"), only if it was taken on the current source of the kernel (same
    sha256); else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    allv = json.load(open(p))
    name = os.path.basename(kernel_file)
    d = allv.get(f"{name}@{workload}") or allv.get(name)
    if not d:
        return None
    sha = hashlib.sha256(open(kernel_file, "rb").read()).hexdigest()
    return d["dram_bytes_per_launch"] if d.get("source_sha256") == sha else None


# ------------------------------------------------------------- CPU oracle

def _oracle_cfg(w):
    import oracle
    return oracle.OracleConfig(head_dim=w.d, rope_dims=w.rope_dims, chunk=w.chunk,
                               window=w.window, n_sinks=w.n_sinks, sched=w.sched,
                               max_slots=w.max_slots, coef=w.coef, expo=w.expo)


def _sample_workload(w, rows):
    """The bounded CPU sample of a workload: `rows` full-length (batch, head) rows,
    drawn as a workload of batch 1 and `rows` heads with the same recipe."""
    return w.with_(B=1, H=rows, name=f"{w.name}[sample B1H{rows}]")


def cpu_oracle_sample(w, heads_per_thread=1, one_thread=True):
    """Time the fp64 oracle on a bounded sample of the workload: one full-length
    (batch, head) row per host core, all cores in parallel.  Returns (record,
    sample) where record's value is tokens/s in the layer's unit (a layer token
    needs all H heads) and sample = (sample workload, oracle debug record)."""
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    nh = min(w.B * w.H, cores * heads_per_thread)
    sub = _sample_workload(w, nh)
    q, k, v, g = wl.prefill_inputs(sub)
    q, k, v, g = q[0], k[0], v[0], g[0]
    ocfg = _oracle_cfg(w)
    t0 = time.perf_counter()
    _, _, odbg = oracle.prefill(ocfg, q, k, v, g, threads=cores)
    dt = time.perf_counter() - t0
    layer_tokens = w.N * q.shape[0] / w.H
    r = dict(value=layer_tokens / dt, unit=UNIT, cores=min(cores, q.shape[0]), kind="oracle",
             sample=f"{q.shape[0]} of {w.B * w.H} (batch, head) rows x {w.N} tokens of "
                    f"{w.name}, one row per thread, {dt:.1f} s wall")
    r["seconds"] = dt
    if one_thread:  # the same oracle on one thread, one row
        t1 = time.perf_counter()
        oracle.prefill(ocfg, q[:1], k[:1], v[:1], g[:1], threads=1)
        dt1 = time.perf_counter() - t1
        r["one_thread"] = {"value": w.N / w.H / dt1, "unit": UNIT, "cores": 1,
                           "sample": f"1 (batch, head) row x {w.N} tokens, {dt1:.1f} s wall"}
    return r, (sub, odbg)


NEAR_TIE = 1e-5


def near_tie_counts(sub, odbg, dev):
    """Fold decisions of the GPU against the oracle on the CPU sample's rows (the
    same seeded inputs, one GPU prefill with a debug record): per row the first
    event where they differ (if any), and whether every differing token there is
    a near tie (oracle top-2 cosine gap, or the event's surprise selection margin,
    below 1e-5).  Counts only; nothing is asserted here."""
    import torch
    import oracle
    from compressed_kv_state_gb300 import kvm
    q, k, v, g = wl.prefill_inputs(sub)
    E = oracle.n_events(_oracle_cfg(sub), sub.N)
    layer = kvm.KvmLayer(layer_config(kvm, sub), device=dev)
    shp = (sub.B, sub.H, max(E, 1), sub.chunk)
    assign = torch.full(shp, -7, dtype=torch.int32, device=dev)
    kind = torch.full(shp, -7, dtype=torch.int32, device=dev)
    dbg = kvm.kvm_debug(assign.data_ptr(), kind.data_ptr(), None, None, E)
    t = lambda a: torch.from_numpy(a).to(dev)
    layer.prefill(t(q).bfloat16(), t(k).bfloat16(), t(v).bfloat16(), t(g), dbg=dbg)
    layer.sync()
    ga, gk = assign.cpu().numpy()[0], kind.cpu().numpy()[0]
    layer.close()
    rows = []
    for h in range(sub.H):
        first, n_tok, near = None, 0, True
        for e in range(E):
            bad = (ga[h, e] != odbg["assign"][h, e]) | (gk[h, e] != odbg["kind"][h, e])
            if bad.any():
                toks = np.nonzero(bad)[0]
                first, n_tok = e, len(toks)
                near = bool(odbg["sel_margin"][h, e] < NEAR_TIE or all(
                    odbg["kind"][h, e, t] == oracle.MERGED and odbg["gap"][h, e, t] < NEAR_TIE
                    for t in toks))
                break
        rows.append((first, n_tok, near))
    div = [r for r in rows if r[0] is not None]
    return {"rows": sub.H, "events_per_row": E, "rows_identical": len(rows) - len(div),
            "rows_diverged": len(div),
            "first_divergent_events": sorted(r[0] for r in div),
            "tokens_differing_at_first_divergence": sum(r[1] for r in div),
            "all_divergences_near_ties": all(r[2] for r in div),
            "sample": sub.name,
            "rule": "assignments and kinds compared event by event from event 0; a row stops "
                    "at its first differing event; near tie = oracle top-2 gap (or surprise "
                    "selection margin) < 1e-5"}


# ------------------------------------------------------------- multi-rank

def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank processes its own rows (weak scaling)."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


# ------------------------------------------------------------------ ours

def layer_config(kvm, w):
    return kvm.make_config(batch=w.B, heads=w.H, rope_dims=w.rope_dims, chunk=w.chunk,
                           window=w.window, n_sinks=w.n_sinks, sched=w.sched,
                           max_slots=w.max_slots, coef=w.coef, expo=w.expo, max_tokens=w.N)


def time_prefill(w, dev, stream, steps, warmup, segments, world=1):
    """Device-resident prefill of workload w: warm-up, then `steps` prefills
    between CUDA events on the launch stream (barrier and synchronize on both
    sides), then a sequential pass that times each kernel on its own."""
    import torch
    from compressed_kv_state_gb300 import kvm
    q, k, v, g = wl.prefill_inputs(w)
    dq = torch.from_numpy(q).to(dev).bfloat16()
    dk = torch.from_numpy(k).to(dev).bfloat16()
    dv = torch.from_numpy(v).to(dev).bfloat16()
    dg = torch.from_numpy(g).to(dev)
    layer = kvm.KvmLayer(layer_config(kvm, w), device=dev)
    out = torch.empty_like(dq)

    def step():
        kvm.kvm_prefill(layer.handle, dq, dk, dv, dg, w.N, out, stream)

    kvm.kvm_layer_set_overlap(layer.handle, segments)
    for _ in range(warmup):
        step()
    layer.sync()
    used_segments = kvm.kvm_layer_get_overlap(layer.handle)
    kvm.kvm_layer_set_timing(layer.handle, True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1)
    tm = kvm.kvm_layer_get_timing(layer.handle)
    kvm.kvm_layer_set_timing(layer.handle, False)
    layer.sync()
    ms = max_over_ranks(ms, world, dev)
    # per-kernel durations: the same step run sequentially (fold chain, then attention)
    kvm.kvm_layer_set_overlap(layer.handle, 0)
    step()
    layer.sync()
    kvm.kvm_layer_set_timing(layer.handle, True)
    for _ in range(max(3, steps // 2)):
        step()
    tseq = kvm.kvm_layer_get_timing(layer.handle)
    kvm.kvm_layer_set_timing(layer.handle, False)
    layer.sync()
    kvm.kvm_layer_set_overlap(layer.handle, segments)
    return dict(ms_step=ms / steps, tm=tm, tseq=tseq, segments=used_segments, layer=layer,
                host=(q, k, v, g), dev=(dq, dk, dv, dg), out=out, step=step)


def prefill_report(w, t, peaks):
    """tokens/s, per-kernel times of the sequential pass, the dominant kernel's
    roofline in the timed step and the whole step against the tensor roofline."""
    aw = attention_work(w)
    ffl = fold_work(w)
    tm, tseq = t["tm"], t["tseq"]
    s_attn = tseq["attn_ms"] / max(1, tseq["attn_launches"])
    s_fold = tseq["fold_ms"] / max(1, tseq["fold_launches"])
    s_other = tseq["other_ms"] / max(1, tseq["other_launches"])
    s_tot = max(1e-9, tseq["attn_ms"] + tseq["fold_ms"] + tseq["other_ms"])
    kernels = {
        "attention": dict(ms_per_launch=s_attn, tflops=aw["flops"] / (s_attn / 1e3) / 1e12,
                          flops_per_launch=aw["flops"], share=tseq["attn_ms"] / s_tot),
        "fold_chain": dict(ms_per_launch=s_fold, tflops=ffl / (s_fold / 1e3) / 1e12,
                           flops_per_launch=ffl, share=tseq["fold_ms"] / s_tot),
        "key_rotation_and_ring": dict(ms_per_launch=s_other, share=tseq["other_ms"] / s_tot),
        "pass": "sequential prefill (fold chain, key rotation + window ring fill, attention), timed "
                "separately",
    }
    # dominant kernel of the timed step.  Overlapped: the fold chain is its critical
    # path (the attention runs beside it); its duration is the chain's span per step
    # (first segment start to last segment end, events on the chain's stream).
    # Sequential: the kernel with the larger share of the step.
    if t["segments"] > 0:
        dom = "fold_chain"
        dom_ms = tm["fold_ms"] / max(1, tm["fold_launches"])
    else:
        dom = "attention" if tm["attn_ms"] >= tm["fold_ms"] else "fold_chain"
        dom_ms = (tm["attn_ms"] / max(1, tm["attn_launches"]) if dom == "attention"
                  else tm["fold_ms"] / max(1, tm["fold_launches"]))
    dom_flops = aw["flops"] if dom == "attention" else ffl
    big = w.max_slots > 256 or w.chunk > 128
    dom_src = os.path.join(ROOT, "compressed_kv_state_gb300", "csrc",
                           "kvm_attn_tc.cu" if dom == "attention" else
                           ("kvm_fold_big.cu" if big else "kvm_fold_tc.cu"))
    ach = dom_flops / (dom_ms / 1e3) / 1e12
    roofline = dict(kernel=dom, bound="tensor", achieved=ach, peak=peaks["bf16"], unit="TFLOP/s",
                    frac=ach / peaks["bf16"], peak_source=f"{peaks['src']} bf16 burst",
                    ms_per_step=dom_ms, traffic=_ncu_traffic(dom_src, w.name))
    ms_step = t["ms_step"]
    step_roof = {"flops": aw["flops"] + ffl, "ms_per_step": ms_step,
                 "achieved": (aw["flops"] + ffl) / (ms_step / 1e3) / 1e12,
                 "peak": peaks["bf16"], "unit": "TFLOP/s",
                 "frac": (aw["flops"] + ffl) / (ms_step / 1e3) / 1e12 / peaks["bf16"],
                 "peak_source": f"{peaks['src']} bf16 burst",
                 "flops_4d_count": aw["flops_4d"] + ffl,
                 "frac_4d_count": (aw["flops_4d"] + ffl) / (ms_step / 1e3) / 1e12 / peaks["bf16"]}
    flops = {"attention": aw["flops"], "attention_4d_count": aw["flops_4d"], "fold_similarity": ffl}
    return kernels, roofline, step_roof, flops


def run_ours(args, rank, world, local_rank):
    import torch
    from compressed_kv_state_gb300 import kvm

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    clocks = Clocks(local_rank)
    clocks.start()
    time.sleep(0.3)
    t = time_prefill(W, dev, stream, args.steps, args.warmup, args.segments, world)
    layer = t["layer"]
    q, k, v, g = t["host"]
    dq, dk, dv, dg = t["dev"]
    out = t["out"]
    segments = t["segments"]
    ms_step = t["ms_step"]
    value = job_throughput(W.B * W.N, world, ms_step)

    # end to end through the C ABI: pinned host inputs in, output back to host, every
    # step.  Pipelined like a server: step i+1's host-to-device copies (three copy
    # streams) and step i-1's device-to-host read overlap step i's prefill; device
    # inputs and outputs are double-buffered, and events order every reuse.
    hq = torch.from_numpy(q).bfloat16().pin_memory()
    hk = torch.from_numpy(k).bfloat16().pin_memory()
    hv = torch.from_numpy(v).bfloat16().pin_memory()
    hg = torch.from_numpy(g).pin_memory()
    houts = [torch.empty(out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dins = [(dq, dk, dv, dg), tuple(torch.empty_like(x) for x in (dq, dk, dv, dg))]
    douts = [out, torch.empty_like(out)]
    s_in = [torch.cuda.Stream(dev) for _ in range(3)]
    s_out = torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    ev_in = [[ev() for _ in range(3)] for _ in range(2)]     # inputs of set b landed
    ev_used = [ev() for _ in range(2)]                         # prefill of set b done
    ev_read = [ev() for _ in range(2)]                         # output of set b read back
    started = [False, False]

    def e2e_step(i):
        b = i & 1
        tq, tk, tv, tg = dins[b]
        for j, (src, dst) in enumerate(((hq, tq), (hk, tk), ((hv, hg), (tv, tg)))):
            st = s_in[j]
            if started[b]:
                st.wait_event(ev_used[b])  # the previous prefill on this set read its inputs
            with torch.cuda.stream(st):
                if j < 2:
                    dst.copy_(src, non_blocking=True)
                else:
                    dst[0].copy_(src[0], non_blocking=True)
                    dst[1].copy_(src[1], non_blocking=True)
            ev_in[b][j].record(st)
        for j in range(3):
            stream.wait_event(ev_in[b][j])
        if started[b]:
            stream.wait_event(ev_read[b])  # the previous output of this set was read back
        kvm.kvm_prefill(layer.handle, tq, tk, tv, tg, W.N, douts[b], stream)
        ev_used[b].record(stream)
        s_out.wait_event(ev_used[b])
        with torch.cuda.stream(s_out):
            houts[b].copy_(douts[b], non_blocking=True)
        ev_read[b].record(s_out)
        started[b] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    ke2e = max(3, args.steps // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for j in range(3):
        s_in[j].wait_event(e0)
    for i in range(ke2e):
        e2e_step(i)
    for b in range(2):
        stream.wait_event(ev_read[b])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = e0.elapsed_time(e1) / ke2e
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hg))
    d2h = houts[0].numel() * houts[0].element_size()
    # the pipelined outputs equal the device-resident step's output
    e2e_same = bool(torch.equal(houts[(ke2e - 1) & 1], out.cpu())) if ke2e > 0 else None

    # the host link alone: the same copies on the same streams with no prefill, so the
    # end-to-end step reads against what the link carries in that time
    def copies_only(i):
        b = i & 1
        tq, tk, tv, tg = dins[b]
        with torch.cuda.stream(s_in[0]):
            tq.copy_(hq, non_blocking=True)
        with torch.cuda.stream(s_in[1]):
            tk.copy_(hk, non_blocking=True)
        with torch.cuda.stream(s_in[2]):
            tv.copy_(hv, non_blocking=True)
            tg.copy_(hg, non_blocking=True)
        with torch.cuda.stream(s_out):
            houts[b].copy_(douts[b], non_blocking=True)

    copies_only(0)
    torch.cuda.synchronize(dev)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for st in (*s_in, s_out):
        st.wait_event(c0)
    for i in range(ke2e):
        copies_only(i)
    for st in (*s_in, s_out):
        j = torch.cuda.Event()
        j.record(st)
        stream.wait_event(j)
    c1.record(stream)
    torch.cuda.synchronize(dev)
    ms_link = c0.elapsed_time(c1) / ke2e
    launches = t["tm"]["kernels"]  # every kernel the library launched in the timed region
    timing_main = dict(ms_step=ms_step, tm=t["tm"], tseq=t["tseq"], segments=segments)
    del dins, douts, t
    layer.close()
    torch.cuda.synchronize(dev)

    peaks = _peaks()
    # the other prefill workloads, each timed the same way in this run
    others = {}
    if not args.no_other_workloads:
        for key, w2 in PREFILL.items():
            if w2.name == W.name:
                continue
            t2 = time_prefill(w2, dev, stream, max(3, args.steps // 4), args.warmup, args.segments, world)
            kern2, roof2, step2, fl2 = prefill_report(w2, t2, peaks)
            others[w2.name] = {"value": job_throughput(w2.B * w2.N, world, t2["ms_step"]), "unit": UNIT,
                               "ms_per_step": t2["ms_step"], "steps": max(3, args.steps // 4),
                               "roofline": roof2, "step_tensor_roofline": step2, "kernels": kern2,
                               "algorithmic_flops_per_step": fl2,
                               "overlap": {"fold_segments": t2["segments"]},
                               "config": workload_config(w2, world)}
            t2["layer"].close()
            del t2
            torch.cuda.synchronize(dev)
    decode = None if args.no_decode else run_decode(dev, stream)
    layer_fwd = None if args.no_layer else run_layer(dev, stream, max(3, args.steps // 2), args.segments)
    bwd = None if args.no_backward else run_backward(dev, stream, max(3, args.steps // 4))
    clk = clocks.stop()

    kernels, roofline, step_roof, flops = prefill_report(W, timing_main, peaks)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(world),
        "roofline": roofline,
        "kernels": kernels,
        "algorithmic_flops_per_step": flops,
        # the whole step against the tensor roofline: attention + similarity FLOPs per step time
        "step_tensor_roofline": step_roof,
        "e2e": {"value": W.B * W.N / (ms_e2e / 1e3), "unit": UNIT, "ms_per_step": ms_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": "step i+1's host-to-device copies and step i-1's read-back overlap "
                             "step i's prefill (double-buffered device inputs and outputs)",
                "output_matches_device_step": e2e_same,
                "link": {"copies_only_ms_per_step": ms_link,
                         "gbs": (h2d + d2h) / (ms_link / 1e3) / 1e9,
                         "e2e_frac_of_link": ms_link / ms_e2e,
                         "note": "the same host-to-device and device-to-host copies with no "
                                 "prefill; the end-to-end step cannot be shorter"}},
        "gpu_launches": int(launches),
        "overlap": {"fold_segments": segments,
                    "note": "fold segments on one SM partition (green context), attention of "
                            "folded chunks on the other, the rest on all SMs"},
        "clocks": clk,
        "workloads": others,
        "decode": decode,
        "layer_forward": layer_fwd,
        "backward": bwd,
    }
    return line


def run_backward(dev, stream, steps):
    """Backward of the headline prefill at its fold decisions (kvm_prefill_backward):
    one sequential prefill with a decision record, then the backward timed alone
    with CUDA events; fp32 gradients of q, k, v and the gate."""
    import torch
    from compressed_kv_state_gb300 import kvm
    q, k, v, g = wl.prefill_inputs(W)
    rng = np.random.default_rng(11)
    dout = rng.standard_normal(q.shape).astype(np.float32)
    tq, tk, tv, tdo = (torch.from_numpy(x).to(dev).bfloat16() for x in (q, k, v, dout))
    tg = torch.from_numpy(g).to(dev)
    cfg = kvm.make_config(batch=W.B, heads=W.H, rope_dims=W.rope_dims, chunk=W.chunk, window=W.window,
                          n_sinks=W.n_sinks, sched=W.sched, max_slots=W.max_slots, max_tokens=W.N)
    layer = kvm.KvmLayer(cfg, device=dev)
    E = _n_events(W)
    shp = (W.B, W.H, E, W.chunk)
    assign = torch.empty(shp, dtype=torch.int32, device=dev)
    kind = torch.empty(shp, dtype=torch.int32, device=dev)
    rec = kvm.kvm_debug(assign.data_ptr(), kind.data_ptr(), None, None, E)
    out = layer.prefill(tq, tk, tv, tg, stream=stream, dbg=rec)
    nq = (W.B, W.H, W.N, W.d)
    dq, dk, dv = (torch.empty(nq, dtype=torch.float32, device=dev) for _ in range(3))
    dg = torch.empty(nq[:3], dtype=torch.float32, device=dev)
    scratch = torch.empty(kvm.kvm_backward_scratch_bytes(cfg, W.N), dtype=torch.uint8, device=dev)

    def step():
        kvm.kvm_prefill_backward(layer.handle, tq, tk, tv, tg, out, tdo, rec, W.N, dq, dk, dv, dg, scratch,
                                 stream, cfg=cfg)

    for _ in range(2):
        step()
    layer.sync()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    layer.sync()
    ms = e0.elapsed_time(e1) / steps
    aw = attention_work(W)
    flops = 2.5 * aw["flops_4d"]  # five products of 2d per (query, key) pair against two forward
    tf = flops / (ms / 1e3) / 1e12
    layer.close()
    # bf16 layers run the five products on the tensor cores (tcgen05 for chunks a multiple
    # of 128, fp32 accumulators in tensor memory): the roofline is the measured bf16 burst
    # rate (the backward is timed alone)
    pk = _peaks()
    peak = pk["bf16"]
    return {"ms_per_call": ms, "steps": steps, "value": W.B * W.N / (ms / 1e3), "unit": "tokens/s",
            "algorithmic_flops": flops,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                         "peak_source": f"bf16 burst (of {pk['src']})",
                         "fp32_fma_frac": tf / fp32_simt_peak_tflops()},
            "finite": bool(torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
                           and torch.isfinite(dg).all()),
            "note": "fold decisions from the forward's record are constants (no gradient through the "
                    "winner-take-all assignment); 128-query tiles, 128-key blocks by TMA, the five "
                    "products on tcgen05 (fp32 accumulators in tensor memory; P and dS as bf16), "
                    "fp32 softmax-gradient and read-row gradients, half a warp per slot for the "
                    "state sweep"}


def fp32_simt_peak_tflops():
    """Nominal fp32 FMA rate: 152 SMs x 128 fp32 lanes x 2 FLOP x 2070 MHz."""
    return 152 * 128 * 2 * 2.070e9 / 1e12


def _n_events(w):
    nchunks = -(-w.N // w.chunk)
    return max(0, nchunks - w.window // w.chunk - 1)


def run_layer(dev, stream, steps, segments=-1, d_model=768):
    """Whole-layer forward of the same workload as a d_model = 768 layer (12 heads of
    64, the pages' 120M-like shape): tensor-core input projection with fused gate,
    the KVM attention, output projection.  Random bf16 weights; inputs in HBM."""
    import torch
    from compressed_kv_state_gb300 import kvm
    peaks = _peaks()
    x, w_in, w_out = wl.layer_inputs(W, d_model)
    tx = torch.from_numpy(x).to(dev).bfloat16()
    tin = torch.from_numpy(w_in).to(dev).bfloat16()
    tout = torch.from_numpy(w_out).to(dev).bfloat16()
    cfg = kvm.make_config(batch=W.B, heads=W.H, rope_dims=W.rope_dims, chunk=W.chunk, window=W.window,
                          n_sinks=W.n_sinks, sched=W.sched, max_slots=W.max_slots, max_tokens=W.N)
    layer = kvm.KvmLayer(cfg, device=dev)
    kvm.kvm_layer_set_overlap(layer.handle, segments)
    y = torch.empty((W.B, W.N, d_model), dtype=torch.bfloat16, device=dev)
    scratch = torch.empty(kvm.kvm_forward_scratch_bytes(cfg, d_model, W.N), dtype=torch.uint8, device=dev)

    def step():
        kvm.kvm_layer_forward(layer.handle, d_model, tx, tin, tout, W.N, y, scratch, stream)

    for _ in range(3):
        step()
    layer.sync()
    kvm.kvm_layer_set_timing(layer.handle, True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    tm = kvm.kvm_layer_get_timing(layer.handle)
    kvm.kvm_layer_set_timing(layer.handle, False)
    layer.sync()
    Hd = W.H * W.d
    proj_flops = 2.0 * W.B * W.N * d_model * (3 * Hd + W.H) + 2.0 * W.B * W.N * Hd * d_model
    proj_ms = tm["proj_ms"] / max(1, steps)
    tf = proj_flops / (proj_ms / 1e3) / 1e12
    layer.close()
    return {"d_model": d_model, "value": W.B * W.N / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
            "projections": {"ms_per_step": proj_ms, "flops_per_step": proj_flops, "tflops": tf,
                            "frac_of_bf16_peak": tf / peaks["bf16"], "peak": peaks["bf16"],
                            "note": "two launches per step (input and output projection), "
                                    "times summed; measured bf16 burst peak"}}


def run_decode(dev, stream):
    """Decode sweep: 128 steps from a chunk boundary with an imported state of
    n = 256, 512, 1024 slots (B=64, H=16, window 512, bf16)."""
    import torch
    from compressed_kv_state_gb300 import kvm
    peaks = _peaks()
    res = {}
    for n, dw in wl.DECODE.items():
        state, (wk, wv, wg), (q, k, v, g) = wl.decode_inputs(dw)
        cfg = kvm.make_config(batch=dw.B, heads=dw.H, rope_dims=dw.rope_dims, chunk=dw.chunk,
                              window=dw.window, n_sinks=dw.n_sinks, sched=kvm.KVM_SCHED_FIXED,
                              max_slots=n, max_tokens=dw.pos0 + dw.steps)
        layer = kvm.KvmLayer(cfg, device=dev)
        L = dw.window + dw.chunk
        idx = (dw.pos0 - L + np.arange(L)) % L
        bufs = layer.state_buffers(dev)
        bufs["sum_k"][:, :, :n] = torch.from_numpy(state["sum_k"]).to(dev)
        bufs["sum_v"][:, :, :n] = torch.from_numpy(state["sum_v"]).to(dev)
        bufs["counts"][:, :, :n] = torch.from_numpy(state["counts"]).to(dev)
        bufs["rho"][:, :, :n] = torch.from_numpy(state["rho"]).to(dev)
        rk = np.zeros_like(wk); rv = np.zeros_like(wv); rg = np.zeros_like(wg)
        rk[:, :, idx], rv[:, :, idx], rg[:, :, idx] = wk, wv, wg
        bufs["ring_k"].copy_(torch.from_numpy(rk).bfloat16())
        bufs["ring_v"].copy_(torch.from_numpy(rv).bfloat16())
        bufs["ring_g"].copy_(torch.from_numpy(rg))
        bufs.update(n_slots=n, n_overflow=state["t"], pos=dw.pos0)
        dq = torch.from_numpy(q).to(dev).bfloat16()
        dk = torch.from_numpy(k).to(dev).bfloat16()
        dv = torch.from_numpy(v).to(dev).bfloat16()
        dg = torch.from_numpy(g).to(dev)
        out = torch.empty(dw.B, dw.H, dw.d, dtype=torch.bfloat16, device=dev)
        times = []
        for rep in range(2):  # first pass warms up; second is timed
            layer.import_state(bufs)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(dw.steps + 1)]
            evs[0].record(stream)
            for s in range(dw.steps):
                kvm.kvm_decode_step(layer.handle, dq[s], dk[s], dv[s], dg[s], out, stream)
                evs[s + 1].record(stream)
            torch.cuda.synchronize(dev)
            times = [evs[s].elapsed_time(evs[s + 1]) * 1e3 for s in range(dw.steps)]
        layer.sync()
        nb = times[1:]
        med = statistics.median(nb)
        mid = 1 + int(np.argsort(nb)[len(nb) // 2])
        byt = decode_bytes(dw, mid, n)
        res[f"n{n}"] = dict(boundary_us=times[0], median_us=med, mean_us=float(np.mean(times)),
                            hbm_frac=byt / (med * 1e-6) / (peaks["hbm"] * 1e9),
                            bytes_median_step=byt, peak_gbs=peaks["hbm"])
        layer.close()
    return res


# ------------------------------------------------------------- reference

KEYS = {"plain": "N(0,1) keys", "repeat5": "5% repeated keys", "needles10": "10 planted needle keys",
        "neardup20": "20% near-duplicate keys"}


def workload_config(w, world):
    in_bytes = w.B * w.H * w.N * (3 * w.d * 2 + 4)  # bf16 q, k, v and the fp32 gate
    cfg = {"workload": w.name, "batch": w.B, "heads": w.H, "seq_len": w.N,
           "head_dim": w.d, "chunk": w.chunk, "window": w.window,
           "slots": w.max_slots, "sinks": w.n_sinks, "rope_dims": w.rope_dims,
           "growth": "fixed" if w.sched == 0 else f"power law: {w.n_sinks} + ceil({w.coef:g} t^{w.expo:g})",
           "keys": KEYS.get(w.keys, w.keys),
           "l2": f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB), no flush",
           "parallelism": f"rows (batch x head) independent, {world} replica(s)"}
    return cfg


def bench_config(world):
    """The workload both arms report (the reference arm times a sample of it)."""
    return workload_config(W, world)


def run_reference(args):
    """The oracle as it stands, on the host cores: each step is a bounded sample
    of the same workload (one full-length row per core)."""
    for _ in range(args.warmup):
        cpu_oracle_sample(W, one_thread=False)
    secs = []
    for _ in range(args.steps):  # timed: the oracle call of each step (not its input generation)
        r, _ = cpu_oracle_sample(W, one_thread=False)
        secs.append(r.pop("seconds"))
    wall = sum(secs)
    tokens_per_step = W.N * r["cores"] / W.H
    value = tokens_per_step * args.steps / wall
    cb = dict(value=value, unit=UNIT, cores=r["cores"], kind="oracle", sample=r["sample"])
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": bench_config(int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-layer", action="store_true", help="skip the whole-layer forward line")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward line")
    ap.add_argument("--segments", type=int, default=-1,
                    help="fold segments of the overlapped prefill (0: sequential, <0: automatic)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="run the same workload with another batch size (profiling a smaller case)")
    ap.add_argument("--workload", choices=sorted(PREFILL), default="fixed8k",
                    help="headline prefill workload (the others are reported under 'workloads')")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="time only the headline prefill workload")
    args = ap.parse_args()
    global W
    W = PREFILL[args.workload]
    if args.batch is not None:
        W = W.with_(B=args.batch, name=W.name.replace(f"B{W.B}", f"B{args.batch}"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu:
            import torch
            dev = torch.device("cuda", local_rank)
            cb, (sub, odbg) = cpu_oracle_sample(W)
            cb.pop("seconds")
            line["cpu_baseline"] = cb
            line["near_ties"] = near_tie_counts(sub, odbg, dev)
            for w2 in PREFILL.values():
                rec = line["workloads"].get(w2.name)
                if rec is None:
                    continue
                cb2, (sub2, odbg2) = cpu_oracle_sample(w2, one_thread=False)
                cb2.pop("seconds")
                rec["cpu_baseline"] = cb2
                rec["near_ties"] = near_tie_counts(sub2, odbg2, dev)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
