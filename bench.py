#!/usr/bin/env python3
"""Decode-attention benchmark over the block-quantised KV cache (one JSON line on stdout).

A step is one pass of the whole hot path over one batch: for every layer, quantise-on-
append of the new K/V row of each sequence, then split-K decode attention with its split
merge, all in one kernel per layer (kvq_append_decode).  Each step is one CUDA-graph replay.  Inputs are
seeded synthetic tensors shaped like the pages' models (see synthetic.py); caches are
filled and resident in HBM before the timed region starts.

Headline (value): KV-read GB/s of the 10-layer hybrid shape (Hkv 2, Hq 16, D 256) with
q8_0 K / q8_0 V at 65,536 context.  The line also carries the per-(KV type, context)
sweep (steps/s, KV GB/s, % of HBM peak), the decode kernel's roofline, an end-to-end
number with host buffers, the CPU oracle baseline and the SM clocks seen.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference] [--cells headline|default]
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
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic as syn  # noqa: E402

METRIC = "KV-read GB/s (% of GB300 HBM peak) and decode-attn steps/s vs ctx per KV type"
BPV = {"f16": 2.0, "q8_0": 34 / 32, "q4_0": 18 / 32, "q4_1": 20 / 32, "q5_0": 22 / 32, "q5_1": 24 / 32}
L2_BYTES = 129 * 10**6
HBM_FALLBACK = 6800.0


def row_bytes(wl) -> float:
    """Algorithmic KV bytes per (position, layer) of one sequence: Hkv * D * (bpv_K + bpv_V)."""
    return wl.n_kv_heads * wl.head_dim * (BPV[wl.type_k] + BPV[wl.type_v])


def step_kv_bytes(wl, lens) -> float:
    return wl.layers * sum(lens) * row_bytes(wl)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK, "fallback"


def headline_workload():
    return syn.hybrid(65536, "q8_0", "q8_0")


def sweep_workloads(which: str):
    cells = [headline_workload()]
    if which == "headline":
        return cells
    for ctx in (4096, 16384, 32768, 65536):
        for tk, tv in (("q8_0", "q8_0"), ("f16", "f16")):
            wl = syn.hybrid(ctx, tk, tv)
            if wl != cells[0]:
                cells.append(wl)
    for ctx in (65536, 131072):
        cells.append(syn.dense14b(ctx, "q8_0", "q4_0"))
        cells.append(syn.dense14b(ctx, "f16", "f16"))
    cells.append(syn.dense14b(131072, "q4_0", "q4_0"))
    cells.append(syn.dense14b(262144, "q4_0", "q4_0"))
    cells.append(syn.dense14b(262144, "q8_0", "q8_0"))
    for tk, tv in (("q8_0", "q5_0"), ("q5_0", "q5_0"), ("q5_1", "q5_1"), ("q4_1", "q4_1"), ("q5_1", "q4_0")):
        cells.append(syn.dense14b(131072, tk, tv))
    cells.append(syn.multi_session())
    return cells


# ----------------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1, margin=0.05):
        sel = [s for (t, s) in self.samples if t0 - margin <= t <= t1 + margin and len(s) >= 9]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi sample in the timed window"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in sel if num(s[1]) is not None]
        smax = [num(s[2]) for s in sel if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in sel for i in range(4) if s[5 + i].lower().startswith("active")})
        pw = [num(s[3]) for s in sel if num(s[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(sel), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------------------
class Cell:
    """L per-layer caches filled to the workload's lengths, plus static step buffers."""

    def __init__(self, kvq, torch, wl, extra_rows: int, stream):
        self.kvq, self.torch, self.wl, self.stream = kvq, torch, wl, stream
        cap = ((max(wl.lengths) + extra_rows + 15) // 16) * 16
        self.caches = []
        dev = torch.device("cuda", torch.cuda.current_device())
        with torch.cuda.stream(stream):
            for layer in range(wl.layers):
                c = kvq.KVCache(wl.batch, wl.n_kv_heads, wl.head_dim, cap, wl.type_k, wl.type_v, device=dev)
                for b in range(wl.batch):
                    n = wl.lengths[b]
                    if n == 0:
                        continue
                    K = torch.stack([syn.kv_rows(wl, syn.KIND_K, layer, b, h, 0, n) for h in range(wl.n_kv_heads)])
                    V = torch.stack([syn.kv_rows(wl, syn.KIND_V, layer, b, h, 0, n) for h in range(wl.n_kv_heads)])
                    c.append(K[None], V[None], b0=b, stream=stream)
                    del K, V
                self.caches.append(c)
            L, B = wl.layers, wl.batch
            q = torch.stack([syn.queries(wl, layer) for layer in range(L)])
            news = [syn.new_rows(wl, layer, 0) for layer in range(L)]
            knew = torch.stack([k for k, _ in news])
            vnew = torch.stack([v for _, v in news])
            # a step's inputs (q, new K, new V) and results (out, lse) each in one flat buffer,
            # so that a host round trip is one copy in and one copy out
            nq, nk, nv = q.numel(), knew.numel(), vnew.numel()
            self.inputs = torch.empty(nq + nk + nv, device=dev, dtype=torch.float32)
            self.q = self.inputs[:nq].view(q.shape)
            self.knew = self.inputs[nq:nq + nk].view(knew.shape)
            self.vnew = self.inputs[nq + nk:].view(vnew.shape)
            self.q.copy_(q)
            self.knew.copy_(knew)
            self.vnew.copy_(vnew)
            del q, knew, vnew, news
            self.results = torch.empty(nq + L * B * wl.n_q_heads, device=dev, dtype=torch.float32)
            self.out = self.results[:nq].view(self.q.shape)
            self.lse = self.results[nq:].view(L, B, wl.n_q_heads)
            self.splits = self.caches[0].auto_splits(wl.n_q_heads)
            self.ws = self.caches[0].workspace(wl.n_q_heads, self.splits)  # layers run in order: one workspace
        torch.cuda.synchronize()
        self.lens = list(wl.lengths)

    def launch_step(self, events=None):
        """Enqueue one step (append + decode per layer) on self.stream."""
        for layer, c in enumerate(self.caches):
            if events is not None:
                events[layer][0].record(self.stream)
            c.append_decode(self.knew[layer], self.vnew[layer], self.q[layer], scale=self.wl.scale,
                            n_splits=self.splits, out=self.out[layer], lse=self.lse[layer], workspace=self.ws,
                            stream=self.stream)
            if events is not None:
                events[layer][1].record(self.stream)

    def executed(self, n_steps):
        self.lens = [x + n_steps for x in self.lens]

    def free(self):
        self.caches.clear()


def make_event(torch, external):
    if external:
        return torch.cuda.Event(enable_timing=True, external=True)
    return torch.cuda.Event(enable_timing=True)


def launch_ctas(cell):
    """CTAs of one decode launch of a cell: splits x KV heads x sequences x row groups."""
    wl = cell.wl
    return cell.splits * wl.n_kv_heads * wl.batch * ((wl.G + 7) // 8)


STAMPS_PER_CTA = 2


def stamp_spans(stamps, n_launch, layers, ctas):
    """Per-launch timing from the CTA timer stamps of the last replay of each stamp graph
    (per CTA: start, exit): span = last CTA exit - first CTA start (includes the overlap
    with the neighbouring layers under programmatic dependent launch); gap = this launch's
    last exit - the previous launch's last exit (the time a layer adds to the step)."""
    st = stamps.view(n_launch, ctas, STAMPS_PER_CTA).double()
    starts, ends = st[:, :, 0].min(dim=1).values, st[:, :, 1].max(dim=1).values
    spans = ((ends - starts) * 1e-3).tolist()  # us
    gaps = []
    for g in range(n_launch // layers):
        e = ends[g * layers:(g + 1) * layers]
        gaps += ((e[1:] - e[:-1]) * 1e-3).tolist()
    return spans, gaps


def run_cell(kvq, torch, wl, steps, warmup, peak, sampler=None, e2e=False, n_event_graphs=16, n_stamp_graphs=4):
    stream = torch.cuda.Stream()
    extra = 1 + warmup + 3 * steps + (warmup + steps if e2e else 0) + 8
    cell = Cell(kvq, torch, wl, extra, stream)
    L = wl.layers
    # eager warm-up step (also configures the kernels outside any capture)
    cell.launch_step()
    torch.cuda.synchronize()
    cell.executed(1)
    try:
        make_event(torch, True)
        external = True
    except TypeError:
        external = False
    n_eg = min(steps, n_event_graphs) if external else 0
    ev_sets = [[(make_event(torch, True), make_event(torch, True)) for _ in range(L)] for _ in range(n_eg)]
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain, stream=stream):
        cell.launch_step()
    g_ev = []
    for k in range(n_eg):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            cell.launch_step(ev_sets[k])
        g_ev.append(g)
    # graphs whose launches write per-CTA timer stamps (no events: the same schedule as g_plain)
    ctas = launch_ctas(cell)
    n_sg = min(steps, n_stamp_graphs)
    stamps = torch.zeros(n_sg * L * ctas * STAMPS_PER_CTA, dtype=torch.int64, device=stream.device)
    kvq.set_launch_stamps(stamps, n_sg * L, ctas)
    g_st = []
    try:
        for k in range(n_sg):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                cell.launch_step()
            g_st.append(g)
    finally:
        kvq.set_launch_stamps(None)
    torch.cuda.synchronize()
    for _ in range(warmup):
        g_plain.replay()
    torch.cuda.synchronize()
    cell.executed(warmup)
    lens0 = list(cell.lens)
    # timed region 1 (the step time): event-free graph replays, so consecutive kernels can
    # overlap through programmatic dependent launch exactly as in production
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for k in range(steps):
            g_plain.replay()
        e1.record(stream)
    e1.synchronize()
    wall1 = time.time()
    ms_total = e0.elapsed_time(e1)
    cell.executed(steps)
    ms_step = ms_total / steps
    # timed region 2 (the kernel time): the same steps with CUDA events recorded around every
    # decode launch; event nodes serialise the launches, so this pass gives per-launch
    # durations (conservative: each includes its own launch latency), not the step time
    if n_eg:
        with torch.cuda.stream(stream):
            for k in range(steps):
                g_ev[k % n_eg].replay()
        torch.cuda.synchronize()
        cell.executed(steps)
    # timed region 3: the same steps through the stamp graphs (timer stamps per CTA)
    ms_stamp = None
    if n_sg:
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s0.record(stream)
            for k in range(steps):
                g_st[k % n_sg].replay()
            s1.record(stream)
        s1.synchronize()
        ms_stamp = s0.elapsed_time(s1) / steps
        cell.executed(steps)
    # mean lengths over the timed steps (each step appends one row before its decode)
    mean_lens = [x + (steps + 1) / 2.0 for x in lens0]
    bytes_step = step_kv_bytes(wl, mean_lens)
    res = {
        "workload": wl.name, "layers": L, "batch": wl.batch, "n_q_heads": wl.n_q_heads,
        "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim, "kv": f"{wl.type_k}/{wl.type_v}",
        "ctx": list(wl.lengths) if wl.batch > 1 else wl.lengths[0], "splits": cell.splits,
        "steps_per_s": 1000.0 / ms_step, "ms_per_step": ms_step,
        "kv_gbs": bytes_step / (ms_step * 1e-3) / 1e9, "kv_bytes_per_step": bytes_step,
        "l2": "inputs larger than L2" if bytes_step > 4 * L2_BYTES else "set within 4x L2: L2-assisted",
    }
    res["pct_hbm_peak"] = 100.0 * res["kv_gbs"] / peak
    res["_wall"] = (wall0, wall1)
    # the step holds nothing but decode launches (one per layer): its CUDA-event time over
    # the timed region / layers is the kernel's average in-step launch duration
    res["decode_instep_us"] = ms_step * 1e3 / L
    if n_sg:
        spans, gaps = stamp_spans(stamps, n_sg * L, L, ctas)
        res["stamps"] = {"span_us_mean": statistics.fmean(spans), "span_us_median": statistics.median(spans),
                         "gap_us_mean": statistics.fmean(gaps) if gaps else None,
                         "launches": len(spans), "ms_per_step_stamp_pass": ms_stamp,
                         "how": "%globaltimer per CTA (start, exit) in event-free graph replays; span = first "
                                "start to last exit of a launch (overlaps its neighbours under programmatic "
                                "dependent launch), gap = last exit of a launch - last exit of the previous one"}
    if n_eg:
        durs = []
        for k in range(n_eg):
            for layer in range(L):
                a, b = ev_sets[k][layer]
                durs.append(a.elapsed_time(b))
        avg_ms = sum(durs) / len(durs)
        per_launch_bytes = bytes_step / L
        res["decode_us"] = avg_ms * 1e3
        res["decode_gbs"] = per_launch_bytes / (avg_ms * 1e-3) / 1e9
        res["decode_launches_timed"] = len(durs)
        res["roofline_timing"] = ("CUDA events around every decode launch, in a second timed pass of the same "
                                  "steps (event nodes serialise launches; the step time comes from the event-free pass)")
    if e2e:
        pin = dict(pin_memory=True)
        in_h = torch.empty(cell.inputs.shape, dtype=torch.float32, **pin)  # q, new K, new V
        res_h = torch.empty(cell.results.shape, dtype=torch.float32, **pin)  # out, lse
        in_h.copy_(cell.inputs)
        torch.cuda.synchronize()

        def e2e_step():
            cell.inputs.copy_(in_h, non_blocking=True)
            g_plain.replay()
            res_h.copy_(cell.results, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(warmup):
                e2e_step()
            torch.cuda.synchronize()
            cell.executed(warmup)
            lens_e = list(cell.lens)
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(steps):
                e2e_step()
            f1.record(stream)
        f1.synchronize()
        cell.executed(steps)
        ms_e = f0.elapsed_time(f1) / steps
        b_e = step_kv_bytes(wl, [x + (steps + 1) / 2.0 for x in lens_e])
        h2d = in_h.numel() * 4
        d2h = res_h.numel() * 4
        res["e2e"] = {"value": b_e / (ms_e * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": ms_e,
                      "how": "pinned-host inputs (q, new K, new V) copied in, graph step, outputs (out, lse) copied out, every step: one copy each way"}
    for c in cell.caches:
        if c.read_error() != 0:
            res["device_error"] = True
    cell.free()
    del g_plain, g_ev, g_st
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_rotating(kvq, torch, wl, steps, warmup, peak):
    """A cell whose step set is within 4x L2, timed over R copies of its caches used in turn
    (R x set > 4x L2), so that each step reads its KV from HBM rather than from L2."""
    one = step_kv_bytes(wl, list(wl.lengths))
    R = int(math.ceil(4 * L2_BYTES / one)) + 1
    stream = torch.cuda.Stream()
    extra = 1 + warmup + steps + 8
    cells = [Cell(kvq, torch, wl, extra, stream) for _ in range(R)]
    for c in cells:
        c.launch_step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in cells:
            c.launch_step()
    torch.cuda.synchronize()
    reps = max(1, steps // R)
    for _ in range(max(1, warmup // R)):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / (reps * R)
    bytes_step = step_kv_bytes(wl, [x + 2 + max(1, warmup // R) + reps / 2.0 for x in wl.lengths])
    err = any(c2.read_error() for c in cells for c2 in c.caches)
    for c in cells:
        c.free()
    del g, cells
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    r = {"copies": R, "set_bytes": R * one, "ms_per_step": ms, "steps_per_s": 1000.0 / ms,
         "kv_gbs": bytes_step / (ms * 1e-3) / 1e9, "pct_hbm_peak": 100.0 * bytes_step / (ms * 1e-3) / 1e9 / peak,
         "steps": reps * R}
    if err:
        r["device_error"] = True
    return r


def run_window_cell(kvq, torch, wl, window, steps, warmup, peak):
    """Position-axis mixed cache (f16 window of the last `window` tokens + quantised tail):
    one step = for every layer, kvq_window_append_decode: the new row into the window (the
    oldest window row evicted into the tail) and decode over both regions with one exact
    merge, in one launch; the layers of a step form one CUDA graph."""
    stream = torch.cuda.Stream()
    L, B = wl.layers, wl.batch
    ctx = wl.lengths[0]
    extra = 1 + warmup + steps + 8
    caches = []
    with torch.cuda.stream(stream):
        for layer in range(L):
            c = kvq.WindowedCache(B, wl.n_kv_heads, wl.head_dim, window, ((ctx - window + extra + 15) // 16) * 16,
                                  wl.type_k, wl.type_v, stream=stream)
            for b in range(B):
                K = torch.stack([syn.kv_rows(wl, syn.KIND_K, layer, b, h, 0, ctx) for h in range(wl.n_kv_heads)])
                V = torch.stack([syn.kv_rows(wl, syn.KIND_V, layer, b, h, 0, ctx) for h in range(wl.n_kv_heads)])
                c.tail.append(K[None, :, :ctx - window].contiguous(), V[None, :, :ctx - window].contiguous(), b0=b,
                              stream=stream)
                c.window.append(K[None, :, ctx - window:].contiguous(), V[None, :, ctx - window:].contiguous(), b0=b,
                                stream=stream)
                del K, V
            caches.append(c)
        q = torch.stack([syn.queries(wl, layer) for layer in range(L)]).contiguous()
        news = [syn.new_rows(wl, layer, 0) for layer in range(L)]
        knew = torch.stack([k[:, :, 0] for k, _ in news]).contiguous()
        vnew = torch.stack([v[:, :, 0] for _, v in news]).contiguous()
        out = torch.empty_like(q)
        lse = torch.empty((L, B, wl.n_q_heads), device=q.device)
        ws = caches[0].workspace(wl.n_q_heads)
    torch.cuda.synchronize()

    def step():
        for layer, c in enumerate(caches):
            c.append_decode(knew[layer], vnew[layer], q[layer], scale=wl.scale, out=out[layer], lse=lse[layer],
                            workspace=ws, stream=stream)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    D, H = wl.head_dim, wl.n_kv_heads
    bpv = {"f16": 2.0, "q8_0": 34 / 32, "q4_0": 18 / 32}
    n_tail = ctx - window + 1 + warmup + steps / 2.0  # mean tail length over the timed steps
    bytes_step = L * B * H * D * (window * 4.0 + n_tail * (bpv[wl.type_k] + bpv[wl.type_v]))
    err = any(c.window.read_error() or c.tail.read_error() for c in caches)
    family = wl.name.split("-")[0]
    res = {"workload": f"{family}-{L}L-window{window}-f16+{wl.type_k}-{wl.type_v}-ctx{ctx}", "layers": L, "batch": B,
           "n_q_heads": wl.n_q_heads, "n_kv_heads": H, "head_dim": D, "kv": f"f16 window + {wl.type_k}/{wl.type_v} tail",
           "ctx": ctx, "window": window, "steps_per_s": 1000.0 / ms, "ms_per_step": ms,
           "kv_gbs": bytes_step / (ms * 1e-3) / 1e9, "kv_bytes_per_step": bytes_step,
           "pct_hbm_peak": 100.0 * bytes_step / (ms * 1e-3) / 1e9 / peak,
           "step": "per layer: one launch appends the row (evicting the oldest window row into the tail) "
                   "and decodes over both regions (window and tail splits in one grid, one exact merge)"}
    if err:
        res["device_error"] = True
    del g
    caches.clear()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_verify_cell(kvq, torch, wl, n_q, steps, warmup, peak):
    """Draft verify: one step = kvq_decode_verify of n_q queries per sequence on every
    layer (the draft rows are the last n_q cache rows); the layers form one CUDA graph."""
    stream = torch.cuda.Stream()
    cell = Cell(kvq, torch, wl, 0, stream)
    L, B = wl.layers, wl.batch
    gen = torch.Generator(device="cuda").manual_seed(n_q)
    q = torch.randn((L, B, n_q, wl.n_q_heads, wl.head_dim), generator=gen, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((L, B, n_q, wl.n_q_heads), device="cuda")
    b = __import__("ctypes").c_size_t()
    kvq._check(kvq.lib.kvq_verify_workspace_size(cell.caches[0].handle, n_q, wl.n_q_heads, 0,
                                                 __import__("ctypes").byref(b)), "kvq_verify_workspace_size")
    ws = torch.zeros(b.value, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()

    def step():
        for layer, c in enumerate(cell.caches):
            c.verify(q[layer], scale=wl.scale, out=out[layer], lse=lse[layer], workspace=ws, stream=stream)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    torch.cuda.synchronize()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    bytes_step = step_kv_bytes(wl, list(wl.lengths))
    res = {"workload": f"verify-nq{n_q}-{wl.name}", "layers": L, "batch": B, "n_q_heads": wl.n_q_heads,
           "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim, "kv": f"{wl.type_k}/{wl.type_v}",
           "ctx": wl.lengths[0] if B == 1 else list(wl.lengths), "n_q": n_q, "steps_per_s": 1000.0 / ms,
           "ms_per_step": ms, "kv_gbs": bytes_step / (ms * 1e-3) / 1e9, "kv_bytes_per_step": bytes_step,
           "pct_hbm_peak": 100.0 * bytes_step / (ms * 1e-3) / 1e9 / peak,
           "step": f"per layer: verify of {n_q} draft queries per sequence (causal within the draft)"}
    if any(c.read_error() for c in cell.caches):
        res["device_error"] = True
    cell.free()
    del g
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def chunk_quantise(kvq, torch, wl, reps=20, warmup=3):
    """The 4096-row prefill-chunk quantise of one layer: fp32 K,V [1,Hkv,4096,D] -> cache."""
    n = 4096
    cap = n * (reps + warmup)
    c = kvq.KVCache(1, wl.n_kv_heads, wl.head_dim, cap, wl.type_k, wl.type_v)
    K = torch.stack([syn.kv_rows(wl, syn.KIND_K, 0, 0, h, 0, n) for h in range(wl.n_kv_heads)])[None].contiguous()
    V = torch.stack([syn.kv_rows(wl, syn.KIND_V, 0, 0, h, 0, n) for h in range(wl.n_kv_heads)])[None].contiguous()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            c.append(K, V, stream=stream)
    torch.cuda.synchronize()
    # the timed appends form one CUDA graph, so that host launch overhead is not timed
    c.set_lengths([0], stream=stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            c.append(K, V, stream=stream)
    c.set_lengths([0], stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        g.replay()
        e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    err = c.read_error()
    rb = 2 * n * wl.n_kv_heads * wl.head_dim * 4
    wb = n * row_bytes(wl)
    r = {"rows": n, "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim, "kv": f"{wl.type_k}/{wl.type_v}",
         "us_per_chunk": ms * 1e3, "bytes_read": rb, "bytes_written": wb,
         "gbs": (rb + wb) / (ms * 1e-3) / 1e9, "timing": f"{reps} appends of one chunk in one CUDA graph"}
    if err:
        r["device_error"] = True
    return r


# ----------------------------------------------------------------------------------------
# the CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------------------
def oracle_cell(wl, layer=0):
    """Natural-layout oracle cache of one layer (setup, untimed) + the step's new rows."""
    import oracle
    import torch
    n = wl.lengths[0]
    extra = 64
    # the GPU arm's generator where a GPU is present (the same values as that arm); else the
    # host's (other values of the same distribution: the oracle's time depends on sizes only)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    K = torch.stack([syn.kv_rows(wl, syn.KIND_K, layer, 0, h, 0, n, device=dev) for h in range(wl.n_kv_heads)])
    V = torch.stack([syn.kv_rows(wl, syn.KIND_V, layer, 0, h, 0, n, device=dev) for h in range(wl.n_kv_heads)])
    kc, ks = oracle.quantize(wl.type_k, K.cpu().numpy(), n_threads=0)
    vc, vs = oracle.quantize(wl.type_v, V.cpu().numpy(), n_threads=0)

    def grow(a):
        pad = np.zeros((a.shape[0], extra) + a.shape[2:], a.dtype)
        return np.concatenate([a, pad], axis=1)
    kc, ks, vc, vs = grow(kc), grow(ks), grow(vc), grow(vs)
    q = syn.queries(wl, layer, device=dev).cpu().numpy()[0]
    kn, vn = syn.new_rows(wl, layer, 0, device=dev)
    return {"kc": kc, "ks": ks, "vc": vc, "vs": vs, "n": n, "q": q,
            "kn": kn.cpu().numpy()[0, :, 0], "vn": vn.cpu().numpy()[0, :, 0]}


def oracle_step(wl, st):
    """One layer of one step on the CPU oracle: quantise the new row, attend over the cache."""
    import oracle
    n = st["n"]
    kc1, ks1 = oracle.quantize(wl.type_k, st["kn"], n_threads=0)
    vc1, vs1 = oracle.quantize(wl.type_v, st["vn"], n_threads=0)
    st["kc"][:, n], st["vc"][:, n] = kc1, vc1
    if st["ks"].shape[-1]:
        st["ks"][:, n] = ks1
    if st["vs"].shape[-1]:
        st["vs"][:, n] = vs1
    st["n"] = n + 1 if n + 1 < st["kc"].shape[1] else n
    oracle.attention(wl.type_k, st["kc"], st["ks"], wl.type_v, st["vc"], st["vs"], n + 1, st["q"], wl.scale,
                     n_threads=0)
    return (n + 1) * row_bytes(wl)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def oracle_attend_rate(wl, st, n_threads, budget_s):
    """GB/s of the oracle's fp64 attention over the cell's cache (one layer per call)."""
    import oracle
    n = st["n"]
    oracle.attention(wl.type_k, st["kc"], st["ks"], wl.type_v, st["vc"], st["vs"], n, st["q"], wl.scale,
                     n_threads=n_threads)
    t0 = time.perf_counter()
    k = 0
    while True:
        oracle.attention(wl.type_k, st["kc"], st["ks"], wl.type_v, st["vc"], st["vs"], n, st["q"], wl.scale,
                         n_threads=n_threads)
        k += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"gbs": k * n * row_bytes(wl) / dt / 1e9, "s_per_layer": dt / k, "calls": k}


def oracle_quantise_rate(n_threads, budget_s, rows=1024):
    """Rows/s of the oracle's quantiser on the 14B shape's K (q8_0) and V (q4_0) rows
    (8 KV heads x 128 values per row and plane)."""
    import oracle
    rng = np.random.default_rng(7)
    K = rng.standard_normal((8, rows, 128)).astype(np.float32)
    V = rng.standard_normal((8, rows, 128)).astype(np.float32)
    oracle.quantize("q8_0", K, n_threads=n_threads)
    t0 = time.perf_counter()
    k = 0
    while True:
        oracle.quantize("q8_0", K, n_threads=n_threads)
        oracle.quantize("q4_0", V, n_threads=n_threads)
        k += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"rows_per_s": k * rows / dt, "gbs": k * rows * 8 * 128 * 4 * 2 / dt / 1e9}


def cpu_baseline(wl, budget_s=10.0):
    st = oracle_cell(wl)
    oracle_step(wl, st)  # warm
    t0 = time.perf_counter()
    nbytes, nsteps = 0.0, 0
    while True:
        nbytes += oracle_step(wl, st)
        nsteps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cores = cpu_cores()
    # the same oracle single-threaded and on all cores (thread count set explicitly each call)
    detail = {"attention_1_thread": oracle_attend_rate(wl, st, 1, budget_s / 2),
              "attention_all_cores": oracle_attend_rate(wl, st, cores, budget_s / 4),
              "quantise_1_thread": oracle_quantise_rate(1, budget_s / 8),
              "quantise_all_cores": oracle_quantise_rate(cores, budget_s / 8),
              "scaled": f"the oracle runs one layer of {wl.name}; a {wl.layers}-layer step takes "
                        f"{wl.layers} x that (GB/s is the same)"}
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{nsteps} single-layer decode steps (1-row quantise + fp64 attention of all "
                      f"{wl.n_q_heads} query heads over {wl.lengths[0]}+ rows) of {wl.name}; GB/s of the "
                      f"same algorithmic KV bytes, OpenMP over query heads",
            "seconds": dt, "detail": detail}


# ----------------------------------------------------------------------------------------
def decode_kernel_sha() -> str:
    """sha256 over the decode kernel's sources (kernel template, decode launches, shared header)."""
    h = hashlib.sha256()
    for name in ("kvq_decode_kernel.cuh", "kvq_decode.cu", "kvq_internal.cuh"):
        with open(os.path.join(ROOT, "quantised_kv_long_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_from_profiles(wl, path=None):
    """ncu DRAM bytes per decode launch recorded in profiles/, if the kernel source is unchanged."""
    path = path or os.path.join(ROOT, "profiles", "decode_traffic.txt")
    try:
        sha = decode_kernel_sha()
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("decode kernel sha256") != sha or kv.get("workload") != wl.name:
            return None
        return float(kv["dram bytes per launch (read+write)"])
    except Exception:
        return None


def short_name(r):
    """A short cell label: shape, KV types, context."""
    w = r["workload"]
    fam = "hyb" if w.startswith("hybrid") else ("ms16" if w.startswith("multi") else "d48")
    if w.startswith("verify"):
        fam = "vfy" + str(r.get("n_q", "")) + "-" + ("hyb" if "hybrid" in w else "d48")
    kv = r["kv"].replace("_0", "").replace("_1", "1").replace("f16 window + ", "w+").replace(" tail", "")
    ctx = r["ctx"] if isinstance(r["ctx"], int) else "mix"
    return f"{fam} {kv} {ctx // 1024}K" if isinstance(ctx, int) else f"{fam} {kv} {ctx}"


def compact_cells(sweep, chunk):
    """[label, steps/s, KV GB/s, % of HBM peak] per cell (+ rotating-buffer % where taken)."""
    out = []
    for r in sweep:
        row = [short_name(r), round(r["steps_per_s"], 1), round(r["kv_gbs"]), round(r["pct_hbm_peak"], 1)]
        if "rotating" in r:
            row.append(round(r["rotating"]["pct_hbm_peak"], 1))
        out.append(row)
    if chunk:
        out.append(["chunk4096 q8/q4", round(chunk["us_per_chunk"], 1), round(chunk["gbs"]), None])
    return out


def max_over_ranks(dist, value, device):
    """The largest per-rank value (a step time): the whole job is as slow as its slowest rank.
    Every rank gets the result."""
    import torch
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, bytes_per_rank_step, ms_per_step):
    """Whole-job KV-read GB/s: each of the `world` replicas reads its own bytes every step,
    and a step lasts the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--cells", choices=["headline", "default"], default="default")
    ap.add_argument("--sweep-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None, help="run just this sweep workload (by name) as the timed cell")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (profiling captures)")
    ap.add_argument("--cell", choices=["verify4", "verify16", "window", "chunk"], default=None,
                    help="time only this extra cell on the --only workload (default: the headline) and print it")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = headline_workload()
    if args.only:
        named = {w.name: w for w in sweep_workloads("default")}
        if args.only not in named:
            raise SystemExit(f"unknown workload {args.only!r}; one of: {', '.join(named)}")
        wl = named[args.only]
        args.cells = "headline"
    if args.layers:
        import dataclasses
        wl = dataclasses.replace(wl, layers=args.layers, name=f"{wl.name}-{args.layers}L")

    if args.impl == "reference":
        if rank != 0:
            return 0
        # the oracle on the host cores: each step is one layer of the headline step (bounded sample)
        st = oracle_cell(wl)
        for _ in range(args.warmup):
            oracle_step(wl, st)
        t0 = time.perf_counter()
        nbytes = 0.0
        for _ in range(args.steps):
            nbytes += oracle_step(wl, st)
        dt = time.perf_counter() - t0
        v = nbytes / dt / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": wl.name + " (one of 10 layers per step)", "layers": 1, "batch": 1,
                           "n_q_heads": wl.n_q_heads, "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim,
                           "ctx": wl.lengths[0], "kv": f"{wl.type_k}/{wl.type_v}"},
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
                                 "sample": "one layer of the headline step per step: 1-row quantise + fp64 "
                                           "attention of all query heads"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import quantised_kv_long_gb300 as kvq

    peak, peak_kind = measured_peaks()
    if args.cell:  # one extra cell alone (profiling captures)
        if args.cell.startswith("verify"):
            r = run_verify_cell(kvq, torch, wl, int(args.cell[6:]), args.steps, args.warmup, peak)
        elif args.cell == "window":
            r = run_window_cell(kvq, torch, wl, 4096, args.steps, args.warmup, peak)
        else:
            r = chunk_quantise(kvq, torch, syn.multi_session(), reps=args.steps, warmup=args.warmup)
        if rank == 0:
            print(json.dumps({"cell": args.cell, "result": r}), flush=True)
        return 0
    gpu_id = os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0] if world == 1 else str(local_rank)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.3)

    # headline cell: barrier + synchronize on both sides of the timed region, max over ranks
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    head = run_cell(kvq, torch, wl, args.steps, args.warmup, peak, e2e=True)
    torch.cuda.synchronize()
    ms = head["ms_per_step"]
    if world > 1:
        ms = max_over_ranks(dist, ms, "cuda")
        dist.barrier()
    wall0, wall1 = head.pop("_wall")
    clocks = sampler.summary(wall0, wall1)

    sweep = [dict(head)]
    if args.cells == "default":
        for w in sweep_workloads("default")[1:]:
            r = run_cell(kvq, torch, w, args.sweep_steps, max(3, min(args.warmup, 5)), peak)
            r.pop("_wall")
            if r["kv_bytes_per_step"] <= 4 * L2_BYTES:
                r["rotating"] = run_rotating(kvq, torch, w, max(args.sweep_steps, 24), 6, peak)
            sweep.append(r)
        sweep.append(run_window_cell(kvq, torch, syn.hybrid(65536, "q8_0", "q8_0"), 4096, args.sweep_steps,
                                     max(3, min(args.warmup, 5)), peak))
        sweep.append(run_window_cell(kvq, torch, syn.dense14b(131072, "q8_0", "q4_0"), 4096, args.sweep_steps,
                                     max(3, min(args.warmup, 5)), peak))
        for n_q in (4, 16):
            sweep.append(run_verify_cell(kvq, torch, syn.hybrid(65536, "q8_0", "q8_0"), n_q, args.sweep_steps,
                                         max(3, min(args.warmup, 5)), peak))
        sweep.append(run_verify_cell(kvq, torch, syn.dense14b(131072, "q8_0", "q4_0"), 4, args.sweep_steps,
                                     max(3, min(args.warmup, 5)), peak))
        chunk = chunk_quantise(kvq, torch, syn.multi_session())
    else:
        chunk = None
    sampler.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    if rank != 0:
        return 0
    value = job_value(world, step_kv_bytes(wl, [wl.lengths[0]]), ms) if world > 1 else head["kv_gbs"]
    bpl = head["kv_bytes_per_step"] / wl.layers  # algorithmic bytes per launch (mean length)
    achieved = bpl / (head["decode_instep_us"] * 1e-6) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": traffic_from_profiles(wl),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, burst copy)" if peak_kind == "measured"
            else "fallback 6800 GB/s",
            "kernel": "decode_kernel, fused-append mode (1-row quantise-append + split-K decode + split merge)",
            "bytes_per_launch": bpl,
            "per_unit": f"{row_bytes(wl):.0f} B per (position, layer): Hkv*D*(bpv_K+bpv_V)",
            "launch_us": head["decode_instep_us"],
            "timing": "CUDA events over the timed region of event-free graph replays on the launching stream; "
                      "the region holds only decode_kernel launches (one per layer), so region time / launches "
                      "is the kernel's average in-step launch duration",
            "serialised_events": {"launch_us": head.get("decode_us"), "achieved": head.get("decode_gbs"),
                                  "frac": head["decode_gbs"] / peak if head.get("decode_gbs") else None,
                                  "how": "CUDA events around every launch (event nodes serialise the launches)"},
            "stamps": head.get("stamps")}
    if head.get("stamps") and head["stamps"]["span_us_mean"] > 0:  # 0: the kernel wrote no stamps
        sp = head["stamps"]["span_us_mean"]
        roof["stamps"]["span_achieved"] = bpl / (sp * 1e-6) / 1e9
        roof["stamps"]["span_frac"] = roof["stamps"]["span_achieved"] / peak
    e2e = head.pop("e2e")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 mma / fp32 accumulate over q8_0 codes", "data": "synthetic",
        "config": {"workload": wl.name, "layers": wl.layers, "batch": wl.batch, "n_q_heads": wl.n_q_heads,
                   "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim, "ctx": wl.lengths[0],
                   "kv": f"{wl.type_k}/{wl.type_v}", "steps_per_s": head["steps_per_s"],
                   "pct_hbm_peak": head["pct_hbm_peak"], "splits": head["splits"],
                   "l2": "inputs larger than L2 (KV per step >> 129 MB), no flush",
                   "step": "per layer: one kernel = 1-row quantise-append + split-K decode + split merge; "
                           "the layers of a step form one CUDA graph",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": wl.layers * args.steps, "clocks": clocks,
        "sweep": sweep, "chunk_quantise": chunk,
    }
    # the per-cell table once more, compact and last (a reader of only the line's tail sees it)
    cells = compact_cells(sweep, chunk)
    line["config"]["cells"] = cells
    line["cells"] = cells
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
