"""Benchmark: the verify window's grouped routed-expert decode, 48 layers in one CUDA graph.

Workload (the decode-window configuration): 48 layers, each with its own 128 experts, top-8
routing, n_embd 2560, n_ff 768, CB3 gate/up and NL4 down weights (16.4 GB resident pool, seeded
synthetic bytes), window sizes T = 1, 2, 3, 4. Per layer the graph runs the whole hot path:
routing/grouping, activation q8_1, grouped gate/up, fused SwiGLU + q8_1, grouped down, chained
with programmatic dependent launch; every kernel waits for the previous layer before reading.

The gate/up pool is held in the CB3X slot layout, transcoded once at load time from the CB3 pool
(the same integers; load-time re-encoding as in #3455 "GP100 (sm_60): 4-bit slots for resident
IQ2_S / IQ3_XXS / IQ3_S gate/up experts"); the native-layout window (CB3 read directly) is timed
too and reported in "native_layout". Bandwidth figures count the CB3 format's bytes (algorithmic
bytes); the slot layout streams 4/3 of that for gate/up.

One step = one launch of each of the four window graphs (T = 1..4). value = mean microseconds
per window over the four T (lower is better); per-T microseconds and weight-stream bandwidth are
in "per_T". Every window reads >= 1 GB of weights, far more than L2 (129 MB), so no flush is
needed between launches.

--impl reference times the CPU oracle instead (bounded sample: one layer per T per step,
scaled to a 48-layer window).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WL = synth.WORKLOADS["window48"]
GU_T, DN_T = WL.pairs[0]
XT = synth.CB3X  # slot layout the gate/up pool is transcoded to at load
TS = (1, 2, 3, 4)
METRIC = "us_per_verify_window_48L"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def routing_for(layer, T):
    return synth.routing(T, WL.k, WL.E, WL.seed * 1000 + layer * 10 + T + 5)


def job_ms(local_ms, world, device):
    """The whole job's time: the slowest rank's (replicas run independent windows; the timed region
    is bracketed by barriers on every rank)."""
    if world <= 1:
        return float(local_ms)
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def us_per_window(total_ms, windows_per_rank, world):
    """Microseconds per window over every rank's windows (the replicas' aggregate throughput)."""
    return total_ms * 1e3 / (windows_per_rank * world)


def acts_for(layer, T):
    return synth.activations(T, WL.N, WL.seed * 1000 + layer * 10 + T, WL.outliers)


def weight_bytes_per_window(T):
    gu_b = synth.blob_bytes(GU_T, 2 * WL.F, WL.N)
    dn_b = synth.blob_bytes(DN_T, WL.N, WL.F)
    groups = [len(np.unique(routing_for(l, T))) for l in range(WL.layers)]
    return sum(groups) * (gu_b + dn_b), sum(groups) * gu_b, groups


# ------------------------------------------------------------------ clocks

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev):
        self.dev = dev
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        self.f.seek(0)
        rows = [l.strip().split(", ") for l in self.f.read().splitlines() if l.strip()]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if len(r) > 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) > 8 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) > 8 for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ our arm

def make_pools(m, dev):
    """The window's resident weights: per layer 128 experts' CB3 gate/up and NL4 down blobs (seeded,
    16.4 GB), the gate/up pool transcoded at load into CB3X slots (12.8 GB), the pointer tables and
    the codebooks."""
    gu_b = synth.blob_bytes(GU_T, 2 * WL.F, WL.N)
    dn_b = synth.blob_bytes(DN_T, WL.N, WL.F)
    pool_gu = torch.empty((WL.layers, WL.E, gu_b), dtype=torch.uint8, device=dev)
    pool_dn = torch.empty((WL.layers, WL.E, dn_b), dtype=torch.uint8, device=dev)
    for l in range(WL.layers):
        pool_gu[l] = synth.weight_blobs(GU_T, 2 * WL.F, WL.N, WL.E, synth.derive_key(WL.seed, l, GU_T, 0), dev)
        pool_dn[l] = synth.weight_blobs(DN_T, WL.N, WL.F, WL.E, synth.derive_key(WL.seed, l, DN_T, 1), dev)
    tab = lambda p, l: torch.tensor([p[l, x].data_ptr() for x in range(WL.E)], dtype=torch.int64, device=dev)
    tab_gu = [tab(pool_gu, l) for l in range(WL.layers)]
    tab_dn = [tab(pool_dn, l) for l in range(WL.layers)]
    cb_gu = torch.from_numpy(synth.codebook(GU_T, WL.seed * 7 + 1).ravel().copy()).to(dev)
    cb_dn = torch.from_numpy(synth.codebook(DN_T, WL.seed * 7 + 2).ravel().copy()).to(dev)
    # load-time transcoding of the gate/up pool into the slot layout
    xb = synth.blob_bytes(XT, 2 * WL.F, WL.N)
    pool_gx = torch.empty((WL.layers, WL.E, xb), dtype=torch.uint8, device=dev)
    tab_gx = [tab(pool_gx, l) for l in range(WL.layers)]
    terr = torch.zeros(1, dtype=torch.int32, device=dev)
    for l in range(WL.layers):
        m.transcode_cb(GU_T, cb_gu, XT, WL.N, 2 * WL.F, tab_gu[l], tab_gx[l], terr)
    torch.cuda.synchronize()
    if int(terr.item()):
        raise RuntimeError(f"transcoding error bits {int(terr.item())}")
    return dict(pool_gu=pool_gu, pool_dn=pool_dn, pool_gx=pool_gx, tab_gu=tab_gu, tab_dn=tab_dn, tab_gx=tab_gx,
                cb_gu=cb_gu, cb_dn=cb_dn)


class Window:
    """Device state of one T: inputs, routing outputs, scratch and the captured 48-layer graph.

    fused: each layer is one moe_expert_layer launch (routing, q8_1, gate/up, SwiGLU + q8_1, down);
    otherwise each layer is moe_route_group + moe_quantize_q8_1 + moe_expert_grouped (5 launches),
    or, with grouped_fused, moe_route_group + moe_quantize_q8_1 + moe_expert_grouped_fused (3)."""

    def __init__(self, m, T, tab_gu, tab_dn, cb_gu, cb_dn, dev, gu_type=GU_T, fused=True, grouped_fused=False):
        self.T = T
        self.fused = fused
        self.grouped_fused = grouped_fused
        L, n = WL.layers, T * WL.k
        i32 = dict(dtype=torch.int32, device=dev)
        self.ids_h = torch.from_numpy(np.stack([routing_for(l, T) for l in range(L)])).pin_memory()
        self.x_h = torch.from_numpy(np.stack([acts_for(l, T) for l in range(L)])).pin_memory()
        self.out_h = torch.empty((L, n, WL.N), dtype=torch.float32).pin_memory()
        self.ids = self.ids_h.to(dev)
        self.x = self.x_h.to(dev)
        self.ge = torch.zeros((L, n), **i32)
        self.gs = torch.zeros((L, n + 1), **i32)
        self.ng = torch.zeros((L, 1), **i32)
        self.es = torch.zeros((L, n), **i32)
        self.ed = torch.zeros((L, n), **i32)
        self.xq = torch.zeros((L, T, WL.N // 32, 36), dtype=torch.uint8, device=dev)
        self.gu = torch.zeros((n, 2 * WL.F), dtype=torch.float32, device=dev)
        self.hq = torch.zeros((n, WL.F // 32, 36), dtype=torch.uint8, device=dev)
        self.out = torch.zeros((L, n, WL.N), dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, **i32)
        self.gu_type = gu_type
        self.calls = [m.ExpertCall(gu_type, cb_gu, DN_T, cb_dn, WL.N, WL.F, tab_gu[l], tab_dn[l], WL.E, self.ge[l],
                                   self.gs[l], self.ng[l], n, 0, n, self.xq[l], self.es[l], self.ed[l], self.gu,
                                   self.hq, self.out[l], self.err, m.F_PDL) for l in range(L)]
        # a pair of counter halves: layer l uses half l % 2 and zeroes the other (48 layers: the
        # halves alternate across graph replays too)
        self.sync = torch.zeros(2 * m.layer_sync_ints(T, WL.k, WL.F), **i32)
        if grouped_fused:  # one-launch expert calls on alternate halves of their own sync pair
            self.gsync = torch.zeros(2 * m.grouped_fused_sync_ints(n, n, WL.F), **i32)
            for l, c in enumerate(self.calls):
                c.c.flags = m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if l % 2 else 0)
        self.lcalls = [m.LayerCall(gu_type, cb_gu, DN_T, cb_dn, WL.N, WL.F, tab_gu[l], tab_dn[l], WL.E, self.ids[l],
                                   self.x[l], self.out[l], self.gu, self.hq, self.sync, self.err,
                                   m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if l % 2 else 0))
                       for l in range(L)]
        self.m = m
        self.graph = None

    def run_layers(self, stream=None):
        m = self.m
        if self.fused:
            for l in range(WL.layers):
                self.lcalls[l](stream)
            return
        for l in range(WL.layers):
            m.route_group(self.ids[l], WL.E, 0, self.ge[l], self.gs[l], self.ng[l], self.es[l], self.ed[l],
                          self.err, stream=stream)
            m.quantize_q8_1(self.x[l], self.xq[l], stream=stream)
            if self.grouped_fused:
                self.calls[l].call_fused(self.gsync, stream)
            else:
                self.calls[l](stream)

    def capture(self):
        self.run_layers()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            self.run_layers()
        self.graph = g
        return g


def launches_per_window(fused=True):
    return WL.layers * (1 if fused else 5)  # one fused launch, or route, quantize, gate/up, SwiGLU+q8_1, down


def run_ours(args, rank, world):
    import quantized_routed_expert_grouped_gb300 as m
    from quantized_routed_expert_grouped_gb300 import build as cuda_build

    cuda_build.build()
    m.lib()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    hbm_peak, peak_kind = peaks()
    t0 = time.time()
    P = make_pools(m, dev)
    tab_gu, tab_dn, tab_gx, cb_gu, cb_dn = P["tab_gu"], P["tab_dn"], P["tab_gx"], P["cb_gu"], P["cb_dn"]
    setup_s = time.time() - t0

    # headline: fused layer launches on the slot layout; compared: the separate-kernel window on the
    # same layout, and the fused window reading CB3 directly
    wins = {T: Window(m, T, tab_gx, tab_dn, None, cb_dn, dev, gu_type=XT) for T in TS}
    sepv = {T: Window(m, T, tab_gx, tab_dn, None, cb_dn, dev, gu_type=XT, fused=False) for T in TS}
    gfv = {T: Window(m, T, tab_gx, tab_dn, None, cb_dn, dev, gu_type=XT, fused=False, grouped_fused=True) for T in TS}
    natv = {T: Window(m, T, tab_gu, tab_dn, cb_gu, cb_dn, dev) for T in TS}
    every = list(wins.values()) + list(sepv.values()) + list(gfv.values()) + list(natv.values())
    for w in every:
        w.capture()
    torch.cuda.synchronize()
    for w in every:
        if int(w.err.item()):
            raise RuntimeError(f"device error bits {int(w.err.item())}")
    for T in TS:  # the fused window reproduces the separate kernels bit for bit
        if not torch.equal(wins[T].out.view(torch.int32), sepv[T].out.view(torch.int32)):
            raise RuntimeError(f"fused and separate windows differ at T={T}")
        if not torch.equal(gfv[T].out.view(torch.int32), sepv[T].out.view(torch.int32)):
            raise RuntimeError(f"one-launch and three-launch expert calls differ at T={T}")

    s = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        for T in TS:
            wins[T].graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    # ---- timed region: K steps, each the four window graphs; per-T events
    per_t = {T: [] for T in TS}
    clocks = Clocks(dev.index)
    clocks.start()
    t_start, t_end = ev(), ev()
    torch.cuda.synchronize()
    t_start.record(s)
    for _ in range(args.steps):
        for T in TS:
            a, b = ev(), ev()
            a.record(s)
            wins[T].graph.replay()
            b.record(s)
            per_t[T].append((a, b))
    t_end.record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = job_ms(total_ms, world, dev)
    us_t = {T: float(np.median([a.elapsed_time(b) * 1e3 for a, b in per_t[T]])) for T in TS}
    value = us_per_window(total_ms, args.steps * len(TS), world)
    bytes_t = {T: weight_bytes_per_window(T) for T in TS}
    per_T = {str(T): {"us": round(us_t[T], 2), "weight_bytes": bytes_t[T][0],
                      "GBps": round(bytes_t[T][0] / (us_t[T] * 1e-6) / 1e9, 1),
                      "frac_of_measured_hbm": round(bytes_t[T][0] / (us_t[T] * 1e-6) / 1e9 / hbm_peak, 4),
                      "groups_per_layer": round(float(np.mean(bytes_t[T][2])), 2)} for T in TS}

    # ---- the comparison windows, timed the same way after the headline run
    def time_windows(ws):
        ts = {T: [] for T in TS}
        for _ in range(args.warmup):
            for T in TS:
                ws[T].graph.replay()
        for _ in range(args.steps):
            for T in TS:
                a, b = ev(), ev()
                a.record(s)
                ws[T].graph.replay()
                b.record(s)
                ts[T].append((a, b))
        torch.cuda.synchronize()
        res = {}
        for T in TS:
            us = float(np.median([a.elapsed_time(b) * 1e3 for a, b in ts[T]]))
            res[str(T)] = {"us": round(us, 2), "GBps": round(bytes_t[T][0] / (us * 1e-6) / 1e9, 1),
                           "frac_of_measured_hbm": round(bytes_t[T][0] / (us * 1e-6) / 1e9 / hbm_peak, 4)}
        return res

    separate = time_windows(sepv)
    grouped_fused = time_windows(gfv)
    native = time_windows(natv)

    # ---- dominant kernel: the fused layer kernel (T = 4 window: 48 launches per graph)
    roof = layer_roofline(wins[4], bytes_t[4], hbm_peak, peak_kind, s)
    breakdown = {f"T{T}": step_breakdown(m, sepv[T], s) for T in (1, 4)}

    # ---- end to end: pinned host inputs -> device, the window graphs, outputs -> host
    e2e = end_to_end(wins, args, s, world, dev)
    sparse = sparse_calls(m, dev)
    sweep = call_sweep(m, dev, hbm_peak)
    qsa = qsa_sweep(m, dev)

    launches = args.steps * len(TS) * launches_per_window(True)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "us/window", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8 dp4a + fp32", "data": "synthetic",
        "config": {"workload": "window48: 48 layers x 128 experts, top-8, n_embd 2560, n_ff 768, CB3 gate/up + "
                               "NL4 down (16.4 GB pool), T=1..4, one CUDA graph per T",
                   "layout": "gate/up held as CB3X slots (CB3 transcoded at load, same integers); down NL4",
                   "launch": "one fused launch per layer (routing, q8_1, gate/up, SwiGLU + q8_1, down), PDL-chained, "
                  "alternate counter halves",
                   "l2": "inputs larger than L2 (>= 1 GB of weights per window), no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "per_T": per_T,
        "separate_kernels": {"launch": "route + quantize + gate/up + SwiGLU/q8_1 + down per layer", "per_T": separate},
        "grouped_fused_call": {"launch": "route + quantize + moe_expert_grouped_fused (one launch) per layer",
                               "per_T": grouped_fused},
        "native_layout": {"gate_up": "CB3 (read directly), fused launches", "per_T": native},
        "roofline": roof, "step_us_per_layer_alone": breakdown, "second_call_cost": sparse, "calls": sweep, "qsa_block_scores": qsa, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
        "setup_s": round(setup_s, 1),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(sample_layers=args.cpu_layers)
    return line


# DRAM read + write bytes of one fused layer launch at T = 4 (layer 0, 29 groups), from an ncu
# capture of `bench.py --case --case-fused --case-slot` (stored here, not measured by this run);
# reported only while the kernel sources hash to the ones the capture was taken on (else null:
# the counters are stale).
LAYER_TRAFFIC_T4 = {"bytes": 95_313_408, "sources": ("layer.cuh", "gemv.cuh", "common.cuh", "q8_1.cuh", "route.cuh"),
                    "sha1": "28d94235ab10bf903c617c6a3d048e449e099dcd"}


def layer_traffic():
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "quantized_routed_expert_grouped_gb300", "csrc")
    for f in LAYER_TRAFFIC_T4["sources"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return LAYER_TRAFFIC_T4["bytes"] if h.hexdigest() == LAYER_TRAFFIC_T4["sha1"] else None


def sparse_calls(m, dev, reps=20):
    """Per-call cost of the second (PCIe) call of a layer on the sparse workload's geometry (64
    experts, top-8, T = 4, n_embd 2560, n_ff 768, CB2 gate/up, NL4 down): a CUDA graph of 48
    moe_expert_grouped calls (gate/up, SwiGLU + q8_1, down chained with PDL), each with a
    device-side n_groups of 0 (empty) or 1 (one group of 2 entries numbered after the first call's
    32, scattered destinations, its own expert from a 558 MB pool read cold), with grid_groups 0
    (the capacity) and 1; then ("fused") the same calls as one moe_expert_grouped_fused launch
    each, and the residency split: each call's expert copied from pinned host memory into a device
    staging slot (moe_stage_blobs) before its call, copies and calls in one graph; and both one-group
    forms again with the gate/up blobs as CB2X slots (transcoded at load, the same integers).
    Microseconds per call from CUDA events around graph replays."""
    wl = synth.WORKLOADS["sparse"]
    gu_t, dn_t = wl.pairs[0]
    E, calls, n = 256, 48, 4 * wl.k
    cap_e = n + 2
    pool_gu = synth.weight_blobs(gu_t, 2 * wl.F, wl.N, E, synth.derive_key(wl.seed, 0, gu_t, 0), dev)
    pool_dn = synth.weight_blobs(dn_t, wl.N, wl.F, E, synth.derive_key(wl.seed, 0, dn_t, 1), dev)
    tab = lambda p: torch.tensor([p[x].data_ptr() for x in range(E)], dtype=torch.int64, device=dev)
    tab_gu, tab_dn = tab(pool_gu), tab(pool_dn)
    cb_gu = torch.from_numpy(synth.codebook(gu_t, wl.seed * 7 + 1).ravel().copy()).to(dev)
    cb_dn = torch.from_numpy(synth.codebook(dn_t, wl.seed * 7 + 2).ravel().copy()).to(dev)
    i32 = dict(dtype=torch.int32, device=dev)
    xq = m.quantize_q8_1(torch.from_numpy(synth.activations(4, wl.N, wl.seed, 0.0)).to(dev))
    gs = torch.tensor([n, n + 2] + [0] * (n - 1), **i32)
    es = torch.full((cap_e,), -7, **i32)
    ed = torch.full((cap_e,), -7, **i32)
    es[n:n + 2] = torch.tensor([3, 1], **i32)
    ed[n:n + 2] = torch.tensor([n + 4, 2], **i32)
    gu = torch.zeros((cap_e, 2 * wl.F), dtype=torch.float32, device=dev)
    hq = torch.zeros((cap_e, wl.F // 32, 36), dtype=torch.uint8, device=dev)
    out = torch.zeros((n + 6, wl.N), dtype=torch.float32, device=dev)
    err = torch.zeros(1, **i32)
    res = {}
    for ng, gg in ((0, 0), (1, 0), (0, 1), (1, 1)):
        ngt = torch.full((1,), ng, **i32)
        ges = [torch.tensor([(5 * c) % E] + [0] * (n - 1), **i32) for c in range(calls)]
        cs = [m.ExpertCall(gu_t, cb_gu, dn_t, cb_dn, wl.N, wl.F, tab_gu, tab_dn, E, ges[c], gs, ngt, n, gg, cap_e, xq,
                           es, ed, gu, hq, out, err, m.F_PDL) for c in range(calls)]
        for c in cs:
            c()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for c in cs:
                c()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        if int(err.item()):
            raise RuntimeError(f"sparse calls: device error bits {int(err.item())}")
        key = ("empty" if ng == 0 else "one_group_2_entries") + ("_grid_groups_1" if gg else "")
        res[key] = round(a.elapsed_time(b) * 1e3 / (reps * calls), 2)
    res.update({"unit": "us/call", "calls_per_graph": calls, "launches_per_call": 3})

    def graph_us(run):
        run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            run()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        if int(err.item()):
            raise RuntimeError(f"sparse calls: device error bits {int(err.item())}")
        return round(a.elapsed_time(b) * 1e3 / (reps * calls), 2)

    # the same calls in one fused launch each (moe_expert_grouped_fused, alternate sync halves)
    sync = torch.zeros(2 * m.grouped_fused_sync_ints(n, cap_e, wl.F), **i32)
    fused = {}
    for ng in (0, 1):
        ngt = torch.full((1,), ng, **i32)
        ges = [torch.tensor([(5 * c) % E] + [0] * (n - 1), **i32) for c in range(calls)]
        cs = [m.ExpertCall(gu_t, cb_gu, dn_t, cb_dn, wl.N, wl.F, tab_gu, tab_dn, E, ges[c], gs, ngt, n, 0, cap_e, xq,
                           es, ed, gu, hq, out, err, m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if c % 2 else 0))
              for c in range(calls)]
        fused["empty" if ng == 0 else "one_group_2_entries"] = graph_us(lambda: [c.call_fused(sync) for c in cs])
    # the residency split: each call's expert is host-resident (pinned), copied into a device
    # staging slot (moe_stage_blobs: the copy kernel for these pinned blobs) before its one-launch
    # call, all in the graph
    host_gu = [synth.weight_blobs(gu_t, 2 * wl.F, wl.N, 1, synth.derive_key(wl.seed, 0, gu_t, 0), "cpu",
                                  first_blob=(7 * c) % E)[0].pin_memory() for c in range(calls)]
    host_dn = [synth.weight_blobs(dn_t, wl.N, wl.F, 1, synth.derive_key(wl.seed, 0, dn_t, 1), "cpu",
                                  first_blob=(7 * c) % E)[0].pin_memory() for c in range(calls)]
    slot_gu = torch.empty(host_gu[0].numel(), dtype=torch.uint8, device=dev)
    slot_dn = torch.empty(host_dn[0].numel(), dtype=torch.uint8, device=dev)
    stab_gu = torch.full((E,), slot_gu.data_ptr(), dtype=torch.int64, device=dev)
    stab_dn = torch.full((E,), slot_dn.data_ptr(), dtype=torch.int64, device=dev)
    ngt = torch.ones(1, **i32)
    ges = [torch.tensor([(7 * c) % E] + [0] * (n - 1), **i32) for c in range(calls)]
    cs = [m.ExpertCall(gu_t, cb_gu, dn_t, cb_dn, wl.N, wl.F, stab_gu, stab_dn, E, ges[c], gs, ngt, n, 0, cap_e, xq,
                       es, ed, gu, hq, out, err, m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if c % 2 else 0))
          for c in range(calls)]

    def staged():
        for c in range(calls):
            m.stage_blobs([host_gu[c], host_dn[c]], [slot_gu, slot_dn])
            cs[c].call_fused(sync)
    fused["host_staged_one_group_2_entries"] = graph_us(staged)
    fused["host_staged_bytes_per_call"] = int(host_gu[0].numel() + host_dn[0].numel())
    # the same one-group calls on CB2X slots (the gate/up blobs transcoded at load time, the same
    # integers): device-resident, and staged from host memory (host blobs transcoded once, untimed)
    xb = synth.blob_bytes(synth.CB2X, 2 * wl.F, wl.N)
    terr = torch.zeros(1, **i32)
    pool_gx = torch.empty((E, xb), dtype=torch.uint8, device=dev)
    m.transcode_cb(gu_t, cb_gu, synth.CB2X, wl.N, 2 * wl.F, tab_gu, tab(pool_gx), terr)
    tab_gx = tab(pool_gx)
    ges5 = [torch.tensor([(5 * c) % E] + [0] * (n - 1), **i32) for c in range(calls)]
    cx = [m.ExpertCall(synth.CB2X, None, dn_t, cb_dn, wl.N, wl.F, tab_gx, tab_dn, E, ges5[c], gs, ngt, n, 0, cap_e,
                       xq, es, ed, gu, hq, out, err, m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if c % 2 else 0))
          for c in range(calls)]
    fused["one_group_2_entries_cb2x_slots"] = graph_us(lambda: [c.call_fused(sync) for c in cx])
    one = lambda t: torch.tensor([t.data_ptr()], dtype=torch.int64, device=dev)
    host_gx = []
    for c in range(calls):
        src, dst = host_gu[c].to(dev), torch.empty(xb, dtype=torch.uint8, device=dev)
        m.transcode_cb(gu_t, cb_gu, synth.CB2X, wl.N, 2 * wl.F, one(src), one(dst), terr)
        host_gx.append(dst.cpu().pin_memory())
    torch.cuda.synchronize()
    if int(terr.item()):
        raise RuntimeError(f"sparse calls: transcoder error bits {int(terr.item())}")
    slot_gx = torch.empty(xb, dtype=torch.uint8, device=dev)
    stab_gx = torch.full((E,), slot_gx.data_ptr(), dtype=torch.int64, device=dev)
    csx = [m.ExpertCall(synth.CB2X, None, dn_t, cb_dn, wl.N, wl.F, stab_gx, stab_dn, E, ges[c], gs, ngt, n, 0, cap_e,
                        xq, es, ed, gu, hq, out, err, m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if c % 2 else 0))
           for c in range(calls)]

    def staged_x():
        for c in range(calls):
            m.stage_blobs([host_gx[c], host_dn[c]], [slot_gx, slot_dn])
            csx[c].call_fused(sync)
    fused["host_staged_one_group_2_entries_cb2x_slots"] = graph_us(staged_x)
    fused["host_staged_bytes_per_call_cb2x_slots"] = int(host_gx[0].numel() + host_dn[0].numel())
    fused.update({"unit": "us/call", "calls_per_graph": calls, "launches_per_call": 1})
    res["fused"] = fused
    return res


def _routings(wl, calls, seed):
    return [synth.routing(wl.T[0], wl.k, wl.E, seed * 1000 + c) for c in range(calls)]


def _layer_graph(m, lcalls, reps):
    """Microseconds per call of a CUDA graph of the given fused layer calls (PDL-chained,
    alternating the halves of one counter pair), replayed `reps` times."""
    for c in lcalls:
        c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for c in lcalls:
            c()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (reps * len(lcalls))


def call_sweep(m, dev, hbm_peak, reps=10, calls=16):
    """One fused layer call (moe_expert_layer) per routing, timed in a CUDA graph of `calls`
    calls with distinct seeded routings, on
      - the verify workload (T = 4, 64 experts, top-8, n_embd 2560, n_ff 768, CB2 gate/up read
        directly and as CB2X slots, NL4 down): the 139.6 MB pool replicated 8 times (1.1 GB), call
        c on replica c % 8, so every call reads cold;
      - the format sweep (T = 4, 256 experts, top-8, n_embd 4096, n_ff 1536, activations with 1 %
        outliers x20): each of the 8 (gate/up, down) pairs on its own 256-expert pool (1.8-5.1 GB).
    Per case: microseconds per call, the algorithmic weight bytes of the calls' groups (gate/up +
    down blobs of their experts, as stored), GB/s and the fraction of the measured HBM peak."""
    out = {}
    i32 = dict(dtype=torch.int32, device=dev)

    def run(wl, gu_t, dn_t, pools, cb_gu, cb_dn, algo_gu_t, tag):
        n = wl.T[0] * wl.k
        ids = _routings(wl, calls, wl.seed + 7)
        x = [torch.from_numpy(synth.activations(wl.T[0], wl.N, wl.seed * 100 + c, wl.outliers)).to(dev)
             for c in range(calls)]
        idt = [torch.from_numpy(r).to(dev) for r in ids]
        outs = torch.zeros((calls, n, wl.N), dtype=torch.float32, device=dev)
        gu = torch.zeros((n, 2 * wl.F), dtype=torch.float32, device=dev)
        hq = torch.zeros((n, wl.F // 32, 36), dtype=torch.uint8, device=dev)
        sync = torch.zeros(2 * m.layer_sync_ints(wl.T[0], wl.k, wl.F), **i32)
        err = torch.zeros(1, **i32)
        lc = []
        for c in range(calls):
            tg, td = pools[c % len(pools)]
            lc.append(m.LayerCall(gu_t, cb_gu, dn_t, cb_dn, wl.N, wl.F, tg, td, wl.E, idt[c], x[c], outs[c], gu, hq,
                                  sync, err, m.F_PDL | m.F_SYNC_PAIR | (m.F_SYNC_ODD if c % 2 else 0)))
        us = _layer_graph(m, lc, reps)
        if int(err.item()):
            raise RuntimeError(f"{tag}: device error bits {int(err.item())}")
        per_expert = synth.blob_bytes(algo_gu_t, 2 * wl.F, wl.N) + synth.blob_bytes(dn_t, wl.N, wl.F)
        groups = float(np.mean([len(np.unique(r)) for r in ids]))
        by = groups * per_expert
        out[tag] = {"us": round(us, 2), "groups": round(groups, 2), "weight_bytes": int(by),
                    "GBps": round(by / (us * 1e-6) / 1e9, 1), "frac_of_measured_hbm": round(by / (us * 1e-6) / 1e9 / hbm_peak, 4)}

    def tables(pool):
        return torch.tensor([pool[x].data_ptr() for x in range(pool.shape[0])], dtype=torch.int64, device=dev)

    # ---- the verify call (CB2 / NL4), 8 replicas of its pool
    wl = synth.WORKLOADS["verify"]
    gu_t, dn_t = wl.pairs[0]
    cb_gu = torch.from_numpy(synth.codebook(gu_t, wl.seed * 7 + 1).ravel().copy()).to(dev)
    cb_dn = torch.from_numpy(synth.codebook(dn_t, wl.seed * 7 + 2).ravel().copy()).to(dev)
    reps8 = []
    for r in range(8):
        pg = synth.weight_blobs(gu_t, 2 * wl.F, wl.N, wl.E, synth.derive_key(wl.seed, r, gu_t, 0), dev)
        pd = synth.weight_blobs(dn_t, wl.N, wl.F, wl.E, synth.derive_key(wl.seed, r, dn_t, 1), dev)
        reps8.append((pg, pd))
    run(wl, gu_t, dn_t, [(tables(pg), tables(pd)) for pg, pd in reps8], cb_gu, cb_dn, gu_t, "verify_CB2_NL4")
    xs = []
    terr = torch.zeros(1, **i32)
    for pg, pd in reps8:
        px = torch.empty((wl.E, synth.blob_bytes(synth.CB2X, 2 * wl.F, wl.N)), dtype=torch.uint8, device=dev)
        m.transcode_cb(gu_t, cb_gu, synth.CB2X, wl.N, 2 * wl.F, tables(pg), tables(px), terr)
        xs.append((px, pd))
    torch.cuda.synchronize()
    run(wl, synth.CB2X, dn_t, [(tables(px), tables(pd)) for px, pd in xs], None, cb_dn, gu_t,
        "verify_CB2X_slots_NL4")
    del reps8, xs
    # ---- the format sweep: 8 pairs
    wl = synth.WORKLOADS["sweep"]
    for gu_t, dn_t in wl.pairs:
        pg = synth.weight_blobs(gu_t, 2 * wl.F, wl.N, wl.E, synth.derive_key(wl.seed, 0, gu_t, 0), dev)
        pd = synth.weight_blobs(dn_t, wl.N, wl.F, wl.E, synth.derive_key(wl.seed, 0, dn_t, 1), dev)
        cg = synth.codebook(gu_t, wl.seed * 7 + 1)
        cd = synth.codebook(dn_t, wl.seed * 7 + 2)
        cg = None if cg is None else torch.from_numpy(np.ascontiguousarray(cg).ravel()).to(dev)
        cd = None if cd is None else torch.from_numpy(np.ascontiguousarray(cd).ravel()).to(dev)
        run(wl, gu_t, dn_t, [(tables(pg), tables(pd))], cg, cd, gu_t,
            f"sweep_{synth.NAMES[gu_t]}_{synth.NAMES[dn_t]}")
        del pg, pd
    torch.cuda.empty_cache()
    out["method"] = (f"CUDA graph of {calls} fused layer calls (distinct seeded routings, PDL-chained), replayed "
                     f"{reps} times; bytes = the groups' gate/up + down blobs as stored")
    return out


def qsa_sweep(m, dev, reps=10, calls=32):
    """QSA decode block scores (moe_qsa_block_scores) at the page's 131k context (32,769 blocks)
    and at 1M tokens (262,145 blocks), T = 1..4: a CUDA graph of `calls` calls over rotating key
    pools (264-275 MB in all, more than L2), microseconds per call and the key + scale bytes it
    reads per microsecond."""
    out = {}
    for ctx, nb in synth.QSA_CONTEXTS.items():
        npool = 8 if nb > 100000 else 64
        pools = [synth.qsa_keys(nb, 500 + i, device=dev) for i in range(npool)]
        for T in (1, 2, 3, 4):
            q = torch.from_numpy(synth.qsa_queries(T, 9)).to(dev)
            sc = torch.empty((T, nb), dtype=torch.float32, device=dev)
            fs = [lambda i=i: m.qsa_block_scores(q, pools[i % npool][0], pools[i % npool][1], sc) for i in range(calls)]
            for f in fs:
                f()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="relaxed"):
                for f in fs:
                    f()
            g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(b) * 1e3 / (reps * calls)
            out[f"{ctx}_T{T}"] = {"us": round(us, 2), "GBps": round(nb * 132 / (us * 1e-6) / 1e9, 1)}
        del pools
    out["method"] = f"CUDA graph of {calls} calls over rotating int8 key pools, replayed {reps} times"
    return out


def layer_roofline(w, bytes_t, hbm_peak, peak_kind, s, reps=10):
    """The fused layer kernel: the T = 4 window graph (48 launches, one per layer) replayed with
    CUDA events on the launching stream; duration per launch = graph time / 48 (consecutive
    launches overlap slightly under PDL). Algorithmic bytes per launch = the CB3 + NL4 blob bytes
    of the layer's groups, averaged over the 48 layers."""
    w.graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(reps):
        w.graph.replay()
    b.record(s)
    torch.cuda.synchronize()
    dur_s = a.elapsed_time(b) * 1e-3 / (reps * WL.layers)
    per_launch = bytes_t[0] / WL.layers
    ach = per_launch / dur_s / 1e9
    streamed = per_launch + bytes_t[1] / WL.layers * (
        synth.blob_bytes(w.gu_type, 2 * WL.F, WL.N) / synth.blob_bytes(GU_T, 2 * WL.F, WL.N) - 1)
    return {"kernel": f"fused layer kernel ({synth.NAMES[w.gu_type]} gate/up slots of CB3, NL4 down, T=4)",
            "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s",
            "frac": round(ach / hbm_peak, 4), "traffic": layer_traffic(),
            "traffic_source": "stored ncu capture of one T=4 launch (dram read + write bytes), null once the "
                              "kernel sources differ from the captured ones", "peak_kind": peak_kind,
            "bytes_per_launch": int(per_launch), "streamed_bytes_per_launch": int(streamed),
            "streamed_GBps": round(streamed / dur_s / 1e9, 1), "us_per_launch": round(dur_s * 1e6, 2)}


def step_breakdown(m, w, s, reps=5):
    """Each step of the window alone: a CUDA graph of that step's 48 launches (no PDL), replayed
    with CUDA events on the launching stream: GPU microseconds per launch. The per-layer sum
    exceeds the window time / 48 because the window graph chains kernels with programmatic
    dependent launch."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    n = w.T * WL.k
    s = None  # launch on the current stream (the capture stream inside torch.cuda.graph)
    steps = {
        "route": lambda l: m.route_group(w.ids[l], WL.E, 0, w.ge[l], w.gs[l], w.ng[l], w.es[l], w.ed[l], w.err,
                                         stream=s),
        "quantize": lambda l: m.quantize_q8_1(w.x[l], w.xq[l], stream=s),
        "gate_up": lambda l: m.grouped_gu(w.gu_type, w.calls[l]._keep[0], WL.N, WL.F, w.calls[l]._keep[2], WL.E,
                                          w.ge[l], w.gs[l], w.ng[l], n, 0, w.xq[l], w.es[l], n, w.gu, w.err,
                                          stream=s),
        "swiglu_q8_1": lambda l: m.swiglu_q8_1(w.gu, WL.F, w.gs[l], w.ng[l], n, n, w.hq, w.err, stream=s),
        "down": lambda l: m.grouped_down(DN_T, w.calls[l]._keep[1], WL.N, WL.F, w.calls[l]._keep[3], WL.E, w.ge[l],
                                         w.gs[l], w.ng[l], n, 0, w.hq, n, w.ed[l], w.out[l], w.err, stream=s),
    }
    out = {}
    for name, f in steps.items():
        for l in range(WL.layers):
            f(l)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for l in range(WL.layers):
                f(l)
        g.replay()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        a, b = ev(), ev()
        a.record(cur)
        for _ in range(reps):
            g.replay()
        b.record(cur)
        torch.cuda.synchronize()
        out[name] = round(a.elapsed_time(b) * 1e3 / (reps * WL.layers), 2)
    return out


def end_to_end(wins, args, s, world, dev):
    """Every step: each window's inputs (x, ids) copied from pinned host memory, its graph
    replayed, its outputs copied back to pinned host memory, all inside the timed region. Inputs
    and outputs move on two streams of their own, ordered by events per window: the graph waits
    for its inputs and for its previous outputs to have left, the outputs leave once the graph is
    done, and the next inputs land once the graph has read the previous ones. So the copies
    overlap the other windows' compute and no copy touches a buffer still in use."""
    steps = max(2, args.steps // 2)
    h2d = sum(w.x_h.numel() * 4 + w.ids_h.numel() * 4 for w in wins.values())
    d2h = sum(w.out_h.numel() * 4 for w in wins.values())
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {T: {k: torch.cuda.Event() for k in ("in", "done", "out")} for T in wins}
    for e in ev.values():  # recorded once, so the first waits pass
        for x in e.values():
            x.record(s)

    def step():
        for T, w in wins.items():
            e = ev[T]
            s_in.wait_event(e["done"])  # the graph has read the previous inputs
            with torch.cuda.stream(s_in):
                w.x.copy_(w.x_h, non_blocking=True)
                w.ids.copy_(w.ids_h, non_blocking=True)
                e["in"].record(s_in)
            s.wait_event(e["in"])
            s.wait_event(e["out"])  # the previous outputs are out
            with torch.cuda.stream(s):
                w.graph.replay()
                e["done"].record(s)
            s_out.wait_event(e["done"])
            with torch.cuda.stream(s_out):
                w.out_h.copy_(w.out, non_blocking=True)
                e["out"].record(s_out)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for _ in range(steps):
        step()
    s.wait_stream(s_out)  # the last outputs are on the host before the end event
    b.record(s)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    ms = job_ms(ms, world, dev)
    return {"value": round(us_per_window(ms, steps * len(wins), world), 3), "unit": "us/window",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "copies": "input and output streams of their own, overlapping other windows' compute"}


# ------------------------------------------------------------------ CPU oracle

def oracle_inputs(o, layer, T):
    """Layer `layer`'s inputs at T for the oracle: routing, activations, the groups' blobs and the
    codebooks (built outside any timed region)."""
    ids = routing_for(layer, T)
    x = acts_for(layer, T)
    r = o.route_group(ids, WL.E)
    key_gu = synth.derive_key(WL.seed, layer, GU_T, 0)
    key_dn = synth.derive_key(WL.seed, layer, DN_T, 1)
    gub = [np.zeros(1, np.uint8)] * WL.E
    dnb = [np.zeros(1, np.uint8)] * WL.E
    for e in r["grp_expert"]:
        gub[e] = synth.weight_blobs(GU_T, 2 * WL.F, WL.N, 1, key_gu, "cpu", first_blob=int(e))[0].numpy()
        dnb[e] = synth.weight_blobs(DN_T, WL.N, WL.F, 1, key_dn, "cpu", first_blob=int(e))[0].numpy()
    return dict(T=T, ids=ids, x=x, r=r, gub=gub, dnb=dnb, cb_gu=synth.codebook(GU_T, WL.seed * 7 + 1),
                cb_dn=synth.codebook(DN_T, WL.seed * 7 + 2))


def oracle_run(o, inp):
    """Seconds the oracle takes for one layer's path on prepared inputs."""
    T, r = inp["T"], inp["r"]
    G, n = r["n_groups"], T * WL.k
    t0 = time.perf_counter()
    xq = o.quantize_q8_1(inp["x"])
    gu = np.zeros((n, 2 * WL.F))
    o.grouped_gemv(GU_T, WL.N, 2 * WL.F, inp["gub"], r["grp_expert"], r["grp_start"], G, xq, ent_in=r["ent_src"],
                   out=gu, cb=inp["cb_gu"])
    hq = np.zeros((n, WL.F // 32, 36), np.uint8)
    o.swiglu_q8_1(gu.astype(np.float32), WL.F, r["grp_start"][0], r["grp_start"][G], hq)
    out = np.zeros((n, WL.N))
    o.grouped_gemv(DN_T, WL.F, WL.N, inp["dnb"], r["grp_expert"], r["grp_start"], G, hq, ent_out=r["ent_dst"],
                   out=out, cb=inp["cb_dn"])
    o.route_group(inp["ids"], WL.E)
    return time.perf_counter() - t0


def oracle_layer(o, layer, T):
    return oracle_run(o, oracle_inputs(o, layer, T))


def cpu_baseline(sample_layers=1):
    import oracle
    o = oracle.get()
    per_t = {}
    for T in TS:
        secs = [oracle_layer(o, l, T) for l in range(sample_layers)]
        per_t[T] = float(np.mean(secs)) * WL.layers * 1e6
    return {"value": round(float(np.mean(list(per_t.values()))), 1), "unit": "us/window", "cores": 1,
            "kind": "oracle",
            "sample": f"{sample_layers} layer(s) per T=1..4 of the 48-layer window, single-threaded C oracle "
                      f"(fp64 block sums), scaled x48 layers",
            "per_T_us": {str(T): round(v, 1) for T, v in per_t.items()}}


def _reference_worker(w, cores, steps, warmup, bar, q):
    """Worker w of the reference arm: per step, layer (step x cores + w) mod 48 at T = 1..4; the
    inputs are built first, then every worker starts the oracle at the same barrier and reports
    its start and end on the host's monotonic clock (shared by all processes)."""
    import oracle
    torch.set_num_threads(1)
    o = oracle.get()
    for step in range(-warmup, steps):
        layer = (max(step, 0) * cores + w) % WL.layers
        inps = [oracle_inputs(o, layer, T) for T in TS]
        bar.wait(timeout=600)  # a worker that died breaks the barrier instead of stalling the rest
        t0 = time.monotonic()
        for inp in inps:
            oracle_run(o, inp)
        q.put((step, w, t0, time.monotonic()))


def reference_procs(requested=None):
    """Oracle processes of the reference arm: `requested`, else the host's cores capped at 48
    (each process holds a layer's blobs for T = 1..4, about 0.2 GB)."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    return max(1, min(requested or min(cores, 48), cores))


def run_reference(args, rank, world):
    """The oracle as it stands, on the host's cores: one spawned process per core (at most 48, or
    --ref-procs); each step evaluates `procs` consecutive layers (mod 48) at T = 1..4, one layer
    per process, all started together. The step's time is the wall time from the barrier's
    release to the last process's end; us per window = that x 48 / (procs x 4)."""
    if rank != 0:
        return None
    import multiprocessing as mp
    cores = reference_procs(args.ref_procs)
    ctx = mp.get_context("spawn")
    bar, q = ctx.Barrier(cores), ctx.Queue()
    procs = [ctx.Process(target=_reference_worker, args=(w, cores, args.steps, args.warmup, bar, q), daemon=True)
             for w in range(cores)]
    for p in procs:
        p.start()
    res = [q.get(timeout=900) for _ in range(cores * (args.steps + args.warmup))]
    for p in procs:
        p.join(timeout=60)
    walls = [max(t1 for st, _, _, t1 in res if st == step) - min(t0 for st, _, t0, _ in res if st == step)
             for step in range(args.steps)]
    value = float(np.mean(walls)) * WL.layers / (cores * len(TS)) * 1e6
    sample = (f"per step: {cores} consecutive layers (mod 48) at each T=1..4, one per process, started together "
              f"(inputs built untimed); wall time from the start to the last process's end, scaled to 48 layers")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us/window", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(float(np.mean(walls)) * 1e3, 2),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "int32 + fp64",
            "data": "synthetic",
            "config": {"workload": "window48: 48 layers x 128 experts, top-8, n_embd 2560, n_ff 768, CB3 gate/up + "
                                   "NL4 down, T=1..4",
                       "l2": "n/a (CPU)", "parallelism": f"{cores} CPU processes"},
            "cpu_baseline": {"value": round(value, 1), "unit": "us/window", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 1), "unit": "us/window", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_case(args):
    """One layer of the window at T = args.case_t, run eagerly a few times: the small case for
    kernel-level profiling (about 0.4 GB on the device)."""
    import quantized_routed_expert_grouped_gb300 as m
    from quantized_routed_expert_grouped_gb300 import build as cuda_build

    cuda_build.build()
    m.lib()
    dev = torch.device("cuda", 0)
    T = args.case_t
    pool_gu = synth.weight_blobs(GU_T, 2 * WL.F, WL.N, WL.E, synth.derive_key(WL.seed, 0, GU_T, 0), dev)
    pool_dn = synth.weight_blobs(DN_T, WL.N, WL.F, WL.E, synth.derive_key(WL.seed, 0, DN_T, 1), dev)
    tab = lambda p: torch.tensor([p[x].data_ptr() for x in range(WL.E)], dtype=torch.int64, device=dev)
    cb_gu = torch.from_numpy(synth.codebook(GU_T, WL.seed * 7 + 1).ravel().copy()).to(dev)
    cb_dn = torch.from_numpy(synth.codebook(DN_T, WL.seed * 7 + 2).ravel().copy()).to(dev)
    n = T * WL.k
    i32 = dict(dtype=torch.int32, device=dev)
    ids = torch.from_numpy(routing_for(0, T)).to(dev)
    x = torch.from_numpy(acts_for(0, T)).to(dev)
    ge, gs, ng = torch.zeros(n, **i32), torch.zeros(n + 1, **i32), torch.zeros(1, **i32)
    es, ed, err = torch.zeros(n, **i32), torch.zeros(n, **i32), torch.zeros(1, **i32)
    xq = torch.zeros((T, WL.N // 32, 36), dtype=torch.uint8, device=dev)
    gu = torch.zeros((n, 2 * WL.F), dtype=torch.float32, device=dev)
    hq = torch.zeros((n, WL.F // 32, 36), dtype=torch.uint8, device=dev)
    out = torch.zeros((n, WL.N), dtype=torch.float32, device=dev)
    gu_type, cbg, tg = GU_T, cb_gu, tab(pool_gu)
    if args.case_slot:
        pool_gx = torch.empty((WL.E, synth.blob_bytes(XT, 2 * WL.F, WL.N)), dtype=torch.uint8, device=dev)
        tx = tab(pool_gx)
        m.transcode_cb(GU_T, cb_gu, XT, WL.N, 2 * WL.F, tg, tx, err)
        gu_type, cbg, tg = XT, None, tx
    call = m.ExpertCall(gu_type, cbg, DN_T, cb_dn, WL.N, WL.F, tg, tab(pool_dn), WL.E, ge, gs, ng, n, 0, n,
                        xq, es, ed, gu, hq, out, err, m.F_PDL)
    sync = torch.zeros(m.layer_sync_ints(T, WL.k, WL.F), **i32)
    lcall = m.LayerCall(gu_type, cbg, DN_T, cb_dn, WL.N, WL.F, tg, tab(pool_dn), WL.E, ids, x, out, gu, hq, sync,
                        err, m.F_PDL)
    for _ in range(args.steps):
        if args.case_fused:
            lcall()
            continue
        m.route_group(ids, WL.E, 0, ge, gs, ng, es, ed, err)
        m.quantize_q8_1(x, xq)
        call()
    torch.cuda.synchronize()
    extra = {}
    if args.case_aux:
        # the kernels around the path, once per step each on the same layer's shapes: router top-k
        # (T x 128 logits), the weighted combine (T x 8 rows of 2560), the load-time transcoding of
        # the layer's 128 CB3 gate/up blobs to CB3X (200 MB read), QSA block scores at 1M tokens,
        # and the staging copies of the residency split
        logits = torch.from_numpy(np.random.default_rng(3).standard_normal((T, WL.E)).astype(np.float32)).to(dev)
        pool_tx = torch.empty((WL.E, synth.blob_bytes(XT, 2 * WL.F, WL.N)), dtype=torch.uint8, device=dev)
        nb = synth.QSA_CONTEXTS["1M"]
        qk, qs = synth.qsa_keys(nb, 77, device=dev)
        qq = torch.from_numpy(synth.qsa_queries(T, 5)).to(dev)
        # the residency split's staging copies: two experts' CB3X gate/up and NL4 down blobs
        # (6.39 MB) from pinned host memory into device slots
        hbl = [torch.zeros(synth.blob_bytes(t, r, c), dtype=torch.uint8, pin_memory=True)
               for t, r, c in ((XT, 2 * WL.F, WL.N), (DN_T, WL.N, WL.F)) * 2]
        sl = [torch.empty(h.numel(), dtype=torch.uint8, device=dev) for h in hbl]
        for _ in range(args.steps):
            tid, tw = m.router_topk(logits, WL.k)
            y = m.combine(out, tid, tw, WL.E)
            m.transcode_cb(GU_T, cb_gu, XT, WL.N, 2 * WL.F, tab(pool_gu), tab(pool_tx), err)
            sc = m.qsa_block_scores(qq, qk, qs)
            m.stage_blobs(hbl, sl)
        torch.cuda.synchronize()
        extra = {"aux": "router_topk, combine, transcode (CB3 -> CB3X, 128 experts), qsa (1M tokens), "
                        "stage_blobs (2 experts, 6.39 MB from pinned host memory)",
                 "y_finite": bool(torch.isfinite(y).all().item()), "scores": int(sc.numel())}
    print(json.dumps({"case": f"one layer of window48 at T={T}" + (" (fused)" if args.case_fused else ""),
                      "err": int(err.item()),
                      "groups": int(ng.item()), **extra}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", action="store_true", help="run the single-layer profiling case instead")
    ap.add_argument("--case-t", type=int, default=4)
    ap.add_argument("--case-slot", action="store_true", help="profiling case with the gate/up pool in slot layout")
    ap.add_argument("--case-fused", action="store_true", help="profiling case with the fused layer launch")
    ap.add_argument("--case-aux", action="store_true",
                    help="profiling case: also run the router, combine, transcoding, QSA and staging kernels")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-layers", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-procs", type=int, default=0,
                    help="reference arm: oracle processes (default: the host's cores, at most 48)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.case:
        run_case(args)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            torch.distributed.init_process_group("nccl")
        line = run_ours(args, rank, world)
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
