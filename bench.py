#!/usr/bin/env python
"""Benchmark of the compressed-KV hot path on GB300.

Default workload (N=1): Llama-3-8B-shaped decode, 32 layers, batch 16,
32 query / 8 KV heads, d = 128, context 32768 per sequence (32640 compressed
4-bit K / 4-bit V tokens in 64-token pages with a random page permutation,
plus a 128-token fp16 window).  One step = for every layer: append one token
per sequence (tq_append_window: the new token enters the fp16 ring window and
the oldest window token is encoded into the packed pages) and one decode
attention over the whole cache (tq_decode_attn).  The context therefore grows
by one token per step; the metric counts the starting context (the run adds
well under 1 % to it).  The 32 layers' caches
(18.5 GB) are resident in HBM before timing; the working set is far larger
than L2, so no flush is needed between iterations.

Printed JSON line: metric = cached tokens scored per second (B * L * T per
step); plus HBM GB/s of the step, the roofline of the dominant kernel (the
split-KV attention kernel, timed in place with CUDA events), bulk-encode
throughput (32 layers x 8 heads x 65536 tokens, K and V, six formats), the
end-to-end number through the public API with host buffers, the CPU oracle
baseline, clocks and the kernel-launch count.

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import tq_inputs as ti  # noqa: E402

METRIC = "compressed-KV decode attn: cached tokens scored/s & HBM GB/s; encode vecs/s"
UNIT = "tokens/s"


# ------------------------------------------------------------------ utils --
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest x over all ranks (the step time the job is charged with);
    x itself when there is no process group."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job rate of N independent replicas: every rank processes the same
    units, the job takes as long as its slowest rank."""
    return world * units_per_rank / (ms_max * 1e-3)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def nvml_index(cuda_index: int) -> int:
    """nvidia-smi index of a CUDA device (CUDA_VISIBLE_DEVICES may remap)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p for p in vis.split(",") if p.strip()]
    if parts and cuda_index < len(parts) and parts[cuda_index].strip().isdigit():
        return int(parts[cuda_index])
    return cuda_index


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def per_token_head_bytes(fmt) -> dict:
    from decode_attention_tq_gb300 import tq_page_layout

    L = tq_page_layout(fmt)
    k = 4 + L["k_code_bytes"] + (4 + L["k_sign_bytes"] if fmt.k_qjl else 0)
    v = 4 + L["v_code_bytes"]
    return {"k": k, "v": v, "page_bytes": L["page_bytes"]}


# ----------------------------------------------------------- decode bench --
class DecodeBench:
    """A resident multi-layer compressed cache and its decode step."""

    def __init__(self, wl: ti.DecodeWorkload, device: str, spare_tokens: int = 0):
        """`spare_tokens`: compressed positions beyond the context that steps
        may append (their pages are allocated in the block tables)."""
        import decode_attention_tq_gb300 as tq

        self.tq = tq
        self.wl = wl
        f = wl.fmt
        self.fmt = f
        B, Hq, H, d, P, W, T = wl.batch, wl.q_heads, wl.kv_heads, f.head_dim, f.page_size, wl.window, wl.context
        comp = wl.comp_tokens
        self.B, self.Hq, self.H, self.W, self.T, self.comp = B, Hq, H, W, T, comp
        self.pages_per_seq = wl.pages_per_seq + (spare_tokens + P - 1) // P
        self.num_pages = B * self.pages_per_seq + 1
        perm = ti.page_permutation(self.num_pages).to(device)
        self.bt = perm[: B * self.pages_per_seq].reshape(B, self.pages_per_seq).contiguous()
        pos = torch.arange(comp, device=device)
        slots = self.bt[:, pos // P] * P + (pos % P)[None, :]
        self.comp_lens = torch.full((B,), comp, dtype=torch.int32, device=device)
        self.win_lens = torch.full((B,), wl.win_tokens, dtype=torch.int32, device=device)
        self.ks = torch.from_numpy(ti.sign_bits(ti.SEED_SIGNS_K, d)).to(device)
        self.vs = torch.from_numpy(ti.sign_bits(ti.SEED_SIGNS_V, d)).to(device)
        self.kcb = tq.kind_codebook(f, 0, device)
        self.vcb = tq.kind_codebook(f, 1, device)
        self.S = torch.from_numpy(ti.gaussian_matrix(ti.SEED_QJL, f.qjl_m, d)).to(device) if f.k_qjl else None
        page_bytes = tq.tq_page_layout(f)["page_bytes"]
        flat_slots = slots.reshape(-1).to(torch.int32).contiguous()
        self.layers = []
        # per-step inputs and outputs of all layers in three contiguous device
        # buffers (q, the appended K and V token, out), so one copy moves them
        nq, nkv = B * Hq * d, B * H * d  # per layer: [q | new K | new V]
        self.io_in = torch.empty((wl.layers, nq + 2 * nkv), dtype=torch.float16, device=device)
        self.io_out = torch.empty((wl.layers, B * Hq * d), dtype=torch.float32, device=device)
        for layer in range(wl.layers):
            pool = torch.zeros(self.num_pages * page_bytes, dtype=torch.uint8, device=device)
            ent = {"pool": pool}
            for kind, name in ((0, "k"), (1, "v")):
                x = ti.kv_history(B, T, H, d, layer, kind, device=device)
                flat = x[:, :comp].reshape(B * comp, H, d).contiguous()
                tq.tq_encode(f, kind, flat, flat_slots, pool, self.num_pages, self.ks if kind == 0 else self.vs,
                             self.kcb if kind == 0 else self.vcb, self.S if kind == 0 else None)
                del flat
                ent[name + "win"] = x[:, comp:].permute(0, 2, 1, 3).contiguous() if W else None
                new = self.io_in[layer, nq + kind * nkv: nq + (kind + 1) * nkv].view(B, H, d)
                new.copy_(x[:, comp - 1])  # the token each step appends
                ent[name + "new"] = new
                del x
            ent["q"] = self.io_in[layer, :nq].view(B, Hq, d)
            ent["q"].copy_(ti.query(B, Hq, d, device=device, seed=ti.SEED_QUERY + 7919 * layer))
            ent["out"] = self.io_out[layer].view(B, Hq, d)
            # per-layer cache counters, advanced on the device by each append
            ent["comp"] = self.comp_lens.clone()
            ent["wlen"] = self.win_lens.clone() if W else None
            ent["whead"] = torch.zeros(B, dtype=torch.int32, device=device) if W else None
            self.layers.append(ent)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()  # generation temporaries go back to the driver
        self.ws = torch.empty(tq.tq_decode_attn_workspace_size(f, B, Hq, self.pages_per_seq, W), dtype=torch.uint8, device=device)
        self.ws_append = torch.empty(tq.tq_append_window_workspace_size(f, B), dtype=torch.uint8, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        bph = per_token_head_bytes(f)
        self.main_bytes = B * H * comp * (bph["k"] + bph["v"]) + B * self.pages_per_seq * 4  # per layer launch
        self.window_bytes = B * H * wl.win_tokens * d * 2 * 2
        self.step_bytes = wl.layers * (self.main_bytes + self.window_bytes + B * Hq * d * (2 + 4))
        self.launches_per_step = wl.layers * 4  # append (roll + K and V encode), prep (with window chunks), main, merge

    def step(self, events=None, append_only=False):
        tq, f = self.tq, self.fmt
        for i, L in enumerate(self.layers):
            tq.tq_append_window(f, L["knew"], L["vnew"], L["kwin"], L["vwin"], L["wlen"], L["whead"], L["comp"], self.bt, L["pool"],
                                self.num_pages, self.ks, self.vs, self.kcb, self.vcb, self.S, workspace=self.ws_append,
                                err_word=self.err)
            if append_only:
                continue
            args = (f, L["q"], L["pool"], self.num_pages, self.bt, L["comp"], L["kwin"], L["vwin"], L["wlen"],
                    self.ks, self.vs, self.kcb, self.vcb, self.S, L["out"], self.ws)
            if events is None:
                tq.tq_decode_attn(*args, err_word=self.err)
            else:
                tq.tq_decode_attn_timed(*args, events[i][0], events[i][1], err_word=self.err)


class KiviDecodeBench:
    """A resident multi-layer KIVI-style cache (the control arm: keys per
    channel over each page, values per token) and its decode step: one
    tq_kivi_decode_attn per layer over the compressed pages plus the fp16
    window.  Keys are encoded a page group at a time (prefill), so this arm
    has no per-token append."""

    def __init__(self, wl: ti.DecodeWorkload, device: str):
        import decode_attention_tq_gb300 as tq

        self.tq = tq
        self.wl = wl
        f = wl.fmt
        self.fmt = f
        B, Hq, H, d, P, W, T = wl.batch, wl.q_heads, wl.kv_heads, f.head_dim, f.page_size, wl.window, wl.context
        comp = wl.comp_tokens
        self.B, self.Hq, self.H, self.W, self.T, self.comp = B, Hq, H, W, T, comp
        self.pages_per_seq = wl.pages_per_seq
        self.num_pages = B * self.pages_per_seq + 1
        perm = ti.page_permutation(self.num_pages).to(device)
        self.bt = perm[: B * self.pages_per_seq].reshape(B, self.pages_per_seq).contiguous()
        pos = torch.arange(comp, device=device)
        slots = self.bt[:, pos // P] * P + (pos % P)[None, :]
        self.comp_lens = torch.full((B,), comp, dtype=torch.int32, device=device)
        self.win_lens = torch.full((B,), wl.win_tokens, dtype=torch.int32, device=device)
        lay = tq.tq_kivi_page_layout(f)
        self.layers = []
        for layer in range(wl.layers):
            pool = torch.zeros(self.num_pages * lay["page_bytes"], dtype=torch.uint8, device=device)
            ent = {"pool": pool}
            for kind, name in ((0, "k"), (1, "v")):
                x = ti.kv_history(B, T, H, d, layer, kind, device=device)
                for b in range(B):
                    xs = x[b, :comp].contiguous()
                    if kind == 0:
                        tq.tq_kivi_encode_keys(f, xs, self.bt[b].contiguous(), pool, self.num_pages)
                    else:
                        tq.tq_kivi_encode_values(f, xs, slots[b].to(torch.int32).contiguous(), pool, self.num_pages)
                ent[name + "win"] = x[:, comp:].permute(0, 2, 1, 3).contiguous() if W else None
                del x
            ent["q"] = ti.query(B, Hq, d, device=device, seed=ti.SEED_QUERY + 7919 * layer)
            ent["out"] = torch.empty((B, Hq, d), dtype=torch.float32, device=device)
            self.layers.append(ent)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        self.ws = torch.empty(tq.tq_kivi_decode_attn_workspace_size(f, B, Hq, self.pages_per_seq, W), dtype=torch.uint8, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        per_tok = 4 * d / P + lay["k_code_bytes"] + 4 + lay["v_code_bytes"]  # K params amortised over the page
        self.main_bytes = int(B * H * comp * per_tok) + B * self.pages_per_seq * 4
        self.window_bytes = B * H * wl.win_tokens * d * 2 * 2
        self.step_bytes = wl.layers * (self.main_bytes + self.window_bytes + B * Hq * d * (2 + 4))
        self.launches_per_step = wl.layers * 3  # prep (with window chunks), main, merge

    def step(self, events=None):
        for i, L in enumerate(self.layers):
            self.tq.tq_kivi_decode_attn(self.fmt, L["q"], L["pool"], self.num_pages, self.bt, self.comp_lens, L["kwin"], L["vwin"],
                                        self.win_lens if self.W else None, L["out"], self.ws, err_word=self.err,
                                        events=None if events is None else events[i])


def time_steps(fn, steps: int, warmup: int, barrier):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    barrier()
    return e0.elapsed_time(e1) / steps  # ms per step


L2_BYTES = 129e6  # GB300 L2 (126 MiB)
NOMINAL_HBM_GBS = 8000.0  # the nominal HBM3e rate the roofline is also reported against


def time_steps_flushed(fn, steps: int, warmup: int, barrier, flush):
    """Per-step device time with L2 flushed (flush() writes a buffer larger
    than L2) before every step, outside the timed interval."""
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        flush()
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    barrier()
    return statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)


def event_pairs(n):
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in evs:  # torch creates the CUDA event on its first record
        a.record()
        b.record()
    return evs


def measure_decode(bench, steps, warmup, barrier, reduce_max, device, use_graph=True, event_steps=5):
    """Step time (graph replay, L2 flushed per step when the working set is
    under 4x L2), clocks during the timed region, and the main kernel's mean
    CUDA-event duration over eager steps."""
    bench.step()
    torch.cuda.synchronize()
    graph = None
    if use_graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            bench.step()
        torch.cuda.current_stream().wait_stream(s)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            bench.step()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else bench.step
    # a working set that L2 could hold is timed step by step with L2 flushed
    # before each step; larger ones stream from HBM anyway
    flush_l2 = bench.step_bytes < 4 * L2_BYTES
    flush = None
    if flush_l2:
        scratch = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=device)
        flush = lambda: scratch.fill_(1)
    with ClockSampler(nvml_index(torch.cuda.current_device())) as clk:
        if flush_l2:
            ms = time_steps_flushed(run, steps, warmup, barrier, flush)
        else:
            ms = time_steps(run, steps, warmup, barrier)
    ms = reduce_max(ms)
    clocks = clk.summary()
    # dominant kernel in place: eager steps with events around the main kernel
    evs = event_pairs(bench.wl.layers)
    durs = []
    for _ in range(max(1, min(steps, event_steps))):
        if flush_l2:
            flush()
        bench.step(events=evs)
        torch.cuda.synchronize()
        durs.extend(a.elapsed_time(b) for a, b in evs)
    main_ms = statistics.mean(durs)
    del graph
    return dict(ms=ms, clocks=clocks, main_ms=main_ms, err=int(bench.err.item()), cuda_graph=use_graph, flush_l2=flush_l2,
                flush=flush)


def l2_note(bench, flush_l2):
    return ("working set %.1f MB < 4x L2: L2 flushed before every timed step, outside the timing" % (bench.step_bytes / 1e6)
            if flush_l2 else "working set (cache %.1f GB) >> L2; no flush" % (bench.step_bytes / 1e9))


def run_decode(args, device, barrier, reduce_max, rank, world):
    wl = {w.name: w for w in ti.DECODE_WORKLOADS}[args.workload]
    if args.layers:
        import dataclasses

        wl = dataclasses.replace(wl, layers=args.layers, name=f"{wl.name}(first {args.layers} layers)")
    t0 = time.time()
    # every step appends one compressed token per sequence: room for all the
    # steps this run makes (both timed arms, warm-ups, captures, event steps)
    bench = DecodeBench(wl, device, spare_tokens=2 * (args.steps + args.warmup) + 80)
    setup_s = time.time() - t0
    m = measure_decode(bench, args.steps, args.warmup, barrier, reduce_max, device, use_graph=not args.no_graph)
    ms, clocks, main_ms, err, flush_l2, flush = m["ms"], m["clocks"], m["main_ms"], m["err"], m["flush_l2"], m["flush"]
    graph = True if not args.no_graph else None

    peak, peak_kind = measured_peaks()
    achieved = bench.main_bytes / (main_ms * 1e-3) / 1e9
    traffic = load_traffic("attn_main", wl.name)

    tokens_per_step = wl.batch * wl.layers * wl.context
    value = job_throughput(tokens_per_step, ms, world)
    res = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8 codes / fp16 operands / f32 accumulate",
        "data": "synthetic (Student-t nu=3 + 4 outlier channels x20, RoPE keys, seeded)",
        "config": {
            "workload": wl.name, "layers": wl.layers, "batch": wl.batch, "q_heads": wl.q_heads, "kv_heads": wl.kv_heads,
            "head_dim": wl.fmt.head_dim, "context": wl.context, "window": wl.window, "page_size": wl.fmt.page_size,
            "k_bits": wl.fmt.k_bits + 0.5 * wl.fmt.k_mixed, "v_bits": wl.fmt.v_bits, "k_qjl": wl.fmt.k_qjl, "step": "per layer: append 1 token/seq + decode attention",
            "l2": l2_note(bench, flush_l2),
            "cuda_graph": graph is not None,
        },
        "hbm_gbs": bench.step_bytes / (ms * 1e-3) / 1e9,
        "token_heads_per_s": value * wl.kv_heads,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "kernel": "attn_main_kernel", "bytes_per_launch": bench.main_bytes, "ms_per_launch": main_ms,
                     "peak_source": peak_kind, "frac_of_nominal_8000_gbs": achieved / NOMINAL_HBM_GBS},
        "gpu_launches": bench.launches_per_step * args.steps,
        "clocks": clocks,
        "setup_s": setup_s,
        "err_word": err,
    }
    return res, bench


def run_break_even(bench, ms_step, steps: int = 8):
    """M7 of the design study ('Append cost and memory-bandwidth tradeoffs'):
    G* = C_append tau_op / (dB_step / BW_eff), the number of future decode
    steps whose bandwidth savings repay one step's append.  C_append tau_op is
    the measured device time of one step's appends (every layer's
    tq_append_window, replayed as one CUDA graph between two events),
    dB_step = T L H d (4 - (b_K + b_V)/8) the bytes one decode step saves
    against an fp16 cache, BW_eff the measured bytes per second of the
    decode step."""
    wl, f = bench.wl, bench.fmt
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bench.step(append_only=True)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bench.step(append_only=True)
    torch.cuda.synchronize()
    g.replay()
    per_step = []
    for _ in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        per_step.append(e0.elapsed_time(e1))
    del g
    t_append_ms = statistics.median(per_step)
    kbits = f.k_bits + 0.5 * f.k_mixed + (f.qjl_m / f.head_dim if f.k_qjl else 0.0)
    d_bytes = wl.context * wl.layers * wl.kv_heads * f.head_dim * (4 - (kbits + f.v_bits) / 8)
    bw_eff = bench.step_bytes / (ms_step * 1e-3)
    saved_ms = d_bytes / bw_eff * 1e3
    return {"append_ms_per_step": t_append_ms, "delta_bytes_per_step": d_bytes, "bw_eff_gbs": bw_eff / 1e9,
            "saved_ms_per_step": saved_ms, "g_star_steps": t_append_ms / saved_ms,
            "how": "append time: one step's appends (every layer) replayed as a CUDA graph between two events, median of 8; "
                   "dB_step from the formula with the format's bits per coordinate (QJL sign bits included); "
                   "BW_eff = step bytes / step time"}


def workload_entry(wl, bench, m, kind: str):
    peak, _ = measured_peaks()
    achieved = bench.main_bytes / (m["main_ms"] * 1e-3) / 1e9
    tokens = wl.batch * wl.layers * wl.context
    f = wl.fmt
    return {
        "ms_per_step": m["ms"], "value": tokens / (m["ms"] * 1e-3), "unit": UNIT, "hbm_gbs": bench.step_bytes / (m["ms"] * 1e-3) / 1e9,
        "main_kernel": kind, "main_us": m["main_ms"] * 1e3, "main_bytes": bench.main_bytes, "main_gbs": achieved, "frac": achieved / peak,
        "frac_of_nominal_8000_gbs": achieved / NOMINAL_HBM_GBS, "clocks": m["clocks"], "l2": l2_note(bench, m["flush_l2"]),
        "cuda_graph": m["cuda_graph"], "err_word": m["err"], "gpu_launches_per_step": bench.launches_per_step,
        "shape": {"layers": wl.layers, "batch": wl.batch, "q_heads": wl.q_heads, "kv_heads": wl.kv_heads, "context": wl.context,
                  "window": wl.window, "page_size": f.page_size, "k_bits": f.k_bits + 0.5 * getattr(f, "k_mixed", 0), "v_bits": f.v_bits,
                  "k_qjl": getattr(f, "k_qjl", 0)},
        "step": "per layer: append 1 token/seq + decode attention" if kind == "attn_main_kernel" else
                "per layer: decode attention (the KIVI arm encodes keys a page group at a time; no per-token append)",
    }


def run_workloads(args, device, barrier, reduce_max, skip_name: str):
    """Every other decode workload (the five configurations' decode shapes,
    the design study's K3.5/V3 mode and the KIVI control arm), each timed the
    same way as the headline line, with fewer steps."""
    out = {}
    steps, warmup = max(3, min(args.steps, 10)), 3
    for wl in ti.DECODE_WORKLOADS + ti.KIVI_WORKLOADS:
        if wl.name == skip_name:
            continue
        kivi = wl in ti.KIVI_WORKLOADS
        bench = KiviDecodeBench(wl, device) if kivi else DecodeBench(wl, device, spare_tokens=2 * (steps + warmup) + 48)
        m = measure_decode(bench, steps, warmup, barrier, reduce_max, device)
        out[wl.name] = workload_entry(wl, bench, m, "kivi_main_kernel" if kivi else "attn_main_kernel")
        del bench, m
        torch.cuda.empty_cache()
    return out


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (same hash)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[f"{kernel}:{workload}"]
    except (OSError, KeyError, ValueError):
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# Sources the split-KV main attention kernel is compiled from: a change in
# any of them invalidates its recorded DRAM traffic.
ATTN_MAIN_SOURCES = ("tq_attn_main.cuh", "tq_attn_k2.cu", "tq_attn_k3.cu", "tq_attn_k4.cu", "tq_internal.cuh", "tq_device.cuh")


def kernel_source_hash() -> str:
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_tq_gb300", "csrc")
    for n in ATTN_MAIN_SOURCES:
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    with open(os.path.join(ROOT, "include", "tq.h"), "rb") as f:
        h.update(b"tq.h" + f.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------- encode bench --
def run_encode(args, device):
    """Bulk encode: 32 layers x 8 heads x 65536 tokens of K and V into 64-token
    pages, for b in {2,3,4} and keys with / without QJL (m = 128)."""
    import decode_attention_tq_gb300 as tq

    wl = ti.BULK_ENCODE_64K
    layers = wl.layers if not args.quick else 4
    H, d, N, P = wl.kv_heads, 128, wl.tokens, wl.page_size
    xs = []
    for layer in range(layers):
        xs.append((ti.kv_history(1, N, H, d, layer, 0, device=device)[0].contiguous(),
                   ti.kv_history(1, N, H, d, layer, 1, device=device)[0].contiguous()))
    num_pages = N // P
    perm = ti.page_permutation(num_pages).to(device)
    pos = torch.arange(N, device=device)
    slots = (perm[pos // P] * P + pos % P).to(torch.int32).contiguous()
    ks = torch.from_numpy(ti.sign_bits(ti.SEED_SIGNS_K, d)).to(device)
    vs = torch.from_numpy(ti.sign_bits(ti.SEED_SIGNS_V, d)).to(device)
    S = torch.from_numpy(ti.gaussian_matrix(ti.SEED_QJL, wl.qjl_m, d)).to(device)
    out = {}
    peak, _ = measured_peaks()
    for b in wl.bits:
        for qjl in wl.qjl_options:
            if args.encode_formats and f"b{b}_qjl{qjl}" not in args.encode_formats.split(","):
                continue
            fmt = ti.Format(d, b, b, qjl, wl.qjl_m, P, H)
            lay = tq.tq_page_layout(fmt)
            pools = [torch.zeros(num_pages * lay["page_bytes"], dtype=torch.uint8, device=device) for _ in range(layers)]
            kcb = tq.device_codebook(b, device)

            def run():
                for layer in range(layers):
                    tq.tq_encode(fmt, 0, xs[layer][0], slots, pools[layer], num_pages, ks, kcb, S if qjl else None)
                    tq.tq_encode(fmt, 1, xs[layer][1], slots, pools[layer], num_pages, vs, kcb, None)

            reps = max(2, args.steps // 3)
            ms = time_steps(run, reps, 2, lambda: None)
            vecs = 2 * layers * N * H
            bph = per_token_head_bytes(fmt)
            algo = layers * N * H * (2 * 256 + bph["k"] + bph["v"])
            out[f"b{b}_qjl{qjl}"] = {"vectors_per_s": vecs / (ms * 1e-3), "ms_per_run": ms, "gbs": algo / (ms * 1e-3) / 1e9,
                                     "frac_hbm": algo / (ms * 1e-3) / 1e9 / peak, "gpu_launches": 2 * layers * reps}
            del pools
    del xs
    torch.cuda.empty_cache()
    return {"workload": wl.name + ("" if layers == wl.layers else f"(first {layers} layers)"), "per_format": out,
            "vectors_per_run": 2 * layers * N * H}


# ------------------------------------------------------------------- e2e --
def run_e2e(args, bench: DecodeBench, graph: bool = True):
    """Same step through the public API with host buffers: every step copies
    all layers' queries and appended K/V tokens from pinned host memory (one
    copy) and reads all layers' outputs back (one copy), inside the timed
    region.  Like the device-resident step it is replayed as a CUDA graph."""
    host_in = bench.io_in.cpu().pin_memory()
    host_out = torch.empty_like(bench.io_out, device="cpu").pin_memory()
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out.numel() * host_out.element_size()

    def step():
        bench.io_in.copy_(host_in, non_blocking=True)
        bench.step()
        host_out.copy_(bench.io_out, non_blocking=True)

    run = step
    if graph:
        step()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        run = g.replay
    ms = time_steps(run, args.steps, args.warmup, lambda: None)
    value = bench.wl.batch * bench.wl.layers * bench.wl.context / (ms * 1e-3)
    out_ok = bool(torch.isfinite(host_out).all())
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "cuda_graph": graph, "outputs_finite": out_ok}


# --------------------------------------------------------------- oracle --
def oracle_sample_setup(wl: ti.DecodeWorkload, n_seq: int, device: str | None, layer: int = 0):
    """Host-side pages of `n_seq` sequences of one layer, encoded by the oracle."""
    import oracle

    f = wl.fmt
    H, d, P, W, T, comp = wl.kv_heads, f.head_dim, f.page_size, wl.window, wl.context, wl.comp_tokens
    gen_dev = device if device else "cpu"
    K = ti.kv_history(n_seq, T, H, d, layer, 0, device=gen_dev).cpu().numpy()
    V = ti.kv_history(n_seq, T, H, d, layer, 1, device=gen_dev).cpu().numpy()
    pps = wl.pages_per_seq
    num_pages = n_seq * pps
    bt = np.arange(num_pages, dtype=np.int32).reshape(n_seq, pps)
    lay = oracle.page_layout(f)
    pool = np.zeros(num_pages * lay["page_bytes"], np.uint8)
    ks, vs = ti.sign_bits(ti.SEED_SIGNS_K, d), ti.sign_bits(ti.SEED_SIGNS_V, d)
    kc, kt = oracle.kind_codebook(f, 0)
    vc, vt = oracle.kind_codebook(f, 1)
    S = ti.gaussian_matrix(ti.SEED_QJL, f.qjl_m, d) if f.k_qjl else None
    jobs = []
    for b in range(n_seq):
        sl = (bt[b, np.arange(comp) // P] * P + np.arange(comp) % P).astype(np.int32)
        jobs.append((0, np.ascontiguousarray(K[b, :comp]), sl, ks, kc, kt, S))
        jobs.append((1, np.ascontiguousarray(V[b, :comp]), sl, vs, vc, vt, None))
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), host_cores())) as ex:
        rcs = list(ex.map(lambda j: oracle.encode(f, j[0], j[1], j[2], pool, num_pages, *j[3:]), jobs))
    assert all(rc == 0 for rc in rcs)
    kwin = np.ascontiguousarray(K[:, comp:].transpose(0, 2, 1, 3)) if W else None
    vwin = np.ascontiguousarray(V[:, comp:].transpose(0, 2, 1, 3)) if W else None
    q = ti.query(n_seq, wl.q_heads, d).numpy()
    return dict(f=f, q=q, pool=pool, num_pages=num_pages, bt=bt, comp=np.full(n_seq, comp, np.int32), kwin=kwin, vwin=vwin,
                wl=np.full(n_seq, wl.win_tokens, np.int32), ks=ks, vs=vs, kc=kc, vc=vc, S=S)


def oracle_time(s, heads, cores):
    """Oracle decode attention for the listed (b*Hq + qh) rows on `cores` threads."""
    import oracle

    chunks = [heads[i::cores] for i in range(cores) if heads[i::cores]]

    def work(hs):
        return oracle.attention(s["f"], s["q"], s["pool"], s["num_pages"], s["bt"], s["comp"], s["kwin"], s["vwin"], s["wl"], s["ks"],
                                s["vs"], s["kc"], s["vc"], s["S"], heads=np.array(hs, np.int32))

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        list(ex.map(work, chunks))
    return time.perf_counter() - t0


def cpu_baseline(wl: ti.DecodeWorkload, device, target_cpu_s: float = 20.0):
    """The oracle as it stands, on a bounded sample: whole sequences (all query
    heads) of layer 0, sized to about `target_cpu_s` seconds of CPU work."""
    cores = host_cores()
    Hq = wl.q_heads
    s = oracle_sample_setup(wl, 1, device)
    probe = oracle_time(s, [0], 1)  # one query head on one core
    rows = int(max(1, target_cpu_s / max(probe, 1e-3)))
    n_seq = int(min(wl.batch, 8, max(1, -(-rows // Hq))))
    if n_seq > 1:
        s = oracle_sample_setup(wl, n_seq, device)
    n_heads = int(min(rows, Hq * n_seq))
    heads = list(range(n_heads))
    dt = oracle_time(s, heads, cores)
    tokens = wl.context * n_heads / Hq  # a sequence-token counts once per layer, all heads included
    return {"value": tokens / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"layer 0: {n_heads} (sequence, query head) rows of {Hq} heads per sequence at context {wl.context}, "
                      f"= {n_heads / Hq:.2f} sequence-layers; {dt:.2f} s wall on {cores} threads "
                      f"(~{n_heads * probe:.0f} s of CPU work)"}


def cpu_baseline_layers(wl: ti.DecodeWorkload, device, budget_s: float):
    """The oracle on whole layers (every sequence and query head), layer after
    layer until the budget is spent or the workload is done: the full step
    when it fits, else the layers it reached (stated in `sample`)."""
    cores = host_cores()
    t_att, layers = 0.0, 0
    t0 = time.perf_counter()
    for layer in range(wl.layers):
        s = oracle_sample_setup(wl, wl.batch, device, layer)
        t_att += oracle_time(s, list(range(wl.batch * wl.q_heads)), cores)
        layers += 1
        if time.perf_counter() - t0 > budget_s:
            break
    value = wl.batch * layers * wl.context / t_att
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"{wl.name}: the full step ({layers} layers)" if layers == wl.layers else
                       f"{wl.name}: {layers} of {wl.layers} layers, every sequence and query head") +
                      f"; {t_att:.2f} s of attention wall time on {cores} threads (encode excluded)"}


def cpu_baseline_slice(wl: ti.DecodeWorkload, device, budget_s: float):
    """The oracle on (sequence, query head) rows of layer 0 of one sequence,
    as many as fit the budget (the long-context shape's layer is minutes of
    CPU work)."""
    cores = host_cores()
    s = oracle_sample_setup(wl, 1, device)
    probe = oracle_time(s, [0], 1)
    n = int(max(1, min(wl.q_heads, budget_s * cores / max(probe, 1e-3))))
    dt = oracle_time(s, list(range(n)), cores)
    return {"value": wl.context * n / wl.q_heads / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{wl.name}: layer 0, sequence 0, {n} of {wl.q_heads} query heads at context {wl.context}; "
                      f"{dt:.2f} s wall on {cores} threads"}


def cpu_baseline_encode(budget_s: float, device):
    """The oracle's encode on vectors of one layer of the bulk-encode workload
    (K with a QJL sketch and V, 3 bits), as many tokens as fit the budget."""
    import oracle

    cores = host_cores()
    wl = ti.BULK_ENCODE_64K
    H, d, P = wl.kv_heads, 128, wl.page_size
    fmt = ti.Format(d, 3, 3, 1, wl.qjl_m, P, H)
    c, t = oracle.make_codebook(3)
    ks, vs = ti.sign_bits(ti.SEED_SIGNS_K, d), ti.sign_bits(ti.SEED_SIGNS_V, d)
    S = ti.gaussian_matrix(ti.SEED_QJL, wl.qjl_m, d)
    NMAX = wl.tokens
    X = [ti.kv_history(1, NMAX, H, d, 0, kind, device=device if device else "cpu")[0].cpu().numpy() for kind in (0, 1)]
    lay = oracle.page_layout(fmt)

    def run(n):
        pool = np.zeros((n // P + 1) * lay["page_bytes"], np.uint8)
        chunks = [(kind, i0) for kind in (0, 1) for i0 in range(0, n, 64)]

        def job(j):
            kind, i0 = j
            i1 = min(n, i0 + 64)
            sl = np.arange(i0, i1, dtype=np.int32)
            return oracle.encode(fmt, kind, X[kind][i0:i1], sl, pool, n // P + 1, ks if kind == 0 else vs, c, t, S if kind == 0 else None)

        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=cores) as ex:
            list(ex.map(job, chunks))
        return time.perf_counter() - t0

    n0 = 64 * cores
    dt0 = run(n0)
    N = int(min(NMAX, max(n0, n0 * budget_s / max(dt0, 1e-3)))) // 64 * 64
    dt = run(N)
    vecs = 2 * N * H
    return {"value": vecs / dt, "unit": "vectors/s", "cores": cores, "kind": "oracle",
            "sample": f"{wl.name}: {N} tokens x {H} heads of K (3-bit + QJL) and V (3-bit), layer 0; {dt:.2f} s wall on {cores} threads"}


def run_cpu_baselines(device):
    """Oracle baselines beyond the headline slice: the single-layer and Qwen
    decode shapes on whole layers, a long-context slice, and the encode."""
    return {
        ti.SINGLE_LAYER_T2K.name: cpu_baseline_layers(ti.SINGLE_LAYER_T2K, device, 10.0),
        ti.QWEN25_3B_T16K.name: cpu_baseline_layers(ti.QWEN25_3B_T16K, device, 15.0),
        ti.LONG_CTX_T128K.name: cpu_baseline_slice(ti.LONG_CTX_T128K, device, 10.0),
        ti.BULK_ENCODE_64K.name: cpu_baseline_encode(8.0, device),
    }


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle, timed on the host cores."""
    wl = {w.name: w for w in ti.DECODE_WORKLOADS}[args.workload]
    if rank != 0:
        return None
    cores = host_cores()
    dev = "cuda" if torch.cuda.is_available() else None
    s = oracle_sample_setup(wl, 1, dev)
    Hq = wl.q_heads
    probe = oracle_time(s, [0], 1)
    budget = max(2.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))  # seconds per step
    n_heads = int(max(1, min(Hq, budget * cores / max(probe, 1e-3))))
    heads = list(range(n_heads))
    for _ in range(args.warmup):
        oracle_time(s, heads, cores)
    times = [oracle_time(s, heads, cores) for _ in range(args.steps)]
    dt = sum(times) / len(times)
    value = wl.context * n_heads / Hq / dt
    sample = f"layer 0, sequence 0, {n_heads} of {Hq} query heads at context {wl.context} per step; {cores} threads"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same recipe)", "config": {"workload": wl.name, "reference": "fp64 CPU oracle (no reference implementation exists)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--workload", default=ti.LLAMA3_8B_T32K.name, choices=[w.name for w in ti.DECODE_WORKLOADS])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-encode", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="only the headline workload (no other decode shapes, no break-even)")
    ap.add_argument("--quick", action="store_true", help="fewer encode layers (development)")
    ap.add_argument("--layers", type=int, default=0, help="decode layers (profiling a small case; 0 = the workload's)")
    ap.add_argument("--encode-only", action="store_true", help="run only the bulk-encode part (profiling)")
    ap.add_argument("--encode-formats", default="", help="comma list such as b4_qjl1 (default: all six)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "tq" else args.warmup

    world, rank, local = dist_info()
    pg = None
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist

    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        if pg:
            pg.barrier()
            pg.destroy_process_group()
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py --impl tq needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    import __graft_entry__

    def barrier():
        if pg:
            pg.barrier()

    # one rank per node compiles (the others would race on the same objects);
    # the rest find the library up to date after the barrier
    if local == 0:
        __graft_entry__.build()
    barrier()
    if local != 0:
        __graft_entry__.build()

    def reduce_max(x):
        return max_over_ranks(x, pg, device)

    if args.encode_only:
        if rank == 0:
            print(json.dumps({"encode": run_encode(args, device)}), flush=True)
        if pg:
            pg.barrier()
            pg.destroy_process_group()
        return
    res, bench = run_decode(args, device, barrier, reduce_max, rank, world)
    if not args.no_e2e:
        e2e = run_e2e(args, bench, graph=not args.no_graph)
        e2e_ms = reduce_max(e2e["ms_per_step"])
        e2e["value"] = job_throughput(bench.wl.batch * bench.wl.layers * bench.wl.context, e2e_ms, world)
        res["e2e"] = e2e
    if not args.no_workloads:
        res["break_even"] = run_break_even(bench, res["ms_per_step"])
    main_name = bench.wl.name
    del bench
    torch.cuda.empty_cache()
    if not args.no_workloads:
        res["workloads"] = run_workloads(args, device, barrier, reduce_max, main_name)
    if not args.no_encode:
        res["encode"] = run_encode(args, device)
    if rank == 0 and world == 1 and not args.no_cpu:
        wl = {w.name: w for w in ti.DECODE_WORKLOADS}[args.workload]
        res["cpu_baseline"] = cpu_baseline(wl, device)
        if not args.no_workloads:
            res["cpu_baselines"] = run_cpu_baselines(device)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
