#!/usr/bin/env python3
"""GVA decode benchmark: cache-read HBM GB/s and microseconds per layer step.

One step = one decode token through a stack of `--layers` layers of the chosen
workload (default: the 350M-class layer, B=8, H=16, G=4, d_h=64, d_n=64, d_r=16,
T=4096, bf16).  Every layer has its own cache (more bytes in total than the 126 MB
L2), and a layer step is: gva_append_cache (the current token at t = L_b - 1) then
gva_decode_attention (absorb, split-K partial, log-sum-exp combine).  The whole step
is captured in one CUDA graph and replayed; time is taken with CUDA events on the
launching stream, max over ranks.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle on the
host cores on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
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

METRIC = "GVA decode cache-read HBM GB/s (% of B300 peak) and μs/step, B=8 T=4096"
SPEC_HBM_GBS = 8000.0          # the "~8 TB/s" B300 HBM figure the target is stated against
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_SUSTAINED = 1400.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return None


def algorithmic_bytes(w, lengths) -> int:
    """Cache bytes one decode of one layer must read: sum_b L_b (G d_h + d_r) x elem."""
    elem = 2 if w.cache_dtype == "bf16" else 4
    return int(sum(int(L) for L in lengths)) * (w.G * w.d_h + w.d_r) * elem


def gqa_bytes(w, lengths) -> int:
    elem = 2 if w.cache_dtype == "bf16" else 4
    return int(sum(int(L) for L in lengths)) * 2 * w.G * w.d_h * elem


# --------------------------------------------------------------------------- #
# distributed plumbing (one process per GPU; weak scaling, no data-path collective)
# --------------------------------------------------------------------------- #
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float, device=None) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(units_per_rank, max_seconds):
    """Whole-job throughput: units processed by all ranks over the slowest rank's time."""
    return units_per_rank / max_seconds


# --------------------------------------------------------------------------- #
# clocks during the timed region
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_marks = {}

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t0 = time.time()

        def rd():
            for line in self.proc.stdout:
                self.lines.append((time.time(), line.strip()))
        self.th = threading.Thread(target=rd, daemon=True)
        self.th.start()

    def mark(self, name):
        self.t_marks[name] = time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.th.join(timeout=2)

    def summary(self, t_from, t_to):
        mhz, mx, reasons = [], None, set()
        names = ("active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap")
        for t, line in self.lines:
            if not (t_from - 0.15 <= t <= t_to + 0.15):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names[1:], f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(mhz)}


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def default_layers(w) -> int:
    """Layers per step: a layer smaller than L2 (126 MB) gets at least 32 distinct layer
    caches and four times L2 in all; a larger layer is streamed from HBM on every call."""
    c_bytes = (w.B * (w.T or sum(w.len_range) // 2)) * (w.G * w.d_h + w.d_r) * 2
    n = max(1, min(64, math.ceil(4 * 126e6 / c_bytes)))
    return max(32, n) if c_bytes < 126e6 else n


def timed_graph(torch, dist, stream, graph, K, W, sampler=None):
    """W untimed replays, then K timed replays of `graph` on `stream` (CUDA events at every
    step boundary), barrier + synchronize on both sides.  Returns (seconds, per-step ms)."""
    for _ in range(W):
        graph.replay()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    if sampler:
        sampler.mark("t0")
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for k in range(K):
            graph.replay()
            ev[k + 1].record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    dist.barrier()
    steps = [ev[k].elapsed_time(ev[k + 1]) for k in range(K)]
    return ev[0].elapsed_time(ev[K]) / 1e3, steps


class LayerStack:
    """`nl` layers of one workload on the device, each with its own cache, queries, maps
    and new-token inputs (the seeded case, copied per layer)."""

    def __init__(self, gva, torch, gva_inputs, name, nl, dev):
        w = gva_inputs.workload(name)
        c = gva_inputs.make_case(w)
        self.w, self.c, self.nl, self.dev = w, c, nl, dev
        self.lengths = c.seq_len.tolist()
        self.dims = gva.Dims(w.B, w.H, w.G, w.d_h, w.d_n, w.d_r,
                             gva.GVA_F32 if w.cache_dtype == "f32" else gva.GVA_BF16,
                             gva.GVA_F32 if w.q_dtype == "f32" else gva.GVA_BF16)
        V0, K0 = c.V.to(dev), c.Kr.to(dev)
        self.V0 = V0
        self.layers = []
        for li in range(nl):
            V = V0.clone() if li else V0
            K = K0.clone() if li else K0
            self.layers.append(dict(
                cache=gva.Cache(self.rows(gva, V), V, K),
                q_nope=c.q_nope.to(dev).clone(), q_rope=c.q_rope.to(dev).clone(),
                M=c.M.to(dev).clone(), v_new=c.v_new.to(dev).clone(),
                k_new=c.k_new.to(dev).clone(),
                out=torch.empty((w.B, w.H, w.d_h), device=dev),
                lse=torch.empty((w.B, w.H), device=dev)))
        self.seq = c.seq_len.to(dev)
        self.pos = (c.seq_len - 1).to(torch.int32).to(dev)
        self.tab = gva.gva_rope_table_fill(int(max(self.lengths)) + 1, w.d_r, w.base).to(dev)
        self.ws = gva.workspace(self.dims, dev)
        self.bytes_layer = algorithmic_bytes(w, self.lengths)

    def rows(self, gva, V):
        c, w, dev = self.c, self.w, self.dev
        offs = c.offsets.to(dev) if c.offsets is not None else None
        bt = c.block_table.to(dev) if c.block_table is not None else None
        return gva.Rows(w.layout, c.num_rows, T_cap=c.T_cap, offsets=offs, block_table=bt,
                        page_size=w.page_size)


def measure_stack(args, dist, torch, gva, gva_inputs, S, stream, sampler, path, with_gqa):
    """Layer step (append + decode) and decode op of every layer of stack S, each as one
    CUDA graph, timed on `stream`; the matched GQA comparator when asked.  Returns the
    workload's figures (microseconds per layer, GB/s, fraction of the measured copy peak)."""
    w, nl = S.w, S.nl
    step_layers = [dict(v_new=L["v_new"], k_rope_new=L["k_new"], q_nope=L["q_nope"],
                        q_rope=L["q_rope"], M=L["M"], cache=L["cache"], out=L["out"],
                        lse=L["lse"]) for L in S.layers]

    def whole_step(_):
        # the library's step call: every layer's append and decode (on the tensor-core
        # path the append shares the absorption's grid: three launches per layer)
        gva.gva_decode_step(S.dims, step_layers, S.pos, S.seq, S.tab, w.scale, S.ws, path=path)

    def layer_calls(L):
        gva.gva_append_cache(S.dims, L["v_new"], L["k_new"], S.pos, None, L["cache"], S.tab)
        gva.gva_decode_attention(S.dims, L["q_nope"], L["q_rope"], L["M"], S.seq, L["cache"],
                                 S.tab, w.scale, L["out"], L["lse"], S.ws, path=path)

    def decode_only(L):
        gva.gva_decode_attention(S.dims, L["q_nope"], L["q_rope"], L["M"], S.seq, L["cache"],
                                 S.tab, w.scale, L["out"], L["lse"], S.ws, path=path)

    g_step = capture_list(torch, stream, [None], whole_step)
    g_calls = capture_list(torch, stream, S.layers, layer_calls)
    g_dec = capture_list(torch, stream, S.layers, decode_only)
    assert gva.gva_get_device_status() == 0
    soak_t = time.time()
    while time.time() - soak_t < args.soak:
        for _ in range(max(1, 64 // nl)):
            g_step.replay()
        torch.cuda.synchronize()
    secs, step_ms = timed_graph(torch, dist, stream, g_step, args.steps, args.warmup, sampler)
    max_secs = dist.max(secs, S.dev)
    dsecs, dec_ms = timed_graph(torch, dist, stream, g_dec, args.steps, max(3, args.warmup))
    dsecs = dist.max(dsecs, S.dev)
    csecs, _ = timed_graph(torch, dist, stream, g_calls, args.steps, max(3, args.warmup))
    csecs = dist.max(csecs, S.dev)
    us_layer = max_secs / (args.steps * nl) * 1e6
    us_decode = dsecs / (args.steps * nl) * 1e6
    achieved = S.bytes_layer / (us_decode * 1e-6) / 1e9
    peaks = measured_peaks()
    hbm_peak = peaks["hbm_gbs"] if peaks else FALLBACK_HBM_GBS
    out = {"layers": nl, "tokens_per_layer": int(sum(S.lengths)), "bytes_per_layer": S.bytes_layer,
           "us_per_layer_step": round(us_layer, 3), "us_per_decode": round(us_decode, 3),
           "us_per_layer_step_separate_calls": round(csecs / (args.steps * nl) * 1e6, 3),
           "median_of_steps": {"us_per_layer_step": round(statistics.median(step_ms) * 1e3 / nl, 3),
                               "us_per_decode": round(statistics.median(dec_ms) * 1e3 / nl, 3),
                               "reps": args.steps},
           "layer_step_gbs": round(aggregate(S.bytes_layer * nl * args.steps * dist.world,
                                             max_secs) / 1e9, 2),
           "decode_gbs": round(achieved, 1), "decode_frac_of_measured_copy": round(achieved / hbm_peak, 4),
           "seconds": max_secs}
    del g_step, g_calls, g_dec
    # The absorption alone (the public gva_absorb_query, which also rotates the positional
    # query), one call per layer in its own graph: what GVA's chain adds to GQA's, before
    # the overlap that programmatic dependent launch gives it inside the decode op.
    qt = torch.empty((w.B, w.H, w.d_h), device=S.dev)
    qr = torch.empty((w.B, w.H, max(1, w.d_r)), device=S.dev)

    def absorb_only(L):
        gva.gva_absorb_query(S.dims, L["q_nope"], L["q_rope"], L["M"], S.seq, S.tab, w.scale,
                             qt, qr)
    g_abs = capture_list(torch, stream, S.layers, absorb_only)
    asecs, _ = timed_graph(torch, dist, stream, g_abs, args.steps, max(3, args.warmup))
    out["absorb_only_us_per_layer"] = round(dist.max(asecs, S.dev) / (args.steps * nl) * 1e6, 3)
    del g_abs

    # the append alone (one new token per sequence and layer), in its own graph
    def append_only(L):
        gva.gva_append_cache(S.dims, L["v_new"], L["k_new"], S.pos, None, L["cache"], S.tab)
    g_app = capture_list(torch, stream, S.layers, append_only)
    psecs, _ = timed_graph(torch, dist, stream, g_app, args.steps, max(3, args.warmup))
    out["append_only_us_per_layer"] = round(dist.max(psecs, S.dev) / (args.steps * nl) * 1e6, 3)
    del g_app
    if not with_gqa:
        return out
    Kq0 = gva_inputs.make_gqa_keys(S.c).to(S.dev)
    qq = gva_inputs.make_gqa_query(S.c).to(S.dev)
    glayers = []
    for li in range(nl):
        glayers.append(dict(kv=gva.KVCache(S.rows(gva, S.V0), Kq0.clone() if li else Kq0,
                                           S.layers[li]["cache"].V), q=qq.clone(),
                            out=torch.empty((w.B, w.H, w.d_h), device=S.dev),
                            lse=torch.empty((w.B, w.H), device=S.dev)))

    def gqa_call(L):
        gva.gva_gqa_decode_attention(S.dims, L["q"], S.seq, L["kv"], 1.0 / math.sqrt(w.d_h),
                                     L["out"], L["lse"], S.ws, path=path)
    gg = capture_list(torch, stream, glayers, gqa_call)
    gsecs, _ = timed_graph(torch, dist, stream, gg, args.steps, max(3, args.warmup))
    us_gqa = dist.max(gsecs, S.dev) / (args.steps * nl) * 1e6
    gb = gqa_bytes(w, S.lengths)
    out["gqa_comparator"] = {"us_per_layer": round(us_gqa, 3), "bytes_per_layer": gb,
                             "gbs": round(gb / (us_gqa * 1e-6) / 1e9, 1),
                             "gva_bytes_saved_pct": round(100 * (1 - S.bytes_layer / gb), 3),
                             "gva_time_saved_pct": round(100 * (1 - us_decode / us_gqa), 1)}
    del glayers, gg, Kq0
    # the MLA-shaped comparator at matched cache bytes (latent width d_c = G d_h)
    mw = gva.MlaDims(w.B, w.H, w.G * w.d_h, w.d_n, w.d_r, w.d_h)
    if w.cache_dtype == "bf16" and gva.gva_mla_workspace_size(mw) > 0:
        mc = gva_inputs.make_mla_case(S.c)
        C0 = mc.C.to(S.dev)
        mws = gva.mla_workspace(mw, S.dev)
        mlayers = []
        for li in range(nl):
            mlayers.append(dict(cache=gva.Cache(S.rows(gva, C0), C0.clone() if li else C0,
                                                S.layers[li]["cache"].K_rope),
                                Wuk=mc.W_uk.to(S.dev), Wuv=mc.W_uv.to(S.dev),
                                out=torch.empty((w.B, w.H, w.d_h), device=S.dev),
                                lse=torch.empty((w.B, w.H), device=S.dev)))

        def mla_call(L):
            gva.gva_mla_decode_attention(mw, S.layers[0]["q_nope"], S.layers[0]["q_rope"],
                                         L["Wuk"], L["Wuv"], S.seq, L["cache"], S.tab, w.scale,
                                         L["out"], L["lse"], mws)
        gm = capture_list(torch, stream, mlayers, mla_call)
        msecs, _ = timed_graph(torch, dist, stream, gm, args.steps, max(3, args.warmup))
        us_mla = dist.max(msecs, S.dev) / (args.steps * nl) * 1e6
        out["mla_comparator"] = {"us_per_layer": round(us_mla, 3), "latent_width": mw.d_c,
                                 "bytes_per_layer": S.bytes_layer,
                                 "gbs": round(S.bytes_layer / (us_mla * 1e-6) / 1e9, 1),
                                 "gva_time_saved_pct": round(100 * (1 - us_decode / us_mla), 1)}
        del mlayers, gm, C0, mws
    return out


def measure_rope_keys(args, dist, torch, gva, gva_inputs, name, stream, dev, sampler):
    """The variant with ordinary RoPE on the reconstructed key (gva_rope_keys_decode_attention)
    on workload `name`'s shape with the query d_n wide and no positional slice: nl decode
    calls on distinct layer caches (more than L2 in all), one CUDA graph, timed on
    `stream`.  It is a dense contraction (2 d_h d_n flops per token and head, the
    algorithmic count), run as two bf16 products per weight (high and low parts)."""
    w = gva_inputs.workload(name)
    nl = default_layers(w)
    c = gva_inputs.make_case(w)
    lengths = c.seq_len.tolist()
    dims = gva.Dims(w.B, w.H, w.G, w.d_h, w.d_n, 0, gva.GVA_BF16,
                    gva.GVA_F32 if w.q_dtype == "f32" else gva.GVA_BF16)
    if gva.gva_rope_keys_workspace_size(dims) == 0:
        return None
    V0 = c.V.to(dev)
    offs = c.offsets.to(dev) if c.offsets is not None else None
    bt = c.block_table.to(dev) if c.block_table is not None else None
    rows = gva.Rows(w.layout, c.num_rows, T_cap=c.T_cap, offsets=offs, block_table=bt,
                    page_size=w.page_size)
    tab = torch.from_numpy(_rope_keys_table(max(128, int(max(lengths)) + 1), w.d_n, w.base)).to(dev)
    seq = c.seq_len.to(dev)
    ws = gva.rope_keys_workspace(dims, dev)
    layers = []
    for li in range(nl):
        layers.append(dict(cache=gva.Cache(rows, V0.clone() if li else V0, None),
                           q=c.q_nope.to(dev).clone(), M=c.M.to(dev).clone(),
                           out=torch.empty((w.B, w.H, w.d_h), device=dev),
                           lse=torch.empty((w.B, w.H), device=dev)))

    def call(L):
        gva.gva_rope_keys_decode_attention(dims, L["q"], L["M"], seq, L["cache"], tab, w.scale,
                                           L["out"], L["lse"], ws)
    g = capture_list(torch, stream, layers, call)
    assert gva.gva_get_device_status() == 0
    secs, step_ms = timed_graph(torch, dist, stream, g, args.steps, max(3, args.warmup), sampler)
    us = dist.max(secs, dev) / (args.steps * nl) * 1e6
    ck = sampler.summary(sampler.t_marks["t0"], sampler.t_marks["t1"])
    tokens = int(sum(int(L) for L in lengths))
    flops = 2.0 * tokens * w.H * w.d_h * w.d_n
    tflops = flops / (us * 1e-6) / 1e12
    peaks = measured_peaks()
    pk = (peaks["bf16_tflops_sustained"] if peaks else FALLBACK_BF16_SUSTAINED)
    cache_bytes = tokens * w.G * w.d_h * 2
    del g, layers, V0, ws
    torch.cuda.empty_cache()
    return {
        "workload": f"{name} shape, RoPE on the reconstructed key: B={w.B} H={w.H} G={w.G} "
                    f"d_h={w.d_h} d_n={w.d_n} (query d_n wide) "
                    + (f"T={w.T}" if w.layout == "contiguous" else f"{w.layout} lengths")
                    + f" bf16 cache; {nl} layer(s) per graph",
        "us_per_decode": round(us, 3),
        "median_us_per_decode": round(statistics.median(step_ms) * 1e3 / nl, 3),
        "flops_per_decode": flops, "cache_bytes_per_decode": cache_bytes,
        "cache_gbs": round(cache_bytes / (us * 1e-6) / 1e9, 1),
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1),
                     "peak": pk, "unit": "TFLOP/s", "frac": round(tflops / pk, 4),
                     "peak_source": ("measured bf16, sustained" if peaks else "fallback"),
                     "mma_flops_issued_frac": round(2 * tflops / pk, 4),
                     "note": "algorithmic flops (2 d_h d_n per token and head); the kernel "
                             "issues two bf16 products per weight (high and low parts)"},
        "launches_per_decode": 3,
        "clocks": ck,
    }


def _rope_keys_table(rows: int, d_n: int, base: float):
    """(cos, sin)(p theta_i) over d_n, fp32 from fp64 (the library's host routine)."""
    import value_only_kv_gva_b300 as gva
    return gva.gva_rope_table_fill(rows, d_n, base).numpy()


def single_pass_floor(gva, torch, dist, stream, dev, nbytes, nl, K, W):
    """The fastest single pass over `nbytes` this GPU gives one kernel in the same launch
    configuration as the decode op: `nl` distinct buffers of `nbytes` (more than L2 in
    all), one read-probe launch each, captured in one CUDA graph.  Microseconds per pass
    and GB/s."""
    n16 = nbytes // 16 * 16
    bufs = [torch.ones(n16 // 4, dtype=torch.int32, device=dev) for _ in range(nl)]
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    g = capture_list(torch, stream, bufs, lambda b: gva.gva_read_probe(b, sink, stream=stream))
    secs, _ = timed_graph(torch, dist, stream, g, K, W)
    us = dist.max(secs, dev) / (K * nl) * 1e6
    del bufs, g
    return {"us_per_pass": round(us, 3), "gbs": round(n16 / (us * 1e-6) / 1e9, 1),
            "bytes": n16, "buffers": nl}


def run_ours(args, dist: Dist):
    import torch

    import gva_inputs
    import value_only_kv_gva_b300 as gva

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    stream = torch.cuda.Stream(device=dev)
    path = args.path
    if args.rope_keys_only:
        sampler = ClockSampler(dev.index if dev.index is not None else 0)
        sampler.start()
        time.sleep(0.3)
        res = {n: measure_rope_keys(args, dist, torch, gva, gva_inputs, n, stream, dev, sampler)
               for n in args.rope_keys}
        sampler.stop()
        if dist.rank == 0:
            print(json.dumps({"rope_keys_variant": res, "steps": args.steps,
                              "warmup": args.warmup}), flush=True)
        dist.close()
        return
    S = LayerStack(gva, torch, gva_inputs, args.workload, args.layers, dev)
    w, nl = S.w, S.nl
    log(f"[bench] workload {w.name}: B={w.B} H={w.H} G={w.G} d_h={w.d_h} d_r={w.d_r} "
        f"tokens={sum(S.lengths)} layers={nl}")
    peaks = measured_peaks()
    hbm_peak = peaks["hbm_gbs"] if peaks else FALLBACK_HBM_GBS

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    t_soak = time.time()
    m = measure_stack(args, dist, torch, gva, gva_inputs, S, stream, sampler, path,
                      not args.no_gqa)
    clocks = sampler.summary(sampler.t_marks.get("t0", t_soak) - args.soak,
                             sampler.t_marks.get("t1", time.time()))
    value = m["layer_step_gbs"]                       # GB/s, all ranks
    ms_per_step = m["seconds"] / args.steps * 1e3
    achieved = m["decode_gbs"]
    read_probe = read_probe_gbs(gva, torch, stream, dev)
    floor = single_pass_floor(gva, torch, dist, stream, dev, S.bytes_layer, nl, args.steps,
                              max(3, args.warmup))

    # end to end through the public API with host buffers (eager calls, pinned copies)
    e2e = run_e2e(args, w, S.c, S.dims, gva, torch, dev, S.layers, S.seq, S.pos, S.tab, S.ws,
                  path, S.bytes_layer, dist)
    c_case = S.c
    del S
    torch.cuda.empty_cache()

    # the other workloads, measured in this process with the same clock sampling: the
    # long-context layer, the paged serving batch and the ragged batch
    others = {}
    if not args.no_others:
        for name in args.others:
            if name == w.name:
                continue
            S2 = LayerStack(gva, torch, gva_inputs, name, default_layers(gva_inputs.workload(name)), dev)
            m2 = measure_stack(args, dist, torch, gva, gva_inputs, S2, stream, sampler, path, True)
            ck = sampler.summary(sampler.t_marks["t0"], sampler.t_marks["t1"])
            w2 = S2.w
            others[name] = {
                "workload": f"{name}: GVA decode layer B={w2.B} H={w2.H} G={w2.G} d_h={w2.d_h} "
                            f"d_n={w2.d_n} d_r={w2.d_r} "
                            + (f"T={w2.T}" if w2.layout == "contiguous" else f"{w2.layout} lengths")
                            + f" {w2.cache_dtype} cache",
                **{k: v for k, v in m2.items() if k != "seconds"},
                "roofline": {"bound": "hbm", "achieved": m2["decode_gbs"], "peak": hbm_peak,
                             "unit": "GB/s", "frac": m2["decode_frac_of_measured_copy"],
                             "peak_source": "measured" if peaks else "fallback",
                             "traffic": profiled_traffic(name) if path in ("auto", "mma") else None},
                "clocks": ck}
            del S2
            torch.cuda.empty_cache()
    rope_keys = {}
    if not args.no_rope_keys:
        for name in args.rope_keys:
            rk = measure_rope_keys(args, dist, torch, gva, gva_inputs, name, stream, dev, sampler)
            if rk:
                rope_keys[name] = rk
    sampler.stop()

    # the CPU oracle on a bounded sample (rank 0 only)
    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_baseline(w, c_case, budget_s=args.cpu_seconds)

    # per layer: the partial and combine kernels, after one fused append + absorption grid
    # (tensor-core path, bf16 cache, d_n 64 or 128) or the append and absorption kernels
    fused = path in ("auto", "mma") and w.cache_dtype == "bf16" and w.d_n in (64, 128)
    launches_per_step = nl * (3 if fused else 4)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if w.cache_dtype == "bf16" else "f32", "data": "synthetic",
        "config": {
            "workload": f"{w.name}: GVA decode layer B={w.B} H={w.H} G={w.G} d_h={w.d_h} "
                        f"d_n={w.d_n} d_r={w.d_r} "
                        + (f"T={w.T}" if w.layout == "contiguous" else f"{w.layout} lengths")
                        + f" {w.cache_dtype} cache; step = append + decode through {nl} layers",
            **{k: v for k, v in m.items() if k not in ("seconds", "layer_step_gbs",
                                                       "decode_gbs",
                                                       "decode_frac_of_measured_copy",
                                                       "gqa_comparator", "mla_comparator")},
            "pct_of_8tbs_spec": round(100 * value / dist.world / SPEC_HBM_GBS, 2),
            "pct_of_measured_copy": round(100 * value / dist.world / hbm_peak, 2),
            "read_probe_gbs": read_probe,
            "decode_pct_of_read_probe": round(100 * achieved / read_probe, 2) if read_probe else None,
            "single_pass_floor": {**floor,
                                  "decode_frac_of_floor": round(floor["us_per_pass"] /
                                                                m["us_per_decode"], 4)},
            "seqs_steps_per_s": round(w.B * dist.world / (ms_per_step * 1e-3), 1),
            "l2": f"inputs larger than L2: {nl} distinct layer caches, "
                  f"{S_bytes_mb(m)} MB",
            "path": path, "accumulate": "fp32", "parallelism": f"replicas x{dist.world}",
            "gqa_comparator": m.get("gqa_comparator"),
            "mla_comparator": m.get("mla_comparator"),
            "other_workloads": others or None,
            "rope_keys_variant": rope_keys or None,
        },
        "roofline": {"bound": "hbm", "kernel": "gva_decode_attention (absorb + split-K "
                     "partial + combine), per call", "achieved": round(achieved, 1),
                     "peak": hbm_peak, "unit": "GB/s",
                     "frac": m["decode_frac_of_measured_copy"],
                     "peak_source": "measured" if peaks else "fallback",
                     "traffic": profiled_traffic(w.name) if path in ("auto", "mma") else None,
                     "traffic_kernel": "decode_mma_kernel, DRAM bytes per launch (ncu)"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def S_bytes_mb(m) -> int:
    return int(round(m["bytes_per_layer"] * m["layers"] / 1e6))


def prefill_work(w, L0, n: int):
    """Algorithmic work of one chunked-prefill call on one layer: every sequence's rows
    (history and chunk) read once, sum_b (L0_b + n)(G d_h + d_r) x elem bytes; and the
    flops of scoring and weighting, each query at position p covering p + 1 positions
    with H (2 d_h + d_r) multiply-adds (the absorption excluded)."""
    elem = 2 if w.cache_dtype == "bf16" else 4
    nbytes = sum(int(l0) + n for l0 in L0) * (w.G * w.d_h + w.d_r) * elem
    pairs = sum(n * (int(l0) + 1) + n * (n - 1) // 2 for l0 in L0)
    return nbytes, 2 * w.H * (2 * w.d_h + w.d_r) * pairs


def _prefill_tc(w, n: int, path: str) -> bool:
    """True when the library's automatic path takes the tcgen05 prefill kernel."""
    rows = n * (w.H // w.G)
    return (path == "auto" and w.cache_dtype == "bf16" and w.d_h in (64, 128)
            and (rows <= 64 or (rows <= 128 and w.d_h == 64)))


def _prefill_chain(w, n: int, path: str, sms: int = 148):
    """The kernels one prefill call launches: (description, launches per call).  The
    tcgen05 kernel merges its history ranges in the last CTA of each (value group,
    sequence) when the ranges' (max, sum) of the group's rows fit its P buffers (at least
    512 M bytes for M query rows per product)."""
    if _prefill_tc(w, n, path):
        rows = n * (w.H // w.G)
        m = 64 if rows <= 64 else 128
        splits = max(2, sms // (w.G * w.B))
        if (2 * rows * splits + 2 * rows) * 4 <= 512 * m:
            return "append + absorb + tcgen05 prefill with the ranges' merge in its last CTAs", 3
        return "append + absorb + tcgen05 prefill partial + merge", 4
    return "view + append + absorb + prefill partial + merge", 5


def _prefill_design(w, n: int, path: str) -> str:
    """Which prefill kernel the library's automatic path takes for this shape."""
    if path != "auto" or w.cache_dtype != "bf16" or w.d_h not in (64, 128):
        return ("each new token run as one entry of a decode batch of B*n entries over a "
                "paged view of the cache")
    if _prefill_tc(w, n, path):
        return ("tcgen05 prefill kernel: one CTA per (history range, value group, sequence) "
                "holds the group's chunk rows, streams 128-token tiles of its rows once "
                "(TMA), S = Q V^T and O += P V accumulate in tensor memory (P's bf16 high and "
                "low parts stacked as one 128-row product), online softmax in 16 warps; "
                "ranges merged by log-sum-exp in the last CTA of each (group, sequence); "
                "a grid of more than one wave starts the longest sequences' ranges first")
    return ("mma.sync prefill kernel: each 16-token slab of a sequence's rows loaded once "
            "per CTA and scored against all the chunk's (query, head) rows, split over the "
            "history and merged by log-sum-exp")


def run_prefill(args, dist: Dist):
    """Causal chunked prefill: one step = gva_prefill_attention (append of n tokens per
    sequence, then the attention of each new token over the history and the chunk up to
    itself) on every layer, the chunk being the last n tokens of each sequence of the
    workload."""
    import numpy as np
    import torch

    import gva_inputs
    import value_only_kv_gva_b300 as gva

    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    dist.init("nccl")
    w = gva_inputs.workload(args.workload)
    c = gva_inputs.make_case(w)
    n = args.prefill
    ch = gva_inputs.make_prefill_chunk(c, n)
    L0 = ch.L0.tolist()
    nl = args.layers
    dims = gva.Dims(w.B, w.H, w.G, w.d_h, w.d_n, w.d_r,
                    gva.GVA_F32 if w.cache_dtype == "f32" else gva.GVA_BF16,
                    gva.GVA_F32 if w.q_dtype == "f32" else gva.GVA_BF16)
    offs = c.offsets.to(dev) if c.offsets is not None else None
    bt = c.block_table.to(dev) if c.block_table is not None else None
    rows = gva.Rows(w.layout, c.num_rows, T_cap=c.T_cap, offsets=offs, block_table=bt,
                    page_size=w.page_size)
    V0, K0 = c.V.to(dev), c.Kr.to(dev)
    d_in = [t.to(dev).unsqueeze(0).expand((nl,) + tuple(t.shape)).contiguous()
            for t in (ch.q_nope, ch.q_rope, ch.v_new, ch.k_new)]
    layers = []
    for li in range(nl):
        V = V0.clone() if li else V0
        K = K0.clone() if li else K0
        layers.append(dict(cache=gva.Cache(rows, V, K), M=c.M.to(dev).clone(), li=li))
    d_out = torch.empty((nl, w.B, n, w.H, w.d_h), device=dev)
    d_lse = torch.empty((nl, w.B, n, w.H), device=dev)
    L0d = ch.L0.to(dev)
    tab = gva.gva_rope_table_fill(int(c.seq_len.max()) + 1, w.d_r, w.base).to(dev)
    ws = gva.prefill_workspace(dims, n, rows, dev)
    path = args.path
    log(f"[bench] prefill {w.name}: B={w.B} n={n} history={sum(L0)} tokens layers={nl}")

    def call(L, stream=None):
        li = L["li"]
        gva.gva_prefill_attention(dims, d_in[0][li], d_in[1][li], L["M"], L0d, d_in[2][li],
                                  d_in[3][li], L["cache"], tab, w.scale, d_out[li], d_lse[li],
                                  ws, path=path, stream=stream)

    stream = torch.cuda.Stream(device=dev)
    graph = capture_list(torch, stream, layers, call)
    assert gva.gva_get_device_status() == 0
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    soak_t = time.time()
    while time.time() - soak_t < args.soak:
        for _ in range(5):
            graph.replay()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    sampler.mark("t0")
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for k in range(args.steps):
            graph.replay()
            ev[k + 1].record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    dist.barrier()
    clocks = sampler.summary(sampler.t_marks["t0"] - args.soak, sampler.t_marks["t1"])
    sampler.stop()
    secs = dist.max(ev[0].elapsed_time(ev[args.steps]) / 1e3, dev)
    step_ms = [ev[k].elapsed_time(ev[k + 1]) for k in range(args.steps)]
    us_call = secs / (args.steps * nl) * 1e6
    nbytes, flops = prefill_work(w, L0, n)
    tokens = w.B * n * nl * args.steps * dist.world
    value = tokens / secs
    peaks = measured_peaks()
    hbm_peak = peaks["hbm_gbs"] if peaks else FALLBACK_HBM_GBS
    tc_peak = peaks.get("bf16_tflops") if peaks else 1800.0
    gbs = nbytes / (us_call * 1e-6) / 1e9
    tflops = flops / (us_call * 1e-6) / 1e12

    # end to end: pinned host chunk inputs in, every layer's outputs out, the recorded plans
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    lp = PackedLoop(torch, dev, (ch.q_nope, ch.q_rope, ch.v_new, ch.k_new), nl, d_out,
                    args.e2e_chunks or 4)
    lp.record(lambda a, b, view: gva.create_prefill_plan(
        dims, n, [dict(q_nope=view(li, 0), q_rope=view(li, 1), M=layers[li]["M"],
                       v_new=view(li, 2), k_rope_new=view(li, 3), cache=layers[li]["cache"],
                       out=d_out[li], lse=d_lse[li]) for li in range(a, b)],
        L0d, tab, w.scale, ws, path=path))
    for _ in range(3):
        lp.step()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        lp.step()
    te = dist.max(time.perf_counter() - t0, dev)
    lp.close()
    e2e = {"value": round(w.B * n * nl * e2e_steps * dist.world / te, 1), "unit": "tokens/s",
           "h2d_bytes_per_step": lp.h2d_bytes, "d2h_bytes_per_step": lp.d2h_bytes,
           "steps": e2e_steps, "chunks": lp.nch,
           "how": lp.how("each the chunk's prefill through a chunk of layers, recorded once "
                         "by gva_prefill_plan_create")}

    cpu = None
    if dist.rank == 0 and not args.no_cpu_baseline:
        import oracle
        nthr = os.cpu_count() or 1
        oracle.set_threads(nthr)
        Vh, Kh = oracle._np(c.V), oracle._np(c.Kr)
        done = 0
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < args.cpu_seconds or done == 0:
            b = done % w.B
            if w.layout == "contiguous":
                Rb = oracle.Rows("ragged", offsets=np.array([b * c.T_cap, (b + 1) * c.T_cap]))
            elif w.layout == "ragged":
                Rb = oracle.Rows("ragged", offsets=c.offsets.numpy()[[b, b + 1]])
            else:
                Rb = oracle.Rows("paged", block_table=c.block_table.numpy()[[b]],
                                 page_size=w.page_size)
            oracle.gva_prefill(ch.q_nope[[b]], ch.q_rope[[b]], c.M, ch.L0[[b]], Rb, Vh, Kh,
                               w.scale, w.base, w.G)
            done += 1
        cs = time.perf_counter() - t0
        cpu = {"value": round(done * n / cs, 2), "unit": "tokens/s", "cores": oracle.get_threads(),
               "kind": "oracle",
               "sample": f"{done} whole chunks of one sequence ({n} queries, all {w.H} heads) "
                         f"of one {w.name} layer, fp64 C oracle with OpenMP over (b, h), "
                         f"{cs:.1f} s"}

    chain, per_call = _prefill_chain(w, n, path, gva.gva_num_sms())
    line = {
        "metric": f"GVA causal chunked prefill, new tokens/s ({w.name} layer, n={n} per "
                  f"sequence)",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.cache_dtype == "bf16" else "f32", "data": "synthetic",
        "config": {
            "workload": f"{w.name}: GVA chunked prefill B={w.B} n={n} H={w.H} G={w.G} "
                        f"d_h={w.d_h} d_n={w.d_n} d_r={w.d_r}, chunk = the last {n} tokens "
                        f"of each sequence; step = one prefill call on each of {nl} layers",
            "layers": nl, "history_tokens": int(sum(L0)), "us_per_layer_call": round(us_call, 3),
            "median_us_per_layer_call": round(statistics.median(step_ms) * 1e3 / nl, 3),
            "bytes_per_layer": nbytes, "flops_per_layer": flops,
            "achieved_tflops": round(tflops, 3),
            "tensor_frac_of_bf16_peak": round(tflops / tc_peak, 5) if tc_peak else None,
            "l2": f"inputs larger than L2: {nl} distinct layer caches", "path": path,
            "design": _prefill_design(w, n, path)},
        "roofline": {"bound": "hbm", "kernel": f"gva_prefill_attention ({chain}), per call",
                     "achieved": round(gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                     "peak_source": "measured" if peaks else "fallback", "traffic": None},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": nl * per_call * args.steps,
        "clocks": clocks,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


# Sources of the tensor-core decode kernel: a DRAM-traffic figure recorded with ncu is
# reported only while these files are unchanged since the capture.
KERNEL_SOURCES = ["decode_mma.cuh", "decode_simt.cuh", "common.cuh"]


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: comments and whitespace are dropped first, so
    that only a change of the code itself invalidates a recorded profile."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "value_only_kv_gva_b300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch of decode_mma_kernel on
    this workload, from the ncu summary under profiles/, or None when there is none or
    the kernel's sources changed since it was taken."""
    import re
    path = os.path.join(ROOT, "profiles", f"decode_mma_{workload}_ncu.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        m = re.search(r"traffic_bytes_per_launch=(\d+) source_hash=([0-9a-f]+)", f.read())
    if not m or m.group(2) != kernel_source_hash():
        return None
    return int(m.group(1))


def capture_list(torch, stream, items, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for it in items:
            fn(it)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for it in items:
                fn(it)
    torch.cuda.synchronize()
    return g


class PackedLoop:
    """The end-to-end loop shared by the decode and prefill legs.  Every layer's inputs
    (the tensors `srcs`, the same for each layer) sit in one 256-byte-aligned region of a
    pinned host buffer and of a device buffer, so a chunk of layers moves in one copy;
    `make_plan(a, b, view)` records layers a..b-1 as one plan, `view(li, k)` being layer
    li's device copy of srcs[k].  A step copies the inputs in, launches the plans and
    copies `d_out` back, all inside the caller's timed region.  With more than one chunk
    the copies overlap the compute: chunk i + 1's inputs arrive on one copy stream while
    chunk i computes, and chunk i's outputs leave on a second while chunk i + 1 computes."""

    def __init__(self, torch, dev, srcs, nl, d_out, nch):
        self.torch = torch
        self.stream = torch.cuda.current_stream()
        self.h2d_s, self.d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        self.srcs = srcs
        self.sizes = [t.numel() * t.element_size() for t in srcs]
        self.offs, o = [], 0
        for n in self.sizes:
            self.offs.append(o)
            o += (n + 255) // 256 * 256
        self.per_layer = o
        self.h_pack = torch.empty((nl, o), dtype=torch.uint8).pin_memory()
        for li in range(nl):
            for t, off, n in zip(srcs, self.offs, self.sizes):
                self.h_pack[li, off:off + n].copy_(t.contiguous().view(-1).view(torch.uint8))
        self.d_pack = torch.empty((nl, o), dtype=torch.uint8, device=dev)
        self.d_out = d_out
        self.h_out = torch.empty(tuple(d_out.shape), dtype=d_out.dtype).pin_memory()
        self.nch = max(1, min(nch, nl))
        bounds = [nl * i // self.nch for i in range(self.nch + 1)]
        self.chunks = [(bounds[i], bounds[i + 1]) for i in range(self.nch)]
        self.ev_in = [torch.cuda.Event() for _ in self.chunks]
        self.ev_done = [torch.cuda.Event() for _ in self.chunks]
        self.plans = []
        self.h2d_bytes = nl * o
        self.d2h_bytes = self.h_out.numel() * self.h_out.element_size()

    def view(self, li, k):
        t = self.srcs[k]
        return self.d_pack[li, self.offs[k]:self.offs[k] + self.sizes[k]].view(t.dtype).view(t.shape)

    def record(self, make_plan):
        self.plans = [make_plan(a, b, self.view) for a, b in self.chunks]

    def step(self):
        torch, stream = self.torch, self.stream
        if self.nch == 1:
            self.d_pack.copy_(self.h_pack, non_blocking=True)
            self.plans[0].launch(stream)
            self.h_out.copy_(self.d_out, non_blocking=True)
            stream.synchronize()
            return
        with torch.cuda.stream(self.h2d_s):
            for i, (a, b) in enumerate(self.chunks):
                self.d_pack[a:b].copy_(self.h_pack[a:b], non_blocking=True)
                self.ev_in[i].record(self.h2d_s)
        for i, (a, b) in enumerate(self.chunks):
            stream.wait_event(self.ev_in[i])
            self.plans[i].launch(stream)
            self.ev_done[i].record(stream)
            with torch.cuda.stream(self.d2h_s):
                self.d2h_s.wait_event(self.ev_done[i])
                self.h_out[a:b].copy_(self.d_out[a:b], non_blocking=True)
        self.d2h_s.synchronize()
        stream.synchronize()

    def close(self):
        for pl in self.plans:
            pl.close()

    def how(self, what):
        h = (f"{self.nch} gva_step_plan_launch C-ABI call(s) per step ({what}); pinned "
             "host->device inputs (one packed copy per chunk of layers) and device->host "
             "outputs of every layer inside the timed region")
        return h + (", on two copy streams overlapping the chunks' compute" if self.nch > 1 else "")


def run_e2e(args, w, c, dims, gva, torch, dev, layers, seq, pos, tab, ws, path, bytes_layer,
            dist):
    """Same metric through the public API (PackedLoop): every step copies its inputs from
    pinned host memory, launches the step plans (gva_step_plan_create recorded each chunk
    of layers' append and decode once; gva_step_plan_launch replays a chunk with one call)
    and reads every layer's output back, all inside the timed region."""
    nl = len(layers)
    d_out = torch.empty((nl, w.B, w.H, w.d_h), dtype=torch.float32, device=dev)
    d_lse = torch.empty((nl, w.B, w.H), dtype=torch.float32, device=dev)
    lp = PackedLoop(torch, dev, (c.q_nope, c.q_rope, c.v_new, c.k_new), nl, d_out,
                    args.e2e_chunks or 1)
    lp.record(lambda a, b, view: gva.create_step_plan(
        dims, [dict(q_nope=view(li, 0), q_rope=view(li, 1), v_new=view(li, 2),
                    k_rope_new=view(li, 3), M=layers[li]["M"], cache=layers[li]["cache"],
                    out=d_out[li], lse=d_lse[li]) for li in range(a, b)],
        pos, seq, tab, w.scale, ws, path=path))
    steps = max(3, min(args.steps, args.e2e_steps))
    for _ in range(3):
        lp.step()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        lp.step()
    t = dist.max(time.perf_counter() - t0, dev)
    lp.close()
    val = bytes_layer * nl * steps * dist.world / t / 1e9
    return {"value": round(val, 2), "unit": "GB/s", "h2d_bytes_per_step": lp.h2d_bytes,
            "d2h_bytes_per_step": lp.d2h_bytes, "steps": steps,
            "ms_per_step": round(t / steps * 1e3, 4), "chunks": lp.nch,
            "how": lp.how("each a chunk of layers' append + decode, recorded once by "
                          "gva_step_plan_create as a CUDA graph")}


def read_probe_gbs(gva, torch, stream, dev, gib: float = 4.0, reps: int = 10):
    """Read-only streaming ceiling of this GPU, measured in the same run: the library's
    probe kernel over a buffer larger than L2, CUDA events on the launching stream."""
    n = int(gib * (1 << 30)) // 16 * 16
    buf = torch.ones(n // 4, dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            gva.gva_read_probe(buf, sink, stream=stream)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            gva.gva_read_probe(buf, sink, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize()
    secs = e0.elapsed_time(e1) * 1e-3 / reps
    del buf
    return round(n / secs / 1e9, 1)


def oracle_sample(w, c, budget_s, threads=None):
    """Run the fp64 oracle over whole sequences of one layer until ~budget_s elapses;
    returns (seconds, cache bytes read, description, threads)."""
    import numpy as np

    import oracle
    rows_all = {"contiguous": None}
    nthr = threads or os.cpu_count() or 1
    oracle.set_threads(nthr)
    V = oracle._np(c.V)
    K = oracle._np(c.Kr)
    done_bytes = 0
    t0 = time.perf_counter()
    nseq = 0
    b = 0
    while time.perf_counter() - t0 < budget_s or nseq == 0:
        sample = [b % w.B]
        if w.layout == "contiguous":
            R = oracle.Rows("ragged", offsets=np.array([sample[0] * c.T_cap, 0]))
        elif w.layout == "ragged":
            R = oracle.Rows("ragged", offsets=np.array([int(c.offsets[sample[0]]), 0]))
        else:
            R = oracle.Rows("paged", block_table=c.block_table.numpy()[sample],
                            page_size=w.page_size)
        sl = c.seq_len.numpy()[sample].astype(np.int64)
        oracle.gva_decode(c.q_nope[sample], c.q_rope[sample], c.M, sl, R, V, K, w.scale, w.base,
                          w.G)
        done_bytes += algorithmic_bytes(w, sl)
        nseq += 1
        b += 1
    secs = time.perf_counter() - t0
    del rows_all
    return secs, done_bytes, nseq, oracle.get_threads()


def oracle_baseline(w, c, budget_s=10.0):
    secs, nbytes, nseq, thr = oracle_sample(w, c, budget_s)
    s1, b1, n1, _ = oracle_sample(w, c, max(1.0, budget_s / 4), threads=1)
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": thr,
            "kind": "oracle",
            "sample": f"{nseq} whole sequences of one {w.name} layer (all {w.H} heads each), "
                      f"fp64 C oracle with OpenMP over (b, h), {secs:.1f} s",
            "single_thread_value": round(b1 / s1 / 1e9, 4),
            "single_thread_sample": f"{n1} whole sequences, 1 thread, {s1:.1f} s"}


def run_reference(args, dist: Dist):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    if dist.world > 1 and dist.rank != 0:
        return
    import gva_inputs
    w = gva_inputs.workload(args.workload)
    c = gva_inputs.make_case(w)
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps))
    for _ in range(args.warmup):
        oracle_sample(w, c, 0.0)
    tot_s = tot_b = 0.0
    nseq = 0
    thr = 1
    for _ in range(args.steps):
        s, b, n, thr = oracle_sample(w, c, per_step)
        tot_s += s
        tot_b += b
        nseq += n
    val = tot_b / tot_s / 1e9
    desc = (f"{nseq} whole sequences of one {w.name} layer over {args.steps} steps "
            f"(~{per_step:.1f} s each), fp64 C oracle, OpenMP over (b, h)")
    line = {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": "GB/s",
            "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: GVA decode layer B={w.B} H={w.H} G={w.G} "
                                   f"d_h={w.d_h} d_r={w.d_r}, oracle on host cores"},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": thr,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="350m",
                    choices=["tiny", "350m", "ragged", "long", "paged"])
    ap.add_argument("--layers", type=int, default=0,
                    help="layers per step (0 = enough distinct caches to exceed L2)")
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "mma"])
    ap.add_argument("--soak", type=float, default=1.0, help="untimed load before timing (s)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="plans per step in the end-to-end leg, the copies overlapping the "
                         "compute; 0: 1 for the decode step (bound by host calls), 4 for the "
                         "prefill (bound by its 32 MB of copies)")
    ap.add_argument("--no-gqa", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--others", nargs="*", default=["long", "paged", "ragged"],
                    help="further workloads measured in the same run (config.other_workloads)")
    ap.add_argument("--no-others", action="store_true")
    ap.add_argument("--no-rope-keys", action="store_true",
                    help="skip the variant with RoPE on the reconstructed key "
                         "(config.rope_keys_variant)")
    ap.add_argument("--rope-keys", nargs="*", default=["350m", "long"],
                    help="workload shapes of config.rope_keys_variant")
    ap.add_argument("--rope-keys-only", action="store_true",
                    help="measure only the variant with RoPE on the reconstructed key and "
                         "print its figures (a profiling aid; not the bench line)")
    ap.add_argument("--prefill", type=int, default=0,
                    help="time the causal chunked prefill of this many new tokens per "
                         "sequence instead of the decode step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.layers == 0:
        import gva_inputs
        args.layers = default_layers(gva_inputs.workload(args.workload))
    dist = Dist()
    if args.impl == "reference":
        run_reference(args, dist)
    elif args.prefill > 0:
        run_prefill(args, dist)
    else:
        run_ours(args, dist)


if __name__ == "__main__":
    main()
