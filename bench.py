#!/usr/bin/env python3
"""Benchmark of the quantized MoE layer on GB300.

One step = one MoE-layer forward at decode batch size (router + top-k,
dispatch, gate/up + SwiGLU, down, combine) on the NVFP4 decode layer:
hidden 2048, 512 routed experts, top-10, intermediate 512, FP8 block-128
shared expert (intermediate 512).  The headline value is algorithmic weight
bytes per second at batch 8 (the bytes of the router, the shared expert and
every distinct routed expert the batch touches, each read once); per-batch
results for 1, 4 and 8 tokens ride along.

Synthetic inputs: N(0, 0.02) FP32 weights quantised per format, N(0, 1) BF16
activations, seeded.  L2 is defeated by rotating R copies of the layer (each
at its own addresses) so one rotation touches at least three times the L2
size, and by a new token batch every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the FP64 CPU oracle (the reference implementation of
this build) on the same workload and metric.  With N > 1 (torchrun), every
rank runs an independent replica (the layer does not shard across ranks in
this build); value sums the ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE-layer weight GB/s & tokens/s at batch 1/8; % of HBM (decode) / FP4 peak"
WORKLOAD = "decode_nvfp4"
FALLBACK_HBM_GBS = 6800.0
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one gate/up launch at batch 8 on the
# decode_nvfp4 workload, from one ncu capture of the current kernel; None while the kernel has
# changed since the counters were taken.
GATEUP_TRAFFIC_BYTES = 93324800  # 90.69 MB read + 2.63 MB written in the full-section capture of gate/up
# kernels one decode layer call launches: router logits (exact, every SM), top-k selection (one CTA
# per token), gate/up, down, combine
DECODE_KERNELS_PER_CALL = 5


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s): the measured burst figure, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def _once(self):
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
            if out.returncode == 0:
                self.rows.append(out.stdout.strip())
        except Exception:
            pass

    def start(self):
        self._once()
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append(line.strip())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        self._once()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_ranks(ms: float, work: float, dist=None, device: str = "cpu"):
    """Whole-job timing over replicas: the slowest rank's time and the sum of every rank's work
    (a single process returns its own numbers)."""
    if dist is None:
        return ms, work
    import torch
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    w = torch.tensor([work], device=device, dtype=torch.float64)
    dist.all_reduce(w)
    return float(t.item()), float(w.item())


def _bytes_per_call(host, cnt_rows):
    """Algorithmic weight bytes of one call from its per-expert pair counts."""
    per_expert = host.expert_bytes()
    fixed = host.router_bytes() + host.shared_bytes()
    return [fixed + int(np.count_nonzero(c)) * per_expert for c in cnt_rows]


def _clone_layer(q, base):
    def clone(qw):
        return q.QWeight(qw.data.clone(), qw.scales.clone(),
                         None if qw.tensor_scale is None else qw.tensor_scale.clone())
    return q.Layer(base.hidden, base.inter, base.n_experts, base.top_k, base.fmt, base.router_w.clone(),
                   None if base.router_bias is None else base.router_bias.clone(), clone(base.gate),
                   clone(base.up), clone(base.down), base.shared_fmt, base.shared_inter,
                   clone(base.shared_gate) if base.shared_gate else None,
                   clone(base.shared_up) if base.shared_up else None,
                   clone(base.shared_down) if base.shared_down else None)


def _median_replays(torch, graph, stream, n):
    """Replay `graph` n times on `stream`, each bracketed by its own CUDA events; ms per replay."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            graph.replay()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def measure_decode(args, name, batches, world, rank, local, dist, peak, peak_kind, headline_T=None):
    """One decode workload: per batch size, K consecutive layer calls (one CUDA graph, rotating
    R layer copies and NB token batches) timed as one measurement, replayed at least 20 times;
    the median replay gives the per-call time.  Per-kernel times come from a second graph with
    event-record nodes between the kernels."""
    import torch
    import quantized_moe_decode_router_gb300 as q
    cfg = synth.CONFIGS[name]
    t0 = time.time()
    host = synth.make_layer(cfg, seed=rank)
    gen_s = time.time() - t0
    base = q.to_device(host, f"cuda:{local}")
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    Tmax = max(batches)
    fixed = host.router_bytes() + host.shared_bytes()
    min_call = fixed + min(cfg.k, cfg.E) * host.expert_bytes()
    layer_bytes = fixed + cfg.E * host.expert_bytes()
    R = args.instances or max(2, min(-(-3 * l2 // min_call), int(args.mem_gb * 1e9 // layer_bytes)))
    layers = [base] + [_clone_layer(q, base) for _ in range(R - 1)]
    NB = args.token_batches
    K = max(1, min(args.steps, 1024))
    stream = torch.cuda.Stream()
    per_exp_gu = sum(m.nbytes() // m.E for m in (host.gate, host.up))
    per_exp_dn = host.down.nbytes() // host.down.E
    s_gu = (host.shared_gate.nbytes() + host.shared_up.nbytes()) if host.shared_gate else 0
    s_dn = host.shared_down.nbytes() if host.shared_gate else 0
    results, extra = {}, {}
    for T in batches:
        xs = [torch.from_numpy(synth.make_tokens(cfg, T, seed=1000 + rank, batch=i).view(np.int16)).cuda()
              for i in range(NB)]
        ys = torch.zeros((T, cfg.H), dtype=torch.int16, device="cuda")
        ws = torch.empty(q.workspace_size(base, Tmax), dtype=torch.uint8, device="cuda")
        q.workspace_init(ws)
        # the library's own routing of every token batch -> touched experts -> algorithmic bytes
        cnt = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
        cnts = []
        for i in range(NB):
            q.moe_route(base, xs[i], T, expert_cnt=cnt, ws=ws)
            cnts.append(cnt.cpu().numpy().copy())
        touched = [int(np.count_nonzero(c)) for c in cnts]
        bytes_b = [fixed + n * host.expert_bytes() for n in touched]
        torch.cuda.synchronize()

        def call(i, s):
            q.moe_decode_forward(layers[i % R], xs[i % NB], T, ys, ws, stream=s)

        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(3):
                call(i, stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(K):
                    call(i, stream)
        bytes_graph = sum(bytes_b[i % NB] for i in range(K))
        warm = max(3, -(-args.warmup // K))
        _median_replays(torch, g, stream, warm)
        reps = max(20, args.replays)
        headline = T == headline_T
        sampler = ClockSampler(local) if headline else None
        if sampler:
            sampler.start()
            time.sleep(0.3)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ms_list = _median_replays(torch, g, stream, reps)
        if dist:
            dist.barrier()
        if sampler:
            extra["clocks"] = sampler.stop()
        ms_med = statistics.median(ms_list)
        ms_all, total_bytes = aggregate_ranks(ms_med, float(bytes_graph), dist, "cuda")
        us_call = ms_all * 1e3 / K
        gbs = total_bytes / (ms_all * 1e-3) / 1e9
        res = {"us_per_layer": round(us_call, 3), "weight_GBps": round(gbs, 1),
               "tokens_per_s": round(world * T * K / (ms_all * 1e-3), 1), "hbm_frac": round(gbs / world / peak, 4),
               "bytes_per_layer": int(np.mean(bytes_b)), "experts_touched": round(float(np.mean(touched)), 1),
               "steps": K, "replays": reps,
               "us_per_layer_min_max": [round(min(ms_list) * 1e3 / K, 3), round(max(ms_list) * 1e3 / K, 3)]}
        # per-kernel times: event-record nodes between the kernels of each call
        n = 64
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
        for row in evs:          # create the CUDA events (torch creates them lazily on first record)
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
        gt = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gt, stream=stream):
            for i in range(n):
                q.moe_decode_forward_timed(layers[i % R], xs[i % NB], T, ys, ws, evs[i], stream=stream)
        for _ in range(2):
            with torch.cuda.stream(stream):
                gt.replay()
        torch.cuda.synchronize()
        dur = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(3)] for i in range(n)])
        avg = dur.mean(axis=0) * 1e3  # us per launch: router (both stages), gate/up, down + combine
        gu_bytes = float(np.mean([touched[i % NB] * per_exp_gu + s_gu for i in range(n)]))
        dn_bytes = float(np.mean([touched[i % NB] * per_exp_dn + s_dn for i in range(n)]))
        rt_bytes = host.router_bytes()
        res["kernel_us"] = {"router": round(avg[0], 3), "gateup": round(avg[1], 3), "down_combine": round(avg[2], 3)}
        res["kernel_hbm_frac"] = {"router": round(rt_bytes / (avg[0] * 1e-6) / 1e9 / peak, 4),
                                  "gateup": round(gu_bytes / (avg[1] * 1e-6) / 1e9 / peak, 4),
                                  "down_combine": round(dn_bytes / (avg[2] * 1e-6) / 1e9 / peak, 4)}
        results[T] = res
        if headline:
            ach = gu_bytes / (avg[1] * 1e-6) / 1e9
            extra["roofline"] = {
                "kernel": "gateup_kernel (decode gate/up + SwiGLU GEMV)", "bound": "hbm", "achieved": round(ach, 1),
                "peak": peak, "peak_kind": f"{peak_kind} (HBM copy, burst)", "unit": "GB/s",
                "frac": round(ach / peak, 4), "traffic": GATEUP_TRAFFIC_BYTES, "bytes_per_launch": int(gu_bytes),
                "kernel_us": res["kernel_us"]}
            # end to end through the public API with host buffers (pinned): K steps per measurement,
            # each step copies its tokens in and its output back
            xh = [torch.from_numpy(synth.make_tokens(cfg, T, seed=2000 + rank, batch=i).view(np.int16)).pin_memory()
                  for i in range(NB)]
            yh = torch.empty((T, cfg.H), dtype=torch.int16).pin_memory()
            xd = torch.empty((T, cfg.H), dtype=torch.int16, device="cuda")

            def e2e_steps(nsteps):
                for i in range(nsteps):
                    xd.copy_(xh[i % NB], non_blocking=True)
                    q.moe_decode_forward(layers[i % R], xd, T, ys, ws)
                    yh.copy_(ys, non_blocking=True)
            e2e_steps(3)
            torch.cuda.synchronize()
            e_ms = []
            for _ in range(5):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                e2e_steps(K)
                e1.record()
                torch.cuda.synchronize()
                e_ms.append(e0.elapsed_time(e1))
            ems = statistics.median(e_ms)
            eb = sum(bytes_b[i % NB] for i in range(K))
            extra["e2e"] = {"value": round(eb / (ems * 1e-3) / 1e9, 1), "unit": "GB/s", "steps": K,
                            "us_per_step": round(ems * 1e3 / K, 2), "tokens_per_s": round(T * K / (ems * 1e-3), 1),
                            "h2d_bytes_per_step": T * cfg.H * 2, "d2h_bytes_per_step": T * cfg.H * 2,
                            "measurements": 5, "statistic": "median"}
        del g, gt
        torch.cuda.synchronize()
    st = q.moe_check(ws)
    if st != 0:
        raise RuntimeError(f"device-side error: {q.status_string(st)}")
    info = {"workload": workload_name(cfg), "instances_rotated": R,
            "l2": f"inputs larger than L2: {R} layer copies rotated, at least {R * min_call / 1e6:.0f} MB "
                  f"touched per rotation vs L2 {l2 / 1e6:.0f} MB",
            "layer_gen_s": round(gen_s, 1), "batches": {str(T): r for T, r in results.items()}}
    del layers, base
    torch.cuda.empty_cache()
    return info, extra


def run_ours(args, world, rank, local):
    import torch
    import quantized_moe_decode_router_gb300 as q
    from quantized_moe_decode_router_gb300 import build as qbuild

    qbuild.build()
    q.load()
    torch.cuda.set_device(local)
    dev_name = torch.cuda.get_device_name(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    peak, peak_kind = _peaks()
    batches = [int(b) for b in args.batches.split(",")]
    Th = max(batches)
    head, extra = measure_decode(args, args.workload, batches, world, rank, local, dist, peak, peak_kind, Th)
    others = {}
    for name in [w for w in args.more_workloads.split(",") if w and w != args.workload]:
        cfg = synth.CONFIGS[name]
        others[name], _ = measure_decode(args, name, list(cfg.batches), world, rank, local, dist, peak, peak_kind)
    hb = head["batches"][str(Th)]
    out = {
        "metric": METRIC, "value": hb["weight_GBps"], "unit": "GB/s", "n_gpus": world,
        "steps": hb["steps"], "warmup": args.warmup, "ms_per_step": round(hb["us_per_layer"] / 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": f"synthetic ({DATA_DESC[args.workload]}; N(0,1) bf16 tokens; seeded)",
        "config": {"workload": f"{head['workload']}, batch {Th} tokens", "batch_tokens": Th,
                   "instances_rotated": head["instances_rotated"], "l2": head["l2"],
                   "timing": f"one measurement = one CUDA graph of {hb['steps']} consecutive layer calls "
                             f"(K = --steps); median of {hb['replays']} measurements",
                   "parallelism": "replicas" if world > 1 else "1 GPU", "gpu": dev_name,
                   "layer_gen_s": head["layer_gen_s"]},
        "tokens_per_s": hb["tokens_per_s"], "hbm_frac": hb["hbm_frac"],
        "batches": head["batches"],
        "workloads": {name: {"workload": o["workload"], "data": DATA_DESC[name], "batches": o["batches"],
                             "instances_rotated": o["instances_rotated"], "l2": o["l2"]}
                      for name, o in others.items()},
        "roofline": extra.get("roofline"), "clocks": extra.get("clocks"), "e2e": extra.get("e2e"),
        "gpu_launches": DECODE_KERNELS_PER_CALL * hb["steps"],
    }
    return out


PREFILL_EXTRA = {
    # the MXFP4 and int4 g64 (+ int8 g64 shared) decode layers at the prefill workload's token count
    "prefill_mxfp4": lambda: synth.CONFIGS["decode_mxfp4"].with_(name="prefill_mxfp4", batches=(4096,)),
    "prefill_int4": lambda: synth.CONFIGS["decode_int4"].with_(name="prefill_int4", batches=(4096,)),
    # the prefill workload's shape with AutoRound int4 g128 routed experts (the fold-scales lever's case)
    "prefill_int4g128": lambda: synth.CONFIGS["prefill_nvfp4"].with_(name="prefill_int4g128",
                                                                     fmt=synth.configs.FMT_INT4_G128),
    # the prefill workload's shape with FP8 b128 routed experts (the FP8-activation lever's case)
    "prefill_fp8": lambda: synth.CONFIGS["prefill_nvfp4"].with_(name="prefill_fp8", fmt=synth.configs.FMT_FP8_B128),
}


# the prefill workloads a default run measures beside prefill_nvfp4
MORE_PREFILL = "prefill_mxfp4,prefill_int4,prefill_int4g128,prefill_fp8"


def prefill_config(name: str):
    return PREFILL_EXTRA[name]() if name in PREFILL_EXTRA else synth.CONFIGS[name]


def _prefill_times(torch, q, lay, xs, T, y, ws, stream, act_quant, reps, G=6, fold_scales=0, fp8_act=0):
    """Median whole-layer time (graph of G calls, `reps` replays) and per-stage event times."""
    NB = len(xs)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(3):
            q.moe_prefill_forward(lay, xs[i % NB], T, y, ws, stream=stream, act_quant=act_quant,
                                  fold_scales=fold_scales, fp8_act=fp8_act)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                q.moe_prefill_forward(lay, xs[i % NB], T, y, ws, stream=stream, act_quant=act_quant,
                                  fold_scales=fold_scales, fp8_act=fp8_act)
        for _ in range(2):
            g.replay()
    torch.cuda.synchronize()
    ms_list = _median_replays(torch, g, stream, reps)
    us = statistics.median(ms_list) * 1e3 / G
    # per-stage times: event-record nodes between the launches
    n = 6
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    gt = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gt, stream=stream):
        for i in range(n):
            q.moe_prefill_forward_timed(lay, xs[i % NB], T, y, ws, evs[i], stream=stream, act_quant=act_quant,
                                        fold_scales=fold_scales, fp8_act=fp8_act)
    with torch.cuda.stream(stream):
        gt.replay()
    torch.cuda.synchronize()
    dur = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(7)] for i in range(n)]).mean(axis=0) * 1e3
    st = q.moe_check(ws)
    if st != 0:
        raise RuntimeError(f"device-side error: {q.status_string(st)}")
    return us, dur


def run_prefill(args, local, peak_bf16, peak_kind, name="prefill_nvfp4", tokens=0, w4a4=True):
    """One prefill workload: whole-layer time through moe_prefill_forward, per-stage event times and the
    grouped GEMMs' tensor throughput, for the exact chain, the W4A4 lever (NVFP4 and MXFP4 layers), the
    fold-scales lever (layers with int8 g64, FP8 b128 or int4 g128 experts) and the FP8-activation lever
    (layers with FP8 b128 experts)."""
    import torch
    import quantized_moe_decode_router_gb300 as q
    cfg = prefill_config(name)
    T = tokens or cfg.batches[0]
    host = synth.make_layer(cfg, seed=0)
    lay = q.to_device(host, f"cuda:{local}")
    NB = 3
    xs = [torch.from_numpy(synth.make_tokens(cfg, T, seed=4000, batch=i).view(np.int16)).cuda() for i in range(NB)]
    y = torch.zeros((T, cfg.H), dtype=torch.int16, device="cuda")
    ws = torch.empty(q.workspace_size(lay, T), dtype=torch.uint8, device="cuda")
    q.workspace_init(ws)
    cnt = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    touched = []
    for i in range(NB):
        q.moe_route(lay, xs[i], T, expert_cnt=cnt, ws=ws)
        touched.append(int(np.count_nonzero(cnt.cpu().numpy())))
    stream = torch.cuda.Stream()
    G = 6
    reps = max(20, args.prefill_steps // G)
    us, dur = _prefill_times(torch, q, lay, xs, T, y, ws, stream, 0, reps, G)
    names = ["router_logits", "router_topk", "dispatch", "gateup_gemm", "h_convert", "down_gemm", "combine"]
    pairs = T * cfg.k
    flops = pairs * 6.0 * cfg.H * cfg.I
    gemm_us = dur[3] + dur[5]
    tflops = flops / (gemm_us * 1e-6) / 1e12
    fp4_peak = peak_bf16 * 13.5 / 2.25   # derived: the measured dense bf16 peak x the nominal FP4/bf16 ratio
    fp4_kind = f"derived: {peak_kind} bf16 burst {peak_bf16} TFLOP/s x 13.5/2.25 (nominal dense FP4/bf16)"
    wbytes = host.router_bytes() + np.mean(touched) * host.expert_bytes()
    zipf = f", Zipf router bias s={cfg.zipf_s}" if cfg.zipf_s else ""
    # the GEMMs' own HBM roofline: at about T*k/E tokens per expert each weight byte feeds few FLOP, so
    # the weight stream bounds them (weight bytes of the touched experts / the GEMM's event time)
    gu_bytes = np.mean(touched) * sum(m.nbytes() // m.E for m in (host.gate, host.up))
    dn_bytes = np.mean(touched) * (host.down.nbytes() // host.down.E)
    if cfg.shared_fmt:
        gu_bytes += host.shared_gate.nbytes() + host.shared_up.nbytes()
        dn_bytes += host.shared_down.nbytes()
    hbm = _peaks()[0]
    gemm_hbm = {"gateup_GBps": round(gu_bytes / (dur[3] * 1e-6) / 1e9, 1),
                "down_GBps": round(dn_bytes / (dur[5] * 1e-6) / 1e9, 1),
                "gateup_frac_hbm": round(gu_bytes / (dur[3] * 1e-6) / 1e9 / hbm, 4),
                "down_frac_hbm": round(dn_bytes / (dur[5] * 1e-6) / 1e9 / hbm, 4),
                "weight_bytes_gateup": int(gu_bytes), "weight_bytes_down": int(dn_bytes),
                "flop_per_weight_byte": round(flops / (gu_bytes + dn_bytes), 1),
                "hbm_bound_tflops": round(flops / (gu_bytes + dn_bytes) * hbm / 1e3, 1)}
    shared = f" + {FMT_TEXT[cfg.shared_fmt]} shared expert I={cfg.shared_I}" if cfg.shared_fmt else ""
    if cfg.shared_fmt:
        flops += T * 6.0 * cfg.H * cfg.shared_I
        tflops = flops / (gemm_us * 1e-6) / 1e12
        wbytes += host.shared_bytes()
    out = {
        "workload": f"{name}: {FMT_TEXT[cfg.fmt]} MoE layer H={cfg.H} E={cfg.E} top-{cfg.k} I={cfg.I}{shared}, "
                    f"{T} tokens{zipf}",
        "us_per_layer": round(us, 1), "tokens_per_s": round(T / (us * 1e-6), 1),
        "kernel_us": {k: round(float(v), 2) for k, v in zip(names, dur)},
        "experts_touched": float(np.mean(touched)),
        "gemm": {"path": f"exact chain: tcgen05 kind::f16, {FMT_TEXT[cfg.fmt]} decoded in shared memory",
                 "flops_per_layer": flops, "achieved_tflops": round(tflops, 1),
                 "frac_f16_peak": round(tflops / peak_bf16, 4), "f16_peak_tflops": peak_bf16,
                 "frac_fp4_peak": round(tflops / fp4_peak, 4), "fp4_peak_tflops": round(fp4_peak, 1),
                 "peak_kind": peak_kind, "fp4_peak_kind": fp4_kind, "hbm": gemm_hbm},
        "weight_GBps": round(wbytes / (us * 1e-6) / 1e9, 1),
        "graph": f"CUDA graph of {G} layer calls; median of {reps} replays",
    }
    aq = {synth.configs.FMT_NVFP4: 1, synth.configs.FMT_MXFP4: 2}.get(cfg.fmt, 0)
    if w4a4 and aq and not cfg.shared_fmt:
        # the W4A4 lever (act_quant 1: NVFP4 activations, 2: MXFP4 activations): block-scaled FP4 GEMMs
        ws4 = torch.empty(q.workspace_size(lay, T, aq), dtype=torch.uint8, device="cuda")
        q.workspace_init(ws4)
        us4, dur4 = _prefill_times(torch, q, lay, xs, T, y, ws4, stream, aq, reps, G)
        gemm4_us = dur4[3] + dur4[5]
        tflops4 = flops / (gemm4_us * 1e-6) / 1e12
        out["w4a4"] = {
            "path": (f"{FMT_TEXT[cfg.fmt]} activations (lever, act_quant={aq}): tcgen05 kind::mxf4nvf4 "
                     f"block-scaled GEMMs ({'UE8M0, scale_vec::2X' if aq == 2 else 'UE4M3, scale_vec::4X'})"),
            "us_per_layer": round(us4, 1), "tokens_per_s": round(T / (us4 * 1e-6), 1),
            "kernel_us": {k: round(float(v), 2) for k, v in zip(
                ["router_logits", "router_topk", "dispatch_quantise", "gateup_gemm", "-", "down_gemm",
                 "combine"], dur4) if k != "-"},
            "achieved_tflops": round(tflops4, 1), "frac_fp4_peak": round(tflops4 / fp4_peak, 4),
            "fp4_peak_tflops": round(fp4_peak, 1), "peak_kind": fp4_kind,
            "hbm": {"gateup_GBps": round(gu_bytes / (dur4[3] * 1e-6) / 1e9, 1),
                    "down_GBps": round(dn_bytes / (dur4[5] * 1e-6) / 1e9, 1),
                    "gateup_frac_hbm": round(gu_bytes / (dur4[3] * 1e-6) / 1e9 / hbm, 4),
                    "down_frac_hbm": round(dn_bytes / (dur4[5] * 1e-6) / 1e9 / hbm, 4)}}
    fold_fmts = (synth.configs.FMT_INT8_G64, synth.configs.FMT_FP8_B128, synth.configs.FMT_INT4_G128)
    on = [w for w, f in (("routed", cfg.fmt), ("shared", cfg.shared_fmt)) if f in fold_fmts]
    if on:
        # the fold-scales lever: group scales folded into BF16 weights, one FP32 accumulator
        usf, durf = _prefill_times(torch, q, lay, xs, T, y, ws, stream, 0, reps, G, fold_scales=1)
        tflf = flops / ((durf[3] + durf[5]) * 1e-6) / 1e12
        out["fold_scales"] = {
            "path": (f"fold-scales lever (fold_scales=1) on the {' and '.join(on)} experts: bf16(code x group "
                     f"scale) weights against BF16 tokens, one FP32 accumulator, tcgen05 kind::f16 bf16 operands"),
            "us_per_layer": round(usf, 1), "tokens_per_s": round(T / (usf * 1e-6), 1),
            "kernel_us": {k: round(float(v), 2) for k, v in zip(names, durf)},
            "achieved_tflops": round(tflf, 1), "frac_f16_peak": round(tflf / peak_bf16, 4),
            "vs_exact_chain": round(us / usf, 3)}
    on8 = [w for w, f in (("routed", cfg.fmt), ("shared", cfg.shared_fmt)) if f == synth.configs.FMT_FP8_B128]
    if on8:
        # the FP8-activation lever: E4M3 x E4M3 MMAs, weight and activation block scales per 128-K group
        us8, dur8 = _prefill_times(torch, q, lay, xs, T, y, ws, stream, 0, reps, G, fp8_act=1)
        tfl8 = flops / ((dur8[3] + dur8[5]) * 1e-6) / 1e12
        fp8_peak = peak_bf16 * 4.5 / 2.25   # derived: the measured dense bf16 peak x the nominal FP8/bf16 ratio
        out["fp8_act"] = {
            "path": (f"FP8-activation lever (fp8_act=1) on the {' and '.join(on8)} experts: per-token 1x128 E4M3 "
                     f"activations, tcgen05 kind::f8f6f4 E4M3 x E4M3, scales per 128-K group in FP32"),
            "us_per_layer": round(us8, 1), "tokens_per_s": round(T / (us8 * 1e-6), 1),
            "kernel_us": {k: round(float(v), 2) for k, v in zip(
                ["router_logits", "router_topk", "dispatch_quantise", "gateup_gemm", "h_quantise", "down_gemm",
                 "combine"], dur8)},
            "achieved_tflops": round(tfl8, 1), "frac_fp8_peak": round(tfl8 / fp8_peak, 4),
            "fp8_peak_tflops": round(fp8_peak, 1),
            "fp8_peak_kind": f"derived: {peak_kind} bf16 burst {peak_bf16} TFLOP/s x 4.5/2.25 (nominal dense FP8/bf16)",
            "vs_exact_chain": round(us / us8, 3)}
    return out


FMT_TEXT = {1: "NVFP4", 2: "MXFP4", 3: "int4 g64", 4: "int8 g64", 5: "FP8 b128", 6: "int4 g128"}
DATA_DESC = {
    "tiny_nvfp4": "N(0,0.02) weights quantised NVFP4",
    "decode_nvfp4": "N(0,0.02) weights quantised NVFP4 routed / FP8 b128 shared",
    "decode_mxfp4": "N(0,0.02) weights quantised MXFP4",
    "decode_int4": "N(0,0.02) weights quantised int4 g64 routed / int8 g64 shared",
    "prefill_nvfp4": "N(0,0.02) weights quantised NVFP4, Zipf router bias s=1.1",
    "prefill_int4g128": "N(0,0.02) weights quantised int4 g128 (AutoRound layout), Zipf router bias s=1.1",
    "prefill_fp8": "N(0,0.02) weights quantised FP8 b128, Zipf router bias s=1.1",
}


def workload_name(cfg) -> str:
    shared = (f" + {FMT_TEXT[cfg.shared_fmt]} shared expert I={cfg.shared_I}" if cfg.shared_fmt else "")
    return f"{cfg.name}: {FMT_TEXT[cfg.fmt]} MoE layer H={cfg.H} E={cfg.E} top-{cfg.k} I={cfg.I}{shared}"


def run_reference(args, seconds_budget: float = 180.0):
    """The oracle, as it stands, timed on the host cores, on the GPU arm's headline
    workload and metric: one step is one whole layer call on one batch of T tokens (the
    router with exact logits, top-k and dispatch, the shared expert, every routed expert
    segment, the weighted combine), successive steps on successive token batches.  W
    untimed steps, then K timed ones, stopping early if the timed steps exceed
    `seconds_budget` (the line reports the steps actually timed).  value = weight bytes
    of the timed calls / time."""
    from oracle import moe as M
    cfg = synth.CONFIGS[args.workload]
    T = max(int(b) for b in args.batches.split(","))
    host = synth.make_layer(cfg, seed=0)

    def step(b):
        x = synth.make_tokens(cfg, T, seed=3000, batch=b)
        ref = M.layer_forward(host, x)
        return host.router_bytes() + host.shared_bytes() + int(np.count_nonzero(ref["expert_cnt"])) * \
            host.expert_bytes()

    for b in range(args.warmup):
        step(b)
    byts, n = 0, 0
    t0 = time.time()
    for b in range(args.steps):
        byts += step(args.warmup + b)
        n += 1
        if time.time() - t0 > seconds_budget:
            break
    dt = time.time() - t0
    cores = len(os.sched_getaffinity(0))
    value = round(byts / dt / 1e9, 4)
    sample = (f"{n} whole layer calls of {T} tokens on {cfg.name} (FP64 numpy oracle, BLAS threads = {cores}; "
              f"{args.warmup} untimed first)")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": n, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / max(1, n), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": f"synthetic ({DATA_DESC[args.workload]}; N(0,1) bf16 tokens; seeded)",
            "config": {"workload": f"{workload_name(cfg)}, batch {T} tokens", "batch_tokens": T,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
                             "seconds": round(dt, 2)},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_cpu_baseline(args, seconds_budget: float = 20.0):
    """The oracle, as it stands, on a bounded sample of the workload (rank 0 only)."""
    from oracle import moe as M
    cfg = synth.CONFIGS[args.workload]
    T = max(int(b) for b in args.batches.split(","))
    host = synth.make_layer(cfg, seed=0)
    n = 0
    byts = 0
    t0 = time.time()
    while True:
        x = synth.make_tokens(cfg, T, seed=3000, batch=n)
        ref = M.layer_forward(host, x)
        byts += host.router_bytes() + host.shared_bytes() + int(np.count_nonzero(ref["expert_cnt"])) * \
            host.expert_bytes()
        n += 1
        if time.time() - t0 > seconds_budget or n >= args.cpu_batches:
            break
    dt = time.time() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": round(byts / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} layer calls of {T} tokens on {cfg.name} (FP64 numpy oracle, BLAS threads = {cores}, "
                      f"decode single-threaded)", "seconds": round(dt, 2), "tokens_per_s": round(n * T / dt, 2)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128, help="layer calls per timed measurement (K)")
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--replays", type=int, default=30, help="timed measurements per batch size (>= 20)")
    ap.add_argument("--more-workloads", default="decode_mxfp4,decode_int4",
                    help="further decode workloads measured at their own batch sizes")
    ap.add_argument("--mem-gb", type=float, default=40.0, help="device memory budget for the rotated layer copies")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--batches", default="1,4,8")
    ap.add_argument("--instances", type=int, default=0)
    ap.add_argument("--token-batches", type=int, default=64)
    ap.add_argument("--cpu-batches", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill workload's measurement")
    ap.add_argument("--prefill-steps", type=int, default=60)
    ap.add_argument("--more-prefill", default=MORE_PREFILL,
                    help="further prefill workloads measured beside prefill_nvfp4 (the exact chain and the levers "
                         "that apply to their formats)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="measure only the prefill workload (e.g. at a small --prefill-tokens for a profiler)")
    ap.add_argument("--prefill-tokens", type=int, default=0, help="token count of the prefill workloads (0: 4096)")
    args = ap.parse_args()
    world, rank, local = _dist()
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return
    if args.prefill_only:
        pk, pkk = _bf16_peak()
        res = {"prefill": run_prefill(args, local, pk, pkk, tokens=args.prefill_tokens)}
        for name in filter(None, args.more_prefill.split(",")):
            res[name] = run_prefill(args, local, pk, pkk, name, tokens=args.prefill_tokens)
        if rank == 0:
            print(json.dumps(res))
        return
    out = run_ours(args, world, rank, local)
    if world == 1 and not args.no_prefill:
        pk, pkk = _bf16_peak()
        out["prefill"] = run_prefill(args, local, pk, pkk, tokens=args.prefill_tokens)
        more = {}
        for name in filter(None, args.more_prefill.split(",")):
            more[name] = run_prefill(args, local, pk, pkk, name, tokens=args.prefill_tokens)
        if more:
            out["prefill_more"] = more
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = run_cpu_baseline(args)
    elif rank == 0:
        out["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
