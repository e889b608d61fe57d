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
# decode_nvfp4 workload, from one ncu capture of the current kernel (read 91.86 MB, write 2.36 MB);
# None once the kernel changes, until the counters are taken again.
GATEUP_TRAFFIC_BYTES = 94_224_128
# kernels one decode layer call launches: router, gate/up, down, combine
DECODE_KERNELS_PER_CALL = 4


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
    cfg = synth.CONFIGS[args.workload]
    t0 = time.time()
    host = synth.make_layer(cfg, seed=rank)
    gen_s = time.time() - t0
    base = q.to_device(host, f"cuda:{local}")
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    batches = [int(b) for b in args.batches.split(",")]
    Tmax = max(batches)
    fixed = host.router_bytes() + host.shared_bytes()
    min_call = fixed + min(cfg.k, cfg.E) * host.expert_bytes()
    R = args.instances or max(2, -(-3 * l2 // min_call))
    layers = [base]

    def clone(qw):
        return q.QWeight(qw.data.clone(), qw.scales.clone(),
                         None if qw.tensor_scale is None else qw.tensor_scale.clone())
    for _ in range(R - 1):
        L = q.Layer(base.hidden, base.inter, base.n_experts, base.top_k, base.fmt, base.router_w.clone(),
                    None if base.router_bias is None else base.router_bias.clone(), clone(base.gate),
                    clone(base.up), clone(base.down), base.shared_fmt, base.shared_inter,
                    clone(base.shared_gate) if base.shared_gate else None,
                    clone(base.shared_up) if base.shared_up else None,
                    clone(base.shared_down) if base.shared_down else None)
        layers.append(L)
    NB = args.token_batches
    stream = torch.cuda.Stream()
    results = {}
    peak, peak_kind = _peaks()
    clocks = None
    roof = None
    e2e = None
    for T in batches:
        xs = [torch.from_numpy(synth.make_tokens(cfg, T, seed=1000 + rank, batch=i).view(np.int16)).cuda()
              for i in range(NB)]
        ys = torch.zeros((T, cfg.H), dtype=torch.int16, device="cuda")
        ws = torch.empty(q.workspace_size(base, Tmax), dtype=torch.uint8, device="cuda")
        q.workspace_init(ws)
        # per-batch routing (the library's own) -> distinct experts -> algorithmic bytes
        cnt = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
        cnts = []
        for i in range(NB):
            q.moe_route(base, xs[i], T, expert_cnt=cnt, ws=ws)
            cnts.append(cnt.cpu().numpy().copy())
        bytes_b = _bytes_per_call(host, cnts)
        torch.cuda.synchronize()

        def call(i, s=None):
            q.moe_decode_forward(layers[i % R], xs[i % NB], T, ys, ws, stream=s)

        # capture one graph of G calls (rotating instances and batches); replay it
        G = min(512, -(-max(R, NB) // R) * R)   # a whole number of rotations, >= NB batches
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for i in range(3):
                call(i, stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(G):
                    call(i, stream)
        bytes_graph = sum(bytes_b[i % NB] for i in range(G))
        steps = args.steps if T == batches[-1] else max(G, args.steps // 4)
        reps = max(1, steps // G)
        steps = reps * G
        warm = max(1, args.warmup // G)
        with torch.cuda.stream(stream):          # replay on the stream the timing events use
            for _ in range(warm):
                g.replay()
        torch.cuda.synchronize()
        headline = T == batches[-1]
        sampler = ClockSampler(local) if headline else None
        if sampler:
            sampler.start()
            time.sleep(0.3)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        ms = ev0.elapsed_time(ev1)
        if sampler:
            clocks = sampler.stop()
        ms, total_bytes = aggregate_ranks(ms, float(bytes_graph * reps), dist, "cuda")
        us_call = ms * 1e3 / steps
        gbs = total_bytes / (ms * 1e-3) / 1e9
        toks = world * T * steps / (ms * 1e-3)
        results[T] = {"us_per_layer": round(us_call, 3), "weight_GBps": round(gbs, 1),
                      "tokens_per_s": round(toks, 1), "hbm_frac": round(gbs / world / peak, 4),
                      "bytes_per_layer": int(np.mean(bytes_b)), "steps": steps}
        # per-kernel live CUDA-event timing on the launch stream (every batch size; the
        # headline batch also gives the roofline of the dominant kernel, gate/up)
        if True:
            n = min(256, max(32, steps // 8))
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
            for row in evs:          # create the CUDA events (torch creates them lazily on first record)
                for e in row:
                    e.record(stream)
            torch.cuda.synchronize()
            gt = torch.cuda.CUDAGraph()         # event-record nodes between the kernels, no host gaps
            with torch.cuda.graph(gt, stream=stream):
                for i in range(n):
                    q.moe_decode_forward_timed(layers[i % R], xs[i % NB], T, ys, ws, evs[i], stream=stream)
            with torch.cuda.stream(stream):
                gt.replay()
            torch.cuda.synchronize()
            dur = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(3)] for i in range(n)])
            avg = dur.mean(axis=0) * 1e3  # us per launch: router, gate/up, down
            per_exp_gu = sum(m.nbytes() // m.E for m in (host.gate, host.up))
            s_gu = (host.shared_gate.nbytes() + host.shared_up.nbytes()) if host.shared_gate else 0
            gu_bytes = np.mean([int(np.count_nonzero(cnts[i % NB])) * per_exp_gu + s_gu for i in range(n)])
            ach = gu_bytes / (avg[1] * 1e-6) / 1e9
            results[T]["kernel_us"] = {"router": round(avg[0], 3), "gateup": round(avg[1], 3), "down": round(avg[2], 3)}
        if headline:
            roof = {"kernel": "gateup_decode_kernel", "bound": "hbm", "achieved": round(ach, 1),
                    "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(ach / peak, 4),
                    "traffic": GATEUP_TRAFFIC_BYTES, "bytes_per_launch": int(gu_bytes),
                    "kernel_us": {"router": round(avg[0], 3), "gateup": round(avg[1], 3), "down": round(avg[2], 3)}}
            # end to end through the public API with host buffers (pinned), one call per step
            ne = min(steps, args.e2e_steps)
            xh = [torch.from_numpy(synth.make_tokens(cfg, T, seed=2000 + rank, batch=i).view(np.int16)).pin_memory()
                  for i in range(min(NB, ne))]
            yh = torch.empty((T, cfg.H), dtype=torch.int16).pin_memory()
            xd = torch.empty((T, cfg.H), dtype=torch.int16, device="cuda")
            for i in range(3):
                xd.copy_(xh[i % len(xh)], non_blocking=True)
                q.moe_decode_forward(layers[i % R], xd, T, ys, ws)
                yh.copy_(ys, non_blocking=True)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(ne):
                xd.copy_(xh[i % len(xh)], non_blocking=True)
                q.moe_decode_forward(layers[i % R], xd, T, ys, ws)
                yh.copy_(ys, non_blocking=True)
            e1.record()
            torch.cuda.synchronize()
            ems = e0.elapsed_time(e1)
            eb = sum(bytes_b[i % NB] for i in range(ne))
            e2e = {"value": round(eb / (ems * 1e-3) / 1e9, 1), "unit": "GB/s", "steps": ne,
                   "us_per_step": round(ems * 1e3 / ne, 2), "tokens_per_s": round(T * ne / (ems * 1e-3), 1),
                   "h2d_bytes_per_step": T * cfg.H * 2, "d2h_bytes_per_step": T * cfg.H * 2}
        del g
        torch.cuda.synchronize()
    st = q.moe_check(ws)
    if st != 0:
        raise RuntimeError(f"device-side error: {q.status_string(st)}")
    Th = batches[-1]
    head = results[Th]
    out = {
        "metric": METRIC, "value": head["weight_GBps"], "unit": "GB/s", "n_gpus": world,
        "steps": head["steps"], "warmup": args.warmup, "ms_per_step": round(head["us_per_layer"] / 1e3, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights quantised NVFP4 / FP8 b128; N(0,1) bf16 tokens)",
        "config": {"workload": workload_name(cfg, Th),
                   "batch_tokens": Th, "instances_rotated": R,
                   "l2": f"inputs larger than L2: {R} layer copies rotated, "
                         f"{R * min_call / 1e6:.0f} MB touched per rotation vs L2 {l2 / 1e6:.0f} MB",
                   "graph": f"CUDA graph of {G} layer calls replayed", "parallelism": "replicas" if world > 1 else "1 GPU",
                   "gpu": dev_name, "layer_gen_s": round(gen_s, 1)},
        "tokens_per_s": head["tokens_per_s"], "hbm_frac": head["hbm_frac"],
        "batches": {str(T): r for T, r in results.items()},
        "roofline": roof, "clocks": clocks, "e2e": e2e, "gpu_launches": DECODE_KERNELS_PER_CALL * head["steps"],
    }
    return out


def run_prefill(args, local, peak_bf16, peak_kind):
    """The prefill workload (NVFP4 layer, 4096 tokens, Zipf-skewed router): whole-layer time through
    moe_prefill_forward, per-kernel event times, and the grouped GEMMs' tensor throughput."""
    import torch
    import quantized_moe_decode_router_gb300 as q
    cfg = synth.CONFIGS["prefill_nvfp4"]
    T = cfg.batches[0]
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
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(3):
            q.moe_prefill_forward(lay, xs[i % NB], T, y, ws, stream=stream)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                q.moe_prefill_forward(lay, xs[i % NB], T, y, ws, stream=stream)
        for _ in range(2):
            g.replay()
    torch.cuda.synchronize()
    reps = max(1, args.prefill_steps // G)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * G)
    # per-kernel times: event-record nodes between the launches
    n = 6
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    gt = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gt, stream=stream):
        for i in range(n):
            q.moe_prefill_forward_timed(lay, xs[i % NB], T, y, ws, evs[i], stream=stream)
    with torch.cuda.stream(stream):
        gt.replay()
    torch.cuda.synchronize()
    dur = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(7)] for i in range(n)]).mean(axis=0) * 1e3
    names = ["router_logits", "router_topk", "dispatch", "gateup_gemm", "h_convert", "down_gemm", "combine"]
    st = q.moe_check(ws)
    if st != 0:
        raise RuntimeError(f"device-side error: {q.status_string(st)}")
    # the W4A4 lever (act_quant = 1): block-scaled FP4 GEMMs, same workload
    ws4 = torch.empty(q.workspace_size(lay, T, 1), dtype=torch.uint8, device="cuda")
    q.workspace_init(ws4)
    g4 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(3):
            q.moe_prefill_forward(lay, xs[i % NB], T, y, ws4, stream=stream, act_quant=1)
        stream.synchronize()
        with torch.cuda.graph(g4, stream=stream):
            for i in range(G):
                q.moe_prefill_forward(lay, xs[i % NB], T, y, ws4, stream=stream, act_quant=1)
        for _ in range(2):
            g4.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g4.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us4 = e0.elapsed_time(e1) * 1e3 / (reps * G)
    evs4 = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n)]
    for row in evs4:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    gt4 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gt4, stream=stream):
        for i in range(n):
            q.moe_prefill_forward_timed(lay, xs[i % NB], T, y, ws4, evs4[i], stream=stream, act_quant=1)
    with torch.cuda.stream(stream):
        gt4.replay()
    torch.cuda.synchronize()
    dur4 = np.array([[evs4[i][j].elapsed_time(evs4[i][j + 1]) for j in range(7)] for i in range(n)]).mean(axis=0) * 1e3
    st = q.moe_check(ws4)
    if st != 0:
        raise RuntimeError(f"device-side error (W4A4): {q.status_string(st)}")
    pairs = T * cfg.k
    flops = pairs * 6.0 * cfg.H * cfg.I
    gemm4_us = dur4[3] + dur4[5]
    tflops4 = flops / (gemm4_us * 1e-6) / 1e12
    gemm_us = dur[3] + dur[5]
    tflops = flops / (gemm_us * 1e-6) / 1e12
    fp4_peak = peak_bf16 * 13.5 / 2.25
    wbytes = host.router_bytes() + np.mean(touched) * host.expert_bytes()
    return {
        "workload": f"prefill_nvfp4: NVFP4 MoE layer H={cfg.H} E={cfg.E} top-{cfg.k} I={cfg.I}, {T} tokens, "
                    f"Zipf router bias s={cfg.zipf_s}",
        "us_per_layer": round(us, 1), "tokens_per_s": round(T / (us * 1e-6), 1),
        "kernel_us": {k: round(float(v), 2) for k, v in zip(names, dur)},
        "experts_touched": float(np.mean(touched)),
        "gemm": {"path": "exact chain: tcgen05 kind::f16, NVFP4 decoded in shared memory",
                 "flops_per_layer": flops, "achieved_tflops": round(tflops, 1),
                 "frac_f16_peak": round(tflops / peak_bf16, 4), "f16_peak_tflops": peak_bf16,
                 "frac_fp4_peak": round(tflops / fp4_peak, 4), "fp4_peak_tflops": round(fp4_peak, 1),
                 "peak_kind": peak_kind},
        "weight_GBps": round(wbytes / (us * 1e-6) / 1e9, 1),
        "graph": f"CUDA graph of {G} layer calls, {reps} replays",
        "w4a4": {"path": "NVFP4 activations (lever, act_quant=1): tcgen05 kind::mxf4nvf4 block-scaled GEMMs",
                 "us_per_layer": round(us4, 1), "tokens_per_s": round(T / (us4 * 1e-6), 1),
                 "kernel_us": {k: round(float(v), 2) for k, v in zip(
                     ["router_logits", "router_topk", "dispatch_quantise", "gateup_gemm", "-", "down_gemm",
                      "combine"], dur4) if k != "-"},
                 "achieved_tflops": round(tflops4, 1), "frac_fp4_peak": round(tflops4 / fp4_peak, 4),
                 "fp4_peak_tflops": round(fp4_peak, 1), "peak_kind": peak_kind},
    }


def workload_name(cfg, T: int) -> str:
    return (f"{cfg.name}: NVFP4 MoE layer H={cfg.H} E={cfg.E} top-{cfg.k} I={cfg.I} "
            f"+ FP8 b128 shared expert I={cfg.shared_I}, batch {T} tokens")


def run_reference(args):
    """The oracle, as it stands, timed on the host cores.  One step is one piece
    of a batch-T layer call, in layer order: the router (exact logits, top-k,
    dispatch), the shared expert, then each routed expert segment (its gate, up
    and down decoded to FP64, the SwiGLU MLP on its token rows, the weighted
    add into the outputs); successive token batches follow one another, so K
    steps cover whole layer calls in proportion.  value = weight bytes of the
    timed pieces / time, the metric of the GPU arm."""
    from oracle import formats as F
    from oracle import moe as M
    cfg = synth.CONFIGS[args.workload]
    T = max(int(b) for b in args.batches.split(","))
    host = synth.make_layer(cfg, seed=0)

    def layer_pieces(batch):
        x = synth.make_tokens(cfg, T, seed=3000, batch=batch)
        X = F.bf16_to_f64(x)
        st = {}

        def router():
            _, _, idx, w = M.route(x, host.router_w, host.router_b, cfg.k)
            st["cnt"], st["off"], st["pair"] = M.dispatch(idx, cfg.E)
            st["w"], st["y"] = w, np.zeros((T, cfg.H))
            return host.router_bytes()
        yield router
        if host.shared_gate is not None:
            def shared():
                Wg, Wu, Wd = (F.decode_qmat(host.shared_gate, 0), F.decode_qmat(host.shared_up, 0),
                              F.decode_qmat(host.shared_down, 0))
                st["y"] += M.swiglu_mlp(Wg, Wu, Wd, X)[1]
                return host.shared_bytes()
            yield shared
        for e in range(cfg.E):
            if st["cnt"][e] == 0:
                continue

            def expert(e=e):
                ps = [int(p) for p in st["pair"][st["off"][e]:st["off"][e + 1]]]
                rows = np.array([p // cfg.k for p in ps])
                Wg, Wu, Wd = F.decode_qmat(host.gate, e), F.decode_qmat(host.up, e), F.decode_qmat(host.down, e)
                P = M.swiglu_mlp(Wg, Wu, Wd, X[rows])[1]
                for i, p in enumerate(ps):
                    t, j = divmod(p, cfg.k)
                    st["y"][t] += float(st["w"][t, j]) * P[i]
                return host.expert_bytes()
            yield expert

    def steps():
        b = 0
        while True:
            yield from layer_pieces(b)
            b += 1

    it = steps()
    for _ in range(args.warmup):
        next(it)()
    byts = 0
    t0 = time.time()
    for _ in range(args.steps):
        byts += next(it)()
    dt = time.time() - t0
    cores = len(os.sched_getaffinity(0))
    value = round(byts / dt / 1e9, 4)
    sample = (f"{args.steps} pieces of batch-{T} layer calls on {cfg.name} (router, shared expert, routed expert "
              f"segments in layer order; FP64 numpy oracle, BLAS threads = {cores})")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, the GPU arm's layer and token recipe)",
            "config": {"workload": workload_name(cfg, T), "batch_tokens": T, "parallelism": "host cores"},
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
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=512)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--batches", default="1,4,8")
    ap.add_argument("--instances", type=int, default=0)
    ap.add_argument("--token-batches", type=int, default=64)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-batches", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill workload's measurement")
    ap.add_argument("--prefill-steps", type=int, default=60)
    args = ap.parse_args()
    world, rank, local = _dist()
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return
    out = run_ours(args, world, rank, local)
    if world == 1 and not args.no_prefill:
        pk, pkk = _bf16_peak()
        out["prefill"] = run_prefill(args, local, pk, pkk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = run_cpu_baseline(args)
    elif rank == 0:
        out["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
